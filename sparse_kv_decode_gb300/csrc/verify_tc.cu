// Multi-query verify on the 5th-generation tensor cores (StD 3.1: the dense
// model checks all gamma drafted positions in one pass over the full cache;
// ByteCross "The Attention Baseline": split-K dense attention), for KV heads
// with 17..64 query rows (R = G * gamma) at d = 128, where the warp-level
// mma.sync path of attn_splitk.cu waits on the latency of its chained MMAs.
//
// The products run transposed, so that the 128 rows of each MMA are keys or
// head dims and never padding (a tcgen05.mma costs at least ~48 cycles
// whatever its N, so the work per key is what the row count M buys):
//   S^T = K Q^T    M = 128 keys of the tile, N = 32 * NG query rows (NG = 1 or
//                  2 groups of 32), K = 128 dims.
//                  A = the K tile, B = the query rows, both K-major with
//                  128-byte swizzle as TMA writes them; S^T in tensor memory
//                  (lane = key), two buffers.
//   softmax        4 * NG warps, one thread per (key, row group): a warp reads
//                  its own quarter of the tensor-memory lanes (keys) and, for
//                  its group, 32 scores per key.  Every row r has one
//                  reference m_r, the same in all threads (shared memory,
//                  double-buffered); a weight is 2^(scale*log2e*s - m_r),
//                  rounded to bf16 into P^T.  The threads vote once per tile
//                  (a named barrier with an OR) on whether some visible score
//                  passed its row's reference by more than 2^8; only then
//                  (always on the first tile) do they reduce the tile's row
//                  maxima, after which one warp per group computes the new
//                  references and rescale factors and the others read the
//                  factors back, to rescale what was accumulated.  So the
//                  unscaled weights stay <= 256.  Each thread sums its keys'
//                  weights per row: l of the rounded weights, which O is
//                  normalised by (the weights O summed), and l_exact of the
//                  unrounded ones, for the log-sum-exp; the sums are reduced
//                  over the threads at the end.  Causal mask: query t of a
//                  row sees keys <= n_prefix + t; interior tiles skip it, and
//                  chunks of rows past R are skipped.
//   O^T += V^T P^T M = 128 head dims, N = 64 (the rows, padded to a 128-byte
//                  swizzle row of P^T), K = 128 keys.  A = the V tile
//                  as TMA wrote it ([keys][dims]: MN-major), B = P^T
//                  ([keys][rows]: MN-major), both 128-byte swizzle.
// Warp 0 and the last warp issue the TMA copies of the K and V tiles, each in
// stages of their own (a K stage frees as soon as its score is done, so K
// copies run well ahead of the scores); one thread of warp 1 the MMAs, the
// score of tile t before the PV product of tile t - 1 so that the softmax of a
// tile overlaps the next score; warps 2 .. 1 + 4 * NG the softmax.  A CTA takes
// one (sequence, KV head) and one chunk of its keys; the chunks of a head form
// clusters of up to 8 CTAs (one CTA per SM, all in one wave) whose partials
// (o, m, l, l_exact) merge through distributed shared memory, and the last
// cluster of a head (ticket) merges the clusters' partials.  Every wait is
// bounded, and the softmax warps leave their loop together, at a shared vote.
#include "sdkv_common.cuh"
#include "sdkv_internal.h"

#include <algorithm>

namespace sdkv {

namespace {

constexpr int kVD = 128;            // head dim
constexpr int kVTK = 128;           // keys per tile: M of the score product
constexpr int kVNQ = 32;            // query rows of a row group (a softmax thread's rows)
constexpr int kVNP = 64;            // N of the PV product: a P^T row is 64 bf16
constexpr int kVRmin = 17;          // fewer rows go to the mma.sync path
constexpr int kVRmax = 64;          // two row groups
constexpr int kVKSt = 3;            // K stages: free once their score is done
constexpr int kVVSt = 2;            // V stages: held until their PV product is done
constexpr int kVMaxCluster = 8;
constexpr int kVBar = 1;            // named barrier of the softmax warps
constexpr float kVRescale = 8.f;    // growth past a row's reference (log2 units) that raises it

template <int NG>
struct VCfg {
    static constexpr int NQ = kVNQ * NG;                     // query rows: N of the score product
    static constexpr int NT = 32 * (3 + 4 * NG);             // warp 0 K copies, 1 MMA, 4*NG softmax, last V copies
    static constexpr int VWARP = 2 + 4 * NG;
    static constexpr int NSOFT = 128 * NG;                   // softmax threads
    static constexpr int Q_B = 2 * NQ * 128;                 // two 64-dim halves of NQ rows
    static constexpr int T_B = 2 * kVTK * 128;               // a K or V tile: two halves of 128 keys
    static constexpr int P_B = kVTK * 128;                   // P^T: 128 keys x 64 bf16
    static constexpr int OFF_Q = 0;
    static constexpr int OFF_K = OFF_Q + Q_B;
    static constexpr int OFF_V = OFF_K + kVKSt * T_B;
    static constexpr int OFF_P = OFF_V + kVVSt * T_B;
    static constexpr int OFF_RED = OFF_P + 2 * P_B;          // [group][4 warps][32 rows] tile maxima
    static constexpr int OFF_M = OFF_RED + NG * 4 * kVNQ * 4;  // [2][NQ] row references (double-buffered)
    static constexpr int OFF_F = OFF_M + 2 * NQ * 4;         // [NQ] rescale factors of a raise, [NG] flags
    static constexpr int OFF_BAR = OFF_F + NQ * 4 + 16;
    static constexpr int NBAR = 2 * kVKSt + 2 * kVVSt + 1 + 2 + 2 + 2 + 1 + 1;
    static constexpr int OFF_TMEM = OFF_BAR + NBAR * 8;
    static constexpr int SMEM = OFF_TMEM + 16;
    static constexpr int SMEM_ALLOC = SMEM + 1024;
    // after the loop the K and V stages hold: the threads' sums [2][128][NQ+1],
    // the output rows o [NQ][128], the rows' records (m, l, l_exact, -) [NQ],
    // and what the cluster's CTAs push: o slices [cs][R][128/cs] and records [8][R]
    static constexpr int LR_LD = NQ + 1;
    static constexpr int OFF_LR = OFF_K;
    static constexpr int OFF_CMB = OFF_LR + 2 * kVTK * LR_LD * 4;
    static constexpr int OFF_SUM = OFF_CMB + NQ * kVD * 4;
    static constexpr int OFF_RCV = OFF_SUM + NQ * 16;
    static constexpr int OFF_RML = OFF_RCV + NQ * kVD * 4;
    static constexpr int END_MERGE = OFF_RML + kVMaxCluster * NQ * 16;
    static constexpr uint32_t TMEM_COLS = NG == 1 ? 128 : 256;   // S^T: two buffers of NQ columns; O^T: 64
    static constexpr uint32_t COL_O = 2 * NQ;
    static constexpr uint32_t IDESC_S = idesc_bf16_f32(kVTK, NQ);
    static constexpr uint32_t IDESC_PV = idesc_bf16_f32_amn_bmn(kVD, kVNP);
    static_assert(SMEM_ALLOC <= 227 * 1024, "shared memory of one CTA");
    static_assert(OFF_K % 1024 == 0 && OFF_V % 1024 == 0 && OFF_P % 1024 == 0, "128-byte swizzle atoms");
    static_assert(END_MERGE <= OFF_P, "the merge buffers fit the K and V stages");
    static_assert(COL_O + kVNP <= TMEM_COLS, "tensor-memory columns");
};

struct VParams {
    int B, Hq, Hkv, G, gamma, R, n_prefix, n_total, chunk, nsplit, cs;
    float scale_log2;
    bf16* o;
    float* lse;
    int* status;
    int* tickets;
    float* part_o;
    float* part_ml;
};

// One step of a warp all-reduce (max) of 32 values per lane by recursive
// halving: lanes without bit W keep rows [0, W) of their slot, lanes with it
// rows [W, 2W), each taking the maximum with its partner (lane ^ W).  After the
// steps W = 16..1, lane i holds the maximum of row i over the warp in x[0].
template <int W>
__device__ __forceinline__ void halve_max(float (&x)[kVNQ], int lane) {
    const bool upper = (lane & W) != 0;
#pragma unroll
    for (int r = 0; r < W; ++r) {
        const float send = upper ? x[r] : x[r + W];
        const float keep = upper ? x[r + W] : x[r];
        x[r] = fmaxf(keep, __shfl_xor_sync(0xffffffffu, send, W));
    }
}

template <int NG>
__global__ void __launch_bounds__(VCfg<NG>::NT, 1)
    verify_tc_kernel(const __grid_constant__ VParams p, const __grid_constant__ CUtensorMap tmq,
                     const __grid_constant__ CUtensorMap tmk, const __grid_constant__ CUtensorMap tmv) {
    using C = VCfg<NG>;
    constexpr int NQ = C::NQ;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem =
        reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(smem);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const uint32_t bar_kf = sbase + C::OFF_BAR;              // [K stage] the K tile landed
    const uint32_t bar_ke = bar_kf + 8 * kVKSt;              // [K stage] its score product is done
    const uint32_t bar_vf = bar_ke + 8 * kVKSt;              // [V stage] the V tile landed
    const uint32_t bar_ve = bar_vf + 8 * kVVSt;              // [V stage] its PV product is done
    const uint32_t bar_q = bar_ve + 8 * kVVSt;               // the query rows landed
    const uint32_t bar_sf = bar_q + 8;                       // [buf] S^T ready
    const uint32_t bar_se = bar_sf + 16;                     // [buf] S^T read by the four softmax warps
    const uint32_t bar_pf = bar_se + 16;                     // [buf] P^T written, O^T rescaled if needed
    const uint32_t bar_pv = bar_pf + 16;                     // one phase per PV product
    const uint32_t bar_od = bar_pv + 8;                      // every product issued is done (one phase)
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_TMEM);
    float* red = reinterpret_cast<float*>(smem + C::OFF_RED);
    float* mref = reinterpret_cast<float*>(smem + C::OFF_M);
    float* fac = reinterpret_cast<float*>(smem + C::OFF_F);
    int* fac_any = reinterpret_cast<int*>(smem + C::OFF_F + NQ * 4);
    __shared__ int s_abort;
    __shared__ int s_last;
    __shared__ int s_issued_k, s_issued_v;   // K and V tiles whose copies were issued

    const int bh = blockIdx.x / p.nsplit, sp = blockIdx.x - (blockIdx.x / p.nsplit) * p.nsplit;
    const int b = bh / p.Hkv, h = bh - (bh / p.Hkv) * p.Hkv;
    const int lo = sp * p.chunk;
    const int hi = max(lo, min(lo + p.chunk, p.n_total));    // trailing chunks may be empty
    const int ntiles = (hi - lo + kVTK - 1) / kVTK;
    const int qrow0 = (b * p.Hq + h * p.G) * p.gamma;        // first query (and output) row of the head
    const int cidx = blockIdx.x, c0 = bh * p.nsplit, nch = p.nsplit;

    // barriers, tensor memory and the first tiles' L2 prefetch do not depend on
    // the previous kernel: set up while it finishes
    if (tid == 0) {
        prefetch_tmap(&tmq);
        prefetch_tmap(&tmk);
        prefetch_tmap(&tmv);
        for (int t = 0; t < kVKSt && t < ntiles; ++t)
#pragma unroll
            for (int hf = 0; hf < 2; ++hf)
#pragma unroll
                for (int r2 = 0; r2 < 2; ++r2) {
                    tma_prefetch_4d(&tmk, hf * 64, lo + t * kVTK + r2 * 64, h, b);
                    tma_prefetch_4d(&tmv, hf * 64, lo + t * kVTK + r2 * 64, h, b);
                }
#pragma unroll
        for (int s = 0; s < kVKSt; ++s) {
            mbar_init(bar_kf + 8 * s, 1);
            mbar_init(bar_ke + 8 * s, 1);
        }
#pragma unroll
        for (int s = 0; s < kVVSt; ++s) {
            mbar_init(bar_vf + 8 * s, 1);
            mbar_init(bar_ve + 8 * s, 1);
        }
        mbar_init(bar_q, 1);
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            mbar_init(bar_sf + 8 * i, 1);
            mbar_init(bar_se + 8 * i, 4 * NG);
            mbar_init(bar_pf + 8 * i, 4 * NG);
        }
        mbar_init(bar_pv, 1);
        mbar_init(bar_od, 1);
        fence_mbar_init();
        s_abort = 0;
        s_issued_k = 0;
        s_issued_v = 0;
    }
    // row references, the same for every thread of a row group: rows past R
    // start at +inf, so that their weights are 0 and they never raise a vote
    for (int i = tid; i < NQ; i += C::NT) mref[i] = i < p.R ? -INFINITY : INFINITY;
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_slot), C::TMEM_COLS);
        tmem_relinquish();
    }
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    griddep_launch();
    griddep_wait();
    volatile int* abort_flag = &s_abort;

    // softmax threads (warps 2 .. 1 + 4*NG): tensor-memory lane L = key L of a
    // tile and (for O^T) head dim L; row group g2 = rows rb .. rb + 31
    const int q4 = warp & 3;
    const int L = 32 * q4 + lane;
    const int g2 = (warp - 2) >> 2, rb = kVNQ * ((warp - 2) >> 2);
    const uint32_t tlane = tmem + (static_cast<uint32_t>(32 * q4) << 16);
    // this thread's sums of rows rb + r; the references are mref[mb * NQ + rb + r]
    float l[kVNQ], le[kVNQ];
#pragma unroll
    for (int r = 0; r < kVNQ; ++r) {
        l[r] = 0.f;
        le[r] = 0.f;
    }
    int mb = 0;
    bool aborted = false;

    if (warp == 0) {
        // ------------------------------------------------------------ K producer
        // the query rows, then K tile t once its stage's previous score is done
        if (lane == 0 && ntiles > 0) {
            mbar_arrive_expect_tx(bar_q, C::Q_B);
#pragma unroll
            for (int hf = 0; hf < 2; ++hf)
                tma_load_2d(sbase + C::OFF_Q + hf * (NQ * 128), &tmq, hf * 64, qrow0, bar_q);
            int nk = 0;
            bool ok = true;
            for (int t = 0; t < ntiles; ++t) {
                const int sk = t % kVKSt;
                if (t >= kVKSt) ok = mbar_wait(bar_ke + 8 * sk, ((t / kVKSt) & 1) ^ 1);
                if (!ok || *abort_flag) break;
                mbar_arrive_expect_tx(bar_kf + 8 * sk, C::T_B);
#pragma unroll
                for (int hf = 0; hf < 2; ++hf)
#pragma unroll
                    for (int r2 = 0; r2 < 2; ++r2)
                        tma_load_4d(sbase + C::OFF_K + sk * C::T_B + hf * (kVTK * 128) + r2 * 8192, &tmk, hf * 64,
                                    lo + t * kVTK + r2 * 64, h, b, bar_kf + 8 * sk);
                nk = t + 1;
            }
            if (!ok) {
                flag_status(p.status, SDKV_DEV_TIMEOUT);
                *abort_flag = 1;
            }
            s_issued_k = nk;
        }
    } else if (warp == C::VWARP) {
        // ------------------------------------------------------------ V producer
        // V tile t once its stage's previous PV product is done
        if (lane == 0 && ntiles > 0) {
            int nv = 0;
            bool ok = true;
            for (int t = 0; t < ntiles; ++t) {
                const int sv = t % kVVSt;
                if (t >= kVVSt) ok = mbar_wait(bar_ve + 8 * sv, ((t / kVVSt) & 1) ^ 1);
                if (!ok || *abort_flag) break;
                mbar_arrive_expect_tx(bar_vf + 8 * sv, C::T_B);
#pragma unroll
                for (int hf = 0; hf < 2; ++hf)
#pragma unroll
                    for (int r2 = 0; r2 < 2; ++r2)
                        tma_load_4d(sbase + C::OFF_V + sv * C::T_B + hf * (kVTK * 128) + r2 * 8192, &tmv, hf * 64,
                                    lo + t * kVTK + r2 * 64, h, b, bar_vf + 8 * sv);
                nv = t + 1;
            }
            if (!ok) {
                flag_status(p.status, SDKV_DEV_TIMEOUT);
                *abort_flag = 1;
            }
            s_issued_v = nv;
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        // S(0), then S(t) followed by PV(t - 1): PV(t - 2) always precedes S(t), so
        // when S(t) is done every PV product before PV(t - 1) is done (a commit
        // arrives only when all earlier products are), which frees P^T buffer
        // t & 1 and is what the softmax's rescale relies on.
        if (lane == 0 && ntiles > 0) {
            // Operand descriptors built once; an offset of o bytes into an operand adds
            // o >> 4 to its descriptor (the start-address field holds address >> 4 in
            // 14 bits, and every shared address here is below 2^18, so nothing carries).
            const uint64_t qd0 = sw128_kmajor_desc(sbase + C::OFF_Q);
            const uint64_t kd0 = sw128_kmajor_desc(sbase + C::OFF_K);
            // V as A, MN-major: M = dims (the two 64-dim halves kVTK * 128 bytes apart),
            // K = keys (8-key groups 1024 bytes apart, 16 keys per step)
            const uint64_t vd0 = sw128_desc(sbase + C::OFF_V, kVTK * 128, 1024);
            // P^T as B, MN-major: N = the 64 columns of a row, K = keys (8-key groups
            // 1024 bytes apart); a single 64-wide N block, so the block stride is unused
            const uint64_t pd0 = sw128_desc(sbase + C::OFF_P, 1024, 1024);
            bool ok = mbar_wait(bar_q, 0);
            for (int t = 0; ok && t <= ntiles; ++t) {
                if (t < ntiles) {
                    // S^T(t) = K(t) Q^T into S buffer t & 1, once the softmax has read S^T(t - 2)
                    const int s = t % kVKSt, sb = t & 1;
                    ok = mbar_wait(bar_kf + 8 * s, (t / kVKSt) & 1);
                    if (ok && t >= 2) ok = mbar_wait(bar_se + 8 * sb, ((t >> 1) - 1) & 1);
                    if (!ok || *abort_flag) break;
                    tc_fence_after();
                    const uint64_t kds = kd0 + static_cast<uint64_t>((s * C::T_B) >> 4);
#pragma unroll
                    for (int ks = 0; ks < kVD / 16; ++ks)
                        tc_mma_bf16(tmem + sb * NQ,
                                    kds + static_cast<uint64_t>(((ks >> 2) * (kVTK * 128) + (ks & 3) * 32) >> 4),
                                    qd0 + static_cast<uint64_t>(((ks >> 2) * (NQ * 128) + (ks & 3) * 32) >> 4),
                                    C::IDESC_S, ks > 0);
                    tc_commit(bar_ke + 8 * s);    // the K stage is free once the score is done
                    tc_commit(bar_sf + 8 * sb);
                }
                if (t >= 1) {
                    // O^T += V(u)^T P^T(u) for the previous tile u, once its weights are written
                    const int u = t - 1, su = u % kVVSt, pb = u & 1;
                    ok = mbar_wait(bar_pf + 8 * pb, (u >> 1) & 1);
                    if (ok) ok = mbar_wait(bar_vf + 8 * su, (u / kVVSt) & 1);
                    if (!ok || *abort_flag) break;
                    tc_fence_after();
                    const uint64_t vds = vd0 + static_cast<uint64_t>((su * C::T_B) >> 4);
                    const uint64_t pds = pd0 + static_cast<uint64_t>((pb * C::P_B) >> 4);
#pragma unroll
                    for (int kk = 0; kk < kVTK / 16; ++kk)
                        tc_mma_bf16(tmem + C::COL_O, vds + static_cast<uint64_t>((kk * 2048) >> 4),
                                    pds + static_cast<uint64_t>((kk * 2048) >> 4), C::IDESC_PV,
                                    (u > 0 || kk > 0) ? 1u : 0u);
                    tc_commit(bar_ve + 8 * su);   // the V stage is free once the product is done
                    tc_commit(bar_pv);
                }
            }
            // one arrival once every product issued above is done (also after a timeout:
            // tensor memory and the operands' shared memory stay until then)
            tc_commit(bar_od);
            if (!ok) {
                flag_status(p.status, SDKV_DEV_TIMEOUT);
                *abort_flag = 1;
            }
        }
    } else {
        // ------------------------------------------------------------ softmax, one thread per (key, row group)
        const float c = p.scale_log2;
        uint8_t* prow0 = smem + C::OFF_P + L * 128;
        // P^T rows start at zero: the columns of padding rows are never written
#pragma unroll
        for (int pb = 0; pb < 2; ++pb)
#pragma unroll
            for (int ch = 0; ch < 8; ++ch)
                *reinterpret_cast<uint4*>(prow0 + pb * C::P_B + ch * 16) = make_uint4(0u, 0u, 0u, 0u);
        for (int t = 0; t < ntiles; ++t) {
            const int sb = t & 1;
            const bool got = mbar_wait(bar_sf + 8 * sb, (t >> 1) & 1);
            if (!got) *abort_flag = 1;
            uint32_t v[kVNQ];
#pragma unroll
            for (int r = 0; r < kVNQ; ++r) v[r] = 0u;
            if (__all_sync(0xffffffffu, got)) {
                tc_fence_after();
                tmem_ld32_sync(tlane + sb * NQ + rb, v);
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar_se + 8 * sb);
            const int tile0 = lo + t * kVTK;
            const int key = tile0 + L;
            // interior tiles: every key inside the chunk and before every row's limit
            const bool full = tile0 + kVTK <= hi && tile0 + kVTK - 1 <= p.n_prefix;
            // bit r: row r sees this key (rows past R see every key, but their
            // reference +inf makes their weights 0)
            uint32_t vis = 0xffffffffu;
            if (!full) {
                const int over = key - p.n_prefix;   // visible to row r iff key < hi and over <= r % gamma
                vis = 0u;
#pragma unroll
                for (int r = 0; r < kVNQ; ++r) vis |= (key < hi && over <= (rb + r) % p.gamma) ? (1u << r) : 0u;
            }
            const float* mc = mref + mb * NQ + rb;   // this group's references (shared-memory broadcast)
            // the largest visible score relative to its row's reference (a tree of maxima)
            float g[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) g[i] = -INFINITY;
#pragma unroll
            for (int k = 0; k < kVNQ / 4; ++k) {   // references 4 at a time (16-byte aligned)
                if (rb + 4 * k >= p.R) break;      // only padding rows from here (warp-uniform)
                const float4 m4 = *reinterpret_cast<const float4*>(mc + 4 * k);
                const float mk[4] = {m4.x, m4.y, m4.z, m4.w};
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int r = 4 * k + i;
                    g[r & 7] = fmaxf(g[r & 7], (vis >> r) & 1u ? fmaf(__uint_as_float(v[r]), c, -mk[i]) : -INFINITY);
                }
            }
            const bool viol = fmaxf(fmaxf(fmaxf(g[0], g[1]), fmaxf(g[2], g[3])), fmaxf(fmaxf(g[4], g[5]), fmaxf(g[6], g[7]))) >
                              kVRescale;
            // one vote per tile; a thread whose wait gave up set the abort flag before it
            const bool any = named_bar_or(kVBar, C::NSOFT, viol);
            if (*abort_flag) {
                aborted = true;
                break;
            }
            if (any) {
                // raise the references of the rows whose tile maximum passed them by more
                // than 2^8: the tile's row maxima over the 128 keys (warp all-reduce of 32
                // rows by recursive halving, then the four warps through shared memory)
                {
                    float x[kVNQ];
#pragma unroll
                    for (int r = 0; r < kVNQ; ++r)
                        x[r] = (vis >> r) & 1u ? __uint_as_float(v[r]) * c : -INFINITY;
                    halve_max<16>(x, lane);
                    halve_max<8>(x, lane);
                    halve_max<4>(x, lane);
                    halve_max<2>(x, lane);
                    halve_max<1>(x, lane);
                    // lane i now holds the warp's maximum of row i (in x[0])
                    red[(4 * g2 + q4) * kVNQ + lane] = x[0];
                }
                named_bar_sync(kVBar, C::NSOFT);
                // the group's first warp, lane r: row rb + r's tile maximum, its new
                // reference (into the other buffer) and its rescale factor
                if (q4 == 0) {
                    const float* rg = red + 4 * kVNQ * g2;
                    const float tm = fmaxf(fmaxf(rg[lane], rg[kVNQ + lane]), fmaxf(rg[2 * kVNQ + lane], rg[3 * kVNQ + lane]));
                    const float mo = mref[mb * NQ + rb + lane];
                    const bool grow = tm > mo + kVRescale;   // mo = -inf: the row's first visible keys
                    const bool scaled = grow && mo != -INFINITY;
                    fac[rb + lane] = scaled ? fast_exp2(mo - tm) : 1.f;
                    mref[(mb ^ 1) * NQ + rb + lane] = grow ? tm : mo;
                    const unsigned any_scaled = __ballot_sync(0xffffffffu, scaled);
                    if (lane == 0) fac_any[g2] = any_scaled != 0u;
                }
                // the factors and new references are written; the old references and
                // the maxima are no longer read
                named_bar_sync(kVBar, C::NSOFT);
                mb ^= 1;
                if (fac_any[g2]) {
                    float f[kVNQ];
#pragma unroll
                    for (int k = 0; k < kVNQ / 4; ++k) {
                        const float4 f4 = *reinterpret_cast<const float4*>(fac + rb + 4 * k);
                        f[4 * k] = f4.x;
                        f[4 * k + 1] = f4.y;
                        f[4 * k + 2] = f4.z;
                        f[4 * k + 3] = f4.w;
                    }
#pragma unroll
                    for (int r = 0; r < kVNQ; ++r) {
                        l[r] *= f[r];
                        le[r] *= f[r];
                    }
                    if (t >= 1) {
                        // S(t) was issued after every PV product but PV(t - 1): wait for that
                        // one, then scale this warp's 32 dims of O^T, 16 rows at a time
                        const bool ok = mbar_wait(bar_pv, (t - 1) & 1);
                        if (!ok) *abort_flag = 1;
                        if (__all_sync(0xffffffffu, ok)) {
                            tc_fence_after();
#pragma unroll
                            for (int hh = 0; hh < 2; ++hh) {
                                uint32_t ov[16];
                                tmem_ld16_sync(tlane + C::COL_O + rb + 16 * hh, ov);
#pragma unroll
                                for (int i = 0; i < 16; ++i)
                                    ov[i] = __float_as_uint(__uint_as_float(ov[i]) * f[16 * hh + i]);
                                tmem_st16_sync(tlane + C::COL_O + rb + 16 * hh, ov);
                            }
                        }
                    }
                }
                // a wait that gave up above set the abort flag: every thread leaves at the
                // next tile's vote (or at the end of the loop), never alone
            }
            // weights rounded to bf16 as the PV product uses them; l sums the same
            // values, le the unrounded ones; P^T row `L` of buffer t & 1, columns rb .. rb + 31
            uint8_t* prow = prow0 + (t & 1) * C::P_B;
            const float* mw = mref + mb * NQ + rb;
#pragma unroll
            for (int k = 0; k < kVNQ / 8; ++k) {   // 16-byte chunk 4*g2 + k: rows rb + 8k .. rb + 8k + 7
                if (rb + 8 * k >= p.R) break;      // only padding rows from here: their weights stay 0
                const float4 ma = *reinterpret_cast<const float4*>(mw + 8 * k);
                const float4 mb4 = *reinterpret_cast<const float4*>(mw + 8 * k + 4);
                const float mk[8] = {ma.x, ma.y, ma.z, ma.w, mb4.x, mb4.y, mb4.z, mb4.w};
                uint32_t pk[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int r = 8 * k + 2 * i;
                    const float x0 = (vis >> r) & 1u ? fast_exp2(fmaf(__uint_as_float(v[r]), c, -mk[2 * i])) : 0.f;
                    const float x1 = (vis >> (r + 1)) & 1u ? fast_exp2(fmaf(__uint_as_float(v[r + 1]), c, -mk[2 * i + 1])) : 0.f;
                    le[r] += x0;
                    le[r + 1] += x1;
                    const __nv_bfloat162 w2 = __floats2bfloat162_rn(x0, x1);
                    const float2 wf = __bfloat1622float2(w2);
                    l[r] += wf.x;
                    l[r + 1] += wf.y;
                    pk[i] = *reinterpret_cast<const uint32_t*>(&w2);
                }
                *reinterpret_cast<uint4*>(prow + (((4 * g2 + k) ^ (L & 7)) << 4)) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
            }
            tc_fence_before();           // the rescale's tensor-memory stores, then
            fence_proxy_async_smem();    // the weights, visible to the tensor cores
            __syncwarp();
            if (lane == 0) mbar_arrive(bar_pf + 8 * (t & 1));
        }
        // the output is final once every product is done
        if (!aborted && ntiles > 0) {
            if (!__all_sync(0xffffffffu, mbar_wait(bar_od, 0))) aborted = true;
            tc_fence_after();
        }
        if (aborted && lane == 0) {
            flag_status(p.status, SDKV_DEV_TIMEOUT);
            *abort_flag = 1;
        }
    }

    // ------------------------------------------------------------------ partials
    const bool stop = __syncthreads_or(aborted || *abort_flag);
    float* lr = reinterpret_cast<float*>(smem + C::OFF_LR);
    float* cmb = reinterpret_cast<float*>(smem + C::OFF_CMB);
    float4* sum = reinterpret_cast<float4*>(smem + C::OFF_SUM);
    if (!stop && warp >= 2 && warp < C::VWARP) {
        // into the K and V stages, which nothing uses any more (every product is
        // done, and each waited for the copy it read): this thread's sums, and its
        // head dim of every output row (O^T lane L), relative to the references
        uint32_t ov[kVNQ];
        if (ntiles > 0) {
            tmem_ld32_sync(tlane + C::COL_O + rb, ov);
        } else {
#pragma unroll
            for (int r = 0; r < kVNQ; ++r) ov[r] = 0u;
        }
#pragma unroll
        for (int r = 0; r < kVNQ; ++r) {
            cmb[(rb + r) * kVD + L] = __uint_as_float(ov[r]);
            lr[L * C::LR_LD + rb + r] = l[r];
            lr[(kVTK + L) * C::LR_LD + rb + r] = le[r];
        }
        if (L == 0) {   // the references are the same in every thread of the group
#pragma unroll
            for (int r = 0; r < kVNQ; ++r) sum[rb + r].x = mref[mb * NQ + rb + r];
        }
    }
    // after a timeout, the products issued so far must finish before their
    // tensor memory and shared-memory operands go away (bounded)
    if (stop && warp == 1 && lane == 0 && ntiles > 0) mbar_wait(bar_od, 0);
    // tensor memory is no longer read: free it before the merges, which may return early
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, C::TMEM_COLS);
    }
    if (stop) {
        // let copies in flight land before the CTA's shared memory goes away (bounded)
        if (tid == 0 && ntiles > 0) {
            mbar_wait(bar_q, 0);
            const int ik = s_issued_k, iv = s_issued_v;
            for (int s = 0; s < kVKSt && s < ik; ++s) {
                const int last_t = ((ik - 1 - s) / kVKSt) * kVKSt + s;
                mbar_wait(bar_kf + 8 * s, (last_t / kVKSt) & 1);
            }
            for (int s = 0; s < kVVSt && s < iv; ++s) {
                const int last_t = ((iv - 1 - s) / kVVSt) * kVVSt + s;
                mbar_wait(bar_vf + 8 * s, (last_t / kVVSt) & 1);
            }
        }
        if (p.cs > 1) {   // the two cluster barriers the other CTAs pass
            cluster_sync_all();
            cluster_sync_all();
        }
        return;
    }
    // each row's sums over the 128 keys' threads: 8 lanes per row, 16 keys each,
    // then a reduction over the 8 lanes (rows of a warp: 4; all lanes take part)
    for (int rr0 = 4 * warp; rr0 < p.R; rr0 += 4 * (C::NT / 32)) {
        const int rr = rr0 + (lane >> 3), part = lane & 7;
        float a = 0.f, e = 0.f;
        if (rr < p.R) {
#pragma unroll 4
            for (int i = part; i < kVTK; i += 8) {
                a += lr[i * C::LR_LD + rr];
                e += lr[(kVTK + i) * C::LR_LD + rr];
            }
        }
#pragma unroll
        for (int o = 4; o >= 1; o >>= 1) {
            a += __shfl_xor_sync(0xffffffffu, a, o);
            e += __shfl_xor_sync(0xffffffffu, e, o);
        }
        if (rr < p.R && part == 0) {
            sum[rr].y = a;
            sum[rr].z = e;
        }
    }
    __syncthreads();

    // ------------------------------------------ this chunk's partial
    // pushed to the cluster ranks that own the dims (once every CTA of the
    // cluster is past its loop: the receiving buffers are in the stages), written
    // as the output (one chunk per head), or written to the workspace
    const int lcs = __ffs(p.cs) - 1;                 // cluster sizes are powers of two
    const int SL = kVD >> lcs;                       // head dims a cluster rank owns
    const uint32_t me = p.cs > 1 ? cluster_ctarank() : 0u;
    if (p.cs > 1) cluster_sync_all();
    for (int e = tid; e < p.R * (kVD / 4); e += C::NT) {
        const int rr = e >> 5, d0 = 4 * (e & 31);
        const float4 a4 = *reinterpret_cast<const float4*>(cmb + rr * kVD + d0);
        const float4 rec = sum[rr];
        const float M = rec.x, Lr = rec.y, Le = rec.z;
        if (p.cs > 1) {
            const int owner = d0 >> (7 - lcs);
            st_dsmem_f4(dsmem_addr(sbase + C::OFF_RCV + ((me * p.R + rr) * SL + (d0 & (SL - 1))) * 4, owner), a4);
            if (d0 == 0)
                for (int rk = 0; rk < p.cs; ++rk)
                    st_dsmem_f4(dsmem_addr(sbase + C::OFF_RML + (me * p.R + rr) * 16, rk), make_float4(M, Lr, Le, 0.f));
        } else if (nch == 1) {
            const float il = Lr > 0.f ? 1.f / Lr : 0.f;
            uint2 packed;
            packed.x = pack_bf16(a4.x * il, a4.y * il);
            packed.y = pack_bf16(a4.z * il, a4.w * il);
            *reinterpret_cast<uint2*>(p.o + static_cast<size_t>(qrow0 + rr) * kVD + d0) = packed;
            if (d0 == 0 && p.lse) p.lse[qrow0 + rr] = Le > 0.f ? (M + fast_log2(Le)) * kLn2 : -INFINITY;
        } else {
            *reinterpret_cast<float4*>(p.part_o + (static_cast<size_t>(cidx) * p.R + rr) * kVD + d0) = a4;
            if (d0 == 0)
                *reinterpret_cast<float4*>(p.part_ml + (static_cast<size_t>(cidx) * p.R + rr) * 4) =
                    make_float4(M, Lr, Le, 0.f);
        }
    }

    if (p.cs > 1) {
        // ------------------------------------------------ merge the cluster's chunks
        // CTA `rank` owns head dims [rank*SL, (rank+1)*SL); every CTA pushed its
        // rows' slices and records into the owners' shared memory before this barrier.
        cluster_sync_all();
        const int CS = p.cs;
        const uint32_t rank = me;
        const int lsl4 = 7 - lcs - 2;                // float4 per row in this slice: 1 << lsl4
        const int sl4 = 1 << lsl4;
        const int gcl = cidx >> lcs, gcl0 = c0 >> lcs, ncl_h = nch >> lcs;
        const float* rcv = reinterpret_cast<const float*>(smem + C::OFF_RCV);
        const float4* rml = reinterpret_cast<const float4*>(smem + C::OFF_RML);
        for (int e = tid; e < p.R * sl4; e += C::NT) {
            const int rr = e >> lsl4;
            const int dd = 4 * (e & (sl4 - 1));
            const int d0 = static_cast<int>(rank) * SL + dd;
            float4 ml4[kVMaxCluster];
            float4 v4[kVMaxCluster];
#pragma unroll
            for (int cc = 0; cc < kVMaxCluster; ++cc) {
                ml4[cc] = make_float4(-INFINITY, 0.f, 0.f, 0.f);
                v4[cc] = make_float4(0.f, 0.f, 0.f, 0.f);
                if (cc < CS) {
                    ml4[cc] = rml[cc * p.R + rr];
                    v4[cc] = *reinterpret_cast<const float4*>(rcv + (cc * p.R + rr) * SL + dd);
                }
            }
            float M = -INFINITY;
#pragma unroll
            for (int cc = 0; cc < kVMaxCluster; ++cc) M = fmaxf(M, ml4[cc].x);
            float Lr = 0.f, Le = 0.f;
            float4 a4 = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
            for (int cc = 0; cc < kVMaxCluster; ++cc) {
                if (ml4[cc].x == -INFINITY) continue;
                const float w = fast_exp2(ml4[cc].x - M);
                Lr += w * ml4[cc].y;
                Le += w * ml4[cc].z;
                a4.x += w * v4[cc].x;
                a4.y += w * v4[cc].y;
                a4.z += w * v4[cc].z;
                a4.w += w * v4[cc].w;
            }
            if (ncl_h == 1) {
                const float il = Lr > 0.f ? 1.f / Lr : 0.f;
                uint2 packed;
                packed.x = pack_bf16(a4.x * il, a4.y * il);
                packed.y = pack_bf16(a4.z * il, a4.w * il);
                *reinterpret_cast<uint2*>(p.o + static_cast<size_t>(qrow0 + rr) * kVD + d0) = packed;
                if (d0 == 0 && p.lse) p.lse[qrow0 + rr] = Le > 0.f ? (M + fast_log2(Le)) * kLn2 : -INFINITY;
            } else {
                *reinterpret_cast<float4*>(p.part_o + (static_cast<size_t>(gcl) * p.R + rr) * kVD + d0) = a4;
                if (dd == 0)   // this rank's copy of the cluster's record
                    *reinterpret_cast<float4*>(p.part_ml + ((static_cast<size_t>(gcl) * CS + rank) * p.R + rr) * 4) =
                        make_float4(M, Lr, Le, 0.f);
            }
        }
        if (ncl_h == 1) return;
        __syncthreads();
        if (tid == 0) {
            // release this CTA's slice of the partial; acquire the other clusters' (if last)
            const int old = atom_add_acq_rel_gpu(p.tickets + bh * kVMaxCluster + rank, 1);
            s_last = (old == ncl_h - 1);
        }
        __syncthreads();
        if (!s_last) return;
        // the last cluster of the head, for its slice: merge the head's cluster partials
        for (int e = tid; e < p.R * sl4; e += C::NT) {
            const int rr = e >> lsl4;
            const int d0 = static_cast<int>(rank) * SL + 4 * (e & (sl4 - 1));
            float mm = -INFINITY, ll = 0.f, lle = 0.f;
            float4 a4 = make_float4(0.f, 0.f, 0.f, 0.f);
            for (int cb = 0; cb < ncl_h; cb += 4) {
                float4 mv[4];
                float4 ov4[4];
#pragma unroll
                for (int u = 0; u < 4; ++u) {   // the batch's loads in flight together
                    const size_t gi = static_cast<size_t>(gcl0) + cb + u;
                    mv[u] = make_float4(-INFINITY, 0.f, 0.f, 0.f);
                    ov4[u] = make_float4(0.f, 0.f, 0.f, 0.f);
                    if (cb + u < ncl_h) {
                        mv[u] = __ldcg(reinterpret_cast<const float4*>(p.part_ml + ((gi * CS + rank) * p.R + rr) * 4));
                        ov4[u] = __ldcg(reinterpret_cast<const float4*>(p.part_o + (gi * p.R + rr) * kVD + d0));
                    }
                }
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    if (mv[u].x == -INFINITY) continue;
                    const float mnew = fmaxf(mm, mv[u].x);
                    const float fa = (mm == -INFINITY) ? 0.f : fast_exp2(mm - mnew);
                    const float fb = fast_exp2(mv[u].x - mnew);
                    ll = ll * fa + mv[u].y * fb;
                    lle = lle * fa + mv[u].z * fb;
                    a4.x = a4.x * fa + ov4[u].x * fb;
                    a4.y = a4.y * fa + ov4[u].y * fb;
                    a4.z = a4.z * fa + ov4[u].z * fb;
                    a4.w = a4.w * fa + ov4[u].w * fb;
                    mm = mnew;
                }
            }
            const float il = ll > 0.f ? 1.f / ll : 0.f;
            uint2 packed;
            packed.x = pack_bf16(a4.x * il, a4.y * il);
            packed.y = pack_bf16(a4.z * il, a4.w * il);
            *reinterpret_cast<uint2*>(p.o + static_cast<size_t>(qrow0 + rr) * kVD + d0) = packed;
            if (d0 == 0 && p.lse) p.lse[qrow0 + rr] = lle > 0.f ? (mm + fast_log2(lle)) * kLn2 : -INFINITY;
        }
        if (tid == 0) atomicExch(p.tickets + bh * kVMaxCluster + rank, 0);
        return;
    }
    if (nch == 1) return;

    // ---------------------------------------------------- no cluster: the last CTA of the head
    __syncthreads();
    if (tid == 0) {
        const int old = atom_add_acq_rel_gpu(p.tickets + bh, 1);   // release this CTA's partial, acquire the others'
        s_last = (old == nch - 1);
    }
    __syncthreads();
    if (!s_last) return;
    // per (row, 4 dims): the head's nch partials, merged online from L2 in batches of 4
    for (int e = tid; e < p.R * (kVD / 4); e += C::NT) {
        const int rr = e / (kVD / 4), d0 = 4 * (e - rr * (kVD / 4));
        float mm = -INFINITY, ll = 0.f, lle = 0.f;
        float4 a4 = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int cb = 0; cb < nch; cb += 4) {
            float4 mv[4];
            float4 ov4[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const size_t gi = static_cast<size_t>(c0) + cb + u;
                mv[u] = make_float4(-INFINITY, 0.f, 0.f, 0.f);
                ov4[u] = make_float4(0.f, 0.f, 0.f, 0.f);
                if (cb + u < nch) {
                    mv[u] = __ldcg(reinterpret_cast<const float4*>(p.part_ml + (gi * p.R + rr) * 4));
                    ov4[u] = __ldcg(reinterpret_cast<const float4*>(p.part_o + (gi * p.R + rr) * kVD + d0));
                }
            }
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                if (mv[u].x == -INFINITY) continue;
                const float mnew = fmaxf(mm, mv[u].x);
                const float fa = (mm == -INFINITY) ? 0.f : fast_exp2(mm - mnew);
                const float fb = fast_exp2(mv[u].x - mnew);
                ll = ll * fa + mv[u].y * fb;
                lle = lle * fa + mv[u].z * fb;
                a4.x = a4.x * fa + ov4[u].x * fb;
                a4.y = a4.y * fa + ov4[u].y * fb;
                a4.z = a4.z * fa + ov4[u].z * fb;
                a4.w = a4.w * fa + ov4[u].w * fb;
                mm = mnew;
            }
        }
        const float il = ll > 0.f ? 1.f / ll : 0.f;
        uint2 packed;
        packed.x = pack_bf16(a4.x * il, a4.y * il);
        packed.y = pack_bf16(a4.z * il, a4.w * il);
        *reinterpret_cast<uint2*>(p.o + static_cast<size_t>(qrow0 + rr) * kVD + d0) = packed;
        if (d0 == 0 && p.lse) p.lse[qrow0 + rr] = lle > 0.f ? (mm + fast_log2(lle)) * kLn2 : -INFINITY;
    }
    if (tid == 0) atomicExch(p.tickets + bh, 0);
}

struct VPlan {
    int nsplit, chunk, cs;
};

// CTAs of this kernel the device holds at once when launched in clusters of cs
// (occupancy query, cached per device and cluster size; one CTA per SM).
template <int NG>
int vtc_capacity(int dev, int num_sms, int cs) {
    using C = VCfg<NG>;
    static std::atomic<int> cache[64][4];   // 0: not queried yet
    const int ci = cs >= 8 ? 3 : cs >= 4 ? 2 : cs >= 2 ? 1 : 0;
    const bool cached = dev >= 0 && dev < 64;
    if (cached) {
        const int v = cache[dev][ci].load(std::memory_order_relaxed);
        if (v > 0) return v;
    }
    int cap = 0;
    if (cs <= 1) {
        int per_sm = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, verify_tc_kernel<NG>, C::NT, C::SMEM_ALLOC) ==
            cudaSuccess)
            cap = per_sm * num_sms;
    } else {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(cs * 16);
        cfg.blockDim = dim3(C::NT);
        cfg.dynamicSmemBytes = C::SMEM_ALLOC;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = cs;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        int ncl = 0;
        if (cudaOccupancyMaxActiveClusters(&ncl, verify_tc_kernel<NG>, &cfg) == cudaSuccess) cap = ncl * cs;
    }
    if (cap <= 0) {
        cudaGetLastError();   // a failed query leaves no sticky error; plan without clusters
        return cs <= 1 ? std::max(num_sms, 1) : 0;
    }
    if (cached) cache[dev][ci].store(cap, std::memory_order_relaxed);
    return cap;
}

// One wave of CTAs: for each cluster size, as many clusters per head (at most
// 8; the last one merges the others' partials) as the device holds at once, and
// the cluster size whose plan covers the most CTAs.  Without clusters the SMs
// are shared among the heads, but the last CTA of a head then merges all its
// chunks' partials from L2 alone, which takes far longer than a cluster merge
// (34 partials: about 20 us): a cluster plan is kept while it covers at least
// half as many CTAs.
// cap[i]: CTAs held at once in clusters of 1 << i.
VPlan verify_plan(int BH, int n_total, const int cap[4]) {
    const int max_split = std::max(1, (n_total + kVTK - 1) / kVTK);
    VPlan pl{};
    pl.cs = 1;
    pl.nsplit = std::min(std::max(1, cap[0] / BH), max_split);
    int best = 0;
    for (int i = 3; i >= 1; --i) {
        const int cs = 1 << i;
        const int k = std::min(8, cap[i] / cs / BH);
        const int nsplit = std::min(k * cs, (max_split / cs) * cs);
        if (nsplit < cs || BH * nsplit <= best) continue;
        best = BH * nsplit;
        if (2 * best >= BH * std::min(std::max(1, cap[0] / BH), max_split)) {
            pl.cs = cs;
            pl.nsplit = nsplit;
        }
    }
    pl.chunk = (n_total + pl.nsplit - 1) / pl.nsplit;
    pl.chunk = ((pl.chunk + kVTK - 1) / kVTK) * kVTK;
    if (pl.cs == 1) pl.nsplit = (n_total + pl.chunk - 1) / pl.chunk;   // clusters keep empty trailing chunks
    return pl;
}

}  // namespace

size_t verify_tc_ws_bytes(int B, int Hq, int Hkv, int d, int n_total, int gamma, int num_sms) {
    const int R = (Hq / Hkv) * gamma;
    if (d != kVD || R < kVRmin || R > kVRmax) return 0;
    (void)n_total;
    // every plan has at most one CTA per SM, or one per head
    const int BH = B * Hkv;
    return attn_ws(nullptr, BH, R, d, std::max(num_sms, BH), 4).bytes;   // records (m, l, l_exact, -)
}

namespace {

template <int NG>
int launch_vtc(VParams& p, const AttnLaunch& a, const CUtensorMap* tmk, const CUtensorMap* tmv, int num_sms,
               const char** why) {
    using C = VCfg<NG>;
    const int BH = a.B * a.Hkv;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    static std::atomic<unsigned long long> attr_set{0};
    if (e == cudaSuccess && !attr_done(attr_set, dev)) {
        e = cudaFuncSetAttribute(verify_tc_kernel<NG>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_ALLOC);
        if (e == cudaSuccess) attr_mark(attr_set, dev);
    }
    if (e != cudaSuccess) {
        *why = cudaGetErrorString(e);
        return SDKV_ERR_CUDA;
    }
    int cap[4];
    for (int i = 0; i < 4; ++i) cap[i] = vtc_capacity<NG>(dev, num_sms, 1 << i);
    const VPlan pl = verify_plan(BH, p.n_total, cap);
    p.nsplit = pl.nsplit;
    p.chunk = pl.chunk;
    p.cs = pl.cs;
    // the query rows as a [B * Hq * gamma][d] matrix, NQ rows per box from the
    // head's first (rows past R are another head's or, past the matrix, zero)
    CUtensorMap tmq;
    const int rc = encode_rows_tmap(&tmq, a.q, static_cast<int64_t>(a.B) * a.Hq * a.gamma, a.d, C::NQ);
    if (rc) {
        *why = "could not encode the query tensor map";
        return rc;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(BH * pl.nsplit);
    cfg.blockDim = dim3(C::NT);
    cfg.dynamicSmemBytes = C::SMEM_ALLOC;
    cfg.stream = a.stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (pl.cs > 1) {
        attr[1].id = cudaLaunchAttributeClusterDimension;
        attr[1].val.clusterDim.x = pl.cs;
        attr[1].val.clusterDim.y = 1;
        attr[1].val.clusterDim.z = 1;
        cfg.numAttrs = 2;
    }
    e = cudaLaunchKernelEx(&cfg, verify_tc_kernel<NG>, p, tmq, *tmk, *tmv);
    if (e != cudaSuccess) {
        *why = cudaGetErrorString(e);
        return SDKV_ERR_CUDA;
    }
    return SDKV_OK;
}

}  // namespace

int launch_verify_tc(const AttnLaunch& a, const CUtensorMap* tmk, const CUtensorMap* tmv, int num_sms,
                     const char** why) {
    const int BH = a.B * a.Hkv;
    const int G = a.Hq / a.Hkv;
    VParams p{};
    p.B = a.B;
    p.Hq = a.Hq;
    p.Hkv = a.Hkv;
    p.G = G;
    p.gamma = a.gamma;
    p.R = G * a.gamma;
    p.n_prefix = a.n_prefix;
    p.n_total = a.n_prefix + a.gamma;
    if (a.d != kVD || p.R < kVRmin || p.R > kVRmax) {
        *why = "the tensor-core verify needs d = 128 and 17 <= (Hq/Hkv) * gamma <= 64";
        return SDKV_ERR_UNSUPPORTED;
    }
    p.scale_log2 = a.scale * kLog2e;
    p.o = static_cast<bf16*>(a.o);
    p.lse = a.lse;
    const AttnWs L = attn_ws(a.ws, BH, p.R, a.d, std::max(num_sms, BH), 4);
    if (a.ws_bytes < L.bytes) {
        *why = "workspace smaller than sdkv_workspace_size(SDKV_OP_DENSE_VERIFY, ...)";
        return SDKV_ERR_WORKSPACE;
    }
    p.status = L.status;
    p.tickets = L.tickets;
    p.part_o = L.part_o;
    p.part_ml = L.part_ml;
    return p.R <= kVNQ ? launch_vtc<1>(p, a, tmk, tmv, num_sms, why) : launch_vtc<2>(p, a, tmk, tmv, num_sms, why);
}

}  // namespace sdkv
