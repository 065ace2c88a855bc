// Observation-window scoring (StD 3.2 argTopK equation; SparseMM observation
// window): for every KV head h and key j,
//     score[j] = (1/W) sum_{g in group(h)} sum_t P_{g,t}[j],
// P_{g,t} = softmax over the keys window query (g, t) can see.  Each window row
// must be normalised over ALL its visible keys before rows are summed, so the
// keys are read twice:
//   pass 1: per row, the running max m and sum l of 2^(x - m) over the keys
//           (x = scale * log2(e) * q.k), one partial (m, l) per key split;
//   pass 2: merges the split partials of its rows into (M, L) in its prologue
//           (overlapping its first tile), then per key sums 2^(x - M - log2 L)
//           over the rows.
//
// Both passes run the 128-row x 128-key x d contraction on the 5th-generation
// tensor cores (tcgen05.mma, bf16 in, fp32 accumulators in tensor memory):
//   pass 1: A = window rows (M = 128), B = key tile (N = 128): accumulator lane =
//           row, so each epilogue thread owns one row and its statistics;
//   pass 2: A = key tile (M = 128), B = window rows (N = 128): accumulator lane =
//           key, so each epilogue thread sums its key's 128 row probabilities.
// Warp roles: warp 0 streams the window rows once and the key tiles through a
// ring of shared-memory stages with TMA (128-byte swizzle); warp 1 allocates
// tensor memory and one of its threads issues the MMAs into a ring of two or
// four accumulator buffers; warps 2..9 read the accumulators (tcgen05.ld) and do the softmax
// arithmetic.  Every wait is bounded.  A CTA covers 128 window rows (one row
// block) and one key split; larger groups or windows use more row blocks, whose
// partial key sums are added in a fixed order by the last one (deterministic).
#include "sdkv_common.cuh"
#include "sdkv_internal.h"

#include <algorithm>

namespace sdkv {

struct ScoreParams {
    int B, Hq, Hkv, G, W, R, n, q_pos0, BH, n_mg, nsplit, chunk;
    float scale_log2, inv_w;
    float* scores;
    int* status;
    int* tick2;       // [BH][nsplit]
    float* st_part;   // [BH][nsplit][R][2]  pass-1 (m, l) per key split
    float* sc_part;   // [n_mg][BH][n]
};

template <int D, int RB, int ST>
struct ScoreCfg {
    static constexpr int ROWS = 128;              // window rows per row block (MMA M or N)
    static constexpr int GROWS = RB * ROWS;       // window rows per CTA: RB row blocks share each K tile
    static constexpr int TK = 128;                // keys per tile (MMA N or M)
    static constexpr int STAGES = ST;             // K stages (three, or five for d = 128 with one row block: chosen at launch)
    static constexpr int HALVES = D / 64;         // 128-byte K-blocks per row
    static constexpr int NEPI = 8;                // epilogue warps
    static constexpr int NET = NEPI * 32;
    static constexpr int NT = NET + 64;           // + producer warp + MMA warp
    static constexpr int TILE_B = TK * D * 2;
    static constexpr int QBLK_B = ROWS * D * 2;   // one row block of window queries
    static constexpr int Q_B = RB * QBLK_B;
    static constexpr int HALF_B = TK * 128;       // one 64-wide K-block of a 128-row operand
    static constexpr int OFF_Q = 0;
    static constexpr int OFF_K = Q_B;
    static constexpr int OFF_CB = OFF_K + STAGES * TILE_B;     // pass 2: -(M + log2 L) per row (GROWS)
    static constexpr int OFF_LIM = OFF_CB + GROWS * 4;         // last visible key per row
    static constexpr int OFF_RED = OFF_LIM + GROWS * 4;        // [GROWS][2] row statistics
    static constexpr int OFF_BAR = OFF_RED + 2 * GROWS * 4;
    // accumulator buffers: four (all 512 columns) for one row block of d = 128,
    // where shared memory already holds the SM to one CTA; otherwise two
    static constexpr int NACC = (D == 128 && RB == 1) ? 4 : 2;
    static constexpr int NBAR = 2 * STAGES + 1 + 2 * NACC;
    static constexpr int OFF_TMEM = OFF_BAR + NBAR * 8;
    static constexpr int SMEM = OFF_TMEM + 16;
    static constexpr int SMEM_ALLOC = SMEM + 1024;
    static constexpr uint32_t TMEM_COLS = NACC * RB * TK;  // NACC accumulator buffers of RB blocks
    static constexpr uint32_t IDESC = idesc_bf16_f32(128, 128);
    static_assert(ROWS == 128 && TK == 128, "one 128x128 MMA shape for both passes");
    static_assert(RB == 1 || RB == 2, "one or two row blocks per CTA");
    static_assert(GROWS <= NET, "one epilogue thread per window row of the CTA");
    static_assert(SMEM_ALLOC <= 227 * 1024, "shared memory of one CTA");
};

template <int D, bool PASS2, int RB, int ST>
__global__ void __launch_bounds__(ScoreCfg<D, RB, ST>::NT, 1)
    score_kernel(const __grid_constant__ ScoreParams p, const __grid_constant__ CUtensorMap tmk,
                 const __grid_constant__ CUtensorMap tmq) {
    using C = ScoreCfg<D, RB, ST>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem =
        reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(smem);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const uint32_t bar_kfull = sbase + C::OFF_BAR;
    const uint32_t bar_kempty = bar_kfull + 8 * C::STAGES;
    const uint32_t bar_q = bar_kempty + 8 * C::STAGES;
    const uint32_t bar_tfull = bar_q + 8;
    const uint32_t bar_tempty = bar_tfull + 8 * C::NACC;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_TMEM);
    __shared__ int s_abort;
    __shared__ int s_last;

    const int mg = blockIdx.x % p.n_mg;
    const int rest = blockIdx.x / p.n_mg;
    const int sp = rest % p.nsplit;
    const int bh = rest / p.nsplit;
    const int b = bh / p.Hkv, h = bh - (bh / p.Hkv) * p.Hkv;
    const int lo = sp * p.chunk;
    const int hi = min(lo + p.chunk, p.n);
    const int ntiles = (hi - lo + C::TK - 1) / C::TK;
    const int row_base = mg * C::GROWS;   // first window row (of R = G * W) of this CTA

    if (!PASS2 && tid == 0) {
        // the first stages' K tiles and this CTA's window rows into L2 while the
        // previous kernel finishes
        prefetch_tmap(&tmk);
        prefetch_tmap(&tmq);
        for (int t = 0; t < C::STAGES && t < ntiles; ++t)
#pragma unroll
            for (int hf = 0; hf < C::HALVES; ++hf) tma_prefetch_4d(&tmk, hf * 64, lo + t * C::TK, h, b);
#pragma unroll
        for (int rb = 0; rb < RB; ++rb)
#pragma unroll
            for (int hf = 0; hf < C::HALVES; ++hf)
                tma_prefetch_2d(&tmq, hf * 64, (b * p.Hq + h * p.G) * p.W + row_base + rb * C::ROWS);
    }
    // barriers and tensor memory are this CTA's own: set up while the previous
    // kernel finishes
    if (tid == 0) {
#pragma unroll
        for (int s = 0; s < C::STAGES; ++s) {
            mbar_init(bar_kfull + 8 * s, 1);
            mbar_init(bar_kempty + 8 * s, 1);
        }
        mbar_init(bar_q, 1);
        for (int i = 0; i < C::NACC; ++i) {
            mbar_init(bar_tfull + 8 * i, 1);
            mbar_init(bar_tempty + 8 * i, C::NEPI / 2);   // one epilogue group per buffer
        }
        fence_mbar_init();
        s_abort = 0;
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_slot), C::TMEM_COLS);
        tmem_relinquish();
    }
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    // Pass 2 always follows pass 1 of the same call, which writes only the row
    // statistics (read by the epilogue) and never K or the window rows.  Its
    // producer and MMA warps therefore start before the grid dependency resolves:
    // every pass-1 CTA has passed its own wait before any pass-2 CTA starts, so
    // the caller's K and window rows are complete, and the first tiles stream
    // from L2 into shared memory and tensor memory while the last pass-1 CTAs
    // finish.  Only the epilogue waits.
    if (!PASS2 || warp >= 2) griddep_wait();
    griddep_launch();
    volatile int* abort_flag = &s_abort;

    if (warp == 0) {
        // ---------------------------------------------------------- TMA producer
        if (lane == 0) {
            prefetch_tmap(&tmk);
            prefetch_tmap(&tmq);
            // window rows of this row block: rows (b*Hq + h*G)*W + row_base ... +127 of
            // the flattened [B*Hq*W][d] window queries (contiguous per KV head)
            const int qrow0 = (b * p.Hq + h * p.G) * p.W + row_base;
            mbar_arrive_expect_tx(bar_q, C::Q_B);
#pragma unroll
            for (int rb = 0; rb < RB; ++rb)
#pragma unroll
                for (int hf = 0; hf < C::HALVES; ++hf)
                    tma_load_2d(sbase + C::OFF_Q + rb * C::QBLK_B + hf * C::HALF_B, &tmq, hf * 64,
                                qrow0 + rb * C::ROWS, bar_q);
            for (int t = 0; t < ntiles; ++t) {
                const int s = t % C::STAGES;
                if (t >= C::STAGES && !mbar_wait(bar_kempty + 8 * s, ((t / C::STAGES) & 1) ^ 1)) {
                    flag_status(p.status, SDKV_DEV_TIMEOUT);
                    *abort_flag = 1;
                    break;
                }
                if (*abort_flag) break;
                mbar_arrive_expect_tx(bar_kfull + 8 * s, C::TILE_B);
#pragma unroll
                for (int hf = 0; hf < C::HALVES; ++hf)
                    tma_load_4d(sbase + C::OFF_K + s * C::TILE_B + hf * C::HALF_B, &tmk, hf * 64, lo + t * C::TK,
                                h, b, bar_kfull + 8 * s);
            }
        }
    } else if (warp == 1) {
        // ---------------------------------------------------------- MMA issuer
        if (lane == 0) {
            bool ok = mbar_wait(bar_q, 0);
            for (int t = 0; ok && t < ntiles; ++t) {
                const int s = t % C::STAGES, buf = t % C::NACC;
                ok = mbar_wait(bar_kfull + 8 * s, (t / C::STAGES) & 1);
                if (ok && t >= C::NACC) ok = mbar_wait(bar_tempty + 8 * buf, ((t / C::NACC) & 1) ^ 1);
                if (!ok || *abort_flag) break;
                tc_fence_after();
                const uint32_t kst = sbase + C::OFF_K + s * C::TILE_B;
#pragma unroll
                for (int rb = 0; rb < RB; ++rb) {
                    // row block rb of this CTA against the K tile, accumulator rb of the buffer
                    const uint32_t d_tmem = tmem + (buf * RB + rb) * C::TK;
                    const uint32_t qblk = sbase + C::OFF_Q + rb * C::QBLK_B;
#pragma unroll
                    for (int ks = 0; ks < D / 16; ++ks) {
                        const uint32_t off = (ks >> 2) * C::HALF_B + (ks & 3) * 32;
                        const uint64_t qd = sw128_kmajor_desc(qblk + off);
                        const uint64_t kd = sw128_kmajor_desc(kst + off);
                        if (PASS2)
                            tc_mma_bf16(d_tmem, kd, qd, C::IDESC, ks > 0);
                        else
                            tc_mma_bf16(d_tmem, qd, kd, C::IDESC, ks > 0);
                    }
                }
                tc_commit(bar_kempty + 8 * s);    // the stage is free once these MMAs are done
                tc_commit(bar_tfull + 8 * buf);   // and the accumulator is ready
            }
            if (!ok) {
                flag_status(p.status, SDKV_DEV_TIMEOUT);
                *abort_flag = 1;
            }
        }
    } else {
        // ---------------------------------------------------------- epilogue
        const int ew = warp - 2;
        const int quad = warp & 3;          // tensor-memory lanes 32*quad .. +31
        const int half = ew >> 2;           // accumulator columns half*64 .. +63
        const int tl = 32 * quad + lane;    // accumulator lane of this thread
        float* cb = reinterpret_cast<float*>(smem + C::OFF_CB);
        int* lim = reinterpret_cast<int*>(smem + C::OFF_LIM);
        float* red = reinterpret_cast<float*>(smem + C::OFF_RED);
        const int et = ew * 32 + lane;      // 0 .. NET-1
        if (et < C::GROWS) {
            const int r = row_base + et;
            lim[et] = (r < p.R) ? p.q_pos0 + r % p.W : -1;
        }
        if constexpr (PASS2) {
            // Row statistics over the key splits of pass 1: TPR threads per row of the
            // CTA, thread et merges splits s = et/GROWS, et/GROWS + TPR, ... of row
            // et%GROWS (up to 16 loads in flight); with two threads per row the two
            // halves meet in shared memory.  The exponent bias of a row is
            // -(M + log2 L), so a key's probability is 2^(c*q.k + bias).
            constexpr int TPR = C::NET / C::GROWS;
            static_assert(TPR == 1 || TPR == 2, "one or two threads per row");
            const int rr = et % C::GROWS, s0 = et / C::GROWS;
            const int r = row_base + rr;
            float mm = -INFINITY, ll = 0.f;
            if (r < p.R) {
                const float* base = p.st_part + (static_cast<size_t>(bh) * p.nsplit * p.R + r) * 2;
                const size_t stride = static_cast<size_t>(p.R) * 2;
                for (int sb = s0; sb < p.nsplit; sb += 16 * TPR) {
                    float2 v2[16];
#pragma unroll
                    for (int u = 0; u < 16; ++u) {
                        const int sidx = sb + TPR * u;
                        v2[u] = sidx < p.nsplit ? __ldcg(reinterpret_cast<const float2*>(base + sidx * stride))
                                                : make_float2(-INFINITY, 0.f);
                    }
                    // the batch's max first, so that its sixteen exponentials are independent
                    float bm = -INFINITY;
#pragma unroll
                    for (int u = 0; u < 16; ++u) bm = fmaxf(bm, v2[u].x);
                    if (bm != -INFINITY) {
                        const float mnew = fmaxf(mm, bm);
                        float acc = (mm == -INFINITY) ? 0.f : ll * fast_exp2(mm - mnew);
#pragma unroll
                        for (int u = 0; u < 16; ++u)
                            acc += (v2[u].x == -INFINITY) ? 0.f : v2[u].y * fast_exp2(v2[u].x - mnew);
                        ll = acc;
                        mm = mnew;
                    }
                }
            }
            if (TPR == 2 && s0 == 1) {
                red[2 * rr] = mm;
                red[2 * rr + 1] = ll;
            }
            named_bar_sync(1, C::NET);
            if (s0 == 0) {
                float M = mm, L = ll;
                if (TPR == 2) {
                    const float m2 = red[2 * rr], l2 = red[2 * rr + 1];
                    M = fmaxf(mm, m2);
                    L = 0.f;
                    if (M != -INFINITY)
                        L = (mm == -INFINITY ? 0.f : ll * fast_exp2(mm - M)) +
                            (m2 == -INFINITY ? 0.f : l2 * fast_exp2(m2 - M));
                }
                cb[rr] = (r < p.R && L > 0.f) ? -(M + fast_log2(L)) : -INFINITY;   // rows past R add nothing
            }
        }
        named_bar_sync(1, C::NET);
        const float c = p.scale_log2;
        // pass 1 state: row tl of each row block
        int my_lim[RB];
        float m_run[RB], l_run[RB];
#pragma unroll
        for (int rb = 0; rb < RB; ++rb) {
            my_lim[rb] = lim[rb * C::ROWS + tl];
            m_run[rb] = -INFINITY;
            l_run[rb] = 0.f;
        }
        bool aborted = false;

        // Epilogue group `half` (warps 2-5 or 6-9) takes the tiles of its parity,
        // i.e. only accumulator buffers of that parity (RB accumulators of 128
        // columns each); the two groups never meet inside the loop.  Columns are read 64 at a
        // time; the buffer is handed back to the MMA issuer as soon as its last
        // columns are loaded.
        for (int t = half; t < ntiles; t += 2) {
            const int buf = t % C::NACC;
            if (!mbar_wait(bar_tfull + 8 * buf, (t / C::NACC) & 1)) {
                aborted = true;
                break;
            }
            tc_fence_after();
            const int key0 = lo + t * C::TK;
            float acc = 0.f;   // pass 2: this key's sum over the rows
#pragma unroll
            for (int rb = 0; rb < RB; ++rb) {
            const uint32_t ta = tmem + (static_cast<uint32_t>(32 * quad) << 16) + (buf * RB + rb) * C::TK;
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
                uint32_t v[64];
                tmem_ld64_sync(ta + hh * 64, v);
                if (rb == RB - 1 && hh == 1) {
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(bar_tempty + 8 * buf);
                }
                if constexpr (!PASS2) {
                    // row tl of row block rb, columns = keys key0 + hh*64 + i
                    if (my_lim[rb] >= 0) {
                        const int kfirst = key0 + hh * 64;
                        const bool full = (kfirst + 63 < hi) && (kfirst + 63 <= my_lim[rb]);
                        float mx = -INFINITY;
                        if (full) {
#pragma unroll
                            for (int i = 0; i < 64; ++i) mx = fmaxf(mx, __uint_as_float(v[i]));
                        } else {
#pragma unroll
                            for (int i = 0; i < 64; ++i) {
                                const int key = kfirst + i;
                                const float x = (key < hi && key <= my_lim[rb]) ? __uint_as_float(v[i]) : -INFINITY;
                                v[i] = __float_as_uint(x);
                                mx = fmaxf(mx, x);
                            }
                        }
                        if (mx != -INFINITY) {
                            const float mnew = fmaxf(m_run[rb], mx * c);
                            // four running sums (lanes i%4) in two paired registers
                            const float2 c2 = make_float2(c, c), nm2 = make_float2(-mnew, -mnew);
                            float2 s01 = make_float2(0.f, 0.f), s23 = s01;
#pragma unroll
                            for (int i = 0; i < 64; i += 4) {
                                const float2 x01 = fma2(make_float2(__uint_as_float(v[i]), __uint_as_float(v[i + 1])), c2, nm2);
                                const float2 x23 = fma2(make_float2(__uint_as_float(v[i + 2]), __uint_as_float(v[i + 3])), c2, nm2);
                                s01 = add2(s01, make_float2(fast_exp2(x01.x), fast_exp2(x01.y)));
                                s23 = add2(s23, make_float2(fast_exp2(x23.x), fast_exp2(x23.y)));
                            }
                            l_run[rb] = l_run[rb] * fast_exp2(m_run[rb] - mnew) + ((s01.x + s01.y) + (s23.x + s23.y));
                            m_run[rb] = mnew;
                        }
                    }
                } else {
                    // lane tl is key key0 + tl; columns are window rows rb*128 + hh*64 + i
                    const int key = key0 + tl;
                    const bool all_rows = key0 + C::TK - 1 <= p.q_pos0;
                    const float2 c2 = make_float2(c, c);
                    float2 s01 = make_float2(0.f, 0.f), s23 = s01;   // running sums of columns i%4
                    if (all_rows) {
                        // every window row sees every key of the tile: no mask
#pragma unroll
                        for (int i = 0; i < 64; i += 4) {
                            const float4 b4 = *reinterpret_cast<const float4*>(cb + rb * C::ROWS + hh * 64 + i);
                            const float2 x01 = fma2(make_float2(__uint_as_float(v[i]), __uint_as_float(v[i + 1])), c2,
                                                    make_float2(b4.x, b4.y));
                            const float2 x23 = fma2(make_float2(__uint_as_float(v[i + 2]), __uint_as_float(v[i + 3])), c2,
                                                    make_float2(b4.z, b4.w));
                            s01 = add2(s01, make_float2(fast_exp2(x01.x), fast_exp2(x01.y)));
                            s23 = add2(s23, make_float2(fast_exp2(x23.x), fast_exp2(x23.y)));
                        }
                    } else {
#pragma unroll
                        for (int i = 0; i < 64; i += 4) {
                            const float4 b4 = *reinterpret_cast<const float4*>(cb + rb * C::ROWS + hh * 64 + i);
                            const int4 l4 = *reinterpret_cast<const int4*>(lim + rb * C::ROWS + hh * 64 + i);
                            const float2 x01 = fma2(make_float2(__uint_as_float(v[i]), __uint_as_float(v[i + 1])), c2,
                                                    make_float2(b4.x, b4.y));
                            const float2 x23 = fma2(make_float2(__uint_as_float(v[i + 2]), __uint_as_float(v[i + 3])), c2,
                                                    make_float2(b4.z, b4.w));
                            const float e0 = key <= l4.x ? fast_exp2(x01.x) : 0.f;
                            const float e1 = key <= l4.y ? fast_exp2(x01.y) : 0.f;
                            const float e2 = key <= l4.z ? fast_exp2(x23.x) : 0.f;
                            const float e3 = key <= l4.w ? fast_exp2(x23.y) : 0.f;
                            s01 = add2(s01, make_float2(e0, e1));
                            s23 = add2(s23, make_float2(e2, e3));
                        }
                    }
                    acc += (s01.x + s01.y) + (s23.x + s23.y);
                }
            }
            }
            if constexpr (PASS2) {
                const int key = key0 + tl;
                if (key < hi) {
                    if (p.n_mg == 1)
                        p.scores[static_cast<size_t>(bh) * p.n + key] = acc * p.inv_w;
                    else
                        p.sc_part[(static_cast<size_t>(mg) * p.BH + bh) * p.n + key] = acc;
                }
            }
        }
        if (aborted && lane == 0) {
            flag_status(p.status, SDKV_DEV_TIMEOUT);
            *abort_flag = 1;
        }
        const bool stop = named_bar_or(1, C::NET, aborted || *abort_flag);
        if (!stop) {
            if constexpr (!PASS2) {
                // merge the two epilogue groups' statistics of each row, store the split's partial
                if (half == 1) {
#pragma unroll
                    for (int rb = 0; rb < RB; ++rb) {
                        red[2 * (rb * C::ROWS + tl)] = m_run[rb];
                        red[2 * (rb * C::ROWS + tl) + 1] = l_run[rb];
                    }
                }
                named_bar_sync(1, C::NET);
                if (half == 0) {
#pragma unroll
                    for (int rb = 0; rb < RB; ++rb) {
                        const float m2 = red[2 * (rb * C::ROWS + tl)], l2 = red[2 * (rb * C::ROWS + tl) + 1];
                        const float M = fmaxf(m_run[rb], m2);
                        float L = 0.f;
                        if (M != -INFINITY)
                            L = (m_run[rb] == -INFINITY ? 0.f : l_run[rb] * fast_exp2(m_run[rb] - M)) +
                                (m2 == -INFINITY ? 0.f : l2 * fast_exp2(m2 - M));
                        const int r = row_base + rb * C::ROWS + tl;
                        if (r < p.R)
                            *reinterpret_cast<float2*>(
                                p.st_part + ((static_cast<size_t>(bh) * p.nsplit + sp) * p.R + r) * 2) = make_float2(M, L);
                    }
                }
            } else if (p.n_mg > 1) {
                __threadfence();
                named_bar_sync(1, C::NET);
                if (et == 0) {
                    const int old = atomicAdd(p.tick2 + bh * p.nsplit + sp, 1);
                    s_last = (old == p.n_mg - 1);
                }
                named_bar_sync(1, C::NET);
                if (s_last) {
                    __threadfence();
                    // each key's row-block partials added in row-block order; four keys
                    // per step (16-byte loads where rows are aligned) and eight row
                    // blocks' loads in flight
                    const bool vec = (p.n % 4) == 0 && (reinterpret_cast<uintptr_t>(p.scores) & 15) == 0;
                    const int k4 = vec ? (hi - lo) / 4 : 0;
                    for (int q = et; q < k4; q += C::NET) {
                        const int key = lo + 4 * q;
                        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
                        for (int g0 = 0; g0 < p.n_mg; g0 += 8) {
                            float4 v4[8];
#pragma unroll
                            for (int u = 0; u < 8; ++u)
                                v4[u] = (g0 + u < p.n_mg)
                                            ? __ldcg(reinterpret_cast<const float4*>(
                                                  p.sc_part + (static_cast<size_t>(g0 + u) * p.BH + bh) * p.n + key))
                                            : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
                            for (int u = 0; u < 8; ++u) {
                                if (g0 + u < p.n_mg) {
                                    acc.x += v4[u].x;
                                    acc.y += v4[u].y;
                                    acc.z += v4[u].z;
                                    acc.w += v4[u].w;
                                }
                            }
                        }
                        *reinterpret_cast<float4*>(p.scores + static_cast<size_t>(bh) * p.n + key) =
                            make_float4(acc.x * p.inv_w, acc.y * p.inv_w, acc.z * p.inv_w, acc.w * p.inv_w);
                    }
                    for (int key = lo + 4 * k4 + et; key < hi; key += C::NET) {
                        float v2 = 0.f;
                        for (int g0 = 0; g0 < p.n_mg; g0 += 8) {
                            float v1[8];
#pragma unroll
                            for (int u = 0; u < 8; ++u)
                                v1[u] = (g0 + u < p.n_mg)
                                            ? __ldcg(p.sc_part + (static_cast<size_t>(g0 + u) * p.BH + bh) * p.n + key)
                                            : 0.f;
#pragma unroll
                            for (int u = 0; u < 8; ++u)
                                if (g0 + u < p.n_mg) v2 += v1[u];
                        }
                        p.scores[static_cast<size_t>(bh) * p.n + key] = v2 * p.inv_w;
                    }
                    if (et == 0) atomicExch(p.tick2 + bh * p.nsplit + sp, 0);
                }
            }
        }
    }

    // ------------------------------------------------------------------ teardown
    if (*abort_flag && tid == 0) {
        // let copies in flight land before the CTA's shared memory goes away (bounded)
        for (int s = 0; s < C::STAGES && s < ntiles; ++s) {
            const int last_t = ((ntiles - 1 - s) / C::STAGES) * C::STAGES + s;
            mbar_wait(bar_kfull + 8 * s, (last_t / C::STAGES) & 1);
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, C::TMEM_COLS);
    }
}

// =====================================================================================
// host side
// =====================================================================================
namespace {

struct ScorePlan {
    int rb, n_mg, nsplit, chunk;
    size_t off_t2, off_sp, off_sc, bytes;
};

ScorePlan score_plan(int B, int Hq, int Hkv, int n, int W, int num_sms) {
    ScorePlan pl{};
    const int BH = B * Hkv;
    const int R = (Hq / Hkv) * W;
    constexpr int ROWS = 128, TK = 128;
    // more than one row block per head: two per CTA, sharing each K tile
    pl.rb = R > ROWS ? 2 : 1;
    pl.n_mg = (R + pl.rb * ROWS - 1) / (pl.rb * ROWS);
    const int target = std::max(num_sms, 1);   // one CTA per SM (tensor memory + 130 KB of stages)
    // splits per (sequence, KV head, row block): as many as fit one wave; a
    // second wave would double the time for the few CTAs that spill into it
    const int units = BH * pl.n_mg;
    int nsplit = units >= target ? 1 : target / units;
    nsplit = std::min(nsplit, std::max(1, (n + TK - 1) / TK));
    int chunk = (n + nsplit - 1) / nsplit;
    chunk = ((chunk + TK - 1) / TK) * TK;
    pl.nsplit = (n + chunk - 1) / chunk;
    pl.chunk = chunk;
    size_t off = kWsHeader;
    pl.off_t2 = off;
    off += sizeof(int) * static_cast<size_t>(BH) * pl.nsplit;
    off = align256(off);
    pl.off_sp = off;
    off = align256(off + sizeof(float) * 2 * static_cast<size_t>(BH) * pl.nsplit * R);
    pl.off_sc = off;
    if (pl.n_mg > 1) off = align256(off + sizeof(float) * static_cast<size_t>(pl.n_mg) * BH * n);
    pl.bytes = off;
    return pl;
}

template <int D, bool PASS2, int RB, int ST>
cudaError_t launch_score_pass(const ScoreParams& p, const CUtensorMap& tmk, const CUtensorMap& tmq, int grid,
                              cudaStream_t st) {
    using C = ScoreCfg<D, RB, ST>;
    auto kern = score_kernel<D, PASS2, RB, ST>;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    static std::atomic<unsigned long long> attr_set{0};  // one bit per device, per instantiation
    if (!attr_done(attr_set, dev)) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_ALLOC);
        if (e != cudaSuccess) return e;
        attr_mark(attr_set, dev);
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(C::NT);
    cfg.dynamicSmemBytes = C::SMEM_ALLOC;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, p, tmk, tmq);
}

}  // namespace

size_t score_ws_bytes(int B, int Hq, int Hkv, int d, int n, int W, int num_sms) {
    (void)d;
    return score_plan(B, Hq, Hkv, n, W, num_sms).bytes;
}

int launch_score(const ScoreLaunch& a, const CUtensorMap* tmk, const CUtensorMap* tmq, int num_sms,
                 const char** why) {
    const ScorePlan pl = score_plan(a.B, a.Hq, a.Hkv, a.n, a.W, num_sms);
    if (a.ws_bytes < pl.bytes) {
        *why = "workspace smaller than sdkv_workspace_size(SDKV_OP_SCORE, ...)";
        return SDKV_ERR_WORKSPACE;
    }
    uint8_t* ws = static_cast<uint8_t*>(a.ws);
    ScoreParams p{};
    p.B = a.B;
    p.Hq = a.Hq;
    p.Hkv = a.Hkv;
    p.G = a.Hq / a.Hkv;
    p.W = a.W;
    p.R = p.G * a.W;
    p.n = a.n;
    p.q_pos0 = a.q_pos0;
    p.BH = a.B * a.Hkv;
    p.n_mg = pl.n_mg;
    p.nsplit = pl.nsplit;
    p.chunk = pl.chunk;
    p.scale_log2 = a.scale * kLog2e;
    p.inv_w = 1.0f / static_cast<float>(a.W);
    p.scores = a.scores;
    p.status = reinterpret_cast<int*>(ws);
    p.tick2 = reinterpret_cast<int*>(ws + pl.off_t2);
    p.st_part = reinterpret_cast<float*>(ws + pl.off_sp);
    p.sc_part = reinterpret_cast<float*>(ws + pl.off_sc);
    const int grid = p.BH * pl.n_mg * pl.nsplit;
    cudaError_t e;
    if (a.d == 128) {
        if (pl.rb == 2) {
            e = launch_score_pass<128, false, 2, 3>(p, *tmk, *tmq, grid, a.stream);
            if (e == cudaSuccess) e = launch_score_pass<128, true, 2, 3>(p, *tmk, *tmq, grid, a.stream);
        } else {
            // K stages with one row block of d = 128: pass 2 fills five stages (and the
            // four accumulators) while pass 1 finishes; pass 1 streams from HBM, where
            // five stages pay off only for long splits (128K: 84.8 -> 83.3 us per
            // layer) and cost time for short ones (32K: 24.6 -> 25.1 us)
            const bool long_split = (pl.chunk + 127) / 128 >= 32;
            e = long_split ? launch_score_pass<128, false, 1, 5>(p, *tmk, *tmq, grid, a.stream)
                           : launch_score_pass<128, false, 1, 3>(p, *tmk, *tmq, grid, a.stream);
            if (e == cudaSuccess) e = launch_score_pass<128, true, 1, 5>(p, *tmk, *tmq, grid, a.stream);
        }
    } else {
        if (pl.rb == 2) {
            e = launch_score_pass<64, false, 2, 3>(p, *tmk, *tmq, grid, a.stream);
            if (e == cudaSuccess) e = launch_score_pass<64, true, 2, 3>(p, *tmk, *tmq, grid, a.stream);
        } else {
            e = launch_score_pass<64, false, 1, 3>(p, *tmk, *tmq, grid, a.stream);
            if (e == cudaSuccess) e = launch_score_pass<64, true, 1, 3>(p, *tmk, *tmq, grid, a.stream);
        }
    }
    if (e != cudaSuccess) {
        *why = cudaGetErrorString(e);
        return SDKV_ERR_CUDA;
    }
    return SDKV_OK;
}

}  // namespace sdkv
