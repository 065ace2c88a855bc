// Gathered decode over many short index lists, packed by list position.
//
// With many (sequence, KV head) lists of a few hundred entries each (SparseMM's
// per-head budgets: 32 heads x batch 8 = 256 lists, most of them 80-250 rows,
// a few of them thousands), one CTA per list chunk spends most of its time in
// its ramp and merge, and the chunks outnumber the slots of one wave.  Here the
// grid is one wave and CTA c takes an equal span of positions of the
// concatenated lists (the CSR index array): the end of one list, whole lists and
// the start of another.  The query rows of up to 16 / R lists (R = Hq / Hkv
// rows each) share the 16 rows of the mma.sync tile, and a key is scored against
// the rows of its own list only (the rows of the other lists see it masked), so
// the lists of a span stream through one pipeline with no flush between them.
// A list that lies inside one span is normalised and written by its CTA; a list
// cut by span ends leaves an unnormalised partial (o, m, l) in every CTA it
// touches, and the last of them to finish (atomic ticket) merges the partials
// with the log-sum-exp rule
//     o = sum_s 2^(m_s - M) o_s / sum_s 2^(m_s - M) l_s,   M = max_s m_s.
// The arithmetic per key is that of the split-K decode (StD 3.2 sparse attention
// over the selected entries; ByteCross "Speedup Across Context" for the gather).
#include "sdkv_common.cuh"
#include "sdkv_internal.h"

#include <algorithm>
#include <climits>

namespace sdkv {

struct PackParams {
    const bf16* q;
    const bf16* k;
    const bf16* v;
    long long sb, sh, sn;
    int Hq, Hkv, G, BH;
    bf16* o;
    float* lse;
    float scale_log2;
    const int* offsets;
    const int* indices;
    long long n_idx;   // entries of indices; 0: the lists are not read before the grid dependency resolves
    int n_cap, min_span;
    int* status;
    int* tickets;
    float* part_o;     // [2 * grid][R][D]: slot 2c holds the list cut by span c's start, 2c + 1 the one cut by its end
    float* part_ml;    // [2 * grid][R][4]: (m, l, -, -), 16-byte records
};

template <int D>
struct PackCfg {
    static constexpr int TK = 64;                // keys per stage
    static constexpr int STAGES = 3;
    static constexpr int KW = 4;                 // consumer warps, one key group each
    static constexpr int NCW = KW, NCT = 32 * NCW;
    static constexpr int NPW = 2;                // gathering warps: one list entry per lane per stage
    static constexpr int NT = NCT + 32 * NPW;
    static constexpr int KPW = TK / KW;          // keys per consumer warp per stage
    static constexpr int ROWS = 16;              // query rows of one pass: lists x R
    static constexpr int TILE_B = TK * 2 * D;
    static constexpr int QPITCH = 2 * D + 16;
    static constexpr int MPITCH = D + 8;
    static constexpr int OFF_K = 0;
    static constexpr int OFF_V = STAGES * TILE_B;
    static constexpr int OFF_Q = 2 * STAGES * TILE_B;
    static constexpr int OFF_ML = OFF_Q + ROWS * QPITCH;     // [KW][ROWS] (m, l)
    static constexpr int OFF_BAR = OFF_ML + KW * ROWS * 2 * 4;
    static constexpr int SMEM = OFF_BAR + 2 * STAGES * 8;
    static constexpr int SMEM_ALLOC = SMEM + 1024;
    // the list offsets are read once into the (still idle) stage buffers
    static constexpr int MAX_LISTS = 2 * STAGES * TILE_B / 4 - 1;
    static_assert(KPW == 16, "one 16-key sub-step per consumer warp and stage");
    static_assert(TK == 32 * NPW, "one list entry per gathering lane per stage");
    static_assert(KW * ROWS * MPITCH * 4 <= 2 * STAGES * TILE_B, "merge rows fit in the stage buffers");
    static_assert(TILE_B % 1024 == 0, "swizzled stages need 1024-byte alignment");
};

constexpr int kPackMaxLists = 2048;   // lists a launch takes (the host checks)
static_assert(PackCfg<64>::MAX_LISTS >= kPackMaxLists && PackCfg<128>::MAX_LISTS >= kPackMaxLists,
              "the offsets fit in the stage buffers");

__device__ __forceinline__ int clamp_pos(long long x, long long lo, long long hi) {
    return static_cast<int>(x < lo ? lo : (x > hi ? hi : x));
}

template <int D>
__global__ void __launch_bounds__(PackCfg<D>::NT) packed_decode_kernel(const __grid_constant__ PackParams p) {
    using C = PackCfg<D>;
    constexpr int TK = C::TK, STAGES = C::STAGES, KW = C::KW;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem =
        reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(smem);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const uint32_t bar_full = sbase + C::OFF_BAR;
    const uint32_t bar_empty = bar_full + STAGES * 8;

    __shared__ int s_cnt[3];        // lists wholly before this span; lists starting before its end; a bad list
    __shared__ int s_cut[2][3];     // lists cut by the span's start / end: (list, start, end); list -1: none
    __shared__ int s_tab[17];       // boundaries of the current pass's lists, clipped to the span
    __shared__ int s_abort;
    __shared__ int s_win[2];        // this CTA merges cut list 0 / 1

    if (tid == 0) {
#pragma unroll
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(bar_full + 8 * s, C::NPW * 32);
            mbar_init(bar_empty + 8 * s, C::NCW);
        }
        fence_mbar_init();
        s_abort = 0;
        s_cnt[0] = s_cnt[1] = s_cnt[2] = 0;
    }
    {
        // Before the grid dependency resolves: the offsets and this CTA's share of
        // the index array (n_idx > 0) into L2.  Prefetches return nothing, and L2 is
        // where every write lands, so a line fetched early is never older than what
        // a later load of it returns.
        const uint8_t* ob = reinterpret_cast<const uint8_t*>(p.offsets);
        const long long obytes = 4ll * (p.BH + 1);
        for (long long x = 128ll * tid; x < obytes; x += 128ll * C::NT) prefetch_l2_line(ob + x);
        if (p.n_idx > 0) {
            const long long ibytes = 4 * p.n_idx;
            const long long per = (ibytes + gridDim.x - 1) / gridDim.x;
            const long long i0 = per * blockIdx.x, i1 = min(ibytes, i0 + per);
            const uint8_t* ib = reinterpret_cast<const uint8_t*>(p.indices);
            for (long long x = i0 + 128ll * tid; x < i1; x += 128ll * C::NT) prefetch_l2_line(ib + x);
        }
    }
    __syncthreads();
    griddep_launch();
    griddep_wait();

    // ------------------------------------------------------------------ the span
    // Span c = positions [off0 + c * cl, off0 + (c + 1) * cl) of the index array;
    // the last CTA's span runs to the end.  Its lists: those that overlap it, and
    // the empty ones whose position falls in it.  With non-decreasing offsets
    // they are the lists [first, end), first = the number of lists that end at
    // or before the span's start (and start before it), end = the number of
    // lists that start before the span's end.
    int* offc = reinterpret_cast<int*>(smem + C::OFF_K);
    for (int i = tid; i <= p.BH; i += C::NT) offc[i] = __ldcg(p.offsets + i);
    __syncthreads();
    const int off0 = offc[0];
    long long total = static_cast<long long>(offc[p.BH]) - off0;
    const bool total_bad = total < 0;
    if (total_bad) total = 0;
    const int ncta = gridDim.x, cta = blockIdx.x;
    long long cl = (total + ncta - 1) / ncta;
    cl = max(static_cast<long long>(p.min_span), (cl + 15) & ~15ll);
    const long long lo_c = off0 + cta * cl;
    const long long hi_c = (cta == ncta - 1) ? LLONG_MAX : lo_c + cl;
    // gathering warps: the list entries of the first stages, loaded ahead of the
    // plan (the first pass starts at the span's start; rows past its end are masked)
    const long long pos_end = off0 + total;
    const bool early = warp >= C::NCW && lo_c < pos_end;
    int idx_ring[STAGES];
    if (early) {
        const int pw = warp - C::NCW;
#pragma unroll
        for (int j = 0; j < STAGES; ++j)
            idx_ring[j] = __ldg(p.indices + min(lo_c + j * TK + pw * 32 + lane, pos_end - 1));
    }
    {
        int n_first = 0, n_end = 0;
        bool bad = false;
        for (int i = tid; i < p.BH; i += C::NT) {
            const int s = offc[i], e = offc[i + 1];
            bad |= e < s;
            n_first += (e <= lo_c && s < lo_c) ? 1 : 0;
            n_end += (s < hi_c) ? 1 : 0;
        }
        bad = __any_sync(0xffffffffu, bad) || total_bad;
        n_first = __reduce_add_sync(0xffffffffu, n_first);
        n_end = __reduce_add_sync(0xffffffffu, n_end);
        if (lane == 0) {
            atomicAdd(&s_cnt[0], n_first);
            atomicAdd(&s_cnt[1], n_end);
            if (bad) s_cnt[2] = 1;
        }
    }
    __syncthreads();
    // Decreasing offsets: every CTA reads all of them, so every CTA sees it and
    // leaves before touching a ticket (the outputs are left unwritten)
    if (s_cnt[2]) {
        if (tid == 0) flag_status(p.status, SDKV_DEV_BAD_LIST);
        return;
    }
    const int first = s_cnt[0], endl = s_cnt[1];
    if (first >= endl) return;   // nothing in this span (uniform)
    if (tid == 0) {
        s_cut[0][0] = s_cut[1][0] = -1;
        const int s = offc[first], e = offc[first + 1];
        if (s < lo_c && e > lo_c) {
            s_cut[0][0] = first;
            s_cut[0][1] = s;
            s_cut[0][2] = e;
        }
        const int l = endl - 1;
        const int s2 = offc[l], e2 = offc[l + 1];
        if (e2 > hi_c && s2 < hi_c && !(l == first && s_cut[0][0] >= 0)) {
            s_cut[1][0] = l;
            s_cut[1][1] = s2;
            s_cut[1][2] = e2;
        }
    }
    // no barrier needed here: s_cut is read after the first pass's barriers

    const int R = p.G;                          // query rows per list (one decode position)
    const int SEGS = C::ROWS / R;               // lists per pass
    const int npass = (endl - first + SEGS - 1) / SEGS;
    const int hi_int = static_cast<int>(min(hi_c, static_cast<long long>(INT_MAX)));
    const int lo_int = static_cast<int>(max(lo_c, static_cast<long long>(INT_MIN)));
    int gt0 = 0;   // stages filled by earlier passes (the mbarrier phases run on across passes)

    const int kw = warp;          // a consumer warp's key group
    const int r0 = lane >> 2;     // its lane's first row (the second is r0 + 8)

    for (int pp = 0; pp < npass; ++pp) {
        const int hA = first + pp * SEGS;
        const int nseg = min(SEGS, endl - hA);
        // the pass's list boundaries, clipped to the span: from the copy of the
        // offsets in the first pass, from L2 in later ones (the stages hold rows then)
        if (tid <= nseg) {
            const int v = (pp == 0) ? offc[hA + tid] : __ldcg(p.offsets + hA + tid);
            s_tab[tid] = clamp_pos(v, lo_int, hi_int);
        }
        __syncthreads();
        const int P0 = s_tab[0];
        const int npos = max(0, s_tab[nseg] - P0);
        const int ntiles = (npos + TK - 1) / TK;
        bool my_abort = false;

        if (warp >= C::NCW) {
            // -------------------------------------------------------------- gather
            // The NPW warps own 32 stage rows each; lane j holds the list entry of
            // its warp's row j, loaded STAGES stages ahead, and the row's list (the
            // cache row's base: sequence and KV head).  CPR lanes copy one row as
            // CPR 16-byte chunks per instruction.
            constexpr int CPR = D / 8;
            constexpr int RPI = 32 / CPR;
            const int pw = warp - C::NCW;
            auto pos_of = [&](int t) { return P0 + min(t * TK + pw * 32 + lane, npos - 1); };
            auto load_idx = [&](int t) -> int { return (t < ntiles) ? __ldg(p.indices + pos_of(t)) : 0; };
            if (!(pp == 0 && early && P0 == lo_c)) {
#pragma unroll
                for (int j = 0; j < STAGES; ++j) idx_ring[j] = load_idx(j);
            }
            for (int t = 0; t < ntiles; ++t) {
                int idx_cur = idx_ring[0];
                if (static_cast<unsigned>(idx_cur) >= static_cast<unsigned>(p.n_cap)) {
                    flag_status(p.status, SDKV_DEV_BAD_INDEX);
                    idx_cur = 0;
                }
#pragma unroll
                for (int j = 0; j + 1 < STAGES; ++j) idx_ring[j] = idx_ring[j + 1];
                idx_ring[STAGES - 1] = load_idx(t + STAGES);
                const int pos = pos_of(t);
                int sg = 0;
#pragma unroll
                for (int j = 1; j < 16; ++j) sg += (j < nseg && s_tab[j] <= pos) ? 1 : 0;
                const int lst = hA + sg;
                const int b = lst / p.Hkv, h = lst - b * p.Hkv;
                const long long roff = b * p.sb + h * p.sh + static_cast<long long>(idx_cur) * p.sn;
                const int gt = gt0 + t;
                const int s = gt % STAGES;
                const uint32_t ph = (gt / STAGES) & 1;
                if (gt >= STAGES) {
                    bool ok = mbar_wait(bar_empty + 8 * s, ph ^ 1);
                    ok = __all_sync(0xffffffffu, ok);
                    if (!ok) {
                        if (lane == 0) {
                            flag_status(p.status, SDKV_DEV_TIMEOUT);
                            atomicExch(&s_abort, 1);
                        }
                        my_abort = true;
                        break;
                    }
                }
                const uint32_t kst = sbase + C::OFF_K + s * C::TILE_B;
                const uint32_t vst = sbase + C::OFF_V + s * C::TILE_B;
                const int chunk = lane % CPR;
#pragma unroll 4
                for (int it = 0; it < 32 / RPI; ++it) {
                    const int rw = it * RPI + lane / CPR;
                    const long long off = __shfl_sync(0xffffffffu, roff, rw) + chunk * 8;
                    const int row = pw * 32 + rw;
                    cp_async_16(sw128_addr<TK>(kst, row, chunk), p.k + off);
                    cp_async_16(sw128_addr<TK>(vst, row, chunk), p.v + off);
                }
                cp_async_mbar_arrive(bar_full + 8 * s);
            }
            cp_async_wait_all();
        } else {
            // ------------------------------------------------------------ consumers
            // query rows of the pass: row r = list (r / R) of the pass, query head r % R
            uint8_t* qs = smem + C::OFF_Q;
            const int nrow = nseg * R;
            for (int e = tid; e < C::ROWS * (D / 8); e += C::NCT) {
                const int r = e / (D / 8), c = e % (D / 8);
                uint4 val = make_uint4(0u, 0u, 0u, 0u);
                if (r < nrow) {
                    const int sg = r / R, j = r - sg * R;
                    const int lst = hA + sg;
                    const int b = lst / p.Hkv, h = lst - b * p.Hkv;
                    val = *reinterpret_cast<const uint4*>(
                        p.q + (static_cast<size_t>(b) * p.Hq + h * p.G + j) * D + c * 8);
                }
                *reinterpret_cast<uint4*>(qs + r * C::QPITCH + c * 16) = val;
            }
            named_bar_sync(1, C::NCT);
            uint32_t qa[D / 16][4];
            {
                const int row = (lane & 7) + (((lane >> 3) & 1) << 3);
#pragma unroll
                for (int ks = 0; ks < D / 16; ++ks)
                    ldsm_x4(qa[ks], pad_addr<C::QPITCH>(sbase + C::OFF_Q, row, 2 * ks + (lane >> 4)));
            }
            // the positions (relative to the pass) each of this lane's two rows may see
            int rlo[2], rhi[2];
#pragma unroll
            for (int i = 0; i < 2; ++i) {
                const int row = r0 + 8 * i;
                rlo[i] = rhi[i] = 0;
                if (row < nrow) {
                    const int sg = row / R;
                    rlo[i] = s_tab[sg] - P0;
                    rhi[i] = max(rlo[i], s_tab[sg + 1] - P0);
                }
            }
            float o_acc[D / 8][4];
#pragma unroll
            for (int j = 0; j < D / 8; ++j) o_acc[j][0] = o_acc[j][1] = o_acc[j][2] = o_acc[j][3] = 0.f;
            float m_r[2] = {-INFINITY, -INFINITY};
            float l_r[2] = {0.f, 0.f};
            bool aborted = false;
            for (int t = 0; t < ntiles; ++t) {
                const int gt = gt0 + t;
                const int s = gt % STAGES;
                const uint32_t ph = (gt / STAGES) & 1;
                if (!__all_sync(0xffffffffu, mbar_wait(bar_full + 8 * s, ph))) {   // warp-uniform
                    aborted = true;
                    break;
                }
                const uint32_t kst = sbase + C::OFF_K + s * C::TILE_B;
                const uint32_t vst = sbase + C::OFF_V + s * C::TILE_B;
                float sacc[2][4];
#pragma unroll
                for (int nt = 0; nt < 2; ++nt) sacc[nt][0] = sacc[nt][1] = sacc[nt][2] = sacc[nt][3] = 0.f;
#pragma unroll
                for (int ks = 0; ks < D / 16; ++ks) {
                    uint32_t kb[4];
                    const int row = kw * C::KPW + (lane & 7) + ((lane >> 4) << 3);
                    ldsm_x4(kb, sw128_addr<TK>(kst, row, 2 * ks + ((lane >> 3) & 1)));
                    mma_bf16_16816(sacc[0], qa[ks], kb[0], kb[1]);
                    mma_bf16_16816(sacc[1], qa[ks], kb[2], kb[3]);
                }
                // log2 domain; a key counts for the rows of its own list only
                const int cpos = t * TK + kw * C::KPW + 2 * (lane & 3);
#pragma unroll
                for (int nt = 0; nt < 2; ++nt) {
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int col = cpos + nt * 8 + (e & 1);
                        const bool valid = col >= rlo[e >> 1] && col < rhi[e >> 1];
                        sacc[nt][e] = valid ? sacc[nt][e] * p.scale_log2 : -INFINITY;
                    }
                }
#pragma unroll
                for (int i = 0; i < 2; ++i) {
                    float mx = fmaxf(fmaxf(sacc[0][2 * i], sacc[0][2 * i + 1]), fmaxf(sacc[1][2 * i], sacc[1][2 * i + 1]));
                    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
                    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
                    const float mnew = fmaxf(m_r[i], mx);
                    const float muse = (mnew == -INFINITY) ? 0.f : mnew;
                    if (mnew != m_r[i]) {
                        const float alpha = fast_exp2(m_r[i] - muse);
                        l_r[i] *= alpha;
#pragma unroll
                        for (int j = 0; j < D / 8; ++j) {
                            o_acc[j][2 * i] *= alpha;
                            o_acc[j][2 * i + 1] *= alpha;
                        }
                        m_r[i] = mnew;
                    }
#pragma unroll
                    for (int nt = 0; nt < 2; ++nt) {
                        sacc[nt][2 * i] = fast_exp2(sacc[nt][2 * i] - muse);
                        sacc[nt][2 * i + 1] = fast_exp2(sacc[nt][2 * i + 1] - muse);
                        l_r[i] += sacc[nt][2 * i] + sacc[nt][2 * i + 1];
                    }
                }
                // P as two bf16 terms, p = hi + lo (about 16 significant bits), so the
                // weights of the PV product match the fp32 sum l
                uint32_t pa[4], pl[4];
                split_bf16(sacc[0][0], sacc[0][1], pa[0], pl[0]);
                split_bf16(sacc[0][2], sacc[0][3], pa[1], pl[1]);
                split_bf16(sacc[1][0], sacc[1][1], pa[2], pl[2]);
                split_bf16(sacc[1][2], sacc[1][3], pa[3], pl[3]);
#pragma unroll
                for (int jj = 0; jj < D / 16; ++jj) {
                    uint32_t vb[4];
                    const int row = kw * C::KPW + (lane & 7) + (((lane >> 3) & 1) << 3);
                    ldsm_x4_t(vb, sw128_addr<TK>(vst, row, 2 * jj + (lane >> 4)));
                    mma_bf16_16816(o_acc[2 * jj], pa, vb[0], vb[1]);
                    mma_bf16_16816(o_acc[2 * jj + 1], pa, vb[2], vb[3]);
                    mma_bf16_16816(o_acc[2 * jj], pl, vb[0], vb[1]);
                    mma_bf16_16816(o_acc[2 * jj + 1], pl, vb[2], vb[3]);
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(bar_empty + 8 * s);
            }
            if (aborted && lane == 0) flag_status(p.status, SDKV_DEV_TIMEOUT);
#pragma unroll
            for (int i = 0; i < 2; ++i) {
                l_r[i] += __shfl_xor_sync(0xffffffffu, l_r[i], 1);
                l_r[i] += __shfl_xor_sync(0xffffffffu, l_r[i], 2);
            }
            my_abort = named_bar_or(1, C::NCT, aborted || *reinterpret_cast<volatile int*>(&s_abort));
            if (!my_abort) {
                // ---------------------------------- merge the key groups of each row
                // each warp rescales its o to the row max over the groups and parks it
                // in the (drained) stage buffers; group kw then sums its slice of the
                // head dims over the groups and writes the list's output or partial
                float* ml = reinterpret_cast<float*>(smem + C::OFF_ML);
                if ((lane & 3) == 0) {
#pragma unroll
                    for (int i = 0; i < 2; ++i) {
                        ml[(kw * C::ROWS + r0 + 8 * i) * 2 + 0] = m_r[i];
                        ml[(kw * C::ROWS + r0 + 8 * i) * 2 + 1] = l_r[i];
                    }
                }
                named_bar_sync(1, C::NCT);
                float* mrg = reinterpret_cast<float*>(smem + C::OFF_K);
#pragma unroll
                for (int i = 0; i < 2; ++i) {
                    const int row = r0 + 8 * i;
                    if (row >= nrow) continue;
                    float M = -INFINITY;
#pragma unroll
                    for (int k2 = 0; k2 < KW; ++k2) M = fmaxf(M, ml[(k2 * C::ROWS + row) * 2]);
                    const float f = (m_r[i] == -INFINITY) ? 0.f : fast_exp2(m_r[i] - M);
                    float* dst = mrg + (kw * C::ROWS + row) * C::MPITCH + 2 * (lane & 3);
#pragma unroll
                    for (int j = 0; j < D / 8; ++j)
                        *reinterpret_cast<float2*>(dst + 8 * j) =
                            make_float2(o_acc[j][2 * i] * f, o_acc[j][2 * i + 1] * f);
                }
                named_bar_sync(1, C::NCT);
                constexpr int SL4 = D / KW / 4;   // float4 per row in this group's dim slice
                for (int e = lane; e < nrow * SL4; e += 32) {
                    const int row = e / SL4;
                    const int d0 = kw * (D / KW) + 4 * (e % SL4);
                    float M = -INFINITY;
#pragma unroll
                    for (int k2 = 0; k2 < KW; ++k2) M = fmaxf(M, ml[(k2 * C::ROWS + row) * 2]);
                    float L = 0.f;
                    float4 a4 = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
                    for (int k2 = 0; k2 < KW; ++k2) {
                        const float mk = ml[(k2 * C::ROWS + row) * 2];
                        L += (mk == -INFINITY) ? 0.f : ml[(k2 * C::ROWS + row) * 2 + 1] * fast_exp2(mk - M);
                        const float4 v4 = *reinterpret_cast<const float4*>(mrg + (k2 * C::ROWS + row) * C::MPITCH + d0);
                        a4.x += v4.x;
                        a4.y += v4.y;
                        a4.z += v4.z;
                        a4.w += v4.w;
                    }
                    const int sg = row / R, j = row - sg * R;
                    const int lst = hA + sg;
                    const int cut = (lst == s_cut[0][0]) ? 0 : (lst == s_cut[1][0]) ? 1 : -1;
                    if (cut < 0) {
                        const int b = lst / p.Hkv, h = lst - b * p.Hkv;
                        const size_t orow = static_cast<size_t>(b) * p.Hq + h * p.G + j;
                        const float il = L > 0.f ? 1.f / L : 0.f;
                        uint2 packed;
                        packed.x = pack_bf16(a4.x * il, a4.y * il);
                        packed.y = pack_bf16(a4.z * il, a4.w * il);
                        *reinterpret_cast<uint2*>(p.o + orow * D + d0) = packed;
                        if (d0 == 0 && p.lse) p.lse[orow] = L > 0.f ? (M + fast_log2(L)) * kLn2 : -INFINITY;
                    } else {
                        const size_t slot = 2 * static_cast<size_t>(cta) + cut;
                        *reinterpret_cast<float4*>(p.part_o + (slot * R + j) * D + d0) = a4;
                        if (d0 == 0)
                            *reinterpret_cast<float4*>(p.part_ml + (slot * R + j) * 4) = make_float4(M, L, 0.f, 0.f);
                    }
                }
            }
        }
        // end of the pass, every thread: the stages and the query rows are free
        // again, and the vote tells everyone whether a wait gave up
        if (named_bar_or(2, C::NT, my_abort)) return;
        gt0 += ntiles;
    }
    if (warp >= C::NCW) return;

    // ---------------------------------------------- lists cut by this span's ends
    // Each CTA a cut list touches leaves one partial and takes one ticket; the
    // last one merges them.  List [s, e) touches the spans ca = span(s) .. cb =
    // span(e - 1); its partial in span c sits in slot 2c when the list starts
    // before span c (cut by its start), else in slot 2c + 1 (cut by its end).
    // Both tickets are taken at once; when this CTA is last for both lists, the
    // two halves of the consumer threads merge one list each.
    auto span_of = [&](long long x) { return static_cast<int>(min((x - off0) / cl, static_cast<long long>(ncta - 1))); };
    named_bar_sync(1, C::NCT);   // this CTA's partials are written
    if (tid < 2) {
        s_win[tid] = 0;
        const int lst = s_cut[tid][0];
        if (lst >= 0) {
            const int nparts = span_of(static_cast<long long>(s_cut[tid][2]) - 1) - span_of(s_cut[tid][1]) + 1;
            const int old = atom_add_acq_rel_gpu(p.tickets + lst, 1);   // release ours, acquire the others'
            s_win[tid] = (old == nparts - 1) ? 1 : 0;
        }
    }
    named_bar_sync(1, C::NCT);
    const int w0 = s_win[0], w1 = s_win[1];
    if (!w0 && !w1) return;
    const bool both = w0 && w1;
    const int ci = both ? (tid >> 6) : (w0 ? 0 : 1);
    const int nth = both ? C::NCT / 2 : C::NCT;          // whole warps either way
    const int lt = both ? (tid & 63) : tid;
    const int bar_id = both ? 3 + ci : 1;
    const int lst = s_cut[ci][0], ls = s_cut[ci][1], le = s_cut[ci][2];
    const int ca = span_of(ls), cb = span_of(static_cast<long long>(le) - 1);
    const int b = lst / p.Hkv, h = lst - b * p.Hkv;
    // Each thread merges one float4 of the output over the partials, loading
    // them from L2 eight at a time (all in flight together); when the output has
    // fewer float4 than the group has threads, SF threads share an item, each
    // taking every SF-th partial, and combine through shared memory; with at
    // most eight partials one thread loads them all at once, and no combine.
    const int R4 = R * (D / 4);                          // float4 of a list's output
    const int per_round = min(R4, nth);
    const int SF = (cb - ca + 1 <= 8) ? 1 : nth / per_round;
    float* red = reinterpret_cast<float*>(smem + C::OFF_K) + ci * (C::NCT * 6);   // [SF][per_round][6]
    for (int base = 0; base < R4; base += per_round) {
        const int item = base + lt % per_round, qq = lt / per_round;
        const bool act = qq < SF && item < R4;
        const int j = item / (D / 4), d0 = 4 * (item % (D / 4));
        float mm = -INFINITY, ll = 0.f;
        float4 a4 = make_float4(0.f, 0.f, 0.f, 0.f);
        if (act) {
            const float* po = p.part_o + static_cast<size_t>(j) * D + d0;
            const float* pm = p.part_ml + static_cast<size_t>(j) * 4;
            for (int c0 = ca + qq; c0 <= cb; c0 += 8 * SF) {
                float4 v4[8];   // (m, l, -, -)
                float4 o4[8];
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    const int c = c0 + u * SF;
                    v4[u] = make_float4(-INFINITY, 0.f, 0.f, 0.f);
                    o4[u] = make_float4(0.f, 0.f, 0.f, 0.f);
                    if (c <= cb) {
                        const size_t slot = 2 * static_cast<size_t>(c) + ((c > ca) ? 0 : 1);
                        v4[u] = __ldcg(reinterpret_cast<const float4*>(pm + slot * R * 4));
                        o4[u] = __ldcg(reinterpret_cast<const float4*>(po + slot * R * D));
                    }
                }
                float M = mm;
#pragma unroll
                for (int u = 0; u < 8; ++u) M = fmaxf(M, v4[u].x);
                if (M == -INFINITY) continue;
                const float f = (mm == -INFINITY) ? 0.f : fast_exp2(mm - M);
                ll *= f;
                a4.x *= f;
                a4.y *= f;
                a4.z *= f;
                a4.w *= f;
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    const float w = (v4[u].x == -INFINITY) ? 0.f : fast_exp2(v4[u].x - M);
                    ll = fmaf(w, v4[u].y, ll);
                    a4.x = fmaf(w, o4[u].x, a4.x);
                    a4.y = fmaf(w, o4[u].y, a4.y);
                    a4.z = fmaf(w, o4[u].z, a4.z);
                    a4.w = fmaf(w, o4[u].w, a4.w);
                }
                mm = M;
            }
        }
        if (SF > 1) {
            if (act) {
                float* r6 = red + (qq * per_round + lt % per_round) * 6;
                r6[0] = mm;
                r6[1] = ll;
                r6[2] = a4.x;
                r6[3] = a4.y;
                r6[4] = a4.z;
                r6[5] = a4.w;
            }
            if (bar_id == 3)
                named_bar_sync(3, C::NCT / 2);
            else if (bar_id == 4)
                named_bar_sync(4, C::NCT / 2);
            else
                named_bar_sync(1, C::NCT);
            if (act && qq == 0) {
                float M = mm;
                for (int q2 = 1; q2 < SF; ++q2) M = fmaxf(M, red[(q2 * per_round + lt % per_round) * 6]);
                if (M != -INFINITY) {
                    const float f = (mm == -INFINITY) ? 0.f : fast_exp2(mm - M);
                    ll *= f;
                    a4.x *= f;
                    a4.y *= f;
                    a4.z *= f;
                    a4.w *= f;
                    for (int q2 = 1; q2 < SF; ++q2) {
                        const float* r6 = red + (q2 * per_round + lt % per_round) * 6;
                        const float w = (r6[0] == -INFINITY) ? 0.f : fast_exp2(r6[0] - M);
                        ll = fmaf(w, r6[1], ll);
                        a4.x = fmaf(w, r6[2], a4.x);
                        a4.y = fmaf(w, r6[3], a4.y);
                        a4.z = fmaf(w, r6[4], a4.z);
                        a4.w = fmaf(w, r6[5], a4.w);
                    }
                    mm = M;
                }
            }
        }
        if (act && qq == 0) {
            const size_t orow = static_cast<size_t>(b) * p.Hq + h * p.G + j;
            const float il = ll > 0.f ? 1.f / ll : 0.f;
            uint2 packed;
            packed.x = pack_bf16(a4.x * il, a4.y * il);
            packed.y = pack_bf16(a4.z * il, a4.w * il);
            *reinterpret_cast<uint2*>(p.o + orow * D + d0) = packed;
            if (d0 == 0 && p.lse) p.lse[orow] = ll > 0.f ? (mm + fast_log2(ll)) * kLn2 : -INFINITY;
        }
    }
    if (lt == 0) atomicExch(p.tickets + lst, 0);
}

namespace {

template <int D>
cudaError_t ensure_pack_attr(int dev) {
    static std::atomic<unsigned long long> attr_set{0};
    if (attr_done(attr_set, dev)) return cudaSuccess;
    const cudaError_t e = cudaFuncSetAttribute(packed_decode_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                               PackCfg<D>::SMEM_ALLOC);
    if (e == cudaSuccess) attr_mark(attr_set, dev);
    return e;
}

// CTAs the device holds at once (occupancy query, once per device), at most
// two per SM: the grid is one wave.
template <int D>
int pack_grid(int dev, int num_sms) {
    static std::atomic<int> cache[64];
    const bool cached = dev >= 0 && dev < 64;
    if (cached) {
        const int v = cache[dev].load(std::memory_order_relaxed);
        if (v > 0) return v;
    }
    int per_sm = 0;
    if (ensure_pack_attr<D>(dev) != cudaSuccess ||
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, packed_decode_kernel<D>, PackCfg<D>::NT,
                                                      PackCfg<D>::SMEM_ALLOC) != cudaSuccess) {
        (void)cudaGetLastError();
        per_sm = 2;
    }
    const int g = std::max(1, std::min(per_sm, 2) * std::max(num_sms, 1));
    if (cached) cache[dev].store(g, std::memory_order_relaxed);
    return g;
}

template <int D>
int launch_packed(const AttnLaunch& a, int num_sms, const char** why) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = ensure_pack_attr<D>(dev);
    if (e != cudaSuccess) {
        *why = cudaGetErrorString(e);
        return SDKV_ERR_CUDA;
    }
    const int grid = pack_grid<D>(dev, num_sms);
    PackParams p{};
    p.q = static_cast<const bf16*>(a.q);
    p.k = static_cast<const bf16*>(a.k);
    p.v = static_cast<const bf16*>(a.v);
    p.sb = a.sb;
    p.sh = a.sh;
    p.sn = a.sn;
    p.Hq = a.Hq;
    p.Hkv = a.Hkv;
    p.G = a.Hq / a.Hkv;
    p.BH = a.B * a.Hkv;
    p.o = static_cast<bf16*>(a.o);
    p.lse = a.lse;
    p.scale_log2 = a.scale * kLog2e;
    p.offsets = a.offsets;
    p.indices = a.indices;
    p.n_idx = a.n_idx;
    p.n_cap = a.n_cap;
    p.min_span = 2 * PackCfg<D>::TK;
    const AttnWs ws = attn_ws(a.ws, p.BH, p.G, D, 2 * grid, 4);
    if (a.ws_bytes < ws.bytes) {
        *why = "workspace smaller than sdkv_workspace_size(SDKV_OP_SPARSE_DECODE, ...)";
        return SDKV_ERR_WORKSPACE;
    }
    p.status = ws.status;
    p.tickets = ws.tickets;
    p.part_o = ws.part_o;
    p.part_ml = ws.part_ml;
    e = launch_pdl(packed_decode_kernel<D>, dim3(grid), dim3(PackCfg<D>::NT), PackCfg<D>::SMEM_ALLOC, a.stream, p);
    if (e != cudaSuccess) {
        *why = cudaGetErrorString(e);
        return SDKV_ERR_CUDA;
    }
    return SDKV_OK;
}

}  // namespace

bool packed_decode_takes(int B, int Hq, int Hkv, int d) {
    const long long BH = static_cast<long long>(B) * Hkv;
    return (d == 64 || d == 128) && Hq % Hkv == 0 && Hq / Hkv <= 16 && BH <= kPackMaxLists;
}

int packed_decode_grid_max(int num_sms) { return 2 * std::max(num_sms, 1); }

int launch_packed_decode(const AttnLaunch& a, int num_sms, const char** why) {
    if (!packed_decode_takes(a.B, a.Hq, a.Hkv, a.d) || a.gamma != 1) {
        *why = "packed decode: unsupported shape";
        return SDKV_ERR_UNSUPPORTED;
    }
    return a.d == 128 ? launch_packed<128>(a, num_sms, why) : launch_packed<64>(a, num_sms, why);
}

}  // namespace sdkv
