// Split-K flash-decode attention for one decode step, dense and sparse.
//
// Dense (StD 3.1 verify, ByteCross split-K baseline): every CTA takes one
// (batch, KV head) and one contiguous range of cache rows; all gamma x G query
// rows of that KV head (the G query heads of the group at the gamma draft
// positions, causal among the drafts) ride on the same pass over the rows, so
// the cache is read exactly once.
// Sparse (StD 3.2, ByteCross "Speedup Across Context"): every CTA takes one
// chunk of one (batch, KV head)'s selected-index list and gathers those rows;
// the contiguous kind streams the same chunks from buffers the rows were
// compacted into (ByteCross's deployment).
//
// CTA layout: producer warps fill a ring of shared-memory stages (128-byte
// swizzle), completing on mbarriers: one warp issuing TMA tensor copies for
// dense and compacted rows, or two warps issuing 16-byte cp.async copies of
// the listed rows (list entries loaded a ring of stages ahead).  The consumer
// warps run QK^T and PV on mma.sync (bf16 in, fp32 accumulate) with an online
// softmax in the log2 domain, each over its own key group of every stage.
// Merging the unnormalised partials (o, m, l) with the log-sum-exp rule
//     o = sum_s 2^(m_s - M) o_s / sum_s 2^(m_s - M) l_s,   M = max_s m_s
// takes up to three levels: the key groups of a CTA in shared memory; the
// CTAs of a cluster (2 to 8) through distributed shared memory, each CTA
// reducing a slice of the head dims; and, when a head spans several clusters
// (or several CTAs without a cluster), the last of them to finish (atomic
// ticket, no waiting) merges their partials from global memory.
#include "sdkv_common.cuh"
#include "sdkv_internal.h"

#include <algorithm>
#include <cstring>
#include <mutex>

namespace sdkv {

struct AttnParams {
    const bf16* q;
    const bf16* k;
    const bf16* v;
    long long sb, sh, sn;
    int B, Hq, Hkv, G, gamma, R;
    bf16* o;
    float* lse;
    float scale_log2;
    // dense
    int n_prefix, n_total, chunk, nsplit;
    int cs, ncl;   // cluster size along the splits of a head, clusters per head (cs = 1: no cluster)
    // sparse
    const int* offsets;
    const int* indices;
    long long n_idx;   // entries of indices; 0: the lists are not read before the grid dependency resolves
    int n_cap, BH, grid_target, min_chunk;
    // workspace
    int* status;
    int* tickets;
    float* part_o;
    float* part_ml;
};

// Kinds of rows a launch streams: the whole cache (dense verify), rows gathered
// through the index lists, or the lists' rows compacted into contiguous buffers.
constexpr int kDense = 0, kGather = 1, kContig = 2;
constexpr int kMaxCluster = 8;     // portable cluster size
template <int D>
constexpr int kLogD = (D == 128) ? 7 : 6;   // log2 of the head dim

template <int D, int MT, int KW, int TK, int STAGES, int KIND>
struct AttnCfg {
    static constexpr int NCW = MT * KW;          // consumer warps: row tiles x key groups
    static constexpr int NCT = NCW * 32;
    static constexpr int NPW = (KIND == kGather) ? 2 : 1;   // producer warps (gathering rows needs more issuers)
    static constexpr int NT = NCT + NPW * 32;
    static constexpr int KPW = TK / KW;          // keys per consumer warp per stage
    static_assert(KPW % 16 == 0, "keys per warp must be a multiple of 16");
    static_assert(D % (4 * KW) == 0, "each key group reduces a slice of the head dims");
    static_assert(D == 64 || D == 128, "head dim");
    static_assert(KIND != kGather || TK == 32 * NPW, "one list entry per producer lane per tile");
    static constexpr int ROWB = 2 * D;
    static constexpr int TILE_B = TK * ROWB;
    static constexpr int QPITCH = 2 * D + 16;
    static constexpr int ROWS = MT * 16;
    static constexpr int MPITCH = D + 8;         // merge rows: conflict-free 64-bit stores
    static constexpr int OFF_K = 0;
    static constexpr int OFF_V = STAGES * TILE_B;
    static constexpr int OFF_Q = 2 * STAGES * TILE_B;
    static constexpr int OFF_ML = OFF_Q + ROWS * QPITCH;          // [KW][ROWS] (m, l)
    // cluster merge: what the peers push to this CTA (its slice of the head dims)
    static constexpr int OFF_RCV = OFF_ML + KW * ROWS * 2 * 4;    // [src][R][D/cs] fp32
    static constexpr int OFF_RML = OFF_RCV + ROWS * D * 4;           // [src][R] (m, l)
    static constexpr int OFF_BAR = OFF_RML + 8 * ROWS * 2 * 4;
    static constexpr int SMEM = OFF_BAR + 2 * STAGES * 8;
    static constexpr int SMEM_ALLOC = SMEM + 1024;
    static_assert((TILE_B % 1024) == 0, "swizzled stages need 1024-byte alignment");
    static_assert(KW * ROWS * MPITCH * 4 <= 2 * STAGES * TILE_B, "merge rows fit in the stage buffers");
    static_assert(2 * STAGES * TILE_B >= ROWS * (8 * D + 12) + ROWS * 16 + 128, "combine area");
};

template <int NT>
__device__ __forceinline__ int block_excl_scan(int v, int* s_scan, int& total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) s_scan[warp] = x;
    __syncthreads();
    if (warp == 0) {
        int w = (lane < NT / 32) ? s_scan[lane] : 0;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, w, o);
            if (lane >= o) w += y;
        }
        if (lane < NT / 32) s_scan[lane] = w;
    }
    __syncthreads();
    const int res = (warp ? s_scan[warp - 1] : 0) + x - v;
    total = s_scan[NT / 32 - 1];
    __syncthreads();
    return res;
}

// Chunk plan of the list decodes, identical in every CTA (all threads call it).
// Chunk length cl = max(min_chunk, ceil(total / (grid_target - cs * BH)) rounded
// up to 16).  Without clusters head i owns max(1, ceil(k_i / cl)) consecutive
// chunk ids of length cl; with clusters of cs CTAs it owns cs * ceil(k_i / (cs *
// cl)) chunks (a whole number of clusters) of balanced length; trailing ones may
// be empty.  Either way the chunk count stays within the grid.  The CTA's work
// item goes to s_work: head, list positions [lo, hi), chunk id, chunks of the
// head, first chunk of the head (s_work[0] = -1: no chunk for this CTA).
template <int NT>
__device__ __forceinline__ void list_plan(const AttnParams& p, int* s_work, int* s_scan, int& s_tot, int& s_off0) {
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int c = blockIdx.x;
    const int cs = p.cs;
    if (p.BH <= 32) {
        // one warp: each lane a head, the chunk ids by a shuffle scan
        if (warp == 0) {
            int start = 0, kh = 0;
            if (lane < p.BH) {
                start = __ldcg(p.offsets + lane);
                kh = __ldcg(p.offsets + lane + 1) - start;
            }
            const int off0 = __shfl_sync(0xffffffffu, start, 0);
            const int total = max(__shfl_sync(0xffffffffu, start + kh, p.BH - 1) - off0, 0);
            const int slots = max(1, p.grid_target - (cs > 1 ? cs * p.BH : 0));
            int cl = static_cast<int>(min((static_cast<long long>(total) + slots - 1) / slots, 1ll << 26));
            cl = max(p.min_chunk, (cl + 15) & ~15);
            int nch = 0, chl = cl;
            if (lane < p.BH) {
                if (kh < 0) {
                    flag_status(p.status, SDKV_DEV_BAD_LIST);
                    kh = 0;
                }
                if (cs > 1) {
                    nch = cs * max(1, (kh + cs * cl - 1) / (cs * cl));
                    chl = (((kh + nch - 1) / nch) + 15) & ~15;
                } else {
                    nch = max(1, (kh + cl - 1) / cl);
                }
            }
            int incl = nch;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int y = __shfl_up_sync(0xffffffffu, incl, o);
                if (lane >= o) incl += y;
            }
            const int first = incl - nch;
            const bool mine = lane < p.BH && c >= first && c < first + nch;
            if (mine) {
                const int j = c - first;
                const int l0 = min(start + j * chl, start + kh);
                s_work[0] = lane;
                s_work[1] = l0;
                s_work[2] = max(l0, min(start + (j + 1) * chl, start + kh));
                s_work[3] = c;
                s_work[4] = nch;
                s_work[5] = first;
            }
            if (__ballot_sync(0xffffffffu, mine) == 0u && lane == 0) s_work[0] = -1;
            if (lane == 0) {
                s_off0 = off0;
                s_tot = total;
            }
        }
        return;
    }
    int start = 0, kh = 0;
    if (tid < p.BH) {
        start = __ldcg(p.offsets + tid);
        kh = __ldcg(p.offsets + tid + 1) - start;
    }
    if (tid == 0) {
        s_off0 = __ldcg(p.offsets);
        s_tot = __ldcg(p.offsets + p.BH) - s_off0;
        s_work[0] = -1;
    }
    __syncthreads();
    const int total = max(s_tot, 0);
    const int slots = max(1, p.grid_target - (cs > 1 ? cs * p.BH : 0));
    int cl = static_cast<int>(min((static_cast<long long>(total) + slots - 1) / slots, 1ll << 26));
    cl = max(p.min_chunk, (cl + 15) & ~15);
    int running = 0;
    for (int base = 0; base < p.BH; base += NT) {
        const int i = base + tid;
        int nch = 0, chl = cl;
        if (base > 0 && i < p.BH) {
            start = __ldcg(p.offsets + i);
            kh = __ldcg(p.offsets + i + 1) - start;
        }
        if (i < p.BH) {
            if (kh < 0) {
                flag_status(p.status, SDKV_DEV_BAD_LIST);
                kh = 0;
            }
            if (cs > 1) {
                nch = cs * max(1, (kh + cs * cl - 1) / (cs * cl));
                chl = (((kh + nch - 1) / nch) + 15) & ~15;
            } else {
                nch = max(1, (kh + cl - 1) / cl);
            }
        }
        int tile_total;
        const int excl = block_excl_scan<NT>(nch, s_scan, tile_total);
        const int first = running + excl;
        if (i < p.BH && c >= first && c < first + nch) {
            const int j = c - first;
            const int l0 = min(start + j * chl, start + kh);
            s_work[0] = i;
            s_work[1] = l0;
            s_work[2] = max(l0, min(start + (j + 1) * chl, start + kh));
            s_work[3] = c;
            s_work[4] = nch;
            s_work[5] = first;
        }
        running += tile_total;
        __syncthreads();
        if (s_work[0] >= 0 || running > c) break;
    }
}

// Key/value tile address of (row, 16-byte chunk) inside one stage: the 128-byte
// swizzled layout TMA writes for dense tiles; gathered rows are placed the same way.
template <int D, int TK, bool SPARSE>
__device__ __forceinline__ uint32_t tile_addr(uint32_t base, int row, int chunk) {
    return sw128_addr<TK>(base, row, chunk);
}

template <int D, int MT, int KW, int TK, int STAGES, int KIND>
__global__ void __launch_bounds__(AttnCfg<D, MT, KW, TK, STAGES, KIND>::NT)
    attn_splitk_kernel(const __grid_constant__ AttnParams p, const __grid_constant__ CUtensorMap tmk,
                       const __grid_constant__ CUtensorMap tmv) {
    using C = AttnCfg<D, MT, KW, TK, STAGES, KIND>;
    constexpr bool SPARSE = (KIND != kDense);    // list-driven chunk plan, no causal limits
    constexpr bool kTwoTermP = (MT == 1);        // P as hi + lo bf16 terms (see the PV product)
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem =
        reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(smem);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const uint32_t bar_full = sbase + C::OFF_BAR;
    const uint32_t bar_empty = bar_full + STAGES * 8;

    // work item: bh, key/position range [lo, hi), chunk id, chunks of the head, first chunk of the head
    __shared__ int s_work[6];
    __shared__ int s_scan[C::NT / 32];
    __shared__ int s_tot;
    __shared__ int s_off0;           // offsets[0]: row 0 of the compacted buffers
    __shared__ int s_abort;
    __shared__ int s_last;

    if constexpr (!SPARSE) {
        // dense: the work item is known from the grid alone, so the first stages'
        // K and V tiles go to L2 while the previous kernel finishes
        if (tid == 0) {
            const int bh = blockIdx.x / p.nsplit, sp = blockIdx.x % p.nsplit;
            const int b = bh / p.Hkv, h = bh - (bh / p.Hkv) * p.Hkv;
            const int lo = sp * p.chunk, hi = min(lo + p.chunk, p.n_total);
            prefetch_tmap(&tmk);
            prefetch_tmap(&tmv);
            for (int t = 0; t < STAGES && lo + t * TK < hi; ++t)
#pragma unroll
                for (int half = 0; half < D / 64; ++half) {
                    tma_prefetch_4d(&tmk, half * 64, lo + t * TK, h, b);
                    tma_prefetch_4d(&tmv, half * 64, lo + t * TK, h, b);
                }
        }
    }
    if (tid == 0) {
        // this CTA's own barriers: independent of the previous kernel
#pragma unroll
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(bar_full + 8 * s, KIND == kGather ? C::NPW * 32 : 1);
            mbar_init(bar_empty + 8 * s, C::NCW);
        }
        fence_mbar_init();
        s_abort = 0;
    }
    if constexpr (!SPARSE) {
        // dense: the work item follows from the grid alone
        if (tid == 0) {
            const int bh = blockIdx.x / p.nsplit, sp = blockIdx.x % p.nsplit;
            s_work[0] = bh;
            s_work[1] = sp * p.chunk;
            s_work[2] = max(sp * p.chunk, min(sp * p.chunk + p.chunk, p.n_total));  // trailing splits may be empty
            s_work[3] = blockIdx.x;
            s_work[4] = p.nsplit;
            s_work[5] = bh * p.nsplit;
        }
    }
    if constexpr (SPARSE) {
        // Before the grid dependency resolves: bring the list offsets and (gathered
        // kind, n_idx > 0) this CTA's share of the index array, 1/grid of
        // indices[0, n_idx), into L2, so the plan and the index loads after the
        // wait hit L2.  Prefetches return nothing, and L2 is where every write
        // lands, so a line fetched early is never older than what a later load of
        // it returns.
        const uint8_t* ob = reinterpret_cast<const uint8_t*>(p.offsets);
        const long long obytes = 4ll * (p.BH + 1);
        for (long long x = 128ll * tid; x < obytes; x += 128ll * C::NT) prefetch_l2_line(ob + x);
        if (KIND == kGather && p.n_idx > 0) {
            const long long ibytes = 4 * p.n_idx;
            const long long per = (ibytes + gridDim.x - 1) / gridDim.x;
            const long long i0 = per * blockIdx.x, i1 = min(ibytes, i0 + per);
            const uint8_t* ib = reinterpret_cast<const uint8_t*>(p.indices);
            for (long long x = i0 + 128ll * tid; x < i1; x += 128ll * C::NT) prefetch_l2_line(ib + x);
        }
    }
    // This CTA's early work is done.  Once every CTA of the grid is past this
    // point, the next kernel on the stream may start its own early work in the
    // slots this grid leaves free; it waits for this grid before using its output.
    griddep_launch();
    griddep_wait();

    if constexpr (SPARSE) list_plan<C::NT>(p, s_work, s_scan, s_tot, s_off0);
    __syncthreads();

    const int bh = s_work[0];
    if (bh < 0) return;  // no chunk for this CTA (uniform)
    const int lo = s_work[1], hi = s_work[2];
    const int cidx = s_work[3], nch = s_work[4], c0 = s_work[5];
    const int b = bh / p.Hkv, h = bh - (bh / p.Hkv) * p.Hkv;
    const int nkeys = hi - lo;
    const int ntiles = (nkeys + TK - 1) / TK;

    // ------------------------------------------------------------------ producer
    if (warp >= C::NCW) {
        if constexpr (KIND == kGather) {
            // Gather: the NPW producer warps own 32 tile rows each; lane j of a warp
            // holds the list entry of its warp's row j, loaded STAGES tiles ahead (a
            // register ring), so the first stages' gathers do not each wait for an
            // index load; CPR lanes copy one row as CPR 16-byte chunks per instruction.
            constexpr int CPR = D / 8;           // 16-byte chunks per row
            constexpr int RPI = 32 / CPR;        // rows per warp instruction
            const int pw = warp - C::NCW;
            const bf16* kb = p.k + b * p.sb + h * p.sh;
            const bf16* vb = p.v + b * p.sb + h * p.sh;
            // the loads are issued early; an entry is checked (a branch on its value)
            // only when its tile is gathered, so no load is waited for where it is issued
            auto load_idx = [&](int t) -> int {
                const int pos = min(lo + t * TK + pw * 32 + lane, hi - 1);
                return (t < ntiles) ? __ldg(p.indices + pos) : 0;
            };
            int idx_ring[STAGES];   // entries of tiles t .. t + STAGES - 1
#pragma unroll
            for (int j = 0; j < STAGES; ++j) idx_ring[j] = load_idx(j);
            for (int t = 0; t < ntiles; ++t) {
                int idx_cur = idx_ring[0];
                if (static_cast<unsigned>(idx_cur) >= static_cast<unsigned>(p.n_cap)) {
                    flag_status(p.status, SDKV_DEV_BAD_INDEX);
                    idx_cur = 0;
                }
#pragma unroll
                for (int j = 0; j + 1 < STAGES; ++j) idx_ring[j] = idx_ring[j + 1];
                idx_ring[STAGES - 1] = load_idx(t + STAGES);
                const int s = t % STAGES;
                const uint32_t ph = (t / STAGES) & 1;
                if (t >= STAGES) {
                    bool ok = mbar_wait(bar_empty + 8 * s, ph ^ 1);
                    ok = __all_sync(0xffffffffu, ok);
                    if (!ok) {
                        if (lane == 0) {
                            flag_status(p.status, SDKV_DEV_TIMEOUT);
                            atomicExch(&s_abort, 1);
                        }
                        break;
                    }
                }
                const uint32_t kst = sbase + C::OFF_K + s * C::TILE_B;
                const uint32_t vst = sbase + C::OFF_V + s * C::TILE_B;
                const int chunk = lane % CPR;
#pragma unroll 4
                for (int it = 0; it < 32 / RPI; ++it) {
                    const int rw = it * RPI + lane / CPR;     // row within this warp's 32
                    const int idx = __shfl_sync(0xffffffffu, idx_cur, rw);
                    const int row = pw * 32 + rw;
                    const size_t off = static_cast<size_t>(idx) * p.sn + chunk * 8;
                    cp_async_16(tile_addr<D, TK, SPARSE>(kst, row, chunk), kb + off);
                    cp_async_16(tile_addr<D, TK, SPARSE>(vst, row, chunk), vb + off);
                }
                cp_async_mbar_arrive(bar_full + 8 * s);
            }
            cp_async_wait_all();
        } else {
            // TMA producer: dense tiles of the cache (4-D map: dims, row, head,
            // sequence) or tiles of the compacted rows (2-D map: dims, row)
            if (lane == 0) {
                prefetch_tmap(&tmk);
                prefetch_tmap(&tmv);
                const int crow0 = (KIND == kContig) ? lo - s_off0 : 0;   // compacted buffers: the chunk's first row
                for (int t = 0; t < ntiles; ++t) {
                    const int s = t % STAGES;
                    const uint32_t ph = (t / STAGES) & 1;
                    if (t >= STAGES && !mbar_wait(bar_empty + 8 * s, ph ^ 1)) {
                        flag_status(p.status, SDKV_DEV_TIMEOUT);
                        atomicExch(&s_abort, 1);
                        break;
                    }
                    mbar_arrive_expect_tx(bar_full + 8 * s, 2 * TK * D * 2);
                    const int row0 = lo + t * TK;
#pragma unroll
                    for (int half = 0; half < D / 64; ++half) {
                        const uint32_t kdst = sbase + C::OFF_K + s * C::TILE_B + half * TK * 128;
                        const uint32_t vdst = sbase + C::OFF_V + s * C::TILE_B + half * TK * 128;
                        if constexpr (KIND == kContig) {
                            tma_load_2d(kdst, &tmk, half * 64, crow0 + t * TK, bar_full + 8 * s);
                            tma_load_2d(vdst, &tmv, half * 64, crow0 + t * TK, bar_full + 8 * s);
                        } else {
                            tma_load_4d(kdst, &tmk, half * 64, row0, h, b, bar_full + 8 * s);
                            tma_load_4d(vdst, &tmv, half * 64, row0, h, b, bar_full + 8 * s);
                        }
                    }
                }
            }
        }
        if (p.cs > 1) cluster_sync_all();   // the consumers' cluster barrier
        return;
    }

    // ------------------------------------------------------------------ consumers
    // Warp cw owns row tile mi = cw % MT and key group kw = cw / MT: keys
    // [kw*KPW, kw*KPW + KPW) of every stage, all head dims.
    const int cw = warp;
    const int mi = cw % MT, kw = cw / MT;

    // query rows of this KV head -> shared memory (row r = g * gamma + t)
    uint8_t* qs = smem + C::OFF_Q;
    for (int e = tid; e < C::ROWS * (D / 8); e += C::NCT) {
        const int r = e / (D / 8), c = e % (D / 8);
        uint4 val = make_uint4(0u, 0u, 0u, 0u);
        if (r < p.R) {
            const int g = r / p.gamma, t = r - (r / p.gamma) * p.gamma;
            const int hq = h * p.G + g;
            val = *reinterpret_cast<const uint4*>(p.q + ((static_cast<size_t>(b) * p.Hq + hq) * p.gamma + t) * D +
                                                  c * 8);
        }
        *reinterpret_cast<uint4*>(qs + r * C::QPITCH + c * 16) = val;
    }
    named_bar_sync(1, C::NCT);

    uint32_t qa[D / 16][4];
    {
        const int row = mi * 16 + (lane & 7) + (((lane >> 3) & 1) << 3);
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks)
            ldsm_x4(qa[ks], pad_addr<C::QPITCH>(sbase + C::OFF_Q, row, 2 * ks + (lane >> 4)));
    }

    const int r0 = mi * 16 + (lane >> 2);
    int lim[2] = {0x7fffffff, 0x7fffffff};
    if constexpr (!SPARSE) {
        lim[0] = p.n_prefix + (r0 % p.gamma);
        lim[1] = p.n_prefix + ((r0 + 8) % p.gamma);
    }

    float o_acc[D / 8][4];
#pragma unroll
    for (int j = 0; j < D / 8; ++j) o_acc[j][0] = o_acc[j][1] = o_acc[j][2] = o_acc[j][3] = 0.f;
    float m_r[2] = {-INFINITY, -INFINITY};
    float l_r[2] = {0.f, 0.f};
    bool aborted = false;

    for (int t = 0; t < ntiles; ++t) {
        const int s = t % STAGES;
        const uint32_t ph = (t / STAGES) & 1;
        if (!mbar_wait(bar_full + 8 * s, ph)) {
            aborted = true;
            break;
        }
        const uint32_t kst = sbase + C::OFF_K + s * C::TILE_B;
        const uint32_t vst = sbase + C::OFF_V + s * C::TILE_B;
        // Scores of all KPW keys of this warp's group first: the sub-steps of 16
        // keys are independent accumulator chains, interleaved over the head dims
        constexpr int NSUB = C::KPW / 16;
        float sacc[2 * NSUB][4];
#pragma unroll
        for (int nt = 0; nt < 2 * NSUB; ++nt) sacc[nt][0] = sacc[nt][1] = sacc[nt][2] = sacc[nt][3] = 0.f;
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
#pragma unroll
            for (int sub = 0; sub < NSUB; ++sub) {
                uint32_t kb[4];
                const int row = kw * C::KPW + sub * 16 + (lane & 7) + ((lane >> 4) << 3);
                ldsm_x4(kb, tile_addr<D, TK, SPARSE>(kst, row, 2 * ks + ((lane >> 3) & 1)));
                mma_bf16_16816(sacc[2 * sub], qa[ks], kb[0], kb[1]);
                mma_bf16_16816(sacc[2 * sub + 1], qa[ks], kb[2], kb[3]);
            }
        }
        // scale into the log2 domain and mask
        const int cpos = t * TK + kw * C::KPW + 2 * (lane & 3);  // position within [lo, hi) of column (0, 0)
#pragma unroll
        for (int nt = 0; nt < 2 * NSUB; ++nt) {
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int col = cpos + nt * 8 + (e & 1);
                bool valid = col < nkeys;
                if constexpr (!SPARSE) valid = valid && (lo + col <= lim[e >> 1]);
                sacc[nt][e] = valid ? sacc[nt][e] * p.scale_log2 : -INFINITY;
            }
        }
        // online softmax per row over the group's keys (rows r0 and r0 + 8; a quad shares a row)
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            float mx = -INFINITY;
#pragma unroll
            for (int nt = 0; nt < 2 * NSUB; ++nt) mx = fmaxf(mx, fmaxf(sacc[nt][2 * i], sacc[nt][2 * i + 1]));
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
            for (int nt = 0; nt < 2 * NSUB; ++nt) {
                sacc[nt][2 * i] = fast_exp2(sacc[nt][2 * i] - muse);
                sacc[nt][2 * i + 1] = fast_exp2(sacc[nt][2 * i + 1] - muse);
                if constexpr (!kTwoTermP) {
                    // the weights the PV product will use, rounded once to bf16
                    sacc[nt][2 * i] = __bfloat162float(__float2bfloat16_rn(sacc[nt][2 * i]));
                    sacc[nt][2 * i + 1] = __bfloat162float(__float2bfloat16_rn(sacc[nt][2 * i + 1]));
                }
                l_r[i] += sacc[nt][2 * i] + sacc[nt][2 * i + 1];
            }
        }
        // One row tile (decode): P as two bf16 terms, p = hi + lo (about 16
        // significant bits), so the weights of the PV product match the fp32
        // sum l even when a few keys carry the whole softmax.  Several row
        // tiles (the gamma-query verify, where the contraction is the limit):
        // P as one bf16 term and l summed from those same rounded weights, so
        // the output is an exactly normalised average with weights within
        // 2^-9 relative of the fp32 ones.
#pragma unroll
        for (int sub = 0; sub < NSUB; ++sub) {
            const float(&x0)[4] = sacc[2 * sub];
            const float(&x1)[4] = sacc[2 * sub + 1];
            uint32_t pa[4], pl[4];
            if constexpr (kTwoTermP) {
                split_bf16(x0[0], x0[1], pa[0], pl[0]);
                split_bf16(x0[2], x0[3], pa[1], pl[1]);
                split_bf16(x1[0], x1[1], pa[2], pl[2]);
                split_bf16(x1[2], x1[3], pa[3], pl[3]);
            } else {
                pa[0] = pack_bf16(x0[0], x0[1]);
                pa[1] = pack_bf16(x0[2], x0[3]);
                pa[2] = pack_bf16(x1[0], x1[1]);
                pa[3] = pack_bf16(x1[2], x1[3]);
            }
            const int krow0 = kw * C::KPW + sub * 16;
#pragma unroll
            for (int jj = 0; jj < D / 16; ++jj) {
                uint32_t vb[4];
                const int row = krow0 + (lane & 7) + (((lane >> 3) & 1) << 3);
                ldsm_x4_t(vb, tile_addr<D, TK, SPARSE>(vst, row, 2 * jj + (lane >> 4)));
                mma_bf16_16816(o_acc[2 * jj], pa, vb[0], vb[1]);
                mma_bf16_16816(o_acc[2 * jj + 1], pa, vb[2], vb[3]);
                if constexpr (kTwoTermP) {
                    mma_bf16_16816(o_acc[2 * jj], pl, vb[0], vb[1]);
                    mma_bf16_16816(o_acc[2 * jj + 1], pl, vb[2], vb[3]);
                }
            }
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
    // uniform decision among the consumers: stop if any of them (or the producer) gave up
    if (named_bar_or(1, C::NCT, aborted || *reinterpret_cast<volatile int*>(&s_abort))) {
        // drain: give every stage's copies a bounded chance to land before exit
        if (tid == 0) {
            for (int s = 0; s < STAGES && s < ntiles; ++s) {
                const int last_t = ((ntiles - 1 - s) / STAGES) * STAGES + s;
                mbar_wait(bar_full + 8 * s, (last_t / STAGES) & 1);
            }
        }
        if (p.cs > 1) cluster_sync_all();
        return;
    }

    // -------------------------------------------------- merge the KW key groups of each row tile
    // Rows below R only.  Each warp rescales its o to the row max over the groups
    // and parks it in shared memory (padded rows: conflict-free 64-bit stores);
    // then group kw sums dims [kw*D/KW, (kw+1)*D/KW) over the groups and writes them.
    float* ml = reinterpret_cast<float*>(smem + C::OFF_ML);
    if ((lane & 3) == 0) {
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            ml[(kw * C::ROWS + r0 + 8 * i) * 2 + 0] = m_r[i];
            ml[(kw * C::ROWS + r0 + 8 * i) * 2 + 1] = l_r[i];
        }
    }
    named_bar_sync(1, C::NCT);
    float* mrg = reinterpret_cast<float*>(smem + C::OFF_K);  // stage buffers are free now
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        const int row = r0 + 8 * i;
        if (row >= p.R) continue;
        float M = -INFINITY;
#pragma unroll
        for (int k2 = 0; k2 < KW; ++k2) M = fmaxf(M, ml[(k2 * C::ROWS + row) * 2]);
        const float f = (m_r[i] == -INFINITY) ? 0.f : fast_exp2(m_r[i] - M);
        float* dst = mrg + (kw * C::ROWS + row) * C::MPITCH + 2 * (lane & 3);
#pragma unroll
        for (int j = 0; j < D / 8; ++j)
            *reinterpret_cast<float2*>(dst + 8 * j) = make_float2(o_acc[j][2 * i] * f, o_acc[j][2 * i + 1] * f);
    }
    named_bar_sync(1, C::NCT);
    {
        constexpr int SL4 = D / KW / 4;              // float4 per row in this group's dim slice
        const int nrow = min(16, p.R - mi * 16);     // valid rows of this row tile
        for (int e = lane; e < nrow * SL4; e += 32) {
            const int row = mi * 16 + e / SL4;
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
            if (p.cs > 1) {
                // push to the cluster CTA that owns these dims (its receive buffer is
                // not used by the main loop, so early pushes are safe); (M, L) to all.
                // Cluster sizes are powers of two: slices by shifts.
                const int lcs = __ffs(p.cs) - 1;
                const int SL = D >> lcs;
                const uint32_t me = cluster_ctarank();
                const int owner = d0 >> (kLogD<D> - lcs);
                st_dsmem_f4(dsmem_addr(sbase + C::OFF_RCV + ((me * p.R + row) * SL + (d0 & (SL - 1))) * 4, owner),
                            a4);
                // every lane of the row holds the same (M, L): lane d0/4 sends it to
                // rank d0/4 (D/4 >= cluster size, so one remote store at most per lane)
                for (int r = d0 / 4; r < p.cs; r += D / 4)
                    st_dsmem_f2(dsmem_addr(sbase + C::OFF_RML + (me * p.R + row) * 8, r), make_float2(M, L));
            } else if (nch == 1) {
                const int g = row / p.gamma, tt = row - (row / p.gamma) * p.gamma;
                const size_t orow = (static_cast<size_t>(b) * p.Hq + h * p.G + g) * p.gamma + tt;
                const float il = L > 0.f ? 1.f / L : 0.f;
                uint2 packed;
                packed.x = pack_bf16(a4.x * il, a4.y * il);
                packed.y = pack_bf16(a4.z * il, a4.w * il);
                *reinterpret_cast<uint2*>(p.o + orow * D + d0) = packed;
                if (d0 == 0 && p.lse) p.lse[orow] = L > 0.f ? (M + fast_log2(L)) * kLn2 : -INFINITY;
            } else {
                *reinterpret_cast<float4*>(p.part_o + (static_cast<size_t>(cidx) * p.R + row) * D + d0) = a4;
                if (d0 == 0)
                    *reinterpret_cast<float2*>(p.part_ml + (static_cast<size_t>(cidx) * p.R + row) * 2) =
                        make_float2(M, L);
            }
        }
    }
    {
        if (p.cs > 1) {
            // ---------------------------------------------- merge the cluster's splits
            // CTA `rank` of the cluster owns head dims [rank*D/cs, (rank+1)*D/cs); every
            // CTA has pushed its rows' slices and (M, L) into the owners' shared
            // memory, so after one cluster barrier the merge reads local memory only.
            // One partial per cluster (or the output, when one cluster covers the
            // head) goes to global memory.
            cluster_sync_all();
            const int CS = p.cs;
            const int lcs = __ffs(CS) - 1;                   // cluster sizes are powers of two
            const int SL = D >> lcs;
            const uint32_t rank = cluster_ctarank();
            const int lsl4 = kLogD<D> - lcs - 2;             // float4 per row in this slice: 1 << lsl4
            const int sl4 = 1 << lsl4;
            const int gcl = cidx >> lcs;                     // global cluster index (partial slot)
            const int gcl0 = c0 >> lcs, ncl_h = nch >> lcs;  // the head's clusters
            const float* rcv = reinterpret_cast<const float*>(smem + C::OFF_RCV);
            const float2* rml = reinterpret_cast<const float2*>(smem + C::OFF_RML);
            for (int e = tid; e < p.R * sl4; e += C::NCT) {
                const int row = e >> lsl4;
                const int dd = 4 * (e & (sl4 - 1));
                const int d0 = static_cast<int>(rank) * SL + dd;
                // unrolled to the largest cluster so that all loads are in flight together
                float2 ml2[kMaxCluster];
                float4 v4[kMaxCluster];
#pragma unroll
                for (int c = 0; c < kMaxCluster; ++c) {
                    ml2[c] = make_float2(-INFINITY, 0.f);
                    v4[c] = make_float4(0.f, 0.f, 0.f, 0.f);
                    if (c < CS) {
                        ml2[c] = rml[c * p.R + row];
                        v4[c] = *reinterpret_cast<const float4*>(rcv + (c * p.R + row) * SL + dd);
                    }
                }
                float M = -INFINITY;
#pragma unroll
                for (int c = 0; c < kMaxCluster; ++c) M = fmaxf(M, ml2[c].x);
                float L = 0.f;
                float4 a4 = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
                for (int c = 0; c < kMaxCluster; ++c) {
                    if (ml2[c].x == -INFINITY) continue;
                    const float w = fast_exp2(ml2[c].x - M);
                    L += w * ml2[c].y;
                    a4.x += w * v4[c].x;
                    a4.y += w * v4[c].y;
                    a4.z += w * v4[c].z;
                    a4.w += w * v4[c].w;
                }
                if (ncl_h == 1) {
                    const int g = row / p.gamma, tt = row - (row / p.gamma) * p.gamma;
                    const size_t orow = (static_cast<size_t>(b) * p.Hq + h * p.G + g) * p.gamma + tt;
                    const float il = L > 0.f ? 1.f / L : 0.f;
                    uint2 packed;
                    packed.x = pack_bf16(a4.x * il, a4.y * il);
                    packed.y = pack_bf16(a4.z * il, a4.w * il);
                    *reinterpret_cast<uint2*>(p.o + orow * D + d0) = packed;
                    if (d0 == 0 && p.lse) p.lse[orow] = L > 0.f ? (M + fast_log2(L)) * kLn2 : -INFINITY;
                } else {
                    *reinterpret_cast<float4*>(p.part_o + (static_cast<size_t>(gcl) * p.R + row) * D + d0) = a4;
                    if (dd == 0)   // this rank's copy of the cluster's (M, L)
                        *reinterpret_cast<float2*>(
                            p.part_ml + ((static_cast<size_t>(gcl) * CS + rank) * p.R + row) * 2) = make_float2(M, L);
                }
            }
            if (ncl_h == 1) return;
            named_bar_sync(1, C::NCT);
            if (tid == 0) {
                // release this CTA's slice of the partial; acquire the other clusters' (if last)
                const int old = atom_add_acq_rel_gpu(p.tickets + bh * 8 + rank, 1);
                s_last = (old == ncl_h - 1);
            }
            named_bar_sync(1, C::NCT);
            if (!s_last) return;
            // last cluster of the head for this slice: merge the head's cluster partials
            for (int e = tid; e < p.R * sl4; e += C::NCT) {
                const int row = e >> lsl4;
                const int d0 = static_cast<int>(rank) * SL + 4 * (e & (sl4 - 1));
                float mm = -INFINITY, ll = 0.f;
                float4 a4 = make_float4(0.f, 0.f, 0.f, 0.f);
                for (int cb = 0; cb < ncl_h; cb += 8) {
                    float2 v2[8];
                    float4 o4[8];
#pragma unroll
                    for (int u = 0; u < 8; ++u) {   // all loads of the batch in flight together
                        const size_t gi = static_cast<size_t>(gcl0) + cb + u;
                        v2[u] = make_float2(-INFINITY, 0.f);
                        o4[u] = make_float4(0.f, 0.f, 0.f, 0.f);
                        if (cb + u < ncl_h) {
                            v2[u] = __ldcg(reinterpret_cast<const float2*>(p.part_ml + ((gi * CS + rank) * p.R + row) * 2));
                            o4[u] = __ldcg(reinterpret_cast<const float4*>(p.part_o + (gi * p.R + row) * D + d0));
                        }
                    }
#pragma unroll
                    for (int u = 0; u < 8; ++u) {
                        if (v2[u].x == -INFINITY) continue;
                        const float mnew = fmaxf(mm, v2[u].x);
                        const float fa = (mm == -INFINITY) ? 0.f : fast_exp2(mm - mnew);
                        const float fb = fast_exp2(v2[u].x - mnew);
                        ll = ll * fa + v2[u].y * fb;
                        a4.x = a4.x * fa + o4[u].x * fb;
                        a4.y = a4.y * fa + o4[u].y * fb;
                        a4.z = a4.z * fa + o4[u].z * fb;
                        a4.w = a4.w * fa + o4[u].w * fb;
                        mm = mnew;
                    }
                }
                const int g = row / p.gamma, tt = row - (row / p.gamma) * p.gamma;
                const size_t orow = (static_cast<size_t>(b) * p.Hq + h * p.G + g) * p.gamma + tt;
                const float il = ll > 0.f ? 1.f / ll : 0.f;
                uint2 packed;
                packed.x = pack_bf16(a4.x * il, a4.y * il);
                packed.y = pack_bf16(a4.z * il, a4.w * il);
                *reinterpret_cast<uint2*>(p.o + orow * D + d0) = packed;
                if (d0 == 0 && p.lse) p.lse[orow] = ll > 0.f ? (mm + fast_log2(ll)) * kLn2 : -INFINITY;
            }
            if (tid == 0) atomicExch(p.tickets + bh * 8 + rank, 0);
            return;
        }
    }
    if (nch == 1) return;

    // -------------------------------------------------- last CTA of the head merges the partials
    named_bar_sync(1, C::NCT);
    if (tid == 0) {
        const int old = atom_add_acq_rel_gpu(p.tickets + bh, 1);   // release this CTA's partial, acquire the others'
        s_last = (old == nch - 1);
    }
    named_bar_sync(1, C::NCT);
    if (!s_last) return;

    // Partials are merged in batches of splits that fit in the (now idle) stage
    // buffers.  Per batch, one round trip: the batch's o blocks and (m, l) pairs are
    // staged with cp.async; then per row the running max / sum are updated online
    // and o = o * 2^(M_old - M_new) + sum_s 2^(m_s - M_new) o_s is accumulated in
    // shared memory.
    constexpr int AREA = 2 * STAGES * C::TILE_B;
    const int R = p.R;
    float* acc = reinterpret_cast<float*>(smem + C::OFF_K);              // [R][D]
    float* rs = acc + R * D;                                              // [R][4]: M, L, factor
    const int per_split = R * (4 * D + 4 + 8);
    const int batch = max(1, (AREA - R * D * 4 - R * 16 - 64) / per_split);
    float* wts = rs + R * 4;                                              // [batch][R]
    float* mls = wts + ((batch * R + 3) & ~3);                            // [batch][R][2]
    uint8_t* stage = reinterpret_cast<uint8_t*>(mls + ((batch * R * 2 + 3) & ~3));   // [batch][R][D]
    const uint32_t stage_s = smem_u32(stage);
    for (int e = tid; e < R * D; e += C::NCT) acc[e] = 0.f;
    for (int e = tid; e < R; e += C::NCT) {
        rs[4 * e] = -INFINITY;
        rs[4 * e + 1] = 0.f;
    }
    for (int s0 = 0; s0 < nch; s0 += batch) {
        const int nb = min(batch, nch - s0);
        const uint8_t* src = reinterpret_cast<const uint8_t*>(p.part_o + static_cast<size_t>(c0 + s0) * R * D);
        const int n16 = nb * R * (D / 4);
        for (int e = tid; e < n16; e += C::NCT) cp_async_16(stage_s + e * 16, src + static_cast<size_t>(e) * 16);
        const float* msrc = p.part_ml + static_cast<size_t>(c0 + s0) * R * 2;
        // L2 loads (other CTAs wrote these records), four per thread in flight together
        for (int e0 = tid; e0 < nb * R; e0 += 4 * C::NCT) {
            float2 v2[4];
#pragma unroll
            for (int u = 0; u < 4; ++u)
                if (e0 + u * C::NCT < nb * R) v2[u] = __ldcg(reinterpret_cast<const float2*>(msrc) + e0 + u * C::NCT);
#pragma unroll
            for (int u = 0; u < 4; ++u)
                if (e0 + u * C::NCT < nb * R) reinterpret_cast<float2*>(mls)[e0 + u * C::NCT] = v2[u];
        }
        cp_async_wait_all();
        named_bar_sync(1, C::NCT);
        for (int row = cw; row < R; row += C::NCW) {
            float mb = -INFINITY;
            for (int sl = lane; sl < nb; sl += 32) mb = fmaxf(mb, mls[2 * (sl * R + row)]);
            mb = warp_max(mb);
            const float Mold = rs[4 * row];
            const float Mnew = fmaxf(Mold, mb);
            float ladd = 0.f;
            for (int sl = lane; sl < nb; sl += 32) {
                const float m = mls[2 * (sl * R + row)];
                const float w = (m == -INFINITY) ? 0.f : fast_exp2(m - Mnew);
                wts[sl * R + row] = w;
                ladd += w * mls[2 * (sl * R + row) + 1];
            }
            ladd = warp_sum(ladd);
            if (lane == 0) {
                const float f = (Mold == -INFINITY) ? 0.f : fast_exp2(Mold - Mnew);
                rs[4 * row] = Mnew;
                rs[4 * row + 1] = rs[4 * row + 1] * f + ladd;
                rs[4 * row + 2] = f;
            }
        }
        named_bar_sync(1, C::NCT);
        const float4* st4 = reinterpret_cast<const float4*>(stage);
        for (int e = tid; e < R * (D / 4); e += C::NCT) {
            const int row = e / (D / 4);
            const float f = rs[4 * row + 2];
            float4 a4 = reinterpret_cast<float4*>(acc)[e];
            a4.x *= f;
            a4.y *= f;
            a4.z *= f;
            a4.w *= f;
            for (int sl = 0; sl < nb; ++sl) {
                const float w = wts[sl * R + row];
                const float4 v4 = st4[sl * R * (D / 4) + e];
                a4.x += w * v4.x;
                a4.y += w * v4.y;
                a4.z += w * v4.z;
                a4.w += w * v4.w;
            }
            reinterpret_cast<float4*>(acc)[e] = a4;
        }
        named_bar_sync(1, C::NCT);
    }
    for (int e = tid; e < R * (D / 4); e += C::NCT) {
        const int row = e / (D / 4), d4 = e - (e / (D / 4)) * (D / 4);
        const float L = rs[4 * row + 1];
        const float il = L > 0.f ? 1.f / L : 0.f;
        const float4 a4 = reinterpret_cast<const float4*>(acc)[e];
        const int g = row / p.gamma, tt = row - (row / p.gamma) * p.gamma;
        const size_t orow = (static_cast<size_t>(b) * p.Hq + h * p.G + g) * p.gamma + tt;
        uint2 packed;
        packed.x = pack_bf16(a4.x * il, a4.y * il);
        packed.y = pack_bf16(a4.z * il, a4.w * il);
        *reinterpret_cast<uint2*>(p.o + orow * D + 4 * d4) = packed;
        if (d4 == 0 && p.lse) p.lse[orow] = L > 0.f ? (rs[4 * row] + fast_log2(L)) * kLn2 : -INFINITY;
    }
    if (tid == 0) atomicExch(p.tickets + bh, 0);
}

// =====================================================================================
// host side
// =====================================================================================
namespace {

constexpr int kDenseTK = 64;
constexpr int kDenseStages = 3;
constexpr int kSparseTK = 64;
constexpr int kSparseStages = 3;

// per-head counters: one per head-dim slice of a cluster merge (at most kMaxCluster)
size_t attn_ticket_bytes(int BH) { return sizeof(int) * static_cast<size_t>(BH) * kMaxCluster; }

struct WsLayout {
    int* status;
    int* tickets;
    float* part_o;
    float* part_ml;
    size_t bytes;
};

// ml_floats: floats of a partial row's softmax record ((m, l), or wider)
WsLayout attn_ws_layout(void* ws, int BH, int R, int d, int max_chunks, int ml_floats = 2) {
    const size_t off_tickets = kWsHeader;
    const size_t off_po = align256(off_tickets + attn_ticket_bytes(BH));
    const size_t off_pml = align256(off_po + sizeof(float) * static_cast<size_t>(max_chunks) * R * d);
    const size_t end = align256(off_pml + sizeof(float) * static_cast<size_t>(max_chunks) * R * ml_floats);
    WsLayout L{};
    L.bytes = end;
    if (ws) {
        uint8_t* base = static_cast<uint8_t*>(ws);
        L.status = reinterpret_cast<int*>(base);
        L.tickets = reinterpret_cast<int*>(base + off_tickets);
        L.part_o = reinterpret_cast<float*>(base + off_po);
        L.part_ml = reinterpret_cast<float*>(base + off_pml);
    }
    return L;
}

struct DensePlan {
    int nsplit, chunk, cs, ncl;
};

// Splits per head fill two CTAs per SM.  With enough splits per head they are
// grouped in clusters of cs CTAs (nsplit a multiple of cs) that merge their
// partials through distributed shared memory; trailing splits past the cache
// may be empty.
DensePlan dense_plan(int BH, int n_total, int num_sms) {
    const int slots = 2 * std::max(num_sms, 1);
    const int max_split = std::max(1, (n_total + kDenseTK - 1) / kDenseTK);
    const int per_head = std::min(std::max(1, slots / BH), max_split);
    DensePlan pl{};
    pl.cs = per_head >= 16 ? 8 : per_head >= 8 ? 4 : per_head >= 4 ? 2 : 1;
    if (pl.cs > 1) {
        // at most 4 clusters per head: the last one merges their partials
        pl.nsplit = std::min((per_head / pl.cs) * pl.cs, 4 * pl.cs);
        pl.chunk = (n_total + pl.nsplit - 1) / pl.nsplit;
        pl.chunk = ((pl.chunk + kDenseTK - 1) / kDenseTK) * kDenseTK;
        pl.ncl = pl.nsplit / pl.cs;
        return pl;
    }
    int nsplit = std::max(1, (slots + BH - 1) / BH);
    nsplit = std::min(nsplit, max_split);
    int chunk = (n_total + nsplit - 1) / nsplit;
    chunk = ((chunk + kDenseTK - 1) / kDenseTK) * kDenseTK;
    pl.nsplit = (n_total + chunk - 1) / chunk;
    pl.chunk = chunk;
    pl.ncl = pl.nsplit;
    return pl;
}

// Largest list-decode grid: two CTAs per SM, a whole number of clusters.  It
// bounds the partial slots of the workspace.
int sparse_grid_target(int num_sms) { return ((2 * std::max(num_sms, 1)) / kMaxCluster) * kMaxCluster; }
int sparse_max_chunks(int BH, int grid_target, int cs) { return cs > 1 ? grid_target : grid_target + BH; }

template <int D, int MT, int KW, int TK, int STAGES, int KIND>
cudaError_t ensure_smem_attr(int dev) {
    using C = AttnCfg<D, MT, KW, TK, STAGES, KIND>;
    static std::atomic<unsigned long long> attr_set{0};  // one bit per device, per instantiation
    if (attr_done(attr_set, dev)) return cudaSuccess;
    const cudaError_t e = cudaFuncSetAttribute(attn_splitk_kernel<D, MT, KW, TK, STAGES, KIND>,
                                               cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_ALLOC);
    if (e == cudaSuccess) attr_mark(attr_set, dev);
    return e;
}

// CTAs of one instantiation that the current device holds at once when they are
// launched in clusters of cs (occupancy query, once per device and cluster
// size).  A grid larger than this runs in two waves, and its last CTAs, which
// start only when others finish, hold back the next kernel's early start.
template <int D, int MT, int KW, int TK, int STAGES, int KIND>
int attn_capacity(int dev, int num_sms, int cs) {
    using C = AttnCfg<D, MT, KW, TK, STAGES, KIND>;
    static std::atomic<int> cache[64][4];   // 0: not queried yet
    const int ci = cs >= 8 ? 3 : cs >= 4 ? 2 : cs >= 2 ? 1 : 0;
    const bool cached = dev >= 0 && dev < 64;
    if (cached) {
        const int v = cache[dev][ci].load(std::memory_order_relaxed);
        if (v > 0) return v;
    }
    int cap = 0;
    if (ensure_smem_attr<D, MT, KW, TK, STAGES, KIND>(dev) == cudaSuccess) {
        auto kern = attn_splitk_kernel<D, MT, KW, TK, STAGES, KIND>;
        if (cs <= 1) {
            int per_sm = 0;
            if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, C::NT, C::SMEM_ALLOC) == cudaSuccess)
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
            if (cudaOccupancyMaxActiveClusters(&ncl, kern, &cfg) == cudaSuccess) cap = ncl * cs;
        }
    }
    if (cap <= 0) {
        (void)cudaGetLastError();   // a failed query leaves no error behind; assume two CTAs per SM
        cap = 2 * std::max(num_sms, 1);
    }
    if (cached) cache[dev][ci].store(cap, std::memory_order_relaxed);
    return cap;
}

template <int D, int MT, int KW, int TK, int STAGES, int KIND>
cudaError_t launch_attn(const AttnParams& p, const CUtensorMap& tmk, const CUtensorMap& tmv, int grid,
                        cudaStream_t st, int cluster = 1) {
    using C = AttnCfg<D, MT, KW, TK, STAGES, KIND>;
    auto kern = attn_splitk_kernel<D, MT, KW, TK, STAGES, KIND>;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    e = ensure_smem_attr<D, MT, KW, TK, STAGES, KIND>(dev);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(C::NT);
    cfg.dynamicSmemBytes = C::SMEM_ALLOC;
    cfg.stream = st;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cluster > 1) {
        attr[1].id = cudaLaunchAttributeClusterDimension;
        attr[1].val.clusterDim.x = cluster;
        attr[1].val.clusterDim.y = 1;
        attr[1].val.clusterDim.z = 1;
        cfg.numAttrs = 2;
    }
    return cudaLaunchKernelEx(&cfg, kern, p, tmk, tmv);
}

AttnParams make_params(const AttnLaunch& a) {
    AttnParams p{};
    p.q = static_cast<const bf16*>(a.q);
    p.k = static_cast<const bf16*>(a.k);
    p.v = static_cast<const bf16*>(a.v);
    p.sb = a.sb;
    p.sh = a.sh;
    p.sn = a.sn;
    p.B = a.B;
    p.Hq = a.Hq;
    p.Hkv = a.Hkv;
    p.G = a.Hq / a.Hkv;
    p.gamma = a.gamma;
    p.R = p.G * a.gamma;
    p.o = static_cast<bf16*>(a.o);
    p.lse = a.lse;
    p.scale_log2 = a.scale * kLog2e;
    return p;
}

}  // namespace

AttnWs attn_ws(void* ws, int BH, int R, int d, int max_chunks, int ml_floats) {
    const WsLayout L = attn_ws_layout(ws, BH, R, d, max_chunks, ml_floats);
    return AttnWs{L.status, L.tickets, L.part_o, L.part_ml, L.bytes};
}

size_t dense_ws_bytes(int B, int Hq, int Hkv, int d, int n_total, int gamma, int num_sms) {
    const int BH = B * Hkv;
    const DensePlan pl = dense_plan(BH, n_total, num_sms);
    const int R = (Hq / Hkv) * gamma;
    const size_t tc = verify_tc_ws_bytes(B, Hq, Hkv, d, n_total, gamma, num_sms);
    return std::max(attn_ws_layout(nullptr, BH, R, d, BH * pl.nsplit).bytes, tc);
}

size_t sparse_ws_bytes(int B, int Hq, int Hkv, int d, int num_sms) {
    const int BH = B * Hkv;
    const int R = Hq / Hkv;
    // the packed decode's partials: 2 per CTA, 16-byte (m, l) records
    return std::max(attn_ws_layout(nullptr, BH, R, d, sparse_grid_target(num_sms) + BH).bytes,
                    attn_ws_layout(nullptr, BH, R, d, 2 * packed_decode_grid_max(num_sms), 4).bytes);
}

int launch_dense_verify(const AttnLaunch& a, const CUtensorMap* tmk, const CUtensorMap* tmv, int num_sms,
                        const char** why) {
    // more than 16 query rows per KV head at d = 128: the tensor-core verify
    if (verify_tc_ws_bytes(a.B, a.Hq, a.Hkv, a.d, a.n_prefix + a.gamma, a.gamma, num_sms) > 0)
        return launch_verify_tc(a, tmk, tmv, num_sms, why);
    AttnParams p = make_params(a);
    const int BH = a.B * a.Hkv;
    p.n_prefix = a.n_prefix;
    p.n_total = a.n_prefix + a.gamma;
    const DensePlan pl = dense_plan(BH, p.n_total, num_sms);
    p.nsplit = pl.nsplit;
    p.chunk = pl.chunk;
    p.cs = pl.cs;
    p.ncl = pl.ncl;
    WsLayout L = attn_ws_layout(a.ws, BH, p.R, a.d, BH * pl.nsplit);
    if (a.ws_bytes < L.bytes) {
        *why = "workspace smaller than sdkv_workspace_size(SDKV_OP_DENSE_VERIFY, ...)";
        return SDKV_ERR_WORKSPACE;
    }
    p.status = L.status;
    p.tickets = L.tickets;
    p.part_o = L.part_o;
    p.part_ml = L.part_ml;
    const int grid = BH * pl.nsplit;
    const int MT = (p.R + 15) / 16;
    cudaError_t e = cudaErrorInvalidValue;
    if (a.d == 128) {
        switch (MT) {
            case 1: e = launch_attn<128, 1, 4, kDenseTK, kDenseStages, kDense>(p, *tmk, *tmv, grid, a.stream, pl.cs); break;
            case 2: e = launch_attn<128, 2, 2, kDenseTK, kDenseStages, kDense>(p, *tmk, *tmv, grid, a.stream, pl.cs); break;
            case 3: e = launch_attn<128, 3, 2, kDenseTK, kDenseStages, kDense>(p, *tmk, *tmv, grid, a.stream, pl.cs); break;
            case 4: e = launch_attn<128, 4, 2, kDenseTK, kDenseStages, kDense>(p, *tmk, *tmv, grid, a.stream, pl.cs); break;
            default: *why = "(Hq/Hkv) * gamma must be <= 64"; return SDKV_ERR_UNSUPPORTED;
        }
    } else {
        switch (MT) {
            case 1: e = launch_attn<64, 1, 4, kDenseTK, kDenseStages, kDense>(p, *tmk, *tmv, grid, a.stream, pl.cs); break;
            case 2: e = launch_attn<64, 2, 2, kDenseTK, kDenseStages, kDense>(p, *tmk, *tmv, grid, a.stream, pl.cs); break;
            case 3: e = launch_attn<64, 3, 2, kDenseTK, kDenseStages, kDense>(p, *tmk, *tmv, grid, a.stream, pl.cs); break;
            case 4: e = launch_attn<64, 4, 2, kDenseTK, kDenseStages, kDense>(p, *tmk, *tmv, grid, a.stream, pl.cs); break;
            default: *why = "(Hq/Hkv) * gamma must be <= 64"; return SDKV_ERR_UNSUPPORTED;
        }
    }
    if (e != cudaSuccess) {
        *why = cudaGetErrorString(e);
        return SDKV_ERR_CUDA;
    }
    return SDKV_OK;
}

namespace {

// Sparse decode over index lists (KIND = kGather: rows gathered from the caches)
// or over the lists' rows compacted into contiguous buffers (KIND = kContig).
// Clusters only when every head can own whole clusters and still leave the grid
// half free for long lists; the grid is what one wave of such clusters holds.
template <int D, int MT, int KW, int KIND>
int list_decode_launch(AttnParams& p, const AttnLaunch& a, const CUtensorMap& tmk, const CUtensorMap& tmv,
                       int num_sms, const char** why) {
    constexpr int TK = kSparseTK, ST = kSparseStages;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) {
        *why = cudaGetErrorString(e);
        return SDKV_ERR_CUDA;
    }
    const int base = sparse_grid_target(num_sms);
    p.cs = 1;
    p.grid_target = base;
    for (int cs = kMaxCluster; cs > 1; cs /= 2) {
        int cap = std::min(base, attn_capacity<D, MT, KW, TK, ST, KIND>(dev, num_sms, cs));
        cap -= cap % cs;
        if (2 * cs * p.BH <= cap) {
            p.cs = cs;
            p.grid_target = cap;
            break;
        }
    }
    // many lists that no cluster plan covers: pack them by list position
    if (KIND == kGather && p.cs == 1 && a.gamma == 1 && packed_decode_takes(a.B, a.Hq, a.Hkv, a.d))
        return launch_packed_decode(a, num_sms, why);
    p.ncl = 1;
    const int max_chunks = sparse_max_chunks(p.BH, p.grid_target, p.cs);
    WsLayout L = attn_ws_layout(a.ws, p.BH, p.R, a.d, max_chunks);
    if (a.ws_bytes < L.bytes) {
        *why = "workspace smaller than sdkv_workspace_size(SDKV_OP_SPARSE_DECODE, ...)";
        return SDKV_ERR_WORKSPACE;
    }
    p.status = L.status;
    p.tickets = L.tickets;
    p.part_o = L.part_o;
    p.part_ml = L.part_ml;
    e = launch_attn<D, MT, KW, TK, ST, KIND>(p, tmk, tmv, max_chunks, a.stream, p.cs);
    if (e != cudaSuccess) {
        *why = cudaGetErrorString(e);
        return SDKV_ERR_CUDA;
    }
    return SDKV_OK;
}

template <int KIND>
int launch_list_decode(const AttnLaunch& a, const CUtensorMap& tmk, const CUtensorMap& tmv, int num_sms,
                       const char** why) {
    AttnParams p = make_params(a);
    p.offsets = a.offsets;
    p.indices = a.indices;
    p.n_idx = a.n_idx;
    p.n_cap = a.n_cap;
    p.BH = a.B * a.Hkv;
    p.min_chunk = 4 * kSparseTK;   // short lists: one cluster per head, no cross-cluster merge
    const int MT = (p.R + 15) / 16;
    if (a.d == 128) {
        switch (MT) {
            case 1: return list_decode_launch<128, 1, 4, KIND>(p, a, tmk, tmv, num_sms, why);
            case 2: return list_decode_launch<128, 2, 2, KIND>(p, a, tmk, tmv, num_sms, why);
            default: *why = "Hq/Hkv must be <= 32"; return SDKV_ERR_UNSUPPORTED;
        }
    }
    switch (MT) {
        case 1: return list_decode_launch<64, 1, 4, KIND>(p, a, tmk, tmv, num_sms, why);
        case 2: return list_decode_launch<64, 2, 2, KIND>(p, a, tmk, tmv, num_sms, why);
        default: *why = "Hq/Hkv must be <= 32"; return SDKV_ERR_UNSUPPORTED;
    }
}

}  // namespace

int launch_sparse_decode(const AttnLaunch& a, int num_sms, const char** why) {
    CUtensorMap dummy;
    memset(&dummy, 0, sizeof(dummy));
    return launch_list_decode<kGather>(a, dummy, dummy, num_sms, why);
}

int launch_sparse_decode_compact(const AttnLaunch& a, const CUtensorMap* tmk, const CUtensorMap* tmv, int num_sms,
                                 const char** why) {
    return launch_list_decode<kContig>(a, *tmk, *tmv, num_sms, why);
}

// -------------------------------------------------------------------------------------
// Scratch for callers that cannot allocate device memory (see
// sdkv_dense_verify_attn_noalloc): a fixed array in the library's own device
// image.  Every GPU that loads the library holds it until the process exits.
// The array's name in host code is only a host-side stand-in; the device address
// comes from cudaGetSymbolAddress, once per device, with that device current.
// -------------------------------------------------------------------------------------
static __device__ __align__(256) uint8_t g_noalloc_scratch[SDKV_NOALLOC_SCRATCH_BYTES];

namespace {

// Unique id of the calling thread's current CUDA context (0 if it cannot be
// read).  A device reset destroys the context the array's address belongs to;
// the next context has another id, so the address is looked up again.
unsigned long long current_ctx_id() {
    using GetCurrent = CUresult (*)(CUcontext*);
    using GetId = CUresult (*)(CUcontext, unsigned long long*);
    static GetCurrent get_current = nullptr;
    static GetId get_id = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_current = reinterpret_cast<GetCurrent>(p);
        p = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_id = reinterpret_cast<GetId>(p);
    });
    CUcontext ctx = nullptr;
    unsigned long long id = 0;
    if (get_current && get_id && get_current(&ctx) == CUDA_SUCCESS && ctx && get_id(ctx, &id) == CUDA_SUCCESS)
        return id;
    return 0;
}

// Device address of the array on the current device: looked up with
// cudaGetSymbolAddress once per device and context, cached after that.
int noalloc_scratch(void** out, const char** why) {
    static std::mutex mu;
    static void* dev_ptr[64] = {};
    static unsigned long long dev_ctx[64] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) {
        *why = cudaGetErrorString(e);
        return SDKV_ERR_CUDA;
    }
    if (dev < 0 || dev >= 64) {
        *why = "device ordinal above 63";
        return SDKV_ERR_UNSUPPORTED;
    }
    // 0 before the thread has a current context: the lookup below creates it,
    // and the next call, seeing the real id, looks the address up once more
    const unsigned long long ctx = current_ctx_id();
    std::lock_guard<std::mutex> lock(mu);
    if (!dev_ptr[dev] || dev_ctx[dev] != ctx) {
        void* ptr = nullptr;
        e = cudaGetSymbolAddress(&ptr, g_noalloc_scratch);
        if (e != cudaSuccess || ptr == nullptr) {
            *why = e != cudaSuccess ? cudaGetErrorString(e) : "cudaGetSymbolAddress returned null";
            return SDKV_ERR_CUDA;
        }
        dev_ptr[dev] = ptr;
        dev_ctx[dev] = ctx;
    }
    *out = dev_ptr[dev];
    return SDKV_OK;
}

}  // namespace

int dense_verify_noalloc(const AttnLaunch& a_in, const CUtensorMap* tmk, const CUtensorMap* tmv, int num_sms,
                         const char** why) {
    const size_t need = dense_ws_bytes(a_in.B, a_in.Hq, a_in.Hkv, a_in.d, a_in.n_prefix + a_in.gamma, a_in.gamma,
                                       num_sms);
    if (need > static_cast<size_t>(SDKV_NOALLOC_SCRATCH_BYTES)) {
        *why = "shape needs more scratch than the fixed SDKV_NOALLOC_SCRATCH_BYTES array of "
               "sdkv_dense_verify_attn_noalloc holds (use sdkv_dense_verify_attn with a workspace)";
        return SDKV_ERR_UNSUPPORTED;
    }
    void* ptr = nullptr;
    int rc = noalloc_scratch(&ptr, why);
    if (rc) return rc;
    // The array keeps the previous call's contents: the status word and the
    // per-head counters must start at zero.
    cudaError_t e = cudaMemsetAsync(ptr, 0, kWsHeader + align256(attn_ticket_bytes(a_in.B * a_in.Hkv)), a_in.stream);
    if (e != cudaSuccess) {
        *why = cudaGetErrorString(e);
        return SDKV_ERR_CUDA;
    }
    AttnLaunch a = a_in;
    a.ws = ptr;
    a.ws_bytes = SDKV_NOALLOC_SCRATCH_BYTES;
    return launch_dense_verify(a, tmk, tmv, num_sms, why);
}

int noalloc_status(int32_t* status, cudaStream_t st, const char** why) {
    void* ptr = nullptr;
    int rc = noalloc_scratch(&ptr, why);
    if (rc) return rc;
    cudaError_t e = cudaMemcpyAsync(status, ptr, sizeof(int32_t), cudaMemcpyDeviceToHost, st);
    if (e == cudaSuccess) e = cudaMemsetAsync(ptr, 0, sizeof(int32_t), st);
    if (e == cudaSuccess) e = cudaStreamSynchronize(st);
    if (e != cudaSuccess) {
        *why = cudaGetErrorString(e);
        return SDKV_ERR_CUDA;
    }
    return SDKV_OK;
}

}  // namespace sdkv
