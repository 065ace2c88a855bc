// Kernels around the hot path: list builders, row compaction and the SpecVLM
// token selection.
//
//   window_lists    attention sinks plus the recent window (StD baselines,
//                   "Streaming"; ByteCross "The Attention Baseline")
//   append_drafts   a draft step's lists: the base selection plus the positions
//                   drafted so far (StD 3.1)
//   draft_lists     the lists of all gamma draft steps of a round in one launch
//   compact_kv      the selected rows of every head gathered once into
//                   contiguous buffers (ByteCross "Speedup Across Context")
//   specvlm         importance = mean of the verifier's attention maps; Stage I
//                   top-P retention of the attention mass, Stage II uniform
//                   subsample of the rest (SpecVLM post, "The SpecVLM Method")
#include "sdkv_common.cuh"
#include "sdkv_internal.h"

#include <algorithm>

namespace sdkv {

// ============================================================================ lists
__global__ void window_lists_kernel(int BH, int n, int n_sink, int n_recent, int k, int* offsets, int* indices) {
    griddep_wait();   // the lists may still be read by the previous kernel
    griddep_launch();
    const long long e = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
    const int s1 = min(n_sink, n);
    const int w0 = max(n - n_recent, s1);
    if (e <= BH) offsets[e] = static_cast<int>(e) * k;
    if (e < static_cast<long long>(BH) * k) {
        const int j = static_cast<int>(e % k);
        indices[e] = (j < s1) ? j : w0 + (j - s1);
    }
}

__global__ void append_drafts_kernel(const int* base_offsets, const int* base_indices, int BH, int n_pos, int n_new,
                                     int* offsets, int* indices) {
    griddep_wait();   // the base lists come from, and the new ones may be read by, earlier kernels
    griddep_launch();
    const int i = blockIdx.x;
    if (i >= BH) return;
    const int b0 = base_offsets[0];
    const int st = base_offsets[i], len = base_offsets[i + 1] - st;
    const int out0 = (st - b0) + i * n_new;
    if (threadIdx.x == 0) {
        offsets[i] = out0;
        if (i == BH - 1) offsets[BH] = out0 + len + n_new;
    }
    constexpr int U = 8;   // loads in flight per thread
    for (int e0 = threadIdx.x; e0 < len + n_new; e0 += U * blockDim.x) {
        int val[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int e = e0 + u * blockDim.x;
            val[u] = (e < len) ? base_indices[st + e] : n_pos + (e - len);
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int e = e0 + u * blockDim.x;
            if (e < len + n_new) indices[out0 + e] = val[u];
        }
    }
}

// Every draft step's lists of one round: set t (grid y) is the base CSR with
// n_pos .. n_pos + t appended to each list; entries at or past `stride` in a
// set are not written.
__global__ void draft_lists_kernel(const int* base_offsets, const int* base_indices, int BH, int n_pos,
                                   long long stride, int* offsets, int* indices) {
    griddep_wait();
    griddep_launch();
    const int i = blockIdx.x, t = blockIdx.y, n_new = t + 1;
    const int b0 = base_offsets[0];
    const int st = base_offsets[i], len = base_offsets[i + 1] - st;
    const long long out0 = static_cast<long long>(st - b0) + static_cast<long long>(i) * n_new;
    int* set_off = offsets + static_cast<size_t>(t) * (BH + 1);
    int* set_idx = indices + static_cast<size_t>(t) * stride;
    if (threadIdx.x == 0) {
        set_off[i] = static_cast<int>(out0);
        if (i == BH - 1) set_off[BH] = static_cast<int>(out0 + len + n_new);
    }
    constexpr int U = 8;   // loads in flight per thread
    for (int e0 = threadIdx.x; e0 < len + n_new; e0 += U * blockDim.x) {
        int val[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int e = e0 + u * blockDim.x;
            val[u] = (e < len) ? base_indices[st + e] : n_pos + (e - len);
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int e = e0 + u * blockDim.x;
            const long long o = out0 + e;
            if (e < len + n_new && o < stride) set_idx[o] = val[u];
        }
    }
}

// ============================================================================ compaction
// CTA c copies flat list positions [c*CH, (c+1)*CH): one warp per row, 16-byte
// chunks, K chunks on the first D/8 lanes of a row group and V on the next.
constexpr int kCompactRows = 128;

template <int D>
__global__ void __launch_bounds__(256) compact_kv_kernel(const bf16* __restrict__ k, const bf16* __restrict__ v,
                                                          long long sb, long long sh, long long sn, int n_cap, int Hkv,
                                                          int BH, const int* offsets, const int* indices,
                                                          long long rows_cap, bf16* k_out, bf16* v_out, int* status) {
    constexpr int CPR = D / 8;                  // 16-byte chunks of a K (or V) row
    constexpr int LPR = 2 * CPR;                // lanes per row: K chunks, then V chunks
    constexpr int RPW = 32 / LPR;               // rows per warp instruction
    constexpr int WROWS = kCompactRows / 8;     // list positions per warp (8 warps)
    constexpr int NIT = WROWS / RPW;            // copies in flight per lane
    static_assert(WROWS <= 32 && WROWS % RPW == 0, "one list position per lane for the look-up");
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int off0 = __ldg(offsets);
    const long long total = __ldg(offsets + BH) - off0;
    const long long pw = static_cast<long long>(blockIdx.x) * kCompactRows + warp * WROWS;
    // lane j < WROWS looks up position pw + j: its list entry and its head (the
    // first head whose list ends after the position)
    int my_idx = 0, my_b = 0, my_h = 0, my_ok = 0;
    if (lane < WROWS) {
        const long long p = pw + lane;
        if (p < total) {
            if (p >= rows_cap) {
                flag_status(status, SDKV_DEV_BAD_LIST);
            } else {
                int idx = indices[off0 + p];   // in flight during the head search
                int lo = 0, hi = BH;
                while (lo < hi) {
                    const int mid = (lo + hi) >> 1;
                    if (__ldg(offsets + mid + 1) - off0 > p) hi = mid; else lo = mid + 1;
                }
                if (static_cast<unsigned>(idx) >= static_cast<unsigned>(n_cap)) {
                    flag_status(status, SDKV_DEV_BAD_INDEX);
                    idx = 0;
                }
                my_idx = idx;
                my_b = lo / Hkv;
                my_h = lo - my_b * Hkv;
                my_ok = 1;
            }
        }
    }
    // every row's chunk is loaded before any is stored
    const int sub = lane / LPR, cl = lane % LPR;
    const bool is_v = cl >= CPR;
    const int ch = is_v ? cl - CPR : cl;
    uint4 buf[NIT];
#pragma unroll
    for (int it = 0; it < NIT; ++it) {
        const int r = it * RPW + sub;
        const int idx = __shfl_sync(0xffffffffu, my_idx, r);
        const int b = __shfl_sync(0xffffffffu, my_b, r);
        const int h = __shfl_sync(0xffffffffu, my_h, r);
        const int ok = __shfl_sync(0xffffffffu, my_ok, r);
        buf[it] = make_uint4(0u, 0u, 0u, 0u);
        if (ok) {
            const bf16* src = (is_v ? v : k) + b * sb + h * sh + static_cast<long long>(idx) * sn + ch * 8;
            buf[it] = __ldg(reinterpret_cast<const uint4*>(src));
        }
    }
#pragma unroll
    for (int it = 0; it < NIT; ++it) {
        const int r = it * RPW + sub;
        if (__shfl_sync(0xffffffffu, my_ok, r)) {
            bf16* dst = (is_v ? v_out : k_out) + (pw + r) * D + ch * 8;
            *reinterpret_cast<uint4*>(dst) = buf[it];
        }
    }
}

// ============================================================================ SpecVLM
__global__ void importance_kernel(const float* __restrict__ scores, int units, int n, float inv_units,
                                  float* __restrict__ importance) {
    const int b = blockIdx.y;
    const int j = blockIdx.x * blockDim.x + threadIdx.x;
    if (j >= n) return;
    const float* s = scores + static_cast<size_t>(b) * units * n + j;
    float acc = 0.f;
    constexpr int kBatch = 32;   // loads in flight; the adds stay in unit order
    for (int u0 = 0; u0 < units; u0 += kBatch) {
        float x[kBatch];
#pragma unroll
        for (int q = 0; q < kBatch; ++q) x[q] = (u0 + q < units) ? __ldg(s + static_cast<size_t>(u0 + q) * n) : 0.f;
#pragma unroll
        for (int q = 0; q < kBatch; ++q)
            if (u0 + q < units) acc += x[q];
    }
    importance[static_cast<size_t>(b) * n + j] = acc * inv_units;
}

constexpr int kSpecNT = 1024;
constexpr int kSpecSmemKeys = 16384;       // keys in shared memory up to this many video tokens
constexpr int kSpecMaxTokens = 1 << 20;    // the sampled-rank bitmap lives in shared memory
constexpr int kSpecSmemMax = 4 * ((1 << 20) / 32);

struct SpecParams {
    const float* importance;
    int n, v_lo, v_hi, keep_lo, keep_hi, cap;
    double lam_r, r;
    int* indices;
    int* counts;
    int* status;
    uint32_t* keys_ws;   // [B][nV] when the keys do not fit shared memory
    uint8_t* flags_ws;   // [B][nV] likewise
    bool keys_in_smem;
};

// exclusive scan of one value per thread over the CTA (int64); returns the prefix, sets *total
__device__ long long cta_excl_scan(long long v, long long* s_w, long long* total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    long long x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const long long y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) s_w[warp] = x;
    __syncthreads();
    if (warp == 0) {
        long long w = (lane < kSpecNT / 32) ? s_w[lane] : 0;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const long long y = __shfl_up_sync(0xffffffffu, w, o);
            if (lane >= o) w += y;
        }
        s_w[lane] = w;
    }
    __syncthreads();
    const long long res = (warp ? s_w[warp - 1] : 0) + x - v;
    *total = s_w[kSpecNT / 32 - 1];
    __syncthreads();
    return res;
}

// The mass of a score in [0, 2^31) from its fp32 bits: score * 2^32 rounded to
// the nearest integer, ties to even.  The score is man * 2^(ex - 150) with a
// 24-bit significand, so the scaled value man * 2^(ex - 118) is exact and the
// rounding is decided on the bits shifted out.
__device__ __forceinline__ long long mass_of_bits(uint32_t bits) {
    const int ex = static_cast<int>(bits >> 23);
    if (ex == 0) return 0;                                            // subnormal: far below 1/2
    const unsigned long long man = (bits & 0x7fffffu) | 0x800000u;
    const int sh = ex - 118;
    if (sh >= 0) return static_cast<long long>(man << sh);
    const int s = -sh;
    if (s > 24) return 0;                                             // man < 2^24 <= 2^(s-1): below 1/2
    const unsigned long long q = man >> s, rem = man & ((1ull << s) - 1ull), half = 1ull << (s - 1);
    return static_cast<long long>(q + ((rem > half || (rem == half && (q & 1ull))) ? 1ull : 0ull));
}

__global__ void __launch_bounds__(kSpecNT, 1) specvlm_select_kernel(const __grid_constant__ SpecParams p) {
    extern __shared__ __align__(16) uint8_t dyn[];
    __shared__ long long s_w[kSpecNT / 32];
    __shared__ unsigned s_cnt[256];
    __shared__ unsigned s_mlo[256], s_mhi[256];   // per-digit mass: low word (wraps carried) and high word
    __shared__ unsigned s_digit, s_cnt_above;
    __shared__ long long s_above, s_j;
    __shared__ double s_target, s_I;
    __shared__ long long s_kcap;
    const int b = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int nV = p.v_hi - p.v_lo;
    const int nW = (nV + 31) >> 5;
    uint32_t* taken = reinterpret_cast<uint32_t*>(dyn);   // [nW] bitmap of the sampled leftover ranks
    uint32_t* keys = p.keys_in_smem ? taken + nW : p.keys_ws + static_cast<size_t>(b) * nV;
    uint8_t* fl = p.keys_in_smem ? reinterpret_cast<uint8_t*>(taken + nW + nV)
                                 : p.flags_ws + static_cast<size_t>(b) * nV;   // 0, 1 = V_R, 2 = V_U
    const float* a = p.importance + static_cast<size_t>(b) * p.n + p.v_lo;

    // keys = fp32 bits of the score shifted left by one (the sign bit is 0, so
    // the first digit is the exponent): larger key, larger score.  Scores
    // outside [0, 2^31) and NaN count as zero mass; -0 equals +0.
    long long mloc = 0;
    constexpr int kLoads = 8;   // loads in flight per thread
    for (int e0 = tid; e0 < nV; e0 += kLoads * kSpecNT) {
        float xs[kLoads];
#pragma unroll
        for (int q = 0; q < kLoads; ++q) {
            const int e = e0 + q * kSpecNT;
            xs[q] = e < nV ? a[e] : 0.f;
        }
#pragma unroll
        for (int q = 0; q < kLoads; ++q) {
            const int e = e0 + q * kSpecNT;
            if (e >= nV) break;
            float x = xs[q];
            if (!(x >= 0.f && x < 2147483648.f)) {
                flag_status(p.status, SDKV_DEV_BAD_LIST);
                x = 0.f;
            }
            const uint32_t bits = __float_as_uint(x) & 0x7fffffffu;
            keys[e] = bits << 1;
            mloc += mass_of_bits(bits);
        }
    }
    for (int w = tid; w < nW; w += kSpecNT) taken[w] = 0u;
    for (int i = tid; i < 256; i += kSpecNT) {
        s_cnt[i] = 0u;
        s_mlo[i] = 0u;
        s_mhi[i] = 0u;
    }
    long long S = 0;
    cta_excl_scan(mloc, s_w, &S);   // also orders the stores above before every later read
    if (tid == 0) s_target = p.lam_r * static_cast<double>(S);
    __syncthreads();
    const double target = s_target;

    // ---- Stage I.  In the order (score descending, lower token first) V_R ends
    // at the first token where the running mass reaches the target.  Its key T
    // is found 8 bits at a time: per digit of the keys that share the prefix so
    // far, their count and mass; the digit whose range crosses the target is
    // the next digit of T.  Then the keys above T are all in V_R, and of the
    // keys equal to T (equal masses) the lowest j tokens complete it.
    const bool stage1 = target > 0.0;
    uint32_t T = 0u;
    long long j = 0;
    long long c = 0;   // |V_R|
    if (stage1) {
        uint32_t prefix = 0u, pmask = 0u;
        long long above = 0;
        unsigned cnt_above = 0u, cnt_T = 0u;
#pragma unroll 1
        for (int sh = 24; sh >= 0; sh -= 8) {
            if (tid == 0) {   // overwritten by the crossing digit, which always exists
                s_digit = 0u;
                s_above = above;
                s_cnt_above = cnt_above;
            }
            for (int e = tid; e < nV; e += kSpecNT) {
                const uint32_t u = keys[e];
                if ((u & pmask) == prefix) {
                    const unsigned d = (u >> sh) & 0xffu;
                    const unsigned long long m = static_cast<unsigned long long>(mass_of_bits(u >> 1));
                    const unsigned lo = static_cast<unsigned>(m);
                    unsigned hi = static_cast<unsigned>(m >> 32);
                    atomicAdd(&s_cnt[d], 1u);
                    const unsigned old = atomicAdd(&s_mlo[d], lo);
                    if (old + lo < old) ++hi;   // this add wrapped the low word
                    if (hi) atomicAdd(&s_mhi[d], hi);
                }
            }
            __syncthreads();
            if (warp == 0) {
                // lane owns digits 255 - 8*lane .. 248 - 8*lane (descending)
                long long m8[8], msum = 0;
                unsigned c8[8], csum = 0;
#pragma unroll
                for (int q = 0; q < 8; ++q) {
                    const int d = 255 - 8 * lane - q;
                    m8[q] = static_cast<long long>((static_cast<unsigned long long>(s_mhi[d]) << 32) | s_mlo[d]);
                    c8[q] = s_cnt[d];
                    msum += m8[q];
                    csum += c8[q];
                }
                long long mx = msum;
                unsigned cx = csum;
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    const long long ym = __shfl_up_sync(0xffffffffu, mx, o);
                    const unsigned yc = __shfl_up_sync(0xffffffffu, cx, o);
                    if (lane >= o) {
                        mx += ym;
                        cx += yc;
                    }
                }
                long long mb = above + mx - msum;
                unsigned cb = cnt_above + cx - csum;
#pragma unroll
                for (int q = 0; q < 8; ++q) {
                    const long long mn = mb + m8[q];
                    if (static_cast<double>(mb) < target && static_cast<double>(mn) >= target) {
                        s_digit = 255 - 8 * lane - q;
                        s_above = mb;
                        s_cnt_above = cb;
                    }
                    mb = mn;
                    cb += c8[q];
                }
            }
            __syncthreads();
            const unsigned d = s_digit & 0xffu;
            above = s_above;
            cnt_above = s_cnt_above;
            cnt_T = s_cnt[d];
            prefix |= d << sh;
            pmask |= 0xffu << sh;
            __syncthreads();   // every thread has read this pass's histogram
            for (int i = tid; i < 256; i += kSpecNT) {
                s_cnt[i] = 0u;
                s_mlo[i] = 0u;
                s_mhi[i] = 0u;
            }
            __syncthreads();
        }
        T = prefix;
        if (tid == 0) {
            // the fewest keys equal to T (mass mT > 0 each) that reach the target
            const long long mT = mass_of_bits(T >> 1);
            long long jj = static_cast<long long>(cnt_T);
            if (mT > 0) {
                const double est = ceil((target - static_cast<double>(above)) / static_cast<double>(mT));
                if (est < static_cast<double>(cnt_T)) jj = static_cast<long long>(est);
            }
            jj = max(1ll, min(jj, static_cast<long long>(cnt_T)));
            while (jj > 1 && static_cast<double>(above + (jj - 1) * mT) >= target) --jj;
            while (jj < static_cast<long long>(cnt_T) && static_cast<double>(above + jj * mT) < target) ++jj;
            s_j = jj;
        }
        __syncthreads();
        j = s_j;
        c = static_cast<long long>(cnt_above) + j;
    }

    // ---- token order: each thread a contiguous block of V; fl[e] = 1 for V_R
    const int per = (nV + kSpecNT - 1) / kSpecNT;
    const int i0 = min(nV, tid * per), i1 = min(nV, i0 + per);
    const int j32 = static_cast<int>(j);
    int eq_local = 0;
    if (stage1)
        for (int e = i0; e < i1; ++e) eq_local += (keys[e] == T) ? 1 : 0;
    long long tot_eq = 0;
    const int eq0 = static_cast<int>(cta_excl_scan(eq_local, s_w, &tot_eq));
    int left_local = 0;
    {
        int eqr = eq0;   // keys equal to T before this token
        for (int e = i0; e < i1; ++e) {
            const uint32_t u = keys[e];
            bool in1 = false;
            if (stage1 && u >= T) {
                in1 = (u > T) || (eqr < j32);
                eqr += (u == T) ? 1 : 0;
            }
            fl[e] = in1 ? 1 : 0;
            left_local += in1 ? 0 : 1;
        }
    }
    long long L = 0;
    const int rank0 = static_cast<int>(cta_excl_scan(left_local, s_w, &L));   // L = |V| - |V_R|

    // ---- Stage II: the leftover ranks floor(k I) < L, k = 0, 1, ...  floor(k I)
    // never decreases in k, and I >= 1/|V| when positive, so k <= |V| + 2 covers them
    if (tid == 0) {
        const double I0 = static_cast<double>(nV - c) / ((1.0 - p.r) * static_cast<double>(nV));
        long long kcap = -1;
        if (I0 > 0.0) {
            const double kc = ceil(static_cast<double>(L) / I0) + 1.0;
            kcap = kc < static_cast<double>(nV + 2) ? static_cast<long long>(kc) : nV + 2;
        }
        s_I = I0;
        s_kcap = kcap;
    }
    __syncthreads();
    const double I = s_I;
    {
        const long long kcap = s_kcap;
        for (long long k = tid; k <= kcap; k += kSpecNT) {
            const double pos = floor(static_cast<double>(k) * I);
            if (pos < static_cast<double>(L)) {
                const int ip = static_cast<int>(pos);
                atomicOr(&taken[ip >> 5], 1u << (ip & 31));
            }
        }
    }
    __syncthreads();

    // ---- output: V_R u V_U ascending, with the always-kept range before or after V
    int keep_local = 0;
    {
        int rr = rank0;   // leftover rank of the next leftover token
        for (int e = i0; e < i1; ++e) {
            if (!fl[e]) {
                if ((taken[rr >> 5] >> (rr & 31)) & 1u) fl[e] = 2;
                ++rr;
            }
            keep_local += fl[e] ? 1 : 0;
        }
    }
    long long nkeep = 0;
    const long long out0 = cta_excl_scan(keep_local, s_w, &nkeep);
    const int nk = p.keep_hi - p.keep_lo;
    const bool keep_first = p.keep_hi <= p.v_lo;
    int* out = p.indices + static_cast<size_t>(b) * p.cap;
    if (p.keys_in_smem) {
        // the keys are no longer needed: stage V's part of the list there, then
        // copy it out with consecutive threads on consecutive entries
        __syncthreads();
        int* stage = reinterpret_cast<int*>(keys);
        int o = static_cast<int>(out0);
        for (int e = i0; e < i1; ++e)
            if (fl[e]) stage[o++] = p.v_lo + e;
        __syncthreads();
        int* dst = out + (keep_first ? nk : 0);
        for (int i = tid; i < static_cast<int>(nkeep); i += kSpecNT) dst[i] = stage[i];
    } else {
        int o = (keep_first ? nk : 0) + static_cast<int>(out0);
        for (int e = i0; e < i1; ++e)
            if (fl[e]) out[o++] = p.v_lo + e;
    }
    const long long kbase = keep_first ? 0 : nkeep;
    for (int e = tid; e < nk; e += kSpecNT) out[kbase + e] = p.keep_lo + e;
    if (tid == 0) p.counts[b] = static_cast<int>(nkeep + nk);
}

// ============================================================================ host

size_t specvlm_ws_bytes(int B, int nV) {
    size_t bytes = kWsHeader;
    if (nV > kSpecSmemKeys) {
        bytes += align256(sizeof(uint32_t) * static_cast<size_t>(B) * nV);   // keys
        bytes += align256(static_cast<size_t>(B) * nV);                      // flags
    }
    return bytes;
}

int launch_window_lists(int B, int Hkv, int n, int n_sink, int n_recent, int* offsets, int* indices,
                        cudaStream_t st, const char** why) {
    const int BH = B * Hkv;
    const int k = std::min(n, n_sink + n_recent);
    const long long work = std::max<long long>(static_cast<long long>(BH) * k, BH + 1);
    const int grid = static_cast<int>((work + 255) / 256);
    const cudaError_t e = launch_pdl(window_lists_kernel, dim3(grid), dim3(256), 0, st, BH, n, n_sink, n_recent, k,
                                     offsets, indices);
    if (e != cudaSuccess) {
        *why = cudaGetErrorString(e);
        return SDKV_ERR_CUDA;
    }
    return SDKV_OK;
}

int launch_append_drafts(const int* base_offsets, const int* base_indices, int BH, int n_pos, int n_new,
                         int* offsets, int* indices, cudaStream_t st, const char** why) {
    const cudaError_t e = launch_pdl(append_drafts_kernel, dim3(BH), dim3(128), 0, st, base_offsets, base_indices, BH,
                                     n_pos, n_new, offsets, indices);
    if (e != cudaSuccess) {
        *why = cudaGetErrorString(e);
        return SDKV_ERR_CUDA;
    }
    return SDKV_OK;
}

int launch_draft_lists(const int* base_offsets, const int* base_indices, int BH, int n_pos, int gamma,
                       long long stride, int* offsets, int* indices, cudaStream_t st, const char** why) {
    const cudaError_t e = launch_pdl(draft_lists_kernel, dim3(BH, gamma), dim3(128), 0, st, base_offsets, base_indices,
                                     BH, n_pos, stride, offsets, indices);
    if (e != cudaSuccess) {
        *why = cudaGetErrorString(e);
        return SDKV_ERR_CUDA;
    }
    return SDKV_OK;
}

int launch_compact_kv(const CompactLaunch& a, const char** why) {
    const int BH = a.B * a.Hkv;
    const long long blocks = (a.rows_cap + kCompactRows - 1) / kCompactRows;
    if (blocks <= 0) return SDKV_OK;
    if (blocks > 0x7fffffffLL) {
        *why = "rows_cap too large";
        return SDKV_ERR_UNSUPPORTED;
    }
    int* status = static_cast<int*>(a.ws);
    const bf16* k = static_cast<const bf16*>(a.k);
    const bf16* v = static_cast<const bf16*>(a.v);
    bf16* ko = static_cast<bf16*>(a.k_out);
    bf16* vo = static_cast<bf16*>(a.v_out);
    if (a.d == 128)
        compact_kv_kernel<128><<<static_cast<int>(blocks), 256, 0, a.stream>>>(
            k, v, a.sb, a.sh, a.sn, a.n_cap, a.Hkv, BH, a.offsets, a.indices, a.rows_cap, ko, vo, status);
    else
        compact_kv_kernel<64><<<static_cast<int>(blocks), 256, 0, a.stream>>>(
            k, v, a.sb, a.sh, a.sn, a.n_cap, a.Hkv, BH, a.offsets, a.indices, a.rows_cap, ko, vo, status);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) {
        *why = cudaGetErrorString(e);
        return SDKV_ERR_CUDA;
    }
    return SDKV_OK;
}

int launch_specvlm(const SpecLaunch& a, const char** why) {
    const int nV = a.v_hi - a.v_lo;
    if (nV > kSpecMaxTokens) {
        *why = "more than 2^20 video tokens";
        return SDKV_ERR_UNSUPPORTED;
    }
    uint8_t* ws = static_cast<uint8_t*>(a.ws);
    SpecParams p{};
    p.importance = a.importance;
    p.n = a.n;
    p.v_lo = a.v_lo;
    p.v_hi = a.v_hi;
    p.keep_lo = a.keep_lo;
    p.keep_hi = a.keep_hi;
    p.cap = nV + (a.keep_hi - a.keep_lo);
    p.lam_r = a.lam_r;
    p.r = a.r;
    p.indices = a.indices;
    p.counts = a.counts;
    p.status = reinterpret_cast<int*>(ws);
    p.keys_in_smem = nV <= kSpecSmemKeys;
    if (!p.keys_in_smem) {
        p.keys_ws = reinterpret_cast<uint32_t*>(ws + kWsHeader);
        p.flags_ws = ws + kWsHeader + align256(sizeof(uint32_t) * static_cast<size_t>(a.B) * nV);
    }
    dim3 grid_imp((a.n + 255) / 256, a.B);
    importance_kernel<<<grid_imp, 256, 0, a.stream>>>(a.scores, a.units, a.n, 1.0f / static_cast<float>(a.units),
                                                      a.importance);
    cudaError_t e = cudaGetLastError();
    if (e == cudaSuccess) {
        const int nW = (nV + 31) / 32;
        const int smem = 4 * nW + (p.keys_in_smem ? 5 * nV : 0);   // bitmap, then keys and flags
        static std::atomic<unsigned long long> attr_set{0};  // one bit per device
        int dev = 0;
        e = cudaGetDevice(&dev);
        if (e == cudaSuccess && !attr_done(attr_set, dev)) {
            e = cudaFuncSetAttribute(specvlm_select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSpecSmemMax);
            if (e == cudaSuccess) attr_mark(attr_set, dev);
        }
        if (e == cudaSuccess) {
            specvlm_select_kernel<<<a.B, kSpecNT, smem, a.stream>>>(p);
            e = cudaGetLastError();
        }
    }
    if (e != cudaSuccess) {
        *why = cudaGetErrorString(e);
        return SDKV_ERR_CUDA;
    }
    return SDKV_OK;
}

}  // namespace sdkv
