// Kernels around the hot path: list builders, row compaction and the SpecVLM
// token selection.
//
//   window_lists    attention sinks plus the recent window (StD baselines,
//                   "Streaming"; ByteCross "The Attention Baseline")
//   append_drafts   a draft step's lists: the base selection plus the positions
//                   drafted so far (StD 3.1)
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
    const int i = blockIdx.x;
    if (i >= BH) return;
    const int b0 = base_offsets[0];
    const int st = base_offsets[i], len = base_offsets[i + 1] - st;
    const int out0 = (st - b0) + i * n_new;
    if (threadIdx.x == 0) {
        offsets[i] = out0;
        if (i == BH - 1) offsets[BH] = out0 + len + n_new;
    }
    for (int e = threadIdx.x; e < len + n_new; e += blockDim.x)
        indices[out0 + e] = (e < len) ? base_indices[st + e] : n_pos + (e - len);
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
    const long long p0 = static_cast<long long>(blockIdx.x) * kCompactRows;
    const int off0 = __ldg(offsets);
    const long long total = __ldg(offsets + BH) - off0;
    constexpr int CPR = D / 8;                  // 16-byte chunks of a K (or V) row
    constexpr int RPW = 32 / (2 * CPR);         // rows per warp instruction
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int sub = lane / (2 * CPR), cl = lane % (2 * CPR);
    const bool is_v = cl >= CPR;
    const int ch = is_v ? cl - CPR : cl;
    for (int r = warp * RPW + sub; r < kCompactRows; r += (blockDim.x / 32) * RPW) {
        const long long p = p0 + r;
        if (p >= total) break;
        if (p >= rows_cap) {
            flag_status(status, SDKV_DEV_BAD_LIST);
            break;
        }
        // the head holding position p: the first whose list ends after p
        int lo = 0, hi = BH;
        while (lo < hi) {
            const int mid = (lo + hi) >> 1;
            if (__ldg(offsets + mid + 1) - off0 > p) hi = mid; else lo = mid + 1;
        }
        const int i = lo;
        const int b = i / Hkv, h = i - (i / Hkv) * Hkv;
        int idx = indices[off0 + p];
        if (static_cast<unsigned>(idx) >= static_cast<unsigned>(n_cap)) {
            flag_status(status, SDKV_DEV_BAD_INDEX);
            idx = 0;
        }
        const bf16* src = (is_v ? v : k) + b * sb + h * sh + static_cast<long long>(idx) * sn + ch * 8;
        bf16* dst = (is_v ? v_out : k_out) + p * D + ch * 8;
        *reinterpret_cast<uint4*>(dst) = __ldg(reinterpret_cast<const uint4*>(src));
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
    for (int u = 0; u < units; ++u) acc += s[static_cast<size_t>(u) * n];   // units in order
    importance[static_cast<size_t>(b) * n + j] = acc * inv_units;
}

constexpr int kSpecNT = 1024;
constexpr int kSpecSmemKeys = 16384;   // sort in shared memory up to this many keys

struct SpecParams {
    const float* importance;
    int n, v_lo, v_hi, keep_lo, keep_hi, cap;
    double lam_r, r;
    int* indices;
    int* counts;
    int* status;
    unsigned long long* keys_ws;   // [B][N2] when the keys do not fit shared memory
    unsigned char* flags_ws;       // [B][nV]
    int N2;
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

// The mass of a score: the nearest multiple of 2^-32, as an integer.
__device__ __forceinline__ long long mass_of_key(unsigned long long key) {
    const uint32_t bits = ~static_cast<uint32_t>(key >> 32);
    return __double2ll_rn(static_cast<double>(__uint_as_float(bits)) * 4294967296.0);
}

__global__ void __launch_bounds__(kSpecNT, 1) specvlm_select_kernel(const __grid_constant__ SpecParams p) {
    extern __shared__ __align__(16) uint8_t dyn[];
    __shared__ long long s_w[kSpecNT / 32];
    __shared__ int s_first;
    const int b = blockIdx.x, tid = threadIdx.x;
    const int nV = p.v_hi - p.v_lo, N2 = p.N2;
    unsigned long long* keys = p.keys_in_smem ? reinterpret_cast<unsigned long long*>(dyn)
                                              : p.keys_ws + static_cast<size_t>(b) * N2;
    unsigned char* flag = p.flags_ws + static_cast<size_t>(b) * nV;
    const float* a = p.importance + static_cast<size_t>(b) * p.n + p.v_lo;

    // keys: (~score bits, token) ascending = score descending, lower token first;
    // NaN and negative scores count as zero mass; padding sorts last
    for (int e = tid; e < N2; e += kSpecNT) {
        unsigned long long key = ~0ull;
        if (e < nV) {
            float x = a[e];
            if (!(x >= 0.f)) {
                flag_status(p.status, SDKV_DEV_BAD_LIST);
                x = 0.f;
            }
            const uint32_t bits = __float_as_uint(x) & 0x7fffffffu;   // -0 -> +0
            key = (static_cast<unsigned long long>(~bits) << 32) | static_cast<uint32_t>(e);
        }
        keys[e] = key;
    }
    for (int e = tid; e < nV; e += kSpecNT) flag[e] = 0;
    __syncthreads();
    // bitonic sort, ascending
    for (int kk = 2; kk <= N2; kk <<= 1) {
        for (int j = kk >> 1; j > 0; j >>= 1) {
            for (int i = tid; i < N2; i += kSpecNT) {
                const int ixj = i ^ j;
                if (ixj > i) {
                    const unsigned long long x = keys[i], y = keys[ixj];
                    const bool up = (i & kk) == 0;
                    if ((x > y) == up) {
                        keys[i] = y;
                        keys[ixj] = x;
                    }
                }
            }
            __syncthreads();
        }
    }
    // Stage I: prefix masses over the sorted order (each thread a contiguous block)
    const int per = (nV + kSpecNT - 1) / kSpecNT;
    const int i0 = min(nV, tid * per), i1 = min(nV, i0 + per);
    long long local = 0;
    for (int i = i0; i < i1; ++i) local += mass_of_key(keys[i]);
    long long S = 0;
    const long long before = cta_excl_scan(local, s_w, &S);
    const double target = p.lam_r * static_cast<double>(S);
    if (tid == 0) s_first = nV;
    __syncthreads();
    {
        long long acc = before;
        for (int i = i0; i < i1; ++i) {
            acc += mass_of_key(keys[i]);
            if (static_cast<double>(acc) >= target) {
                atomicMin(&s_first, i);
                break;
            }
        }
    }
    __syncthreads();
    const int c = (target <= 0.0) ? 0 : min(nV, s_first + 1);
    for (int i = tid; i < c; i += kSpecNT) flag[static_cast<uint32_t>(keys[i])] = 1;
    __syncthreads();
    // Stage II: leftover ranks in token order, then the walk floor(k I) decided per token
    long long nleft_local = 0;
    for (int e = i0; e < i1; ++e) nleft_local += flag[e] ? 0 : 1;
    long long L = 0;
    const long long rank0 = cta_excl_scan(nleft_local, s_w, &L);
    const double I = static_cast<double>(nV - c) / ((1.0 - p.r) * static_cast<double>(nV));
    long long rho = rank0;
    long long keep_local = 0;
    for (int e = i0; e < i1; ++e) {
        if (!flag[e]) {
            bool take = false;
            if (I > 0.0) {
                const double kc = floor(static_cast<double>(rho) / I);
                for (double kk = fmax(kc - 1.0, 0.0); kk <= kc + 2.0 && !take; kk += 1.0)
                    take = floor(kk * I) == static_cast<double>(rho);
            }
            if (take) flag[e] = 2;
            ++rho;
        }
        keep_local += flag[e] ? 1 : 0;
    }
    __syncthreads();
    long long nkeep = 0;
    const long long out0 = cta_excl_scan(keep_local, s_w, &nkeep);
    // output: the kept tokens ascending, with the always-kept range before or after V
    const int nk = p.keep_hi - p.keep_lo;
    const bool keep_first = p.keep_hi <= p.v_lo;
    int* out = p.indices + static_cast<size_t>(b) * p.cap;
    const long long vbase = keep_first ? nk : 0;
    long long o = vbase + out0;
    for (int e = i0; e < i1; ++e)
        if (flag[e]) out[o++] = p.v_lo + e;
    const long long kbase = keep_first ? 0 : nkeep;
    for (int e = tid; e < nk; e += kSpecNT) out[kbase + e] = p.keep_lo + e;
    if (tid == 0) p.counts[b] = static_cast<int>(nkeep + nk);
}

// ============================================================================ host
namespace {
int pow2_at_least(int x) {
    int v = 1;
    while (v < x) v <<= 1;
    return v;
}
}  // namespace

size_t specvlm_ws_bytes(int B, int nV) {
    const int N2 = pow2_at_least(std::max(nV, 1));
    size_t bytes = kWsHeader;
    if (N2 > kSpecSmemKeys) bytes += align256(sizeof(unsigned long long) * static_cast<size_t>(B) * N2);
    bytes += align256(static_cast<size_t>(B) * std::max(nV, 1));
    return bytes;
}

int launch_window_lists(int B, int Hkv, int n, int n_sink, int n_recent, int* offsets, int* indices,
                        cudaStream_t st, const char** why) {
    const int BH = B * Hkv;
    const int k = std::min(n, n_sink + n_recent);
    const long long work = std::max<long long>(static_cast<long long>(BH) * k, BH + 1);
    const int grid = static_cast<int>((work + 255) / 256);
    window_lists_kernel<<<grid, 256, 0, st>>>(BH, n, n_sink, n_recent, k, offsets, indices);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) {
        *why = cudaGetErrorString(e);
        return SDKV_ERR_CUDA;
    }
    return SDKV_OK;
}

int launch_append_drafts(const int* base_offsets, const int* base_indices, int BH, int n_pos, int n_new,
                         int* offsets, int* indices, cudaStream_t st, const char** why) {
    append_drafts_kernel<<<BH, 128, 0, st>>>(base_offsets, base_indices, BH, n_pos, n_new, offsets, indices);
    const cudaError_t e = cudaGetLastError();
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
    const int N2 = pow2_at_least(std::max(nV, 1));
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
    p.N2 = N2;
    p.keys_in_smem = N2 <= kSpecSmemKeys;
    size_t off = kWsHeader;
    if (!p.keys_in_smem) {
        p.keys_ws = reinterpret_cast<unsigned long long*>(ws + off);
        off += align256(sizeof(unsigned long long) * static_cast<size_t>(a.B) * N2);
    }
    p.flags_ws = ws + off;
    dim3 grid_imp((a.n + 255) / 256, a.B);
    importance_kernel<<<grid_imp, 256, 0, a.stream>>>(a.scores, a.units, a.n, 1.0f / static_cast<float>(a.units),
                                                      a.importance);
    cudaError_t e = cudaGetLastError();
    if (e == cudaSuccess) {
        const int smem = p.keys_in_smem ? N2 * 8 : 0;
        static unsigned long long attr_set = 0;
        int dev = 0;
        e = cudaGetDevice(&dev);
        if (e == cudaSuccess && (dev >= 64 || !(attr_set & (1ull << dev)))) {
            e = cudaFuncSetAttribute(specvlm_select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     kSpecSmemKeys * 8);
            if (e == cudaSuccess && dev < 64) attr_set |= (1ull << dev);
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
