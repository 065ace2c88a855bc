// Top-K selection and list assembly (StD 3.2 argTopK; SparseMM K = r + b_score
// with the local window kept apart; ByteCross: sinks + highest-scoring
// entries).  One CTA of 1024 threads per (batch, KV head):
//   1. radix select (11 + 11 + 10 bits) on an order-preserving uint32 image of
//      the fp32 scores finds the K-th largest key T and how many candidates
//      equal to T are taken (need_eq);
//   2. a single ordered sweep over the candidates writes, in ascending index
//      order, every candidate > T and the first need_eq candidates == T (the
//      lower indices win ties), next to the sinks and the recent window.
// The result is exact: the same fp32 scores always give the same list.
#include "sdkv_common.cuh"
#include "sdkv_internal.h"

namespace sdkv {

namespace {

constexpr int kSelThreads = 1024;
constexpr int kSelItems = 8;  // consecutive candidates per thread per sweep tile

// Order-preserving image of an fp32 score: larger score -> larger key;
// -0.0 equals +0.0; NaN maps to 0, below every number.
__device__ __forceinline__ uint32_t score_key(float f) {
    if (f != f) return 0u;
    if (f == 0.f) f = 0.f;
    const uint32_t u = __float_as_uint(f);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// inclusive scan over the block; returns the exclusive prefix, total in `total`
__device__ __forceinline__ unsigned block_scan_u32(unsigned v, unsigned* s_warp, unsigned& total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    unsigned x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const unsigned y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) s_warp[warp] = x;
    __syncthreads();
    if (warp == 0) {
        unsigned w = s_warp[lane];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const unsigned y = __shfl_up_sync(0xffffffffu, w, o);
            if (lane >= o) w += y;
        }
        s_warp[lane] = w;
    }
    __syncthreads();
    const unsigned res = (warp ? s_warp[warp - 1] : 0u) + x - v;
    total = s_warp[31];
    __syncthreads();
    return res;
}

__global__ void __launch_bounds__(kSelThreads)
    select_topk_kernel(const float* __restrict__ scores, int n, int cand_lo, int cand_hi, int n_sink,
                       int n_recent, const int* __restrict__ offsets, int* __restrict__ indices, int* status) {
    __shared__ unsigned hist[2048];
    __shared__ unsigned s_warp[32];
    __shared__ unsigned s_digit, s_gt;

    const int bh = blockIdx.x;
    const int tid = threadIdx.x;
    griddep_wait();
    griddep_launch();

    const int start = offsets[bh];
    const int kh = offsets[bh + 1] - start;
    const int ncand = cand_hi - cand_lo;
    const int K = kh - n_sink - n_recent;
    if (K < 0 || K > ncand) {
        if (tid == 0) flag_status(status, SDKV_DEV_BAD_LIST);
        return;
    }
    int* out = indices + start;
    for (int i = tid; i < n_sink; i += kSelThreads) out[i] = i;
    for (int i = tid; i < n_recent; i += kSelThreads) out[n_sink + K + i] = n - n_recent + i;
    if (K == 0) return;
    const float* sc = scores + static_cast<size_t>(bh) * n + cand_lo;
    if (K == ncand) {
        for (int i = tid; i < ncand; i += kSelThreads) out[n_sink + i] = cand_lo + i;
        return;
    }

    // ---- radix select of the K-th largest key
    uint32_t prefix = 0, pmask = 0;
    unsigned krem = static_cast<unsigned>(K);
    const int shifts[3] = {21, 10, 0};
    const int widths[3] = {11, 11, 10};
#pragma unroll 1
    for (int pass = 0; pass < 3; ++pass) {
        const int sh = shifts[pass];
        const uint32_t dmask = (1u << widths[pass]) - 1u;
        for (int i = tid; i < 2048; i += kSelThreads) hist[i] = 0u;
        __syncthreads();
        for (int i = tid; i < ncand; i += kSelThreads) {
            const uint32_t u = score_key(__ldg(sc + i));
            if ((u & pmask) == prefix) atomicAdd(&hist[(u >> sh) & dmask], 1u);
        }
        __syncthreads();
        // thread t owns digits 2047-2t and 2046-2t (descending order)
        const int d_hi = 2047 - 2 * tid, d_lo = 2046 - 2 * tid;
        const unsigned c_hi = hist[d_hi], c_lo = hist[d_lo];
        unsigned tot;
        const unsigned gt = block_scan_u32(c_hi + c_lo, s_warp, tot);  // keys with a larger digit
        if (gt < krem && krem <= gt + c_hi) {
            s_digit = d_hi;
            s_gt = gt;
        } else if (gt + c_hi < krem && krem <= gt + c_hi + c_lo) {
            s_digit = d_lo;
            s_gt = gt + c_hi;
        }
        __syncthreads();
        prefix |= s_digit << sh;
        pmask |= dmask << sh;
        krem -= s_gt;
        __syncthreads();
    }
    const uint32_t T = prefix;
    const unsigned need_eq = krem;  // >= 1 candidates equal to T are taken

    // ---- ordered sweep: candidates > T, plus the first need_eq equal to T
    unsigned sel_base = 0, eq_base = 0;
    const int tile = kSelThreads * kSelItems;
#pragma unroll 1
    for (int t0 = 0; t0 < ncand; t0 += tile) {
        const int i0 = t0 + tid * kSelItems;
        uint32_t u[kSelItems];
        unsigned ngt = 0, neq = 0;
#pragma unroll
        for (int q = 0; q < kSelItems; ++q) {
            u[q] = (i0 + q < ncand) ? score_key(__ldg(sc + i0 + q)) : 0u;
            const bool inb = i0 + q < ncand;
            ngt += (inb && u[q] > T);
            neq += (inb && u[q] == T);
        }
        // pack the two counts (each <= 8192) into one scan
        unsigned tot;
        const unsigned excl = block_scan_u32((neq << 16) | ngt, s_warp, tot);
        const unsigned gt_excl = excl & 0xffffu, eq_excl = excl >> 16;
        const unsigned gt_tot = tot & 0xffffu, eq_tot = tot >> 16;
        const unsigned rem_eq = (need_eq > eq_base) ? need_eq - eq_base : 0u;  // equal keys still to take
        unsigned pos = sel_base + gt_excl + min(eq_excl, rem_eq);
        unsigned eq_seen = eq_excl;
#pragma unroll
        for (int q = 0; q < kSelItems; ++q) {
            if (i0 + q >= ncand) break;
            bool take = u[q] > T;
            if (u[q] == T) {
                take = eq_seen < rem_eq;
                ++eq_seen;
            }
            if (take) out[n_sink + pos++] = cand_lo + i0 + q;
        }
        sel_base += gt_tot + min(eq_tot, rem_eq);
        eq_base += eq_tot;
    }
}

}  // namespace

size_t select_ws_bytes(int B, int Hkv, int n) {
    (void)B;
    (void)Hkv;
    (void)n;
    return kWsHeader;
}

int launch_select(const SelectLaunch& a, const char** why) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(a.B * a.Hkv);
    cfg.blockDim = dim3(kSelThreads);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = a.stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e = cudaLaunchKernelEx(&cfg, select_topk_kernel, a.scores, a.n, a.cand_lo, a.cand_hi, a.n_sink,
                                       a.n_recent, a.offsets, a.indices, static_cast<int*>(a.ws));
    if (e != cudaSuccess) {
        *why = cudaGetErrorString(e);
        return SDKV_ERR_CUDA;
    }
    return SDKV_OK;
}

}  // namespace sdkv
