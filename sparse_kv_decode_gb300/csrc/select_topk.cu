// Top-K selection and list assembly (StD 3.2 argTopK; SparseMM K = r + b_score
// with the local window kept apart; ByteCross: sinks + highest-scoring
// entries).  A cluster of 8 CTAs (512 threads each) per (batch, KV head):
//   1. CTA r of the cluster maps its eighth of the candidates' fp32 scores to an
//      order-preserving uint32 key (larger score -> larger key) kept in shared
//      memory;
//   2. four 8-bit radix passes find the K-th largest key T and how many
//      candidates equal to T are taken (need_eq): every CTA counts its keys
//      (per-warp histograms, four lane-skewed copies so that scores crowding
//      into a few exponent bins do not serialise the atomics), the eight CTA
//      histograms are added through distributed shared memory, and every CTA
//      derives the same digit;
//   3. an ordered sweep writes, in ascending index order, every candidate > T
//      and the first need_eq candidates == T (lower indices win ties), each CTA
//      placing its segment after the counts of the lower-ranked CTAs.
// The result is exact: the same fp32 scores always give the same list.
#include "sdkv_common.cuh"
#include "sdkv_internal.h"

namespace sdkv {

namespace {

constexpr int kCS = 8;                          // CTAs per head (portable cluster size)
constexpr int kSelThreads = 512;
constexpr int kSelWarps = kSelThreads / 32;
constexpr int kSkew = 4;                        // histogram copies per warp
constexpr int kSelKeysPerCta = 32 * 1024;       // shared-memory keys per CTA
constexpr int kOffHist = kSelKeysPerCta * 4;
constexpr int kOffCHist = kOffHist + kSelWarps * kSkew * 256 * 4;   // [2][256] this CTA's histogram
constexpr int kOffTot = kOffCHist + 2 * 256 * 4;                      // [256] cluster histogram
constexpr int kOffCnt = kOffTot + 256 * 4;                            // [2] this CTA's (gt, eq)
constexpr int kSelSmem = kOffCnt + 16;

// Order-preserving image of an fp32 score: larger score -> larger key;
// -0.0 equals +0.0; NaN maps to 0, below every number.
__device__ __forceinline__ uint32_t score_key(float f) {
    if (f != f) return 0u;
    if (f == 0.f) f = 0.f;
    const uint32_t u = __float_as_uint(f);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ __forceinline__ uint32_t ld_dsmem_u32(uint32_t addr) {
    uint32_t v;
    asm volatile("ld.shared::cluster.u32 %0, [%1];" : "=r"(v) : "r"(addr) : "memory");
    return v;
}

__global__ void __cluster_dims__(kCS, 1, 1) __launch_bounds__(kSelThreads, 1)
    select_topk_kernel(const float* __restrict__ scores, int n, int cand_lo, int cand_hi, int n_sink,
                       int n_recent, const int* __restrict__ offsets, int* __restrict__ indices, int* status) {
    extern __shared__ __align__(16) uint8_t smem[];
    uint32_t* keys = reinterpret_cast<uint32_t*>(smem);
    unsigned* wh = reinterpret_cast<unsigned*>(smem + kOffHist);     // [warp][copy][256]
    unsigned* chist = reinterpret_cast<unsigned*>(smem + kOffCHist);
    unsigned* tot = reinterpret_cast<unsigned*>(smem + kOffTot);
    unsigned* cnt = reinterpret_cast<unsigned*>(smem + kOffCnt);
    __shared__ unsigned s_digit, s_gt;
    __shared__ unsigned s_wgt[kSelWarps], s_weq[kSelWarps], s_pos[kSelWarps], s_eqt[kSelWarps];
    __shared__ unsigned s_cbase[2];   // (equal keys before this CTA, kept candidates before this CTA)

    const int bh = blockIdx.x / kCS;
    const int rank = static_cast<int>(cluster_ctarank());
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    griddep_wait();
    griddep_launch();

    // every decision up to the sweep depends on the head only: uniform in the cluster
    const int start = offsets[bh];
    const int kh = offsets[bh + 1] - start;
    const int ncand = cand_hi - cand_lo;
    const int K = kh - n_sink - n_recent;
    if (K < 0 || K > ncand) {
        if (rank == 0 && tid == 0) flag_status(status, SDKV_DEV_BAD_LIST);
        return;
    }
    int* out = indices + start;
    if (rank == 0) {
        for (int i = tid; i < n_sink; i += kSelThreads) out[i] = i;
        for (int i = tid; i < n_recent; i += kSelThreads) out[n_sink + K + i] = n - n_recent + i;
    }
    if (K == 0) return;
    const int seg = ((ncand + kCS - 1) / kCS + 31) & ~31;
    const int c0 = min(rank * seg, ncand), c1 = min(c0 + seg, ncand);
    const int len = c1 - c0;
    if (K == ncand) {
        for (int i = tid; i < len; i += kSelThreads) out[n_sink + c0 + i] = cand_lo + c0 + i;
        return;
    }
    const float* sc = scores + static_cast<size_t>(bh) * n + cand_lo + c0;
    for (int i0 = tid; i0 < len; i0 += 16 * kSelThreads) {   // 16 loads in flight per thread
        float v[16];
#pragma unroll
        for (int u = 0; u < 16; ++u) {
            const int i = i0 + u * kSelThreads;
            v[u] = (i < len) ? __ldg(sc + i) : 0.f;
        }
#pragma unroll
        for (int u = 0; u < 16; ++u) {
            const int i = i0 + u * kSelThreads;
            if (i < len) keys[i] = score_key(v[u]);
        }
    }

    // ---- radix select of the K-th largest key, 8 bits per pass
    uint32_t prefix = 0, pmask = 0;
    unsigned krem = static_cast<unsigned>(K);
    unsigned* myh = wh + warp * kSkew * 256 + (lane & (kSkew - 1)) * 256;
    int pass = 0;
#pragma unroll 1
    for (int sh = 24; sh >= 0; sh -= 8, ++pass) {
        for (int i = lane; i < kSkew * 256; i += 32) wh[warp * kSkew * 256 + i] = 0u;
        __syncthreads();
#pragma unroll 4
        for (int i = tid; i < len; i += kSelThreads) {
            const uint32_t u = keys[i];
            if ((u & pmask) == prefix) atomicAdd(&myh[(u >> sh) & 0xffu], 1u);
        }
        __syncthreads();
        unsigned* ch = chist + (pass & 1) * 256;   // alternating: peers read the previous one
        if (tid < 256) {
            unsigned c = 0;
#pragma unroll 8
            for (int w = 0; w < kSelWarps * kSkew; ++w) c += wh[w * 256 + tid];
            ch[tid] = c;
        }
        cluster_sync_all();   // every CTA's histogram of this pass is complete
        if (tid < 256) {
            const uint32_t a = smem_u32(ch + tid);
            unsigned c = 0;
#pragma unroll
            for (int r = 0; r < kCS; ++r) c += ld_dsmem_u32(dsmem_addr(a, r));
            tot[tid] = c;
        }
        __syncthreads();
        if (warp == 0) {
            // lane owns digits 255 - 8*lane .. 248 - 8*lane (descending)
            unsigned cnt8[8], sum = 0;
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                cnt8[j] = tot[255 - 8 * lane - j];
                sum += cnt8[j];
            }
            unsigned incl = sum;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const unsigned y = __shfl_up_sync(0xffffffffu, incl, o);
                if (lane >= o) incl += y;
            }
            unsigned gt = incl - sum;   // keys with a larger digit than this lane's first
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                if (gt < krem && krem <= gt + cnt8[j]) {
                    s_digit = 255 - 8 * lane - j;
                    s_gt = gt;
                }
                gt += cnt8[j];
            }
        }
        __syncthreads();
        prefix |= s_digit << sh;
        pmask |= 0xffu << sh;
        krem -= s_gt;
    }
    const uint32_t T = prefix;
    const unsigned need_eq = krem;  // >= 1 candidates equal to T are taken in all

    // ---- ordered sweep: warp w owns [w*wseg, (w+1)*wseg) of this CTA's segment
    const int wseg = ((len + kSelWarps - 1) / kSelWarps + 31) & ~31;
    const int w0 = min(warp * wseg, len), w1 = min(w0 + wseg, len);
    unsigned ngt = 0, neq = 0;
#pragma unroll 4
    for (int i = w0 + lane; i < w1; i += 32) {
        const uint32_t u = keys[i];
        ngt += (u > T);
        neq += (u == T);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        ngt += __shfl_xor_sync(0xffffffffu, ngt, o);
        neq += __shfl_xor_sync(0xffffffffu, neq, o);
    }
    if (lane == 0) {
        s_wgt[warp] = ngt;
        s_weq[warp] = neq;
    }
    __syncthreads();
    if (tid == 0) {
        unsigned g = 0, e = 0;
        for (int w = 0; w < kSelWarps; ++w) {
            g += s_wgt[w];
            e += s_weq[w];
        }
        cnt[0] = g;
        cnt[1] = e;
    }
    cluster_sync_all();   // every CTA's (gt, eq) is visible
    if (tid == 0) {
        // the CTAs of lower rank hold the earlier candidates
        unsigned eq_before = 0, kept_before = 0;
        const uint32_t a = smem_u32(cnt);
        for (int r = 0; r < rank; ++r) {
            const unsigned g = ld_dsmem_u32(dsmem_addr(a, r));
            const unsigned e = ld_dsmem_u32(dsmem_addr(a + 4, r));
            const unsigned take = (need_eq > eq_before) ? min(e, need_eq - eq_before) : 0u;
            kept_before += g + take;
            eq_before += e;
        }
        s_cbase[0] = eq_before;
        s_cbase[1] = kept_before;
    }
    __syncthreads();
    if (warp == 0) {
        const unsigned eqw = lane < kSelWarps ? s_weq[lane] : 0u;
        const unsigned gtw = lane < kSelWarps ? s_wgt[lane] : 0u;
        unsigned eq_incl = eqw;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const unsigned y = __shfl_up_sync(0xffffffffu, eq_incl, o);
            if (lane >= o) eq_incl += y;
        }
        const unsigned eq_before = s_cbase[0] + eq_incl - eqw;
        const unsigned eq_take = (need_eq > eq_before) ? min(eqw, need_eq - eq_before) : 0u;
        const unsigned sel = gtw + eq_take;
        unsigned sel_incl = sel;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const unsigned y = __shfl_up_sync(0xffffffffu, sel_incl, o);
            if (lane >= o) sel_incl += y;
        }
        if (lane < kSelWarps) {
            s_pos[lane] = s_cbase[1] + sel_incl - sel;
            s_eqt[lane] = eq_take;
        }
    }
    __syncthreads();
    unsigned pos = s_pos[warp];
    const unsigned eq_take = s_eqt[warp];
    unsigned eq_seen = 0;
    const unsigned lt = (1u << lane) - 1u;
    for (int i0 = w0; i0 < w1; i0 += 32) {
        const int i = i0 + lane;
        const bool inb = i < w1;
        const uint32_t u = inb ? keys[i] : 0u;
        const bool is_eq = inb && u == T;
        const unsigned eqf = __ballot_sync(0xffffffffu, is_eq);
        const bool take = inb && (u > T || (is_eq && eq_seen + __popc(eqf & lt) < eq_take));
        const unsigned tf = __ballot_sync(0xffffffffu, take);
        if (take) out[n_sink + pos + __popc(tf & lt)] = cand_lo + c0 + i;
        pos += __popc(tf);
        eq_seen += __popc(eqf);
    }
    cluster_sync_all();   // peers may leave once everyone has read their counts
}

}  // namespace

size_t select_ws_bytes(int B, int Hkv, int n) {
    (void)B;
    (void)Hkv;
    (void)n;
    return kWsHeader;
}

int launch_select(const SelectLaunch& a, const char** why) {
    if (a.cand_hi - a.cand_lo > kCS * kSelKeysPerCta) {
        *why = "more than 262144 candidates per head";
        return SDKV_ERR_UNSUPPORTED;
    }
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    static unsigned long long attr_set = 0;
    if (e == cudaSuccess && (dev >= 64 || !(attr_set & (1ull << dev)))) {
        e = cudaFuncSetAttribute(select_topk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSelSmem);
        if (e == cudaSuccess && dev < 64) attr_set |= (1ull << dev);
    }
    if (e != cudaSuccess) {
        *why = cudaGetErrorString(e);
        return SDKV_ERR_CUDA;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(a.B * a.Hkv * kCS);
    cfg.blockDim = dim3(kSelThreads);
    cfg.dynamicSmemBytes = kSelSmem;
    cfg.stream = a.stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, select_topk_kernel, a.scores, a.n, a.cand_lo, a.cand_hi, a.n_sink, a.n_recent,
                           a.offsets, a.indices, static_cast<int*>(a.ws));
    if (e != cudaSuccess) {
        *why = cudaGetErrorString(e);
        return SDKV_ERR_CUDA;
    }
    return SDKV_OK;
}

}  // namespace sdkv
