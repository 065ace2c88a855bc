// Top-K selection and list assembly (StD 3.2 argTopK; SparseMM K = r + b_score
// with the local window kept apart; ByteCross: sinks + highest-scoring
// entries).  A cluster of up to 8 CTAs per (batch, KV head), 512 threads each,
// 1024 when a CTA holds many keys:
//   1. CTA r of the cluster maps its eighth of the candidates' fp32 scores to an
//      order-preserving uint32 key (larger score -> larger key) kept in shared
//      memory;
//   2. four 8-bit radix passes find the K-th largest key T and how many
//      candidates equal to T are taken (need_eq).  In each pass every CTA
//      counts the digit of its keys that match the prefix so far in one
//      shared-memory histogram, stores that histogram into a slot of every CTA
//      of the cluster, and after one cluster barrier every CTA adds the eight
//      slots and derives the same digit;
//   3. the kept histograms also give, for every CTA, how many of its keys are
//      above T and equal to T, so each CTA knows where its segment of the list
//      starts without another exchange; an ordered sweep then writes, in
//      ascending index order, every candidate > T and the first need_eq
//      candidates == T (lower indices win ties).
// All cross-CTA traffic is stores into the peers' shared memory ahead of a
// cluster barrier: after the last barrier no CTA touches another's memory, so
// each leaves as soon as its own part of the list is written.
// The result is exact: the same fp32 scores always give the same list.
#include "sdkv_common.cuh"
#include "sdkv_internal.h"

namespace sdkv {

namespace {

constexpr int kMaxCS = 8;                       // CTAs per head at most (portable cluster size)
constexpr int kSelBigCta = 8192;                 // keys per CTA above which a CTA runs 1024 threads
constexpr int kPasses = 4;                      // 8-bit digits of a 32-bit key
constexpr int kSelKeysPerCta = 32 * 1024;       // shared-memory keys per CTA
template <int CS>
struct SelCfg {
    static constexpr int OFF_HIST = kSelKeysPerCta * 4;                 // [2][256] this CTA's histogram
    static constexpr int OFF_RECV = OFF_HIST + 2 * 256 * 4;             // [pass][rank][256] every CTA's
    static constexpr int OFF_TOT = OFF_RECV + kPasses * CS * 256 * 4;   // [256] cluster histogram
    static constexpr int OFF_MBAR = OFF_TOT + 256 * 4;                 // [pass] arrival of the peers' histograms
    static constexpr int SMEM = OFF_MBAR + kPasses * 8;
};

// Order-preserving image of an fp32 score: larger score -> larger key;
// -0.0 equals +0.0; NaN maps to 0, below every number.
__device__ __forceinline__ uint32_t score_key(float f) {
    if (f != f) return 0u;
    if (f == 0.f) f = 0.f;
    const uint32_t u = __float_as_uint(f);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Split cluster barrier: arrive early (releasing this CTA's barrier set-up),
// wait where it matters.
__device__ __forceinline__ void cluster_arrive_release() {
    asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() {
    asm volatile("barrier.cluster.wait.aligned;" ::: "memory");
}

// 16 bytes into a peer's shared memory; their arrival counts on the peer's mbarrier.
__device__ __forceinline__ void st_async_v4(uint32_t remote_addr, uint4 v, uint32_t remote_bar) {
    asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.v4.b32 [%0], {%1, %2, %3, %4}, [%5];" ::"r"(
                     remote_addr),
                 "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w), "r"(remote_bar)
                 : "memory");
}

__device__ __forceinline__ unsigned warp_sum_u32(unsigned v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

__device__ __forceinline__ unsigned warp_excl_scan_u32(unsigned v, int lane) {
    unsigned incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const unsigned y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
    }
    return incl - v;
}

template <int CS, int NT>
__global__ void __cluster_dims__(CS, 1, 1) __launch_bounds__(NT, 1)
    select_topk_kernel(const float* __restrict__ scores, int n, int cand_lo, int cand_hi, int n_sink,
                       int n_recent, const int* __restrict__ offsets, int* __restrict__ indices, int* status) {
    static_assert(NT == 512 || NT == 1024, "two histogram parities of 256 entries take 512 threads");
    constexpr int kSelThreads = NT, kSelWarps = NT / 32;
    extern __shared__ __align__(16) uint8_t smem[];
    uint32_t* keys = reinterpret_cast<uint32_t*>(smem);
    using C = SelCfg<CS>;
    unsigned* hist = reinterpret_cast<unsigned*>(smem + C::OFF_HIST);   // [pass & 1][256]
    unsigned* recv = reinterpret_cast<unsigned*>(smem + C::OFF_RECV);   // [pass][rank][256]
    unsigned* tot = reinterpret_cast<unsigned*>(smem + C::OFF_TOT);
    __shared__ unsigned s_digit[kPasses], s_gt;
    __shared__ unsigned s_rgt[kSelWarps];   // warp w: keys of rank w/2 above the digits of passes 2(w%2), +1
    __shared__ unsigned s_wgt[kSelWarps], s_weq[kSelWarps], s_pos[kSelWarps], s_eqt[kSelWarps];

    const int bh = blockIdx.x / CS;
    const int rank = static_cast<int>(cluster_ctarank());
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    griddep_wait();
    griddep_launch();

    // this CTA's candidates; their first scores are requested before the list
    // sizes so that the two reads overlap
    const int ncand = cand_hi - cand_lo;
    const int seg = ((ncand + CS - 1) / CS + 31) & ~31;
    const int c0 = min(rank * seg, ncand), c1 = min(c0 + seg, ncand);
    const int len = c1 - c0;
    const float* sc = scores + static_cast<size_t>(bh) * n + cand_lo + c0;
    constexpr int kInFlight = 16;
    float v[kInFlight];
#pragma unroll
    for (int u = 0; u < kInFlight; ++u) {
        const int i = tid + u * kSelThreads;
        v[u] = (i < len) ? __ldg(sc + i) : 0.f;
    }

    // every decision up to the sweep depends on the head only: uniform in the cluster
    const int start = offsets[bh];
    const int kh = offsets[bh + 1] - start;
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
    if (K == ncand) {
        for (int i = tid; i < len; i += kSelThreads) out[n_sink + c0 + i] = cand_lo + c0 + i;
        return;
    }
    // Each pass's histograms arrive by asynchronous stores that count bytes on a
    // per-pass mbarrier of the receiver (all CS slots, this CTA's own included).
    // A peer's shared memory may be written only once that peer has started and
    // set up its mbarriers: arrive now, wait before the first store into a peer.
    const uint32_t mbar0 = smem_u32(smem + C::OFF_MBAR);
    if constexpr (CS > 1) {
        if (tid == 0) {
#pragma unroll
            for (int ps = 0; ps < kPasses; ++ps) mbar_init(mbar0 + 8 * ps, 1);
            fence_mbar_init();
#pragma unroll
            for (int ps = 0; ps < kPasses; ++ps) mbar_arrive_expect_tx(mbar0 + 8 * ps, CS * 256 * 4);
        }
        cluster_arrive_release();
    }
#pragma unroll
    for (int u = 0; u < kInFlight; ++u) {
        const int i = tid + u * kSelThreads;
        if (i < len) keys[i] = score_key(v[u]);
    }
    for (int i0 = tid + kInFlight * kSelThreads; i0 < len; i0 += kInFlight * kSelThreads) {
#pragma unroll
        for (int u = 0; u < kInFlight; ++u) {
            const int i = i0 + u * kSelThreads;
            v[u] = (i < len) ? __ldg(sc + i) : 0.f;
        }
#pragma unroll
        for (int u = 0; u < kInFlight; ++u) {
            const int i = i0 + u * kSelThreads;
            if (i < len) keys[i] = score_key(v[u]);
        }
    }
    if (tid < 512) hist[tid] = 0u;   // both parities (2 * 256 entries)
    __syncthreads();

    // ---- radix select of the K-th largest key, 8 bits per pass
    uint32_t prefix = 0, pmask = 0;
    unsigned krem = static_cast<unsigned>(K);
#pragma unroll 1
    for (int pass = 0; pass < kPasses; ++pass) {
        const int sh = 24 - 8 * pass;
        unsigned* h = hist + (pass & 1) * 256;
#pragma unroll 4
        for (int i = tid; i < len; i += kSelThreads) {
            const uint32_t u = keys[i];
            if ((u & pmask) == prefix) atomicAdd(&h[(u >> sh) & 0xffu], 1u);
        }
        __syncthreads();
        if constexpr (CS > 1) {
            if (pass == 0) cluster_wait();   // every CTA of the cluster is running
        }
        if constexpr (CS > 1) {
            if (tid < 64) {
                // this CTA's histogram into slot [pass][rank] of every CTA of the cluster
                const uint4 c4 = *reinterpret_cast<const uint4*>(h + 4 * tid);
                const uint32_t a = smem_u32(recv + (pass * CS + rank) * 256 + 4 * tid);
#pragma unroll
                for (int r = 0; r < CS; ++r) st_async_v4(dsmem_addr(a, r), c4, dsmem_addr(mbar0 + 8 * pass, r));
            } else if (tid >= 256 && tid < 512) {
                hist[((pass + 1) & 1) * 256 + (tid - 256)] = 0u;   // the next pass's histogram
            }
            // every CTA's histogram of this pass has arrived here (bounded wait; a
            // peer that never sends cannot happen with the uniform control flow)
            if (!mbar_wait(mbar0 + 8 * pass, 0) && tid == 0) flag_status(status, SDKV_DEV_TIMEOUT);
        } else {
            if (tid < 256)
                recv[pass * 256 + tid] = h[tid];
            else if (tid < 512)
                hist[((pass + 1) & 1) * 256 + (tid - 256)] = 0u;   // the next pass's histogram
            __syncthreads();
        }
        if (tid < 256) {
            unsigned c = 0;
#pragma unroll
            for (int r = 0; r < CS; ++r) c += recv[(pass * CS + r) * 256 + tid];
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
            unsigned gt = warp_excl_scan_u32(sum, lane);   // keys with a larger digit than this lane's first
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                if (gt < krem && krem <= gt + cnt8[j]) {
                    s_digit[pass] = 255 - 8 * lane - j;
                    s_gt = gt;
                }
                gt += cnt8[j];
            }
        }
        __syncthreads();
        prefix |= s_digit[pass] << sh;
        pmask |= 0xffu << sh;
        krem -= s_gt;
    }
    const uint32_t T = prefix;
    const unsigned need_eq = krem;  // >= 1 candidates equal to T are taken in all

    // ---- where each CTA's segment of the list starts.  A key is above T when,
    // at the first pass where its digit differs from T's, the digit is larger:
    // rank r holds sum over passes p of its slot-p counts of digits > digit_p.
    if (warp < 2 * CS) {
        const int r = warp >> 1, p0 = (warp & 1) * 2;
        unsigned g = 0;
#pragma unroll
        for (int pp = p0; pp < p0 + 2; ++pp) {
            const unsigned dig = s_digit[pp];
            const unsigned* hr = recv + (pp * CS + r) * 256;
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const unsigned d = lane + 32 * j;   // consecutive lanes, consecutive banks
                if (d > dig) g += hr[d];
            }
        }
        g = warp_sum_u32(g);
        if (lane == 0) s_rgt[warp] = g;
    }
    // ---- this CTA's keys above / equal to T, per warp: warp w owns [w*wseg, (w+1)*wseg)
    const int wseg = ((len + kSelWarps - 1) / kSelWarps + 31) & ~31;
    const int w0 = min(warp * wseg, len), w1 = min(w0 + wseg, len);
    unsigned ngt = 0, neq = 0;
#pragma unroll 8
    for (int i = w0 + lane; i < w1; i += 32) {
        const uint32_t u = keys[i];
        ngt += (u > T);
        neq += (u == T);
    }
    ngt = warp_sum_u32(ngt);
    neq = warp_sum_u32(neq);
    if (lane == 0) {
        s_wgt[warp] = ngt;
        s_weq[warp] = neq;
    }
    __syncthreads();
    if (tid == 0) {
        // the CTAs of lower rank hold the earlier candidates, then the warps of
        // this CTA in order (a short serial walk: at most CS + kSelWarps steps)
        unsigned eq_before = 0, kept_before = 0;
        for (int r = 0; r < rank; ++r) {
            const unsigned g = s_rgt[2 * r] + s_rgt[2 * r + 1];
            const unsigned e = recv[((kPasses - 1) * CS + r) * 256 + s_digit[kPasses - 1]];
            const unsigned take = (need_eq > eq_before) ? min(e, need_eq - eq_before) : 0u;
            kept_before += g + take;
            eq_before += e;
        }
        for (int w = 0; w < kSelWarps; ++w) {
            const unsigned eqw = s_weq[w];
            const unsigned eq_take = (need_eq > eq_before) ? min(eqw, need_eq - eq_before) : 0u;
            s_pos[w] = kept_before;
            s_eqt[w] = eq_take;
            kept_before += s_wgt[w] + eq_take;
            eq_before += eqw;
        }
    }
    __syncthreads();
    unsigned pos = s_pos[warp];
    const unsigned eq_take = s_eqt[warp];
    unsigned eq_seen = 0;
    const unsigned lt = (1u << lane) - 1u;
#pragma unroll 8
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
}

}  // namespace

size_t select_ws_bytes(int B, int Hkv, int n) {
    (void)B;
    (void)Hkv;
    (void)n;
    return kWsHeader;
}

namespace {

// CTAs per head: 8 while every head's cluster fits the GPU at once; with more
// heads, fewer per head (down to 1, one CTA and no cluster) so that all heads
// run in about one wave, as long as a CTA's share fits its shared memory.
int select_cluster_size(int BH, int ncand, int num_sms) {
    int cs = kMaxCS;
    while (cs > 1 && static_cast<long long>(BH) * cs > num_sms && (ncand + cs / 2 - 1) / (cs / 2) <= kSelKeysPerCta)
        cs /= 2;
    return cs;
}

template <int CS, int NT>
cudaError_t launch_select_cs(const SelectLaunch& a) {
    using C = SelCfg<CS>;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    static std::atomic<unsigned long long> attr_set{0};  // one bit per device, per instantiation
    if (e == cudaSuccess && !attr_done(attr_set, dev)) {
        e = cudaFuncSetAttribute(select_topk_kernel<CS, NT>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
        if (e == cudaSuccess) attr_mark(attr_set, dev);
    }
    if (e != cudaSuccess) return e;
    return launch_pdl(select_topk_kernel<CS, NT>, dim3(a.B * a.Hkv * CS), dim3(NT), C::SMEM, a.stream, a.scores,
                      a.n, a.cand_lo, a.cand_hi, a.n_sink, a.n_recent, a.offsets, a.indices, static_cast<int*>(a.ws));
}

}  // namespace

int launch_select(const SelectLaunch& a, const char** why) {
    const int ncand = a.cand_hi - a.cand_lo;
    if (ncand > kMaxCS * kSelKeysPerCta) {
        *why = "more than 262144 candidates per head";
        return SDKV_ERR_UNSUPPORTED;
    }
    cudaError_t e = cudaErrorInvalidValue;
    const int cs = select_cluster_size(a.B * a.Hkv, ncand, std::max(a.num_sms, 1));
    // few keys per CTA: 512 threads reach the barriers sooner; many: 1024 count them faster
    const bool big = (ncand + cs - 1) / cs > kSelBigCta;
    switch (cs) {
        case 1: e = big ? launch_select_cs<1, 1024>(a) : launch_select_cs<1, 512>(a); break;
        case 2: e = big ? launch_select_cs<2, 1024>(a) : launch_select_cs<2, 512>(a); break;
        case 4: e = big ? launch_select_cs<4, 1024>(a) : launch_select_cs<4, 512>(a); break;
        default: e = big ? launch_select_cs<8, 1024>(a) : launch_select_cs<8, 512>(a); break;
    }
    if (e != cudaSuccess) {
        *why = cudaGetErrorString(e);
        return SDKV_ERR_CUDA;
    }
    return SDKV_OK;
}

}  // namespace sdkv
