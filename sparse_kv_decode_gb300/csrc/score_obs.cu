// Observation-window scoring (StD 3.2 argTopK equation; SparseMM observation
// window): for every KV head h and key j,
//     score[j] = (1/W) sum_{g in group(h)} sum_t P_{g,t}[j],
// P_{g,t} = softmax over the keys window query (g, t) can see.  Each window row
// must be normalised over ALL its visible keys before rows are summed, so the
// keys are read twice:
//   pass 1: per row, the running max m and sum l of 2^(x - m) over the keys
//           (x = scale * log2(e) * q.k); partial (m, l) per key split, merged by
//           the last split CTA of the row block (atomic ticket) into (M, 1/L);
//   pass 2: per key, sum over rows of 2^(x - M) / L.
// Both passes: one producer warp streams K tiles with TMA (128-byte swizzle)
// into an mbarrier ring; four consumer warps each own 32 window rows and run
// QK^T on mma.sync.  A CTA covers 128 rows (one row block) and one key split;
// more rows (large groups or windows) use more row blocks, whose partial key
// sums are added in a fixed order by the last row block (deterministic).
#include "sdkv_common.cuh"
#include "sdkv_internal.h"

#include <algorithm>

namespace sdkv {

struct ScoreParams {
    const bf16* q;
    int B, Hq, Hkv, G, W, R, n, q_pos0, BH, n_mg, nsplit, chunk;
    float scale_log2, inv_w;
    float* scores;
    int* status;
    int* tick1;       // [BH][n_mg]
    int* tick2;       // [BH][nsplit]
    float* st_part;   // [BH][nsplit][R][2]
    float* st_final;  // [BH][R][2]  (M, 1/L)
    float* sc_part;   // [n_mg][BH][n]
};

template <int D>
struct ScoreCfg {
    static constexpr int NCW = 4;                 // consumer warps
    static constexpr int MPW = 2;                 // 16-row tiles per consumer warp
    static constexpr int ROWS = NCW * MPW * 16;   // 128 rows per CTA
    static constexpr int NCT = NCW * 32;
    static constexpr int NT = NCT + 32;
    static constexpr int TK = 64;
    static constexpr int STAGES = 4;
    static constexpr int TILE_B = TK * D * 2;
    static constexpr int QPITCH = 2 * D + 16;
    static constexpr int OFF_K = 0;
    static constexpr int OFF_Q = STAGES * TILE_B;
    static constexpr int OFF_RED = OFF_Q + ROWS * QPITCH;
    static constexpr int OFF_BAR = OFF_RED + 2 * NCW * TK * 4;
    static constexpr int SMEM = OFF_BAR + 2 * STAGES * 8;
    static constexpr int SMEM_ALLOC = SMEM + 1024;
    static_assert(TILE_B % 1024 == 0, "swizzled stage alignment");
};

template <int D, bool PASS2>
__global__ void __launch_bounds__(ScoreCfg<D>::NT)
    score_kernel(const __grid_constant__ ScoreParams p, const __grid_constant__ CUtensorMap tmk) {
    using C = ScoreCfg<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem =
        reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(smem);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const uint32_t bar_full = sbase + C::OFF_BAR;
    const uint32_t bar_empty = bar_full + C::STAGES * 8;
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

    griddep_wait();
    if (tid == 0) {
#pragma unroll
        for (int s = 0; s < C::STAGES; ++s) {
            mbar_init(bar_full + 8 * s, 1);
            mbar_init(bar_empty + 8 * s, C::NCW);
        }
        fence_mbar_init();
        s_abort = 0;
    }
    __syncthreads();
    griddep_launch();

    // ------------------------------------------------------------------ producer
    if (warp == C::NCW) {
        if (lane == 0) {
            prefetch_tmap(&tmk);
            for (int t = 0; t < ntiles; ++t) {
                const int s = t % C::STAGES;
                const uint32_t ph = (t / C::STAGES) & 1;
                if (t >= C::STAGES && !mbar_wait(bar_empty + 8 * s, ph ^ 1)) {
                    flag_status(p.status, SDKV_DEV_TIMEOUT);
                    atomicExch(&s_abort, 1);
                    break;
                }
                mbar_arrive_expect_tx(bar_full + 8 * s, C::TILE_B);
#pragma unroll
                for (int half = 0; half < D / 64; ++half)
                    tma_load_4d(sbase + C::OFF_K + s * C::TILE_B + half * C::TK * 128, &tmk, half * 64,
                                lo + t * C::TK, h, b, bar_full + 8 * s);
            }
        }
        return;
    }

    // ------------------------------------------------------------------ consumers
    const int row_base = mg * C::ROWS;  // first window row (of R = G * W) of this CTA
    uint8_t* qs = smem + C::OFF_Q;
    for (int e = tid; e < C::ROWS * (D / 8); e += C::NCT) {
        const int lr = e / (D / 8), c = e % (D / 8);
        const int r = row_base + lr;
        uint4 val = make_uint4(0u, 0u, 0u, 0u);
        if (r < p.R) {
            const int g = r / p.W, t = r - (r / p.W) * p.W;
            const int hq = h * p.G + g;
            val = *reinterpret_cast<const uint4*>(p.q + ((static_cast<size_t>(b) * p.Hq + hq) * p.W + t) * D +
                                                  c * 8);
        }
        *reinterpret_cast<uint4*>(qs + lr * C::QPITCH + c * 16) = val;
    }
    named_bar_sync(1, C::NCT);

    uint32_t qa[C::MPW][D / 16][4];
#pragma unroll
    for (int mt = 0; mt < C::MPW; ++mt) {
        const int row = warp * (C::MPW * 16) + mt * 16 + (lane & 7) + (((lane >> 3) & 1) << 3);
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks)
            ldsm_x4(qa[mt][ks], pad_addr<C::QPITCH>(sbase + C::OFF_Q, row, 2 * ks + (lane >> 4)));
    }

    // rows of this thread: (mt, i) -> local row warp*32 + mt*16 + lane/4 + 8i
    int lim[C::MPW][2];
    float rM[C::MPW][2], rIL[C::MPW][2];  // pass 2: row max and 1/sum
    float m_r[C::MPW][2], l_r[C::MPW][2]; // pass 1: running stats (this thread's columns)
#pragma unroll
    for (int mt = 0; mt < C::MPW; ++mt) {
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            const int r = row_base + warp * (C::MPW * 16) + mt * 16 + (lane >> 2) + 8 * i;
            const int t = r % p.W;
            lim[mt][i] = (r < p.R) ? p.q_pos0 + t : -1;
            m_r[mt][i] = -INFINITY;
            l_r[mt][i] = 0.f;
            rM[mt][i] = 0.f;
            rIL[mt][i] = 0.f;
            if (PASS2 && r < p.R) {
                const float2 st = __ldcg(reinterpret_cast<const float2*>(p.st_final + (static_cast<size_t>(bh) * p.R + r) * 2));
                rM[mt][i] = st.x;
                rIL[mt][i] = st.y;
            }
        }
    }
    float* red = reinterpret_cast<float*>(smem + C::OFF_RED);  // [2][NCW][TK]
    bool aborted = false;

    for (int t = 0; t < ntiles; ++t) {
        const int s = t % C::STAGES;
        const uint32_t ph = (t / C::STAGES) & 1;
        const bool bad = !mbar_wait(bar_full + 8 * s, ph);
        if (bad) aborted = true;
        if (!PASS2 && bad) break;  // pass 1 has no barrier inside the loop
        const uint32_t kst = sbase + C::OFF_K + s * C::TILE_B;
        float* redb = red + (t & 1) * (C::NCW * C::TK);
#pragma unroll 1
        for (int sub = 0; sub < (bad ? 0 : C::TK / 16); ++sub) {
            const int krow0 = sub * 16;
            float sacc[C::MPW][2][4];
#pragma unroll
            for (int mt = 0; mt < C::MPW; ++mt)
#pragma unroll
                for (int nt = 0; nt < 2; ++nt) sacc[mt][nt][0] = sacc[mt][nt][1] = sacc[mt][nt][2] = sacc[mt][nt][3] = 0.f;
#pragma unroll
            for (int ks = 0; ks < D / 16; ++ks) {
                uint32_t kb[4];
                const int row = krow0 + (lane & 7) + ((lane >> 4) << 3);
                ldsm_x4(kb, sw128_addr<C::TK>(kst, row, 2 * ks + ((lane >> 3) & 1)));
#pragma unroll
                for (int mt = 0; mt < C::MPW; ++mt) {
                    mma_bf16_16816(sacc[mt][0], qa[mt][ks], kb[0], kb[1]);
                    mma_bf16_16816(sacc[mt][1], qa[mt][ks], kb[2], kb[3]);
                }
            }
            const int key0 = lo + t * C::TK + krow0 + 2 * (lane & 3);
            if constexpr (!PASS2) {
#pragma unroll
                for (int mt = 0; mt < C::MPW; ++mt) {
#pragma unroll
                    for (int i = 0; i < 2; ++i) {
                        float x[4];
#pragma unroll
                        for (int q4 = 0; q4 < 4; ++q4) {
                            const int nt = q4 >> 1, e = q4 & 1;
                            const int key = key0 + nt * 8 + e;
                            const bool valid = key < hi && key <= lim[mt][i];
                            x[q4] = valid ? sacc[mt][nt][2 * i + e] * p.scale_log2 : -INFINITY;
                        }
                        const float tmax = fmaxf(fmaxf(x[0], x[1]), fmaxf(x[2], x[3]));
                        const float mnew = fmaxf(m_r[mt][i], tmax);
                        if (mnew != -INFINITY) {
                            l_r[mt][i] = l_r[mt][i] * fast_exp2(m_r[mt][i] - mnew) + fast_exp2(x[0] - mnew) +
                                         fast_exp2(x[1] - mnew) + fast_exp2(x[2] - mnew) + fast_exp2(x[3] - mnew);
                            m_r[mt][i] = mnew;
                        }
                    }
                }
            } else {
                float cs[2][2] = {{0.f, 0.f}, {0.f, 0.f}};  // [nt][e] column sums of this thread
#pragma unroll
                for (int mt = 0; mt < C::MPW; ++mt) {
#pragma unroll
                    for (int i = 0; i < 2; ++i) {
#pragma unroll
                        for (int q4 = 0; q4 < 4; ++q4) {
                            const int nt = q4 >> 1, e = q4 & 1;
                            const int key = key0 + nt * 8 + e;
                            const bool valid = key < hi && key <= lim[mt][i];
                            const float x = sacc[mt][nt][2 * i + e] * p.scale_log2 - rM[mt][i];
                            cs[nt][e] += valid ? fast_exp2(x) * rIL[mt][i] : 0.f;
                        }
                    }
                }
#pragma unroll
                for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        float v = cs[nt][e];
                        v += __shfl_xor_sync(0xffffffffu, v, 4);
                        v += __shfl_xor_sync(0xffffffffu, v, 8);
                        v += __shfl_xor_sync(0xffffffffu, v, 16);
                        cs[nt][e] = v;
                    }
                if (lane < 4) {
#pragma unroll
                    for (int nt = 0; nt < 2; ++nt)
                        *reinterpret_cast<float2*>(redb + warp * C::TK + krow0 + nt * 8 + 2 * lane) =
                            make_float2(cs[nt][0], cs[nt][1]);
                }
            }
        }
        __syncwarp();
        if (lane == 0 && !bad) mbar_arrive(bar_empty + 8 * s);
        if constexpr (PASS2) {
            // one barrier per stage; it also makes a timeout in any warp stop all of them
            if (named_bar_or(1, C::NCT, bad)) break;
            if (tid < C::TK) {
                float v = 0.f;
#pragma unroll
                for (int w = 0; w < C::NCW; ++w) v += redb[w * C::TK + tid];
                const int key = lo + t * C::TK + tid;
                if (key < hi) {
                    if (p.n_mg == 1)
                        p.scores[static_cast<size_t>(bh) * p.n + key] = v * p.inv_w;
                    else
                        p.sc_part[(static_cast<size_t>(mg) * p.BH + bh) * p.n + key] = v;
                }
            }
        }
    }
    if (aborted && lane == 0) flag_status(p.status, SDKV_DEV_TIMEOUT);
    if (named_bar_or(1, C::NCT, aborted || *reinterpret_cast<volatile int*>(&s_abort))) {
        if (tid == 0) {
            for (int s = 0; s < C::STAGES && s < ntiles; ++s) {
                const int last_t = ((ntiles - 1 - s) / C::STAGES) * C::STAGES + s;
                mbar_wait(bar_full + 8 * s, (last_t / C::STAGES) & 1);
            }
        }
        return;
    }

    if constexpr (!PASS2) {
        // merge the quad's column subsets into one (m, l) per row, store the split's partial
#pragma unroll
        for (int mt = 0; mt < C::MPW; ++mt) {
#pragma unroll
            for (int i = 0; i < 2; ++i) {
                float m = m_r[mt][i];
                float M = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 1));
                M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, 2));
                float l = (m == -INFINITY) ? 0.f : l_r[mt][i] * fast_exp2(m - M);
                l += __shfl_xor_sync(0xffffffffu, l, 1);
                l += __shfl_xor_sync(0xffffffffu, l, 2);
                const int r = row_base + warp * (C::MPW * 16) + mt * 16 + (lane >> 2) + 8 * i;
                if ((lane & 3) == 0 && r < p.R)
                    *reinterpret_cast<float2*>(p.st_part + ((static_cast<size_t>(bh) * p.nsplit + sp) * p.R + r) * 2) =
                        make_float2(M, l);
            }
        }
        __threadfence();
        named_bar_sync(1, C::NCT);
        if (tid == 0) {
            const int old = atomicAdd(p.tick1 + bh * p.n_mg + mg, 1);
            s_last = (old == p.nsplit - 1);
        }
        named_bar_sync(1, C::NCT);
        if (!s_last) return;
        __threadfence();
        const int r = row_base + tid;  // one consumer thread per row
        if (tid < C::ROWS && r < p.R) {
            const float* base = p.st_part + (static_cast<size_t>(bh) * p.nsplit * p.R + r) * 2;
            const size_t stride = static_cast<size_t>(p.R) * 2;
            float M = -INFINITY;
            for (int s = 0; s < p.nsplit; ++s) M = fmaxf(M, __ldcg(base + s * stride));
            float L = 0.f;
            for (int s = 0; s < p.nsplit; ++s) {
                const float2 ml = __ldcg(reinterpret_cast<const float2*>(base + s * stride));
                if (ml.x != -INFINITY) L += ml.y * fast_exp2(ml.x - M);
            }
            *reinterpret_cast<float2*>(p.st_final + (static_cast<size_t>(bh) * p.R + r) * 2) =
                make_float2(M, L > 0.f ? 1.f / L : 0.f);
        }
        if (tid == 0) atomicExch(p.tick1 + bh * p.n_mg + mg, 0);
    } else {
        if (p.n_mg == 1) return;
        __threadfence();
        named_bar_sync(1, C::NCT);
        if (tid == 0) {
            const int old = atomicAdd(p.tick2 + bh * p.nsplit + sp, 1);
            s_last = (old == p.n_mg - 1);
        }
        named_bar_sync(1, C::NCT);
        if (!s_last) return;
        __threadfence();
        for (int key = lo + tid; key < hi; key += C::NCT) {
            float v = 0.f;
            for (int g2 = 0; g2 < p.n_mg; ++g2)
                v += __ldcg(p.sc_part + (static_cast<size_t>(g2) * p.BH + bh) * p.n + key);
            p.scores[static_cast<size_t>(bh) * p.n + key] = v * p.inv_w;
        }
        if (tid == 0) atomicExch(p.tick2 + bh * p.nsplit + sp, 0);
    }
}

// =====================================================================================
// host side
// =====================================================================================
namespace {

struct ScorePlan {
    int n_mg, nsplit, chunk;
    size_t off_t1, off_t2, off_sp, off_sf, off_sc, bytes;
};

ScorePlan score_plan(int B, int Hq, int Hkv, int n, int W, int num_sms) {
    ScorePlan pl{};
    const int BH = B * Hkv;
    const int R = (Hq / Hkv) * W;
    constexpr int ROWS = 128, TK = 64;
    pl.n_mg = (R + ROWS - 1) / ROWS;
    const int target = 2 * std::max(num_sms, 1);
    int nsplit = std::max(1, (target + BH * pl.n_mg - 1) / (BH * pl.n_mg));
    nsplit = std::min(nsplit, std::max(1, (n + TK - 1) / TK));
    int chunk = (n + nsplit - 1) / nsplit;
    chunk = ((chunk + TK - 1) / TK) * TK;
    pl.nsplit = (n + chunk - 1) / chunk;
    pl.chunk = chunk;
    size_t off = kWsHeader;
    pl.off_t1 = off;
    off += sizeof(int) * static_cast<size_t>(BH) * pl.n_mg;
    pl.off_t2 = off;
    off += sizeof(int) * static_cast<size_t>(BH) * pl.nsplit;
    off = align256(off);
    pl.off_sp = off;
    off = align256(off + sizeof(float) * 2 * static_cast<size_t>(BH) * pl.nsplit * R);
    pl.off_sf = off;
    off = align256(off + sizeof(float) * 2 * static_cast<size_t>(BH) * R);
    pl.off_sc = off;
    if (pl.n_mg > 1) off = align256(off + sizeof(float) * static_cast<size_t>(pl.n_mg) * BH * n);
    pl.bytes = off;
    return pl;
}

template <int D, bool PASS2>
cudaError_t launch_score_pass(const ScoreParams& p, const CUtensorMap& tmk, int grid, cudaStream_t st) {
    using C = ScoreCfg<D>;
    auto kern = score_kernel<D, PASS2>;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    static unsigned long long attr_set = 0;
    if (dev >= 64 || !(attr_set & (1ull << dev))) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_ALLOC);
        if (e != cudaSuccess) return e;
        if (dev < 64) attr_set |= (1ull << dev);
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
    return cudaLaunchKernelEx(&cfg, kern, p, tmk);
}

}  // namespace

size_t score_ws_bytes(int B, int Hq, int Hkv, int d, int n, int W, int num_sms) {
    (void)d;
    return score_plan(B, Hq, Hkv, n, W, num_sms).bytes;
}

int launch_score(const ScoreLaunch& a, const CUtensorMap* tmk, int num_sms, const char** why) {
    const ScorePlan pl = score_plan(a.B, a.Hq, a.Hkv, a.n, a.W, num_sms);
    if (a.ws_bytes < pl.bytes) {
        *why = "workspace smaller than sdkv_workspace_size(SDKV_OP_SCORE, ...)";
        return SDKV_ERR_WORKSPACE;
    }
    uint8_t* ws = static_cast<uint8_t*>(a.ws);
    ScoreParams p{};
    p.q = static_cast<const bf16*>(a.q_obs);
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
    p.tick1 = reinterpret_cast<int*>(ws + pl.off_t1);
    p.tick2 = reinterpret_cast<int*>(ws + pl.off_t2);
    p.st_part = reinterpret_cast<float*>(ws + pl.off_sp);
    p.st_final = reinterpret_cast<float*>(ws + pl.off_sf);
    p.sc_part = reinterpret_cast<float*>(ws + pl.off_sc);
    const int grid = p.BH * pl.n_mg * pl.nsplit;
    cudaError_t e;
    if (a.d == 128) {
        e = launch_score_pass<128, false>(p, *tmk, grid, a.stream);
        if (e == cudaSuccess) e = launch_score_pass<128, true>(p, *tmk, grid, a.stream);
    } else {
        e = launch_score_pass<64, false>(p, *tmk, grid, a.stream);
        if (e == cudaSuccess) e = launch_score_pass<64, true>(p, *tmk, grid, a.stream);
    }
    if (e != cudaSuccess) {
        *why = cudaGetErrorString(e);
        return SDKV_ERR_CUDA;
    }
    return SDKV_OK;
}

}  // namespace sdkv
