// C ABI of libsdkv: argument checking, head budgets (host), tensor-map setup
// and dispatch to the kernels.  See include/sdkv.h for the contract.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <cmath>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <string>
#include <vector>

#include "../../include/sdkv.h"
#include "sdkv_internal.h"

namespace sdkv {
namespace {

thread_local std::string g_last_error;

int fail(int code, const std::string& msg) {
    g_last_error = msg;
    return code;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int check_kv(const void* k, const void* v, const int64_t s[3], int d) {
    if (!k || (v == nullptr && k == nullptr)) return fail(SDKV_ERR_INVALID_ARG, "null K/V pointer");
    if (!aligned16(k) || (v && !aligned16(v))) return fail(SDKV_ERR_INVALID_ARG, "K/V not 16-byte aligned");
    if (!s) return fail(SDKV_ERR_INVALID_ARG, "null kv_strides");
    for (int i = 0; i < 3; ++i)
        if (s[i] <= 0 || (s[i] % 8) != 0)
            return fail(SDKV_ERR_INVALID_ARG, "kv_strides must be positive multiples of 8 elements");
    if (s[2] < d) return fail(SDKV_ERR_INVALID_ARG, "row stride smaller than d");
    return SDKV_OK;
}

int check_heads(int B, int Hq, int Hkv, int d) {
    if (B <= 0 || Hq <= 0 || Hkv <= 0) return fail(SDKV_ERR_INVALID_ARG, "B, Hq, Hkv must be positive");
    if (Hq % Hkv != 0) return fail(SDKV_ERR_INVALID_ARG, "Hq must be a multiple of Hkv");
    if (d != 64 && d != 128) return fail(SDKV_ERR_UNSUPPORTED, "head dim d must be 64 or 128");
    return SDKV_OK;
}

int check_ws(const void* ws, size_t have, size_t need) {
    if (!ws) return fail(SDKV_ERR_INVALID_ARG, "null workspace");
    if (!aligned16(ws)) return fail(SDKV_ERR_INVALID_ARG, "workspace not 16-byte aligned");
    if (have < need) return fail(SDKV_ERR_WORKSPACE, "workspace smaller than sdkv_workspace_size()");
    return SDKV_OK;
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static std::once_flag once;
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

}  // namespace

DeviceInfo current_device() {
    static std::mutex mu;
    static std::vector<int> sms;
    DeviceInfo info;
    if (cudaGetDevice(&info.device) != cudaSuccess) return info;
    std::lock_guard<std::mutex> lock(mu);
    if (static_cast<int>(sms.size()) <= info.device) sms.resize(info.device + 1, 0);
    if (sms[info.device] == 0) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, info.device) != cudaSuccess) return info;
        sms[info.device] = n;
    }
    info.num_sms = sms[info.device];
    return info;
}

int encode_kv_tmap(CUtensorMap* map, const void* base, int B, int Hkv, int rows, int d, const int64_t strides[3],
                   int box_rows) {
    auto fn = encode_fn();
    if (!fn) return fail(SDKV_ERR_CUDA, "cuTensorMapEncodeTiled not available from the driver");
    cuuint64_t dims[4] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(rows), static_cast<cuuint64_t>(Hkv),
                          static_cast<cuuint64_t>(B)};
    cuuint64_t gstr[3] = {static_cast<cuuint64_t>(strides[2]) * 2, static_cast<cuuint64_t>(strides[1]) * 2,
                          static_cast<cuuint64_t>(strides[0]) * 2};
    cuuint32_t box[4] = {64u, static_cast<cuuint32_t>(box_rows), 1u, 1u};
    cuuint32_t estr[4] = {1u, 1u, 1u, 1u};
    CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims, gstr, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) {
        char msg[96];
        std::snprintf(msg, sizeof(msg), "cuTensorMapEncodeTiled failed (CUresult %d)", static_cast<int>(r));
        return fail(SDKV_ERR_CUDA, msg);
    }
    return SDKV_OK;
}

int encode_rows_tmap(CUtensorMap* map, const void* base, int64_t rows, int d, int box_rows) {
    auto fn = encode_fn();
    if (!fn) return fail(SDKV_ERR_CUDA, "cuTensorMapEncodeTiled not available from the driver");
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(rows)};
    cuuint64_t gstr[1] = {static_cast<cuuint64_t>(d) * 2};
    cuuint32_t box[2] = {64u, static_cast<cuuint32_t>(box_rows)};
    cuuint32_t estr[2] = {1u, 1u};
    CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, gstr, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) {
        char msg[96];
        std::snprintf(msg, sizeof(msg), "cuTensorMapEncodeTiled failed (CUresult %d)", static_cast<int>(r));
        return fail(SDKV_ERR_CUDA, msg);
    }
    return SDKV_OK;
}

}  // namespace sdkv

using namespace sdkv;

extern "C" {

int32_t sdkv_version(void) { return 102; }

const char* sdkv_last_error(void) { return g_last_error.c_str(); }

int sdkv_head_budgets(const float* s, int32_t n_heads, int64_t total_B, int32_t w, double rho, int32_t cap,
                      int32_t* b_out) {
    if (!s || !b_out) return fail(SDKV_ERR_INVALID_ARG, "null pointer");
    if (n_heads <= 0) return fail(SDKV_ERR_INVALID_ARG, "n_heads must be positive");
    if (w < 0) return fail(SDKV_ERR_INVALID_ARG, "w must be >= 0");
    if (!(rho >= 0.0 && rho <= 1.0)) return fail(SDKV_ERR_INVALID_ARG, "rho must lie in [0, 1]");
    const int64_t N = n_heads;
    if (total_B < N * w) return fail(SDKV_ERR_INVALID_ARG, "total budget below n_heads * w");
    if (cap < 0) return fail(SDKV_ERR_INVALID_ARG, "cap must be >= 0");
    if (cap > 0 && static_cast<int64_t>(cap) * N < total_B)
        return fail(SDKV_ERR_INVALID_ARG, "cap * n_heads below the total budget");
    if (total_B / N > 0x7fffffff) return fail(SDKV_ERR_INVALID_ARG, "budget per head exceeds int32");

    // sum of the scores in index order (float64)
    std::vector<double> sc(N);
    double ssum = 0.0;
    for (int64_t i = 0; i < N; ++i) {
        const double x = static_cast<double>(s[i]);
        if (!(x >= 0.0) || !std::isfinite(x)) return fail(SDKV_ERR_INVALID_ARG, "head scores must be finite and >= 0");
        sc[i] = x;
        ssum += x;
    }
    if (ssum == 0.0) {
        std::fill(sc.begin(), sc.end(), 1.0);
        ssum = static_cast<double>(N);
    }
    // r = rho (B - N w) / N ; B_remain = (B - N w) - rho (B - N w)
    const double base = static_cast<double>(total_B) - static_cast<double>(N) * static_cast<double>(w);
    const double r = rho * base / static_cast<double>(N);
    const double b_remain = base - rho * base;
    std::vector<double> bstar(N);
    for (int64_t i = 0; i < N; ++i) bstar[i] = w + r + b_remain * sc[i] / ssum;

    if (cap > 0) {  // move the excess of capped heads to the others, in proportion to s
        std::vector<char> capped(N, 0);
        while (true) {
            double excess = 0.0;
            bool any = false;
            for (int64_t i = 0; i < N; ++i) {
                if (!capped[i] && bstar[i] > cap) {
                    excess += bstar[i] - cap;
                    bstar[i] = cap;
                    capped[i] = 1;
                    any = true;
                }
            }
            if (!any) break;
            double free_s = 0.0;
            int64_t n_free = 0;
            for (int64_t i = 0; i < N; ++i)
                if (!capped[i]) {
                    free_s += sc[i];
                    ++n_free;
                }
            if (n_free == 0) break;
            for (int64_t i = 0; i < N; ++i)
                if (!capped[i]) bstar[i] += excess * (free_s > 0 ? sc[i] / free_s : 1.0 / n_free);
        }
    }
    // largest-remainder apportionment; equal remainders go to the lower index
    std::vector<int64_t> fl(N);
    int64_t fsum = 0;
    for (int64_t i = 0; i < N; ++i) {
        fl[i] = static_cast<int64_t>(std::floor(bstar[i]));
        fsum += fl[i];
    }
    const int64_t missing = total_B - fsum;
    if (missing < 0 || missing > N) return fail(SDKV_ERR_INVALID_ARG, "budget apportionment out of range");
    std::vector<int64_t> order(N);
    for (int64_t i = 0; i < N; ++i) order[i] = i;
    std::stable_sort(order.begin(), order.end(), [&](int64_t a, int64_t b) {
        return (bstar[a] - fl[a]) > (bstar[b] - fl[b]);
    });
    for (int64_t i = 0; i < missing; ++i) fl[order[i]] += 1;
    for (int64_t i = 0; i < N; ++i) b_out[i] = static_cast<int32_t>(fl[i]);
    g_last_error.clear();
    return SDKV_OK;
}

size_t sdkv_workspace_size(int32_t op, int32_t B, int32_t Hq, int32_t Hkv, int32_t d, int32_t n,
                           int32_t gamma_or_W) {
    const DeviceInfo dev = current_device();
    if (dev.num_sms <= 0) return 0;
    switch (op) {
        case SDKV_OP_SCORE:
            if (B <= 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv || n <= 0 || gamma_or_W <= 0) return 0;
            return score_ws_bytes(B, Hq, Hkv, d, n, gamma_or_W, dev.num_sms);
        case SDKV_OP_SELECT:
            if (B <= 0 || Hkv <= 0) return 0;
            return select_ws_bytes(B, Hkv, n);
        case SDKV_OP_SPARSE_DECODE:
            if (B <= 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv) return 0;
            return sparse_ws_bytes(B, Hq, Hkv, d, dev.num_sms);
        case SDKV_OP_DENSE_VERIFY:
            if (B <= 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv || n <= 0 || gamma_or_W <= 0 || n < gamma_or_W) return 0;
            return dense_ws_bytes(B, Hq, Hkv, d, n, gamma_or_W, dev.num_sms);
        case SDKV_OP_COMPACT:
            return SDKV_WS_HEADER_BYTES;
        case SDKV_OP_SPECVLM:
            if (B <= 0 || n < 0 || n > (1 << 20)) return 0;
            return specvlm_ws_bytes(B, n);
        default:
            return 0;
    }
}

int sdkv_score_obs_window(const void* q_obs, const void* k, const int64_t k_strides[3], int32_t B, int32_t Hq,
                          int32_t Hkv, int32_t d, int32_t n, int32_t W, int32_t q_pos0, float scale, float* scores,
                          void* ws, size_t ws_bytes, void* stream) {
    int rc = check_heads(B, Hq, Hkv, d);
    if (rc) return rc;
    if (!q_obs || !scores) return fail(SDKV_ERR_INVALID_ARG, "null q_obs or scores");
    if (!aligned16(q_obs) || !aligned16(scores)) return fail(SDKV_ERR_INVALID_ARG, "q_obs/scores not 16-byte aligned");
    if ((rc = check_kv(k, k, k_strides, d))) return rc;
    if (n <= 0 || W <= 0) return fail(SDKV_ERR_INVALID_ARG, "n and W must be positive");
    if (q_pos0 < 0 || static_cast<int64_t>(q_pos0) + W > n)
        return fail(SDKV_ERR_INVALID_ARG, "window positions must satisfy 0 <= q_pos0 and q_pos0 + W <= n");
    if (static_cast<int64_t>(Hq / Hkv) * W > 4096) return fail(SDKV_ERR_UNSUPPORTED, "(Hq/Hkv) * W must be <= 4096");
    if (!(scale > 0.f) || !std::isfinite(scale)) return fail(SDKV_ERR_INVALID_ARG, "scale must be positive and finite");
    const DeviceInfo dev = current_device();
    if (dev.num_sms <= 0) return fail(SDKV_ERR_CUDA, "no CUDA device");
    if ((rc = check_ws(ws, ws_bytes, score_ws_bytes(B, Hq, Hkv, d, n, W, dev.num_sms)))) return rc;
    CUtensorMap tmk, tmq;
    if ((rc = encode_kv_tmap(&tmk, k, B, Hkv, n, d, k_strides, 128))) return rc;
    if ((rc = encode_rows_tmap(&tmq, q_obs, static_cast<int64_t>(B) * Hq * W, d, 128))) return rc;
    ScoreLaunch a{q_obs, B, Hq, Hkv, d, n, W, q_pos0, scale, scores, ws, ws_bytes, static_cast<cudaStream_t>(stream)};
    const char* why = "";
    rc = launch_score(a, &tmk, &tmq, dev.num_sms, &why);
    if (rc) return fail(rc, why);
    g_last_error.clear();
    return SDKV_OK;
}

int sdkv_select_topk(const float* scores, int32_t B, int32_t Hkv, int32_t n, int32_t cand_lo, int32_t cand_hi,
                     int32_t n_sink, int32_t n_recent, const int32_t* offsets, int32_t* indices, void* ws,
                     size_t ws_bytes, void* stream) {
    if (!scores || !offsets || !indices) return fail(SDKV_ERR_INVALID_ARG, "null pointer");
    if (B <= 0 || Hkv <= 0 || n <= 0) return fail(SDKV_ERR_INVALID_ARG, "B, Hkv, n must be positive");
    if (!(0 <= n_sink && n_sink <= cand_lo && cand_lo <= cand_hi && n_recent >= 0 &&
          static_cast<int64_t>(cand_hi) + n_recent <= n))
        return fail(SDKV_ERR_INVALID_ARG, "need 0 <= n_sink <= cand_lo <= cand_hi <= n - n_recent");
    if (static_cast<int64_t>(B) * Hkv > 0x7fffffff) return fail(SDKV_ERR_INVALID_ARG, "too many heads");
    int rc = check_ws(ws, ws_bytes, select_ws_bytes(B, Hkv, n));
    if (rc) return rc;
    const DeviceInfo dev = current_device();
    if (dev.num_sms <= 0) return fail(SDKV_ERR_CUDA, "no CUDA device");
    SelectLaunch a{scores, B, Hkv, n, cand_lo, cand_hi, n_sink, n_recent, offsets, indices, ws,
                   static_cast<cudaStream_t>(stream), dev.num_sms};
    const char* why = "";
    rc = launch_select(a, &why);
    if (rc) return fail(rc, why);
    g_last_error.clear();
    return SDKV_OK;
}

int sdkv_sparse_decode_attn(const void* q, const void* k, const void* v, const int64_t kv_strides[3], int32_t n_cap,
                            const int32_t* offsets, const int32_t* indices, int64_t n_idx, int32_t B, int32_t Hq,
                            int32_t Hkv, int32_t d, float scale, void* o, float* lse, void* ws, size_t ws_bytes,
                            void* stream) {
    int rc = check_heads(B, Hq, Hkv, d);
    if (rc) return rc;
    if (!q || !o || !offsets || !indices) return fail(SDKV_ERR_INVALID_ARG, "null pointer");
    if (!aligned16(q) || !aligned16(o)) return fail(SDKV_ERR_INVALID_ARG, "q/o not 16-byte aligned");
    if (!v) return fail(SDKV_ERR_INVALID_ARG, "null V pointer");
    if ((rc = check_kv(k, v, kv_strides, d))) return rc;
    if (n_cap <= 0) return fail(SDKV_ERR_INVALID_ARG, "n_cap must be positive");
    if (n_idx < 0) return fail(SDKV_ERR_INVALID_ARG, "n_idx must be >= 0");
    if (Hq / Hkv > 32) return fail(SDKV_ERR_UNSUPPORTED, "Hq/Hkv must be <= 32");
    if (static_cast<int64_t>(B) * Hkv > 65536) return fail(SDKV_ERR_UNSUPPORTED, "B*Hkv must be <= 65536");
    if (!std::isfinite(scale)) return fail(SDKV_ERR_INVALID_ARG, "scale must be finite");
    const DeviceInfo dev = current_device();
    if (dev.num_sms <= 0) return fail(SDKV_ERR_CUDA, "no CUDA device");
    if ((rc = check_ws(ws, ws_bytes, sparse_ws_bytes(B, Hq, Hkv, d, dev.num_sms)))) return rc;
    AttnLaunch a{};
    a.q = q;
    a.k = k;
    a.v = v;
    a.sb = kv_strides[0];
    a.sh = kv_strides[1];
    a.sn = kv_strides[2];
    a.B = B;
    a.Hq = Hq;
    a.Hkv = Hkv;
    a.d = d;
    a.gamma = 1;
    a.o = o;
    a.lse = lse;
    a.scale = scale;
    a.offsets = offsets;
    a.indices = indices;
    a.n_idx = n_idx;
    a.n_cap = n_cap;
    a.ws = ws;
    a.ws_bytes = ws_bytes;
    a.stream = static_cast<cudaStream_t>(stream);
    const char* why = "";
    rc = launch_sparse_decode(a, dev.num_sms, &why);
    if (rc) return fail(rc, why);
    g_last_error.clear();
    return SDKV_OK;
}

int sdkv_dense_verify_attn(const void* q, const void* k, const void* v, const int64_t kv_strides[3], int32_t B,
                           int32_t Hq, int32_t Hkv, int32_t d, int32_t n_prefix, int32_t gamma, float scale, void* o,
                           float* lse, void* ws, size_t ws_bytes, void* stream) {
    int rc = check_heads(B, Hq, Hkv, d);
    if (rc) return rc;
    if (!q || !o) return fail(SDKV_ERR_INVALID_ARG, "null q or o");
    if (!aligned16(q) || !aligned16(o)) return fail(SDKV_ERR_INVALID_ARG, "q/o not 16-byte aligned");
    if (!v) return fail(SDKV_ERR_INVALID_ARG, "null V pointer");
    if ((rc = check_kv(k, v, kv_strides, d))) return rc;
    if (n_prefix < 0 || gamma < 1) return fail(SDKV_ERR_INVALID_ARG, "need n_prefix >= 0 and gamma >= 1");
    if (static_cast<int64_t>(n_prefix) + gamma > 0x7fffffff) return fail(SDKV_ERR_INVALID_ARG, "cache too long");
    if (static_cast<int64_t>(Hq / Hkv) * gamma > 64) return fail(SDKV_ERR_UNSUPPORTED, "(Hq/Hkv) * gamma must be <= 64");
    if (!std::isfinite(scale)) return fail(SDKV_ERR_INVALID_ARG, "scale must be finite");
    const DeviceInfo dev = current_device();
    if (dev.num_sms <= 0) return fail(SDKV_ERR_CUDA, "no CUDA device");
    const int n_total = n_prefix + gamma;
    if ((rc = check_ws(ws, ws_bytes, dense_ws_bytes(B, Hq, Hkv, d, n_total, gamma, dev.num_sms)))) return rc;
    CUtensorMap tmk, tmv;
    if ((rc = encode_kv_tmap(&tmk, k, B, Hkv, n_total, d, kv_strides, 64))) return rc;
    if ((rc = encode_kv_tmap(&tmv, v, B, Hkv, n_total, d, kv_strides, 64))) return rc;
    AttnLaunch a{};
    a.q = q;
    a.k = k;
    a.v = v;
    a.sb = kv_strides[0];
    a.sh = kv_strides[1];
    a.sn = kv_strides[2];
    a.B = B;
    a.Hq = Hq;
    a.Hkv = Hkv;
    a.d = d;
    a.gamma = gamma;
    a.o = o;
    a.lse = lse;
    a.scale = scale;
    a.n_prefix = n_prefix;
    a.ws = ws;
    a.ws_bytes = ws_bytes;
    a.stream = static_cast<cudaStream_t>(stream);
    const char* why = "";
    rc = launch_dense_verify(a, &tmk, &tmv, dev.num_sms, &why);
    if (rc) return fail(rc, why);
    g_last_error.clear();
    return SDKV_OK;
}

int sdkv_dense_verify_attn_noalloc(const void* q, const void* k, const void* v, const int64_t kv_strides[3],
                                   int32_t B, int32_t Hq, int32_t Hkv, int32_t d, int32_t n_prefix, int32_t gamma,
                                   float scale, void* o, float* lse, void* stream) {
    int rc = check_heads(B, Hq, Hkv, d);
    if (rc) return rc;
    if (!q || !o) return fail(SDKV_ERR_INVALID_ARG, "null q or o");
    if (!aligned16(q) || !aligned16(o)) return fail(SDKV_ERR_INVALID_ARG, "q/o not 16-byte aligned");
    if (!v) return fail(SDKV_ERR_INVALID_ARG, "null V pointer");
    if ((rc = check_kv(k, v, kv_strides, d))) return rc;
    if (n_prefix < 0 || gamma < 1) return fail(SDKV_ERR_INVALID_ARG, "need n_prefix >= 0 and gamma >= 1");
    if (static_cast<int64_t>(n_prefix) + gamma > 0x7fffffff) return fail(SDKV_ERR_INVALID_ARG, "cache too long");
    if (static_cast<int64_t>(Hq / Hkv) * gamma > 64) return fail(SDKV_ERR_UNSUPPORTED, "(Hq/Hkv) * gamma must be <= 64");
    if (!std::isfinite(scale)) return fail(SDKV_ERR_INVALID_ARG, "scale must be finite");
    const DeviceInfo dev = current_device();
    if (dev.num_sms <= 0) return fail(SDKV_ERR_CUDA, "no CUDA device");
    const int n_total = n_prefix + gamma;
    CUtensorMap tmk, tmv;
    if ((rc = encode_kv_tmap(&tmk, k, B, Hkv, n_total, d, kv_strides, 64))) return rc;
    if ((rc = encode_kv_tmap(&tmv, v, B, Hkv, n_total, d, kv_strides, 64))) return rc;
    AttnLaunch a{};
    a.q = q;
    a.k = k;
    a.v = v;
    a.sb = kv_strides[0];
    a.sh = kv_strides[1];
    a.sn = kv_strides[2];
    a.B = B;
    a.Hq = Hq;
    a.Hkv = Hkv;
    a.d = d;
    a.gamma = gamma;
    a.o = o;
    a.lse = lse;
    a.scale = scale;
    a.n_prefix = n_prefix;
    a.stream = static_cast<cudaStream_t>(stream);
    const char* why = "";
    rc = dense_verify_noalloc(a, &tmk, &tmv, dev.num_sms, &why);
    if (rc) return fail(rc, why);
    g_last_error.clear();
    return SDKV_OK;
}

int sdkv_dense_verify_attn_noalloc_status(int32_t* status, void* stream) {
    if (!status) return fail(SDKV_ERR_INVALID_ARG, "null pointer");
    const char* why = "";
    const int rc = noalloc_status(status, static_cast<cudaStream_t>(stream), &why);
    if (rc) return fail(rc, why);
    g_last_error.clear();
    return SDKV_OK;
}

int sdkv_workspace_status(void* ws, int32_t* status, void* stream) {
    if (!ws || !status) return fail(SDKV_ERR_INVALID_ARG, "null pointer");
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    cudaError_t e = cudaMemcpyAsync(status, ws, sizeof(int32_t), cudaMemcpyDeviceToHost, st);
    if (e == cudaSuccess) e = cudaStreamSynchronize(st);
    if (e == cudaSuccess) e = cudaMemsetAsync(ws, 0, sizeof(int32_t), st);
    if (e == cudaSuccess) e = cudaStreamSynchronize(st);
    if (e != cudaSuccess) return fail(SDKV_ERR_CUDA, cudaGetErrorString(e));
    g_last_error.clear();
    return SDKV_OK;
}


// ----------------------------------------------------------------------------------------
// next rows
// ----------------------------------------------------------------------------------------
int sdkv_window_lists(int32_t B, int32_t Hkv, int32_t n, int32_t n_sink, int32_t n_recent, int32_t* offsets,
                      int32_t* indices, void* stream) {
    if (!offsets || !indices) return fail(SDKV_ERR_INVALID_ARG, "null pointer");
    if (B <= 0 || Hkv <= 0 || n < 0 || n_sink < 0 || n_recent < 0)
        return fail(SDKV_ERR_INVALID_ARG, "need B, Hkv > 0 and n, n_sink, n_recent >= 0");
    const int64_t k = std::min<int64_t>(n, static_cast<int64_t>(n_sink) + n_recent);
    if (static_cast<int64_t>(B) * Hkv * k > 0x7fffffff) return fail(SDKV_ERR_INVALID_ARG, "lists too long");
    const char* why = "";
    const int rc = launch_window_lists(B, Hkv, n, n_sink, n_recent, offsets, indices,
                                       static_cast<cudaStream_t>(stream), &why);
    if (rc) return fail(rc, why);
    g_last_error.clear();
    return SDKV_OK;
}

int sdkv_append_drafts(const int32_t* base_offsets, const int32_t* base_indices, int32_t BH, int32_t n_pos,
                       int32_t n_new, int32_t* offsets, int32_t* indices, void* stream) {
    if (!base_offsets || !base_indices || !offsets || !indices) return fail(SDKV_ERR_INVALID_ARG, "null pointer");
    if (BH <= 0 || n_pos < 0 || n_new < 0) return fail(SDKV_ERR_INVALID_ARG, "need BH > 0 and n_pos, n_new >= 0");
    if (offsets == base_offsets || indices == base_indices)
        return fail(SDKV_ERR_INVALID_ARG, "output lists must not alias the base lists");
    const char* why = "";
    const int rc = launch_append_drafts(base_offsets, base_indices, BH, n_pos, n_new, offsets, indices,
                                        static_cast<cudaStream_t>(stream), &why);
    if (rc) return fail(rc, why);
    g_last_error.clear();
    return SDKV_OK;
}

int sdkv_draft_lists(const int32_t* base_offsets, const int32_t* base_indices, int32_t BH, int32_t n_pos,
                     int32_t gamma, int64_t stride, int32_t* offsets, int32_t* indices, void* stream) {
    if (!base_offsets || !base_indices || !offsets || !indices) return fail(SDKV_ERR_INVALID_ARG, "null pointer");
    if (BH <= 0 || n_pos < 0 || gamma <= 0 || gamma > 65535 || stride <= 0)
        return fail(SDKV_ERR_INVALID_ARG, "need BH > 0, n_pos >= 0, 0 < gamma <= 65535, stride > 0");
    if (offsets == base_offsets || indices == base_indices)
        return fail(SDKV_ERR_INVALID_ARG, "output lists must not alias the base lists");
    const char* why = "";
    const int rc = launch_draft_lists(base_offsets, base_indices, BH, n_pos, gamma, stride, offsets, indices,
                                      static_cast<cudaStream_t>(stream), &why);
    if (rc) return fail(rc, why);
    g_last_error.clear();
    return SDKV_OK;
}

int sdkv_compact_kv(const void* k, const void* v, const int64_t kv_strides[3], int32_t n_cap,
                    const int32_t* offsets, const int32_t* indices, int32_t B, int32_t Hkv, int32_t d,
                    int64_t rows_cap, void* k_out, void* v_out, void* ws, size_t ws_bytes, void* stream) {
    if (B <= 0 || Hkv <= 0) return fail(SDKV_ERR_INVALID_ARG, "B and Hkv must be positive");
    if (d != 64 && d != 128) return fail(SDKV_ERR_UNSUPPORTED, "head dim must be 64 or 128");
    if (!offsets || !indices || !k_out || !v_out) return fail(SDKV_ERR_INVALID_ARG, "null pointer");
    if (!aligned16(k_out) || !aligned16(v_out)) return fail(SDKV_ERR_INVALID_ARG, "k_out/v_out not 16-byte aligned");
    int rc = check_kv(k, v, kv_strides, d);
    if (rc) return rc;
    if (n_cap <= 0 || rows_cap < 0) return fail(SDKV_ERR_INVALID_ARG, "need n_cap > 0 and rows_cap >= 0");
    if ((rc = check_ws(ws, ws_bytes, SDKV_WS_HEADER_BYTES))) return rc;
    CompactLaunch a{k, v, kv_strides[0], kv_strides[1], kv_strides[2], n_cap, B, Hkv, d, offsets, indices,
                    rows_cap, k_out, v_out, ws, static_cast<cudaStream_t>(stream)};
    const char* why = "";
    rc = launch_compact_kv(a, &why);
    if (rc) return fail(rc, why);
    g_last_error.clear();
    return SDKV_OK;
}

int sdkv_sparse_decode_compact(const void* q, const void* k_c, const void* v_c, int64_t rows_cap,
                               const int32_t* offsets, int32_t B, int32_t Hq, int32_t Hkv, int32_t d, float scale,
                               void* o, float* lse, void* ws, size_t ws_bytes, void* stream) {
    int rc = check_heads(B, Hq, Hkv, d);
    if (rc) return rc;
    if (!q || !o || !offsets || !k_c || !v_c) return fail(SDKV_ERR_INVALID_ARG, "null pointer");
    if (!aligned16(q) || !aligned16(o) || !aligned16(k_c) || !aligned16(v_c))
        return fail(SDKV_ERR_INVALID_ARG, "q/o/k_c/v_c not 16-byte aligned");
    if (rows_cap <= 0 || rows_cap > 0x7fffffff) return fail(SDKV_ERR_INVALID_ARG, "rows_cap must be in [1, 2^31)");
    if (Hq / Hkv > 32) return fail(SDKV_ERR_UNSUPPORTED, "Hq/Hkv must be <= 32");
    if (static_cast<int64_t>(B) * Hkv > 65536) return fail(SDKV_ERR_UNSUPPORTED, "B*Hkv must be <= 65536");
    if (!std::isfinite(scale)) return fail(SDKV_ERR_INVALID_ARG, "scale must be finite");
    const DeviceInfo dev = current_device();
    if (dev.num_sms <= 0) return fail(SDKV_ERR_CUDA, "no CUDA device");
    if ((rc = check_ws(ws, ws_bytes, sparse_ws_bytes(B, Hq, Hkv, d, dev.num_sms)))) return rc;
    CUtensorMap tmk, tmv;
    if ((rc = encode_rows_tmap(&tmk, k_c, rows_cap, d, 64))) return rc;
    if ((rc = encode_rows_tmap(&tmv, v_c, rows_cap, d, 64))) return rc;
    AttnLaunch a{};
    a.q = q;
    a.k = k_c;
    a.v = v_c;
    a.B = B;
    a.Hq = Hq;
    a.Hkv = Hkv;
    a.d = d;
    a.gamma = 1;
    a.o = o;
    a.lse = lse;
    a.scale = scale;
    a.offsets = offsets;
    a.indices = nullptr;
    a.n_idx = 0;   // no index array
    a.n_cap = static_cast<int>(rows_cap);
    a.ws = ws;
    a.ws_bytes = ws_bytes;
    a.stream = static_cast<cudaStream_t>(stream);
    const char* why = "";
    rc = launch_sparse_decode_compact(a, &tmk, &tmv, dev.num_sms, &why);
    if (rc) return fail(rc, why);
    g_last_error.clear();
    return SDKV_OK;
}

int sdkv_specvlm_select(const float* scores, int32_t B, int32_t units, int32_t n, int32_t v_lo, int32_t v_hi,
                        double lam_r, double r, int32_t keep_lo, int32_t keep_hi, float* importance,
                        int32_t* indices, int32_t* counts, void* ws, size_t ws_bytes, void* stream) {
    if (!scores || !importance || !indices || !counts) return fail(SDKV_ERR_INVALID_ARG, "null pointer");
    if (B <= 0 || units <= 0 || n <= 0) return fail(SDKV_ERR_INVALID_ARG, "B, units, n must be positive");
    if (!(0 <= v_lo && v_lo <= v_hi && v_hi <= n)) return fail(SDKV_ERR_INVALID_ARG, "need 0 <= v_lo <= v_hi <= n");
    if (!(0 <= keep_lo && keep_lo <= keep_hi && keep_hi <= n))
        return fail(SDKV_ERR_INVALID_ARG, "need 0 <= keep_lo <= keep_hi <= n");
    if (keep_lo < keep_hi && v_lo < v_hi && !(keep_hi <= v_lo || keep_lo >= v_hi))
        return fail(SDKV_ERR_INVALID_ARG, "the kept range must not overlap the video tokens");
    if (!(lam_r >= 0.0 && lam_r <= 1.0)) return fail(SDKV_ERR_INVALID_ARG, "lam_r must be in [0, 1]");
    if (!(r >= 0.0 && r < 1.0)) return fail(SDKV_ERR_INVALID_ARG, "r must be in [0, 1)");
    if (v_hi - v_lo > (1 << 20)) return fail(SDKV_ERR_UNSUPPORTED, "at most 2^20 video tokens");
    if (static_cast<int64_t>(B) * units * n > (int64_t(1) << 40)) return fail(SDKV_ERR_INVALID_ARG, "scores too large");
    int rc = check_ws(ws, ws_bytes, specvlm_ws_bytes(B, v_hi - v_lo));
    if (rc) return rc;
    SpecLaunch a{scores, B, units, n, v_lo, v_hi, keep_lo, keep_hi, lam_r, r, importance, indices, counts, ws,
                 static_cast<cudaStream_t>(stream)};
    const char* why = "";
    rc = launch_specvlm(a, &why);
    if (rc) return fail(rc, why);
    g_last_error.clear();
    return SDKV_OK;
}

}  // extern "C"
