// Host-side interface between the C ABI layer (sdkv_api.cpp) and the kernel
// translation units.  Not part of the public header.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace sdkv {

struct DeviceInfo {
    int device = -1;
    int num_sms = 0;
};
DeviceInfo current_device();

// Encode a 4-D bf16 tensor map over a KV cache [B][Hkv][rows][d] (d contiguous)
// with a box of (64 elements, box_rows, 1, 1) and 128-byte swizzle.
int encode_kv_tmap(CUtensorMap* map, const void* base, int B, int Hkv, int rows, int d,
                   const int64_t strides[3], int box_rows);

// ---- split-K attention (attn_splitk.cu) --------------------------------------
struct AttnLaunch {
    const void* q;
    const void* k;
    const void* v;
    int64_t sb, sh, sn;
    int B, Hq, Hkv, d, gamma;
    void* o;
    float* lse;
    float scale;
    // dense
    int n_prefix;
    // sparse
    const int32_t* offsets;
    const int32_t* indices;
    int64_t n_idx;   // entries of indices (0: no early reads of the lists)
    int n_cap;
    void* ws;
    size_t ws_bytes;
    cudaStream_t stream;
};
// Workspace of the split-K kernels: status word, per-head tickets (BH x 8), and
// partials o fp32 [max_chunks][R][d] and softmax records [max_chunks][R][ml_floats].
struct AttnWs {
    int* status;
    int* tickets;
    float* part_o;
    float* part_ml;
    size_t bytes;
};
AttnWs attn_ws(void* ws, int BH, int R, int d, int max_chunks, int ml_floats);
size_t dense_ws_bytes(int B, int Hq, int Hkv, int d, int n_total, int gamma, int num_sms);
// gamma-query verify on tcgen05 (verify_tc.cu): d = 128, 16 < (Hq/Hkv) * gamma <= 64.
// verify_tc_ws_bytes is its workspace size, 0 for shapes it does not take.
size_t verify_tc_ws_bytes(int B, int Hq, int Hkv, int d, int n_total, int gamma, int num_sms);
int launch_verify_tc(const AttnLaunch& a, const CUtensorMap* tmk, const CUtensorMap* tmv, int num_sms,
                     const char** why);
size_t sparse_ws_bytes(int B, int Hq, int Hkv, int d, int num_sms);
int launch_dense_verify(const AttnLaunch& a, const CUtensorMap* tmk, const CUtensorMap* tmv,
                        int num_sms, const char** why);
int launch_sparse_decode(const AttnLaunch& a, int num_sms, const char** why);
// gathered decode packed by list position (packed_decode.cu): many short lists,
// Hq/Hkv <= 16, B*Hkv <= 2048, one decode position; 2 partial slots per CTA
bool packed_decode_takes(int B, int Hq, int Hkv, int d);
int packed_decode_grid_max(int num_sms);
int launch_packed_decode(const AttnLaunch& a, int num_sms, const char** why);
// decode over the lists' rows compacted into contiguous [rows][d] buffers (2-D tensor maps)
int launch_sparse_decode_compact(const AttnLaunch& a, const CUtensorMap* tmk, const CUtensorMap* tmv, int num_sms,
                                 const char** why);
// dense verify with its scratch in the library's fixed device array (no allocation)
int dense_verify_noalloc(const AttnLaunch& a, const CUtensorMap* tmk, const CUtensorMap* tmv, int num_sms,
                         const char** why);
// status word of the fixed array on the current device: read, then cleared (synchronous on st)
int noalloc_status(int32_t* status, cudaStream_t st, const char** why);

// ---- observation-window scoring (score_obs.cu) --------------------------------
struct ScoreLaunch {
    const void* q_obs;
    int B, Hq, Hkv, d, n, W, q_pos0;
    float scale;
    float* scores;
    void* ws;
    size_t ws_bytes;
    cudaStream_t stream;
};
size_t score_ws_bytes(int B, int Hq, int Hkv, int d, int n, int W, int num_sms);
int launch_score(const ScoreLaunch& a, const CUtensorMap* tmk, const CUtensorMap* tmq, int num_sms,
                 const char** why);
// 2-D bf16 tensor map over rows x d (row pitch d), box (64, box_rows), 128-byte swizzle
int encode_rows_tmap(CUtensorMap* map, const void* base, int64_t rows, int d, int box_rows);

// ---- top-K selection (select_topk.cu) -------------------------------------------
struct SelectLaunch {
    const float* scores;
    int B, Hkv, n, cand_lo, cand_hi, n_sink, n_recent;
    const int32_t* offsets;
    int32_t* indices;
    void* ws;
    cudaStream_t stream;
    int num_sms;
};
size_t select_ws_bytes(int B, int Hkv, int n);
int launch_select(const SelectLaunch& a, const char** why);

// ---- next rows (next_rows.cu) ------------------------------------------------------
int launch_window_lists(int B, int Hkv, int n, int n_sink, int n_recent, int* offsets, int* indices,
                        cudaStream_t st, const char** why);
int launch_append_drafts(const int* base_offsets, const int* base_indices, int BH, int n_pos, int n_new,
                         int* offsets, int* indices, cudaStream_t st, const char** why);
int launch_draft_lists(const int* base_offsets, const int* base_indices, int BH, int n_pos, int gamma,
                       long long stride, int* offsets, int* indices, cudaStream_t st, const char** why);
struct CompactLaunch {
    const void* k;
    const void* v;
    int64_t sb, sh, sn;
    int n_cap, B, Hkv, d;
    const int32_t* offsets;
    const int32_t* indices;
    long long rows_cap;
    void* k_out;
    void* v_out;
    void* ws;
    cudaStream_t stream;
};
int launch_compact_kv(const CompactLaunch& a, const char** why);
struct SpecLaunch {
    const float* scores;
    int B, units, n, v_lo, v_hi, keep_lo, keep_hi;
    double lam_r, r;
    float* importance;
    int32_t* indices;
    int32_t* counts;
    void* ws;
    cudaStream_t stream;
};
size_t specvlm_ws_bytes(int B, int nV);
int launch_specvlm(const SpecLaunch& a, const char** why);

}  // namespace sdkv
