/*
 * sdkv.h -- C ABI of the sparse-KV decode attention library (libsdkv.so).
 *
 * The library computes the decode-step attention hot path of per-head sparse
 * KV selection on an NVIDIA GB300 (sm_103a):
 *
 *   sdkv_head_budgets        per-head cache budgets (host)
 *   sdkv_score_obs_window    observation-window scores of every cached key
 *   sdkv_select_topk         sinks + top-K + recent window, as ascending lists
 *   sdkv_sparse_decode_attn  attention of one query per head over its list
 *   sdkv_dense_verify_attn   attention of gamma causal queries over the cache
 *
 * Conventions shared by every call:
 *  - Pointers marked "device" are CUDA device pointers, "host" are host
 *    pointers.  The caller owns every buffer; the library never allocates,
 *    frees or synchronises (except sdkv_workspace_status, which is a
 *    synchronous diagnostic).
 *  - GPU calls are asynchronous on `stream` (a cudaStream_t passed as void*;
 *    NULL = the legacy default stream).  They may be captured in CUDA graphs.
 *  - Tensors are bf16 (2-byte bfloat16) unless stated.  Device pointers must
 *    be 16-byte aligned.  The head dimension d must be 64 or 128.
 *  - K and V caches have the logical shape [B][Hkv][n_cap][d] with the head
 *    dimension contiguous; kv_strides = {batch, head, row} strides in
 *    ELEMENTS, each a multiple of 8 (16 bytes), row stride >= d.
 *  - GQA: query head hq reads KV head hq / (Hq / Hkv) (contiguous groups);
 *    Hq must be a multiple of Hkv.
 *  - Workspace: every GPU call takes a device scratch buffer `ws` of at least
 *    sdkv_workspace_size(...) bytes.  Its first SDKV_WS_HEADER_BYTES hold a
 *    device status word and per-head counters: they must be zero before the
 *    first call that uses the buffer (e.g. cudaMemset once after allocation),
 *    and every call leaves the counters at zero again.  Calls that may run at
 *    the same time must use different workspaces.
 *  - Return value: SDKV_OK or a negative SDKV_ERR_* code; a human-readable
 *    message for the last failure of the calling thread is returned by
 *    sdkv_last_error().  Argument errors are detected on the host before any
 *    launch.  Errors that only the device can see (an index outside the
 *    cache, a list that does not fit, a wait that ran out) set the status
 *    word in the workspace header; the call still completes and its outputs
 *    for the affected heads are unspecified.  Read and clear it with
 *    sdkv_workspace_status.
 *
 * Sources (the pages this library follows):
 *  [StD]       "Sparse-to-Dense: A Free Lunch for Lossless Acceleration of
 *              Video Understanding in LLMs", sections 3.1-3.3.
 *  [ByteCross] "Where Activation Sparsity and KV-Cache Sparsity Cross in LLM
 *              Decoding", sections "The Byte Crossover", "Speedup Across
 *              Context", "The Attention Baseline".
 *  [SparseMM]  "小谈SparseMM，利用多模态大模型中视觉头的稀疏性优化KV Cache",
 *              methodology section (budget formulas, observation window).
 */
#ifndef SDKV_H
#define SDKV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define SDKV_OK                   0
#define SDKV_ERR_INVALID_ARG     -1  /* bad pointer, size, stride or alignment */
#define SDKV_ERR_UNSUPPORTED     -2  /* shape outside what the kernels implement (d, group size ...) */
#define SDKV_ERR_CUDA            -3  /* a CUDA runtime/driver call failed */
#define SDKV_ERR_WORKSPACE       -4  /* ws_bytes smaller than sdkv_workspace_size */

/* device status word values (see sdkv_workspace_status) */
#define SDKV_DEV_OK               0
#define SDKV_DEV_TIMEOUT          1  /* a bounded wait inside a kernel ran out (about 1 s) */
#define SDKV_DEV_BAD_INDEX        2  /* a list entry outside [0, n_cap) */
#define SDKV_DEV_BAD_LIST         3  /* list lengths do not fit sinks + candidates + recent */

#define SDKV_WS_HEADER_BYTES   256   /* status word + reserved; counters follow */

/* operation ids for sdkv_workspace_size */
#define SDKV_OP_SCORE             1
#define SDKV_OP_SELECT            2
#define SDKV_OP_SPARSE_DECODE     3
#define SDKV_OP_DENSE_VERIFY      4
#define SDKV_OP_COMPACT           5
#define SDKV_OP_SPECVLM           6

/*
 * Per-head cache budgets.  [SparseMM] methodology: with N heads, total budget
 * B, local window w and uniform share rho,
 *     r        = rho (B - N w) / N
 *     B_remain = B - N w - rho (B - N w)
 *     b_i      = w + r + B_remain * s_i / sum_j s_j
 * The real b_i are turned into integers that sum to B exactly by
 * largest-remainder apportionment (ties to the lower index i).  If cap > 0 no
 * head gets more than cap: the excess of capped heads is shared among the
 * others in proportion to s, repeated until none exceeds the cap.  sum(s) is a
 * float64 sum in index order; all-zero scores count as uniform.  The top-K
 * count of head i is then b_i - w (the local window is kept apart).
 *
 *   s       host float[n_heads], finite, >= 0 (flat index layer * H + head)
 *   total_B budget B, >= n_heads * w
 *   w       local window per head, >= 0
 *   rho     uniform share in [0, 1]
 *   cap     per-head maximum (e.g. the cache length) or 0 for none;
 *           cap * n_heads must be >= B
 *   b_out   host int32[n_heads] (written)
 * Host only, synchronous.  Returns SDKV_ERR_INVALID_ARG on bad input.
 */
int sdkv_head_budgets(const float* s, int32_t n_heads, int64_t total_B, int32_t w,
                      double rho, int32_t cap, int32_t* b_out);

/*
 * Bytes of workspace an operation needs for the given shape.
 *   op = SDKV_OP_SCORE:         (B, Hq, Hkv, d, n, W)       W = window length
 *   op = SDKV_OP_SELECT:        (B, 0, Hkv, 0, n, 0)
 *   op = SDKV_OP_SPARSE_DECODE: (B, Hq, Hkv, d, 0, 0)
 *   op = SDKV_OP_DENSE_VERIFY:  (B, Hq, Hkv, d, n, gamma)   n = n_prefix + gamma
 *   op = SDKV_OP_COMPACT:       (any)                       status word only
 *   op = SDKV_OP_SPECVLM:       (B, 0, 0, 0, nV, 0)         nV = v_hi - v_lo
 * sdkv_sparse_decode_compact uses the SDKV_OP_SPARSE_DECODE size.
 * Queries the current device's SM count.  Returns 0 for an invalid request.
 */
size_t sdkv_workspace_size(int32_t op, int32_t B, int32_t Hq, int32_t Hkv, int32_t d,
                           int32_t n, int32_t gamma_or_W);

/*
 * Observation-window scores.  [StD] 3.2 (mean attention of the text queries
 * to each key, GQA scores summed over the group) and [SparseMM] observation
 * window (last 32 queries):
 *     score[b][h][j] = (1/W) sum_{g in group(h)} sum_{t<W} P[b][h*G+g][t][j]
 *     P[.][t][j]     = softmax over keys j <= q_pos0 + t of scale * q_t . k_j
 * Window query t sits at position q_pos0 + t and sees keys 0 .. q_pos0 + t;
 * keys it cannot see contribute 0.
 *
 *   q_obs     device bf16 [B][Hq][W][d], contiguous
 *   k         device bf16 K cache (see conventions), rows 0 .. n-1 are read
 *   k_strides host int64[3] element strides {batch, head, row}
 *   n         keys scored, 1 <= n
 *   W         window length, 1 <= W; q_pos0 >= 0 and q_pos0 + W <= n
 *   scale     logit scale (usually 1/sqrt(d))
 *   scores    device float [B][Hkv][n], contiguous (written)
 * Needs Hq/Hkv * W <= 4096.
 */
int sdkv_score_obs_window(const void* q_obs, const void* k, const int64_t k_strides[3],
                          int32_t B, int32_t Hq, int32_t Hkv, int32_t d, int32_t n,
                          int32_t W, int32_t q_pos0, float scale, float* scores,
                          void* ws, size_t ws_bytes, void* stream);

/*
 * Top-K selection and list assembly.  [StD] 3.2 argTopK over the candidate
 * (visual) keys; [SparseMM] K = r + b_score, the local window kept apart;
 * [ByteCross] "Speedup Across Context": four sinks plus the highest-scoring
 * entries of each KV head.
 * For every (b, h), with k_h = offsets[bh+1] - offsets[bh] and
 * K_h = k_h - n_sink - n_recent, the list indices[offsets[bh] .. +k_h) is
 *     [0, n_sink)  +  top K_h of [cand_lo, cand_hi)  +  [n - n_recent, n)
 * in ascending order.  Candidates rank by score descending, equal scores by
 * lower index first; -0.0 equals +0.0; NaN ranks below every number.
 *
 *   scores   device float [B][Hkv][n] (as written by sdkv_score_obs_window)
 *   cand_lo, cand_hi  candidate range; needs
 *            0 <= n_sink <= cand_lo <= cand_hi <= n - n_recent
 *   offsets  device int32 [B*Hkv + 1], non-decreasing
 *   indices  device int32 [offsets[B*Hkv]] (written)
 * A head whose K_h is outside [0, cand_hi - cand_lo] sets SDKV_DEV_BAD_LIST and
 * its list is left unwritten.
 */
int sdkv_select_topk(const float* scores, int32_t B, int32_t Hkv, int32_t n,
                     int32_t cand_lo, int32_t cand_hi, int32_t n_sink, int32_t n_recent,
                     const int32_t* offsets, int32_t* indices,
                     void* ws, size_t ws_bytes, void* stream);

/*
 * Sparse decode attention over per-head index lists.  [StD] 3.2: the sparse
 * model loads only the retained KV entries; [ByteCross] "The Byte Crossover":
 * unselected entries stay allocated but unread.  For each (b, hq), with S the
 * list of KV head h = hq / G:
 *     o[b][hq]   = sum_{j in S} softmax_j(scale q . k_j) v_j
 *     lse[b][hq] = log sum_{j in S} exp(scale q . k_j)        (natural log)
 * An empty list gives o = 0 and lse = -inf.  Split-K over chunks of the lists
 * with a log-sum-exp combine; with many lists (more than the clusters of one
 * wave cover, Hq/Hkv <= 16, B*Hkv <= 2048) each CTA takes an equal span of the
 * concatenated lists instead, several short lists at once.  fp32 accumulation,
 * bf16 output.
 *
 *   q        device bf16 [B][Hq][d], contiguous
 *   k, v     device bf16 caches (see conventions), kv_strides shared
 *   n_cap    rows per head present in k and v; list entries must lie in
 *            [0, n_cap) (others set SDKV_DEV_BAD_INDEX and read row 0)
 *   offsets, indices  device int32 CSR lists per (b, h), as from sdkv_select_topk;
 *            offsets non-decreasing (a decrease sets SDKV_DEV_BAD_LIST and leaves
 *            o and lse unspecified)
 *   n_idx    number of int32 entries the `indices` array holds (its length), or
 *            0.  With n_idx > 0 the kernel, while the previous kernel on
 *            `stream` finishes, prefetches the offsets and indices[0, n_idx)
 *            into L2 (prefetches read nothing back; the lists are loaded only
 *            after that kernel has finished).  n_idx = 0 skips the prefetch.
 *   o        device bf16 [B][Hq][d] (written)
 *   lse      device float [B][Hq] (written) or NULL
 * Needs Hq/Hkv <= 32 and B*Hkv <= 65536.
 */
int sdkv_sparse_decode_attn(const void* q, const void* k, const void* v,
                            const int64_t kv_strides[3], int32_t n_cap,
                            const int32_t* offsets, const int32_t* indices, int64_t n_idx,
                            int32_t B, int32_t Hq, int32_t Hkv, int32_t d, float scale,
                            void* o, float* lse, void* ws, size_t ws_bytes, void* stream);

/*
 * Dense multi-query verify attention.  [StD] 3.1: the dense model verifies the
 * gamma drafted tokens in parallel with one read of the full cache;
 * [ByteCross] "The Attention Baseline": split-K dense decode.  The cache holds
 * n_prefix + gamma rows; query t (t < gamma) sits at position n_prefix + t and
 * attends keys 0 .. n_prefix + t:
 *     o[b][hq][t]   = sum_{j <= n_prefix+t} softmax_j(scale q_t . k_j) v_j
 *     lse[b][hq][t] = log sum_{j <= n_prefix+t} exp(scale q_t . k_j)
 * gamma = 1 with n_prefix = n - 1 is the dense decode over n keys.
 *
 *   q        device bf16 [B][Hq][gamma][d], contiguous
 *   k, v     device bf16 caches with at least n_prefix + gamma rows
 *   o        device bf16 [B][Hq][gamma][d] (written)
 *   lse      device float [B][Hq][gamma] (written) or NULL
 * Needs (Hq/Hkv) * gamma <= 64, n_prefix >= 0, gamma >= 1.
 */
int sdkv_dense_verify_attn(const void* q, const void* k, const void* v,
                           const int64_t kv_strides[3], int32_t B, int32_t Hq, int32_t Hkv,
                           int32_t d, int32_t n_prefix, int32_t gamma, float scale,
                           void* o, float* lse, void* ws, size_t ws_bytes, void* stream);

/*
 * Dense multi-query verify attention that allocates nothing.  The pages have
 * no counterpart of this call; it exists for callers that cannot hand the
 * library a workspace: programs whose device memory is owned by a pool they
 * cannot draw from at this point (an inference server that fixes its memory
 * at start-up, a plugin host that forbids cudaMalloc, a latency-critical loop
 * where an allocation's implicit synchronisation would stall the stream).
 *
 * Computes exactly what sdkv_dense_verify_attn computes, with the same
 * arguments except ws / ws_bytes.  Its scratch (split-K partials, per-head
 * counters, status word) lives in one fixed device array of
 * SDKV_NOALLOC_SCRATCH_BYTES inside the library, present on every GPU that
 * loads the library until the process exits.  A shape that needs more scratch
 * than that returns SDKV_ERR_UNSUPPORTED (use sdkv_dense_verify_attn then).
 *  - The first call on a device looks up the array's device address (once per
 *    device, with that device current); make that first call before any
 *    stream capture.  The address belongs to the device's current CUDA
 *    context: after a device reset (cudaDeviceReset, from any runtime in the
 *    process) the next call, in the new context, looks it up again, so that
 *    call too belongs before any capture.
 *  - Each call clears the counters and status word it needs (an asynchronous
 *    memset on `stream`, not an allocation) and calls no cudaMalloc/cudaFree.
 *  - Every call on a device uses that device's one copy of the array: calls
 *    that may overlap on the same GPU (for example on different streams) race
 *    on it and give wrong results.  Serialise them.
 * Device-side errors (a bounded wait that ran out) set the array's status
 * word: read it with sdkv_dense_verify_attn_noalloc_status before the next
 * call clears it.  Argument errors are reported as for sdkv_dense_verify_attn.
 */
#define SDKV_NOALLOC_SCRATCH_BYTES (8u << 20)   /* 8 MiB */
int sdkv_dense_verify_attn_noalloc(const void* q, const void* k, const void* v,
                                   const int64_t kv_strides[3], int32_t B, int32_t Hq,
                                   int32_t Hkv, int32_t d, int32_t n_prefix, int32_t gamma,
                                   float scale, void* o, float* lse, void* stream);

/*
 * Synchronous diagnostic for sdkv_dense_verify_attn_noalloc: waits for
 * `stream`, copies the status word of the current device's fixed array to
 * *status (one of SDKV_DEV_*), then clears it.  Allocates nothing.
 */
int sdkv_dense_verify_attn_noalloc_status(int32_t* status, void* stream);

/*
 * Synchronous diagnostic: waits for `stream`, copies the device status word of
 * the workspace to *status (one of SDKV_DEV_*), then clears it.
 */
int sdkv_workspace_status(void* ws, int32_t* status, void* stream);

/* Message of the calling thread's last failed call ("" if none). */
const char* sdkv_last_error(void);

/* Library ABI version (major * 100 + minor). */
int32_t sdkv_version(void);

/* ---------------------------------------------------------------------------
 * Around the hot path: list builders, compaction, SpecVLM selection.
 * ------------------------------------------------------------------------- */

/*
 * Sink-plus-recent lists, no scoring.  [StD] baselines ("Streaming": a draft
 * model with streaming attention); [ByteCross] "The Attention Baseline" (a
 * sink-plus-recent window timed against dense decoding).  Every (b, h) keeps
 * rows [0, min(n_sink, n)) and [max(n - n_recent, min(n_sink, n)), n), so each
 * list has k = min(n, n_sink + n_recent) entries, ascending.
 *   offsets  device int32[B*Hkv + 1] (written: i * k)
 *   indices  device int32[B*Hkv*k]   (written)
 * Asynchronous on `stream`; no workspace.  Feed the lists to
 * sdkv_sparse_decode_attn unchanged.
 */
int sdkv_window_lists(int32_t B, int32_t Hkv, int32_t n, int32_t n_sink, int32_t n_recent,
                      int32_t* offsets, int32_t* indices, void* stream);

/*
 * Draft-step lists.  [StD] 3.1: the sparse model proposes gamma tokens one at a
 * time; draft step t attends the base selection plus the t + 1 positions
 * drafted so far, whose KV rows it has just appended to the cache.  Each list
 * of the base CSR followed by n_pos, n_pos + 1, ..., n_pos + n_new - 1:
 *   offsets[i] = (base_offsets[i] - base_offsets[0]) + i * n_new
 *   base_*   device CSR of BH lists (every base entry below n_pos keeps the
 *            new lists ascending)
 *   offsets  device int32[BH + 1], indices device int32[total + BH * n_new]
 *            (written; must not alias the base arrays)
 * Asynchronous on `stream`; no workspace.
 */
int sdkv_append_drafts(const int32_t* base_offsets, const int32_t* base_indices, int32_t BH,
                       int32_t n_pos, int32_t n_new, int32_t* offsets, int32_t* indices,
                       void* stream);

/*
 * All draft-step lists of one StD round in one launch.  [StD] 3.1: draft step
 * t = 0 .. gamma - 1 attends the base selection plus n_pos .. n_pos + t.  Set
 * t is exactly what sdkv_append_drafts writes with n_new = t + 1:
 *   offsets  device int32[gamma][BH + 1]; set t at offsets + t * (BH + 1)
 *   indices  device int32[gamma][stride]; set t at indices + t * stride, with
 *            stride >= (base_offsets[BH] - base_offsets[0]) + BH * gamma
 *            (entries at or past stride are not written)
 *   base_*   device CSR of BH lists, entries below n_pos; outputs must not
 *            alias them
 * Asynchronous on `stream`; no workspace.  One launch replaces gamma calls of
 * sdkv_append_drafts.
 */
int sdkv_draft_lists(const int32_t* base_offsets, const int32_t* base_indices, int32_t BH, int32_t n_pos,
                     int32_t gamma, int64_t stride, int32_t* offsets, int32_t* indices, void* stream);

/*
 * Contiguous compaction of the selected rows.  [ByteCross] "Speedup Across
 * Context": after selection the kept entries are gathered into a contiguous
 * buffer that every later step reads in one kernel call.  Row
 * offsets[i] - offsets[0] + j of k_out / v_out is row indices[offsets[i] + j]
 * of KV head (b, h) = (i / Hkv, i % Hkv) of the caches.
 *   k, v, kv_strides, n_cap, offsets, indices  as for sdkv_sparse_decode_attn
 *            (entries outside [0, n_cap) set SDKV_DEV_BAD_INDEX and copy row 0)
 *   rows_cap rows k_out and v_out hold; list rows past it are skipped and set
 *            SDKV_DEV_BAD_LIST
 *   k_out, v_out  device bf16 [rows_cap][d] (written), 16-byte aligned
 *   ws       workspace of at least sdkv_workspace_size(SDKV_OP_COMPACT, ...)
 * Asynchronous on `stream`.  Reads and writes 4*d bytes per listed row.
 */
int sdkv_compact_kv(const void* k, const void* v, const int64_t kv_strides[3], int32_t n_cap,
                    const int32_t* offsets, const int32_t* indices, int32_t B, int32_t Hkv,
                    int32_t d, int64_t rows_cap, void* k_out, void* v_out, void* ws,
                    size_t ws_bytes, void* stream);

/*
 * Sparse decode over compacted rows: the attention of sdkv_sparse_decode_attn,
 * where the rows of list i are the contiguous rows [offsets[i] - offsets[0],
 * offsets[i+1] - offsets[0]) of k_c / v_c (as written by sdkv_compact_kv).
 * Streamed with tensor copies, no index reads.
 *   rows_cap rows of k_c / v_c (the tensor maps' extent; rows past it read 0)
 *   other arguments as for sdkv_sparse_decode_attn; workspace of at least
 *   sdkv_workspace_size(SDKV_OP_SPARSE_DECODE, ...)
 */
int sdkv_sparse_decode_compact(const void* q, const void* k_c, const void* v_c, int64_t rows_cap,
                               const int32_t* offsets, int32_t B, int32_t Hq, int32_t Hkv,
                               int32_t d, float scale, void* o, float* lse, void* ws,
                               size_t ws_bytes, void* stream);

/*
 * SpecVLM token selection.  [SpecVLM] "The SpecVLM Method": the importance of
 * token j is the mean of the verifier's attention maps (all layers and heads)
 *     a_j = (1/units) sum_u scores[b][u][j]        (fp32, units in order)
 * Stage I keeps the shortest prefix V_R of the video tokens V = [v_lo, v_hi),
 * ordered by a_j descending (equal a_j: lower j first), whose mass reaches
 * lam_r times the mass of V (top-P).  Stage II walks the other video tokens in
 * index order at the interval I = (|V| - |V_R|) / ((1 - r)|V|) and keeps the
 * ones at positions floor(k I), k = 0, 1, ...  The list is V_R u V_U plus the
 * always-kept range [keep_lo, keep_hi) (e.g. the text tokens), ascending.
 * Exact decisions: every mass is a_j rounded to the nearest multiple of 2^-32
 * and summed as an integer; lam_r * S, I and k * I are float64.
 *   scores     device float [B][units][n]; importance values outside
 *              [0, 2^31) and NaN count as 0 and set SDKV_DEV_BAD_LIST
 *   lam_r      in [0, 1];  r (pruning ratio) in [0, 1)
 *   keep range disjoint from V
 *   importance device float [B][n] (written)
 *   indices    device int32 [B][(v_hi - v_lo) + (keep_hi - keep_lo)] (written;
 *              the first counts[b] entries of row b are the list)
 *   counts     device int32 [B] (written)
 *   ws         workspace of at least sdkv_workspace_size(SDKV_OP_SPECVLM, B, 0,
 *              0, 0, v_hi - v_lo, 0)
 * Asynchronous on `stream`.  One CTA per sequence; Stage I is a radix search
 * for the crossing on the score bits (counts and masses per digit), Stage II
 * enumerates floor(k I).  Up to 16384 video tokens keep their keys in shared
 * memory, more in the workspace (at most 2^20).
 */
int sdkv_specvlm_select(const float* scores, int32_t B, int32_t units, int32_t n,
                        int32_t v_lo, int32_t v_hi, double lam_r, double r,
                        int32_t keep_lo, int32_t keep_hi, float* importance,
                        int32_t* indices, int32_t* counts, void* ws, size_t ws_bytes,
                        void* stream);

#ifdef __cplusplus
}
#endif

#endif /* SDKV_H */
