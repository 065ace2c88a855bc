"""sparse_kv_decode_gb300: decode-step attention over per-head sparse KV selections on GB300.

The compute lives in libsdkv.so (hand-written CUDA for sm_103a behind the C ABI
of include/sdkv.h); this package is its thin Python binding plus the byte
account used to report achieved bandwidth.
"""
from ._lib import (  # noqa: F401
    OP_COMPACT,
    OP_DENSE_VERIFY,
    OP_SPECVLM,
    OP_SCORE,
    OP_SELECT,
    OP_SPARSE_DECODE,
    SdkvError,
    dense_verify_attn,
    head_budgets,
    lib,
    new_workspace,
    score_obs_window,
    select_topk,
    sparse_decode_attn,
    version,
    workspace_size,
    workspace_status,
    window_lists,
    append_drafts,
    draft_lists,
    compact_kv,
    sparse_decode_compact,
    specvlm_select,
)
