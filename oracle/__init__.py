"""Plain fp64 CPU oracle for the sparse-KV decode hot path.

TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the bench's CPU
baseline leg may import this package; the product path never does, and the
CUDA library shares no code with it.

Every function here restates, in numpy float64, what the pages define:

  head_budgets      SparseMM post, methodology section: b = w + r + b_score,
                    r = rho (B - N w) / N, B_remain = B - N w - rho (B - N w),
                    b_score = B_remain s / sum(s).
  score_obs_window  StD section 3.2 (argTopK equation; GQA scores summed over
                    the group) and SparseMM's observation window (last 32
                    queries, averaged attention weight per key).
  select_topk       StD section 3.2 argTopK; SparseMM K = r + b_score (the
                    local window kept apart); ByteCross "Speedup Across
                    Context" (four sinks kept).
  sparse_decode     StD section 3.2 / ByteCross byte crossover: attention of
                    one query over the selected keys only.
  dense_verify      StD section 3.1: gamma drafted positions verified in one
                    pass over the full cache, causal among the drafts.
  window_lists      StD baselines ("Streaming") / ByteCross "The Attention
                    Baseline": attention sinks plus the recent window.
  compact_kv,       ByteCross "Speedup Across Context": selected entries
  sparse_decode_    gathered into a contiguous buffer read by every later step.
  compact
  specvlm_*         SpecVLM post, "The SpecVLM Method": top-P retention of the
                    verifier's attention mass, then uniform subsampling.
  append_drafts     StD 3.1: the draft steps' lists grow by the drafted tokens.

Pins (tests/test_oracle_pins.py) tie each function to closed forms,
invariants, brute force and printed values; none is "parity unpinned".
"""
from .sdkv_oracle import (  # noqa: F401
    budget_terms,
    head_budgets_real,
    head_budgets,
    score_obs_window,
    select_topk,
    sparse_decode,
    dense_verify,
    to_f64,
    window_lists,
    compact_kv,
    sparse_decode_compact,
    specvlm_importance,
    specvlm_select,
    append_drafts,
    MASS_FRAC_BITS,
)
