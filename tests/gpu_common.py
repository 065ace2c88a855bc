"""Helpers shared by the GPU parity tests: tolerances and comparisons against
the fp64 oracle."""
import math

import numpy as np
import torch

# Attention outputs (bf16 inputs, fp32 accumulation, bf16 output): the bar the
# method's contract sets for every output tensor.
O_MAX_ABS = 1e-2
O_MEAN_ABS = 1e-3
# Log-sum-exp (fp32 output): logits carry fp32 rounding of bf16 products summed
# over d <= 128 terms (|error| ~ 1e-5 for |logit| ~ 10) plus the approximate
# exp2/log2 (relative 2^-22); the multi-query verify sums bf16-rounded weights
# (relative 2^-9 each, at most 2^-10 in lse for a two-key prefix, ~1e-4 over
# thousands of keys).  2e-3 leaves margin over all of these.
LSE_MAX_ABS = 2e-3
# Window scores (fp32): each score sums G*W probabilities; relative 1e-3 is the
# tolerance the selection rule is stated with.
SCORE_REL = 1e-3
# Top-K gap rule: index sets must be identical where the K-th and (K+1)-th
# oracle scores differ by more than this relative gap.
GAP_REL = 1e-3


def f64(t):
    return t.detach().to("cpu").to(torch.float64).numpy()


def assert_attn_close(o_gpu, o_ref, what=""):
    o = f64(o_gpu)
    diff = np.abs(o - o_ref)
    assert np.isfinite(o).all(), what + ": non-finite output"
    assert diff.max() <= O_MAX_ABS, "%s: max-abs %.3g" % (what, diff.max())
    assert diff.mean() <= O_MEAN_ABS, "%s: mean-abs %.3g" % (what, diff.mean())
    return diff.max(), diff.mean()


def assert_lse_close(l_gpu, l_ref, what=""):
    l = f64(l_gpu)
    fin = np.isfinite(l_ref)
    assert np.array_equal(np.isfinite(l), fin), what + ": -inf pattern differs"
    if fin.any():
        d = np.abs(l[fin] - l_ref[fin]).max()
        assert d <= LSE_MAX_ABS, "%s: lse max-abs %.3g" % (what, d)


def assert_scores_close(s_gpu, s_ref, what=""):
    s = f64(s_gpu)
    scale = max(np.abs(s_ref).max(), 1e-30)
    rel = np.abs(s - s_ref) / np.maximum(np.abs(s_ref), 1e-3 * scale)
    assert rel.max() <= SCORE_REL, "%s: score rel err %.3g" % (what, rel.max())


def check_selection_gap_rule(idx_gpu, offsets, s_ref, n, cand_lo, cand_hi, n_sink, n_recent):
    """GPU lists (from GPU scores) against oracle fp64 scores.  Where the oracle's
    K-th / (K+1)-th candidate gap exceeds GAP_REL, the set must equal the
    oracle's; otherwise it must hold every clear winner, only near-threshold
    candidates, exactly K distinct entries, ascending."""
    import oracle
    idx_gpu = np.asarray(idx_gpu)
    offsets = np.asarray(offsets)
    want = oracle.select_topk(s_ref, n, cand_lo, cand_hi, n_sink, n_recent, offsets)
    B, Hkv = s_ref.shape[0], s_ref.shape[1]
    exact = 0
    for b in range(B):
        for h in range(Hkv):
            i = b * Hkv + h
            a, e = offsets[i], offsets[i + 1]
            got = idx_gpu[a:e]
            ref = want[a:e]
            assert (np.diff(got) > 0).all(), "list not ascending"
            K = (e - a) - n_sink - n_recent
            assert list(got[:n_sink]) == list(range(n_sink))
            assert list(got[len(got) - n_recent:]) == list(range(n - n_recent, n))
            if K == 0 or K == cand_hi - cand_lo:
                assert np.array_equal(got, ref)
                exact += 1
                continue
            cs = np.sort(s_ref[b, h, cand_lo:cand_hi])[::-1]
            tK, tK1 = cs[K - 1], cs[K]
            if (tK - tK1) / max(tK, 1e-300) > GAP_REL:
                assert np.array_equal(got, ref), "set differs at (b=%d, h=%d) despite a clear gap" % (b, h)
                exact += 1
            else:
                top = got[n_sink:n_sink + K]
                assert len(np.unique(top)) == K
                sc = s_ref[b, h, top]
                assert (sc >= tK * (1 - GAP_REL)).all()
                must = np.nonzero(s_ref[b, h, cand_lo:cand_hi] > tK * (1 + GAP_REL))[0] + cand_lo
                assert set(must.tolist()) <= set(top.tolist())
    return exact


def csr(lengths, device):
    offs = np.zeros(len(lengths) + 1, np.int64)
    offs[1:] = np.cumsum(lengths)
    return torch.tensor(offs.astype(np.int32), device=device), offs


def scale_of(d):
    return 1.0 / math.sqrt(d)
