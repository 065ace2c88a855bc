"""Pins of the fp64 oracle against what the pages and the mathematics fix.

Each test ties an oracle function to something other than itself: a printed
value, a closed form, an invariant the method states, a special case that
reduces to a textbook result, or brute force on tiny inputs.  Together they
are chosen so that a dropped term, a wrong sign or index, a wrong scale or a
transposed operand in the oracle fails at least one of them.
"""
import itertools
import math
import os

import numpy as np
import pytest

import oracle
from sparse_kv_decode_gb300 import byte_account as ba

RNG = np.random.default_rng(12345)


def _bf16_round(x):
    """Round float64 values to bf16 values (RNE), returned as float64, so the
    small cases use inputs the CUDA path could receive."""
    import torch
    return torch.as_tensor(x, dtype=torch.float64).to(torch.bfloat16).to(torch.float64).numpy()


# ---------------------------------------------------------------------------
# a1 head budgets (SparseMM methodology: b = w + r + B_remain s / sum s)
# ---------------------------------------------------------------------------

def test_budget_terms_sparsemm_workload_closed_form():
    # N = 32 x 32 heads, B = 256 N, w = 32, rho = 0.1:
    # r = 0.1 (262144 - 32768) / 1024 = 22.4 ; B_remain = 0.9 * 229376 = 206438.4
    r, b_rem = oracle.budget_terms(1024, 262144, 32, 0.1)
    assert r == pytest.approx(22.4, rel=1e-15)
    assert b_rem == pytest.approx(206438.4, rel=1e-15)


def test_budget_three_parts_add_up_to_B():
    # N w (local windows) + N r (uniform) + B_remain (score-preferred) = B
    for N, B, w, rho in [(7, 1000, 16, 0.3), (1024, 262144, 32, 0.1), (3, 96, 32, 0.5)]:
        r, b_rem = oracle.budget_terms(N, B, w, rho)
        assert N * w + N * r + b_rem == pytest.approx(B, rel=1e-12)
        assert N * r == pytest.approx(rho * (B - N * w), rel=1e-12)


def test_budget_real_is_affine_in_s():
    # b*_i - (w + r) is proportional to s_i with total B_remain
    s = RNG.lognormal(0, 0.5, 50)
    B, w, rho = 50 * 300, 32, 0.2
    r, b_rem = oracle.budget_terms(50, B, w, rho)
    bs = np.array(oracle.head_budgets_real(s, B, w, rho))
    extra = bs - (w + r)
    assert np.allclose(extra / s, b_rem / s.sum(), rtol=1e-12)
    assert bs.sum() == pytest.approx(B, rel=1e-12)


def test_budget_one_visual_head_takes_the_pool():
    # all score on head 0: b_0 = w + r + B_remain, the rest w + r
    s = np.zeros(8)
    s[0] = 3.0
    B, w, rho = 8 * 100, 20, 0.25
    r, b_rem = oracle.budget_terms(8, B, w, rho)   # r = 0.25*640/8 = 20, b_rem = 480
    assert (r, b_rem) == (20.0, 480.0)
    b = oracle.head_budgets(s, B, w, rho)
    assert list(b) == [20 + 20 + 480] + [40] * 7


def test_budget_sums_to_B_and_floor_of_w_plus_r():
    for trial in range(20):
        N = int(RNG.integers(1, 300))
        w = int(RNG.integers(0, 40))
        B = N * w + int(RNG.integers(0, 100 * N + 1))
        rho = float(RNG.uniform(0, 1))
        s = RNG.lognormal(0, 0.5, N) * np.where(RNG.uniform(size=N) < 0.05, 20, 1)
        b = oracle.head_budgets(s, B, w, rho)
        r, _ = oracle.budget_terms(N, B, w, rho)
        assert b.sum() == B
        assert (b >= w + math.floor(r)).all()


def test_budget_uniform_scores_and_rho_one():
    N, B, w = 37, 37 * 250 + 11, 32
    for s in (np.ones(N), RNG.lognormal(0, 1, N)):
        b = oracle.head_budgets(s, B, w, 1.0)           # rho = 1: every head w + r
        assert set(b.tolist()) <= {B // N, B // N + 1}
        assert b.sum() == B
        # remainders are all equal, so the extra units go to the lowest indices
        assert list(b) == [B // N + 1] * (B % N) + [B // N] * (N - B % N)
    b = oracle.head_budgets(np.full(N, 2.5), B, w, 0.3)
    assert list(b) == [B // N + 1] * (B % N) + [B // N] * (N - B % N)


def test_budget_apportionment_brute_force():
    # largest remainders give the integer vector with sum B closest to b* in
    # squared distance; enumerate every vector within one unit of the floors.
    for trial in range(30):
        N = int(RNG.integers(1, 6))
        w = int(RNG.integers(0, 8))
        B = N * w + int(RNG.integers(0, 40))
        rho = float(RNG.uniform(0, 1))
        s = RNG.uniform(0.1, 3.0, N)
        bs = np.array(oracle.head_budgets_real(s, B, w, rho))
        fl = np.floor(bs).astype(int)
        best = None
        for bump in itertools.product([0, 1], repeat=N):
            cand = fl + np.array(bump)
            if cand.sum() != B:
                continue
            dist = float(((cand - bs) ** 2).sum())
            if best is None or dist < best[0] - 1e-12:
                best = (dist, cand)
        assert best is not None
        assert list(oracle.head_budgets(s, B, w, rho)) == list(best[1])


def test_budget_cap_moves_excess_proportionally():
    # 3 heads, B = 300, w = 0, rho = 0: b* = 300 s / sum s = [150, 100, 50]
    # cap 120: head 0 keeps 120, its excess 30 goes 2:1 to heads 1, 2 -> [120, 120, 60]
    b = oracle.head_budgets([3.0, 2.0, 1.0], 300, 0, 0.0, cap=120)
    assert list(b) == [120, 120, 60]
    # cap 110: second round caps head 1 as well -> [110, 110, 80]
    b = oracle.head_budgets([3.0, 2.0, 1.0], 300, 0, 0.0, cap=110)
    assert list(b) == [110, 110, 80]


def test_budget_rejects_bad_input():
    with pytest.raises(ValueError):
        oracle.head_budgets([1.0, 1.0], 10, 8, 0.1)        # B < N w
    with pytest.raises(ValueError):
        oracle.head_budgets([1.0, -1.0], 100, 8, 0.1)
    with pytest.raises(ValueError):
        oracle.head_budgets([1.0, 1.0], 100, 8, 0.1, cap=40)


# ---------------------------------------------------------------------------
# a2 observation-window scoring (StD 3.2 equation; SparseMM window)
# ---------------------------------------------------------------------------

def _rand_case(B, Hq, Hkv, W, d, n):
    q = _bf16_round(RNG.standard_normal((B, Hq, W, d)))
    k = _bf16_round(RNG.standard_normal((B, Hkv, n, d)))
    return q, k


def test_score_each_row_sums_to_one():
    # every window query's softmax sums to 1, so sum_j score = G * W / W = G
    B, Hq, Hkv, W, d, n = 2, 6, 2, 5, 16, 40
    q, k = _rand_case(B, Hq, Hkv, W, d, n)
    sc = oracle.score_obs_window(q, k, n, q_pos0=n - W)
    assert np.allclose(sc.sum(axis=2), Hq // Hkv, rtol=1e-12)
    assert (sc >= 0).all()


def test_score_zero_queries_closed_form():
    # q = 0: query at position p spreads 1/(p+1) over keys 0..p
    B, Hq, Hkv, W, d, n, p0 = 1, 4, 2, 3, 8, 10, 5
    q = np.zeros((B, Hq, W, d))
    _, k = _rand_case(B, Hq, Hkv, W, d, n)
    sc = oracle.score_obs_window(q, k, n, q_pos0=p0)
    G = Hq // Hkv
    want = np.zeros(n)
    for t in range(W):
        p = p0 + t
        want[: p + 1] += 1.0 / (p + 1)
    want *= G / W
    assert np.allclose(sc[0, 0], want, rtol=1e-13)
    assert np.allclose(sc[0, 1], want, rtol=1e-13)


def test_score_two_keys_logistic_with_scale():
    # d = 4 so scale = 1/2; logits a*b/2 and 0 -> weights sigmoid(ab/2), 1 - that
    a, b = 3.0, 1.25
    q = np.zeros((1, 1, 1, 4)); q[0, 0, 0, 0] = a
    k = np.zeros((1, 1, 2, 4)); k[0, 0, 0, 0] = b
    sc = oracle.score_obs_window(q, k, 2, q_pos0=1)
    p0 = 1.0 / (1.0 + math.exp(-a * b / 2))
    assert sc[0, 0, 0] == pytest.approx(p0, rel=1e-14)
    assert sc[0, 0, 1] == pytest.approx(1 - p0, rel=1e-13)


def test_score_group_is_sum_of_member_heads():
    # GQA: KV head h sums the scores of query heads h*G .. h*G+G-1 (StD 3.2)
    B, Hq, Hkv, W, d, n = 1, 4, 2, 4, 8, 24
    q, k = _rand_case(B, Hq, Hkv, W, d, n)
    sc = oracle.score_obs_window(q, k, n, q_pos0=n - W)
    for h in range(Hkv):
        parts = [oracle.score_obs_window(q[:, [hq]], k[:, [h]], n, q_pos0=n - W)[0, 0]
                 for hq in (2 * h, 2 * h + 1)]
        assert np.allclose(sc[0, h], parts[0] + parts[1], rtol=1e-12)


def test_score_window_is_mean_over_its_queries():
    B, Hq, Hkv, W, d, n = 1, 2, 1, 4, 8, 20
    q, k = _rand_case(B, Hq, Hkv, W, d, n)
    p0 = n - W
    sc = oracle.score_obs_window(q, k, n, q_pos0=p0)
    acc = np.zeros(n)
    for t in range(W):
        acc += oracle.score_obs_window(q[:, :, [t]], k, n, q_pos0=p0 + t)[0, 0]
    assert np.allclose(sc[0, 0], acc / W, rtol=1e-12)


def test_score_brute_force_loops():
    B, Hq, Hkv, W, d, n = 1, 2, 1, 3, 3, 7
    q, k = _rand_case(B, Hq, Hkv, W, d, n)
    p0 = 3
    sc = oracle.score_obs_window(q, k, n, q_pos0=p0, scale=0.7)
    want = [0.0] * n
    for g in range(2):
        for t in range(W):
            last = p0 + t
            logits = []
            for j in range(last + 1):
                dot = 0.0
                for c in range(d):
                    dot += q[0, g, t, c] * k[0, 0, j, c]
                logits.append(0.7 * dot)
            mx = max(logits)
            den = sum(math.exp(x - mx) for x in logits)
            for j in range(last + 1):
                want[j] += math.exp(logits[j] - mx) / den / W
    assert np.allclose(sc[0, 0], want, rtol=1e-12)


# ---------------------------------------------------------------------------
# a3 top-K selection (StD argTopK; sinks + recent)
# ---------------------------------------------------------------------------

def test_select_brute_force_every_K():
    for trial in range(6):
        n = int(RNG.integers(8, 65))
        n_sink = int(RNG.integers(0, 3))
        n_recent = int(RNG.integers(0, 4))
        lo, hi = n_sink, n - n_recent
        # quantised scores so that ties occur
        sc = np.round(RNG.uniform(0, 1, (1, 2, n)) * 6) / 6
        for K in range(0, hi - lo + 1):
            kh = n_sink + K + n_recent
            offs = [0, kh, 2 * kh]
            got = oracle.select_topk(sc, n, lo, hi, n_sink, n_recent, offs)
            for h in range(2):
                ranked = sorted(range(lo, hi), key=lambda j: (-sc[0, h, j], j))
                want = sorted(list(range(n_sink)) + ranked[:K] + list(range(n - n_recent, n)))
                assert list(got[h * kh:(h + 1) * kh]) == want


def test_select_keep_all_and_ties():
    n = 30
    sc = np.zeros((1, 1, n))
    got = oracle.select_topk(sc, n, 0, n, 0, 0, [0, n])
    assert list(got) == list(range(n))
    # all equal: the lowest candidate indices win
    got = oracle.select_topk(sc + 0.5, n, 2, 25, 2, 5, [0, 2 + 7 + 5])
    assert list(got) == [0, 1] + list(range(2, 9)) + list(range(25, 30))


def test_select_nan_ranks_last_and_bad_sizes():
    sc = np.array([[[0.1, np.nan, 0.3, 0.2]]])
    assert list(oracle.select_topk(sc, 4, 0, 4, 0, 0, [0, 3])) == [0, 2, 3]
    sc = np.array([[[np.nan, -np.inf, 0.3, -0.0, 0.0]]])
    assert list(oracle.select_topk(sc, 5, 0, 5, 0, 0, [0, 3])) == [2, 3, 4]
    assert list(oracle.select_topk(sc, 5, 0, 5, 0, 0, [0, 4])) == [1, 2, 3, 4]
    with pytest.raises(ValueError):
        oracle.select_topk(sc, 4, 0, 4, 0, 0, [0, 5])


# ---------------------------------------------------------------------------
# a4 sparse decode, a5 dense verify (StD 3.1 / 3.2)
# ---------------------------------------------------------------------------

def _kvq(B, Hq, Hkv, n, d, gamma=None):
    k = _bf16_round(RNG.standard_normal((B, Hkv, n, d)))
    v = _bf16_round(RNG.standard_normal((B, Hkv, n, d)))
    shape = (B, Hq, d) if gamma is None else (B, Hq, gamma, d)
    q = _bf16_round(RNG.standard_normal(shape))
    return q, k, v


def test_sparse_keep_all_equals_dense():
    # a selection that keeps every entry reads the same bytes as dense decode
    B, Hq, Hkv, n, d = 2, 4, 2, 33, 16
    q, k, v = _kvq(B, Hq, Hkv, n, d)
    offs = np.arange(B * Hkv + 1) * n
    idx = np.tile(np.arange(n), B * Hkv)
    o_s, l_s = oracle.sparse_decode(q, k, v, offs, idx)
    o_d, l_d = oracle.dense_verify(q[:, :, None, :], k, v, n_prefix=n - 1)
    assert np.allclose(o_s, o_d[:, :, 0], rtol=1e-12, atol=1e-14)
    assert np.allclose(l_s, l_d[:, :, 0], rtol=1e-12)


def test_sparse_single_key_and_equal_keys():
    B, Hq, Hkv, n, d = 1, 2, 1, 12, 8
    q, k, v = _kvq(B, Hq, Hkv, n, d)
    o, lse = oracle.sparse_decode(q, k, v, [0, 1], [7])
    assert np.allclose(o[0, 0], v[0, 0, 7], rtol=0, atol=0)
    assert lse[0, 0] == pytest.approx(float(q[0, 0] @ k[0, 0, 7]) / math.sqrt(d), rel=1e-14)
    # all listed keys identical: uniform weights, o = mean of the listed values
    k2 = k.copy()
    k2[0, 0, :] = k[0, 0, 3]
    sel = [1, 4, 5, 9]
    o, lse = oracle.sparse_decode(q, k2, v, [0, 4], sel)
    assert np.allclose(o[0, 1], v[0, 0, sel].mean(axis=0), rtol=1e-13)
    z = float(q[0, 1] @ k[0, 0, 3]) / math.sqrt(d)
    assert lse[0, 1] == pytest.approx(z + math.log(4), rel=1e-13)


def test_sparse_two_keys_closed_form_and_huge_logit():
    d = 4
    q = np.zeros((1, 1, d)); q[0, 0, 0] = 2.0
    k = np.zeros((1, 1, 3, d)); k[0, 0, 0, 0] = 1.0; k[0, 0, 2, 0] = -1.0
    v = np.zeros((1, 1, 3, d)); v[0, 0, 0] = [1, 2, 3, 4]; v[0, 0, 2] = [-4, 0, 4, 8]
    o, lse = oracle.sparse_decode(q, k, v, [0, 2], [0, 2])      # logits +1, -1
    w0 = math.exp(1) / (math.exp(1) + math.exp(-1))
    assert np.allclose(o[0, 0], w0 * v[0, 0, 0] + (1 - w0) * v[0, 0, 2], rtol=1e-14)
    assert lse[0, 0] == pytest.approx(math.log(math.exp(1) + math.exp(-1)), rel=1e-14)
    q[0, 0, 0] = 3000.0                                           # weight -> 1 on key 0
    o, _ = oracle.sparse_decode(q, k, v, [0, 2], [0, 2])
    assert np.allclose(o[0, 0], v[0, 0, 0], rtol=0, atol=0)


def test_sparse_gqa_reads_kv_head_hq_div_G_and_empty_list():
    B, Hq, Hkv, n, d = 1, 4, 2, 6, 4
    q = np.zeros((B, Hq, d))
    k = np.zeros((B, Hkv, n, d))
    v = np.zeros((B, Hkv, n, d))
    v[0, 0] = 1.0
    v[0, 1] = 7.0
    o, _ = oracle.sparse_decode(q, k, v, [0, 2, 4], [0, 1, 2, 3])
    assert np.allclose(o[0, :2], 1.0) and np.allclose(o[0, 2:], 7.0)
    o, lse = oracle.sparse_decode(q, k, v, [0, 0, 2], [2, 3])
    assert np.allclose(o[0, :2], 0.0) and np.isneginf(lse[0, :2]).all()


def test_verify_equals_sequential_decodes():
    # StD 3.1: the parallel verify of gamma drafts is lossless, i.e. each draft
    # position sees exactly what a one-token decode at that position would see
    B, Hq, Hkv, d, gamma, n_prefix = 2, 6, 3, 16, 5, 29
    q, k, v = _kvq(B, Hq, Hkv, n_prefix + gamma, d, gamma=gamma)
    o, lse = oracle.dense_verify(q, k, v, n_prefix)
    for t in range(gamma):
        o1, l1 = oracle.dense_verify(q[:, :, [t]], k, v, n_prefix + t)
        assert np.allclose(o[:, :, t], o1[:, :, 0], rtol=1e-13, atol=1e-15)
        # and a sparse decode over the list 0 .. n_prefix + t
        offs = np.arange(B * Hkv + 1) * (n_prefix + t + 1)
        idx = np.tile(np.arange(n_prefix + t + 1), B * Hkv)
        o2, l2 = oracle.sparse_decode(q[:, :, t], k, v, offs, idx)
        assert np.allclose(o[:, :, t], o2, rtol=1e-12, atol=1e-14)
        assert np.allclose(lse[:, :, t], l2, rtol=1e-12)


def test_verify_zero_query_is_causal_prefix_mean():
    B, Hq, Hkv, d, gamma, n_prefix = 1, 2, 1, 8, 4, 9
    _, k, v = _kvq(B, Hq, Hkv, n_prefix + gamma, d, gamma=gamma)
    q = np.zeros((B, Hq, gamma, d))
    o, lse = oracle.dense_verify(q, k, v, n_prefix)
    for t in range(gamma):
        assert np.allclose(o[0, 0, t], v[0, 0, : n_prefix + t + 1].mean(axis=0), rtol=1e-13)
        assert lse[0, 1, t] == pytest.approx(math.log(n_prefix + t + 1), rel=1e-14)


# ---------------------------------------------------------------------------
# byte account (ByteCross "The Byte Crossover" and "Locating the Crossing")
# ---------------------------------------------------------------------------

def _golden(golden_dir):
    rows = []
    with open(os.path.join(golden_dir, "byte_crossover.txt")) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                rows.append(line.split())
    return rows


def test_byte_crossover_table(golden_dir):
    seen = 0
    for row in _golden(golden_dir):
        if row[0] == "crossover":
            d, dff, nstar, nstar_ff = int(row[2]), int(row[3]), float(row[4]), float(row[5])
            P = ba.projection_params(d, dff, 8, 128)
            assert round(ba.crossover_tokens(P, 8, 128, 0.5, 0.3) / 1024, 1) == nstar
            assert round(ba.crossover_tokens(3 * d * dff, 8, 128, 0.5, 0.3) / 1024, 1) == nstar_ff
            seen += 1
        elif row[0] == "pair":
            d, dff, rp, rkv, nstar = int(row[2]), int(row[3]), float(row[4]), float(row[5]), float(row[6])
            P = ba.projection_params(d, dff, 8, 128)
            assert round(ba.crossover_tokens(P, 8, 128, rp, rkv) / 1024, 1) == nstar
            seen += 1
        elif row[0] == "proj_mb":
            assert round(ba.projection_params(4096, 14336, 8, 128) * 2 / 1e6) == int(row[2])
        elif row[0] == "kv_per_token":
            assert ba.kv_bytes_per_token(8, 128) == int(row[2])
        elif row[0] == "kv_mb":
            assert round(ba.kv_bytes_per_token(8, 128) * int(row[1]) / 1e6) == int(row[2])
    assert seen == 8
