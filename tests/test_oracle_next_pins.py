"""Pins of the oracle's next-row functions (CPU): closed forms, brute force and
invariants that do not retype the functions' own formulas."""
import itertools
import math

import numpy as np
import pytest
import torch

import oracle


def test_window_lists_closed_form_and_overlap():
    offs, idx = oracle.window_lists(2, 3, 1000, 4, 64)
    assert offs.tolist() == [68 * i for i in range(7)]
    want = list(range(4)) + list(range(936, 1000))
    for i in range(6):
        assert idx[offs[i]: offs[i + 1]].tolist() == want
    # sinks and window overlap: every row once
    offs, idx = oracle.window_lists(1, 1, 50, 30, 40)
    assert idx.tolist() == list(range(50))
    offs, idx = oracle.window_lists(1, 2, 5, 0, 0)
    assert offs.tolist() == [0, 0, 0] and idx.size == 0


def test_compact_kv_rows_are_the_listed_rows():
    g = torch.Generator().manual_seed(1)
    B, Hkv, n, d = 2, 3, 40, 8
    k = torch.randn((B, Hkv, n, d), generator=g).to(torch.bfloat16)
    v = torch.randn((B, Hkv, n, d), generator=g).to(torch.bfloat16)
    lens = [3, 0, 7, 1, 40, 5]
    rng = np.random.default_rng(1)
    offs = np.concatenate([[0], np.cumsum(lens)])
    idx = np.concatenate([np.sort(rng.choice(n, L, replace=False)) for L in lens]).astype(np.int32)
    k_c, v_c = oracle.compact_kv(k, v, offs, idx)
    row = 0
    for i, L in enumerate(lens):
        b, h = divmod(i, Hkv)
        for j in idx[offs[i]: offs[i + 1]]:
            assert np.array_equal(k_c[row], k[b, h, j].double().numpy())
            assert np.array_equal(v_c[row], v[b, h, j].double().numpy())
            row += 1
    assert row == k_c.shape[0] == sum(lens)


def test_compact_decode_keep_all_equals_dense_decode():
    # compacting every row in order and decoding over the compacted buffer is
    # the dense single-query decode over the whole cache (a5 with gamma = 1)
    g = torch.Generator().manual_seed(2)
    B, Hq, Hkv, n, d = 2, 4, 2, 33, 16
    k = torch.randn((B, Hkv, n, d), generator=g).to(torch.bfloat16)
    v = torch.randn((B, Hkv, n, d), generator=g).to(torch.bfloat16)
    q = torch.randn((B, Hq, d), generator=g).to(torch.bfloat16)
    offs = np.arange(B * Hkv + 1) * n
    idx = np.tile(np.arange(n), B * Hkv).astype(np.int32)
    k_c, v_c = oracle.compact_kv(k, v, offs, idx)
    o, lse = oracle.sparse_decode_compact(q, k_c, v_c, offs, Hkv)
    od, ld = oracle.dense_verify(q[:, :, None], k, v, n - 1)
    assert np.allclose(o, od[:, :, 0], atol=1e-12) and np.allclose(lse, ld[:, :, 0], atol=1e-12)


def _mass_ints(a):
    return [int(np.rint(float(x) * 2.0 ** oracle.MASS_FRAC_BITS)) for x in a]


def test_specvlm_stage1_is_the_smallest_set_reaching_the_mass():
    # brute force over every subset: the retained prefix has the minimum size of
    # any token set whose mass reaches lam_r of the total
    rng = np.random.default_rng(3)
    for trial in range(30):
        nV = 9
        a = rng.random(nV).astype(np.float32) ** 3
        lam = float(rng.choice([0.2, 0.4, 0.5, 0.77, 0.95]))
        fx = _mass_ints(a)
        target = lam * float(sum(fx))
        best = min(len(c) for m in range(nV + 1) for c in itertools.combinations(range(nV), m)
                   if float(sum(fx[j] for j in c)) >= target)
        out = oracle.specvlm_select(a, 0, nV, lam, 0.999999, nV, nV)
        # with r near 1 the interval is huge: Stage II adds only the first leftover
        retained = len(out) - (1 if len(out) < nV else 0)
        assert retained == best or len(out) == nV, (trial, out, best)


def test_specvlm_stage2_count_and_positions_exact():
    # lam_r = 0 keeps nothing in Stage I; the walk then takes positions floor(k I)
    # with I = 1 / (1 - r): for r = 0.9 every tenth token starting at the first
    a = np.ones(95, dtype=np.float32)
    out = oracle.specvlm_select(a, 0, 95, 0.0, 0.9, 95, 95)
    assert out.tolist() == list(range(0, 95, 10))
    # general case: Stage I is the exact prefix; Stage II walks the leftovers in
    # steps of floor(I) or ceil(I) from the first one, about L / I of them
    rng = np.random.default_rng(4)
    for trial in range(40):
        nV = int(rng.integers(5, 60))
        a = rng.random(nV).astype(np.float32)
        lam, r = float(rng.random()), float(rng.choice([0.5, 0.8, 0.9]))
        out = set(oracle.specvlm_select(a, 0, nV, lam, r, nV, nV).tolist())
        fx = _mass_ints(a)
        order = sorted(range(nV), key=lambda j: (-float(a[j]), j))
        target, acc, c = lam * float(sum(fx)), 0, 0
        while c < nV and float(acc) < target:
            acc += fx[order[c]]
            c += 1
        retained = set(order[:c])
        assert retained <= out
        left = sorted(set(range(nV)) - retained)
        pos = [left.index(x) for x in sorted(out - retained)]
        if not left:
            assert not pos
            continue
        I = float(nV - c) / ((1.0 - r) * float(nV))
        assert pos[0] == 0
        if I >= 1:
            assert all(math.floor(I) <= y - x <= math.ceil(I) for x, y in zip(pos, pos[1:])), (pos, I)
            assert abs(len(pos) - math.ceil(len(left) / I)) <= 1
        else:
            assert pos == list(range(len(left)))


def test_specvlm_extremes():
    a = np.array([0.0, 0.2, 0.0, 0.5, 0.3], dtype=np.float32)
    # lam_r = 1: every token with mass is retained; r = 0 keeps everything
    assert oracle.specvlm_select(a, 0, 5, 1.0, 0.0, 5, 5).tolist() == [0, 1, 2, 3, 4]
    out = oracle.specvlm_select(a, 0, 5, 1.0, 0.9, 5, 7).tolist()
    assert {1, 3, 4} <= set(out) and out[-2:] == [5, 6]
    # ties: lower index first
    b = np.array([0.25, 0.25, 0.25, 0.25], dtype=np.float32)
    assert oracle.specvlm_select(b, 0, 4, 0.5, 0.999999, 4, 4).tolist()[:2] == [0, 1]
    assert oracle.specvlm_importance(np.ones((3, 4, 7))).tolist() == [1.0] * 7


def test_append_drafts_equals_lists_built_per_step():
    bo = np.array([0, 3, 3, 6])
    bi = np.array([0, 2, 5, 1, 4, 6], dtype=np.int32)
    for t in range(4):
        offs, idx = oracle.append_drafts(bo, bi, 10, t + 1)
        for i in range(3):
            want = list(bi[bo[i]: bo[i + 1]]) + list(range(10, 10 + t + 1))
            assert idx[offs[i]: offs[i + 1]].tolist() == want


def test_compact_kv_csr_starting_inside_a_larger_array():
    # the lists may start at offsets[0] > 0 (a slice of a larger CSR): output row
    # 0 is the first listed row, not row offsets[0]
    g = torch.Generator().manual_seed(5)
    k = torch.randn((1, 2, 12, 4), generator=g).to(torch.bfloat16)
    v = torch.randn((1, 2, 12, 4), generator=g).to(torch.bfloat16)
    idx = np.array([9, 9, 9, 1, 4, 7, 0, 11], dtype=np.int32)   # three entries before the lists
    offs = np.array([3, 6, 8])
    k_c, v_c = oracle.compact_kv(k, v, offs, idx)
    assert k_c.shape == (5, 4)
    assert np.array_equal(k_c[0], k[0, 0, 1].double().numpy())
    assert np.array_equal(v_c[4], v[0, 1, 11].double().numpy())
