"""GPU parity of the calls around the hot path, through the C ABI, against the
oracle: list builders and compaction bit-exactly; decode over compacted rows
within the attention tolerances; the SpecVLM selection exactly, given the same
fp32 importance (integer decisions taken on identical inputs)."""
import math

import numpy as np
import pytest
import torch

import oracle
import sparse_kv_decode_gb300 as sk
import workloads
from gpu_common import assert_attn_close, assert_lse_close, csr, f64, scale_of

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from sparse_kv_decode_gb300 import build
    build.build()
    sk.lib()


def _rand(shape, gen, scale=1.0):
    return (scale * torch.randn(shape, generator=gen)).to(torch.bfloat16)


# --------------------------------------------------------------------------- window lists (f2)

@pytest.mark.parametrize("B,Hkv,n,n_sink,n_recent", [
    (1, 8, 32768, 4, 64), (2, 3, 100, 4, 96), (1, 4, 50, 60, 10), (3, 2, 10, 0, 0), (1, 1, 1000, 0, 17)])
def test_window_lists_exact(B, Hkv, n, n_sink, n_recent):
    offs, idx = sk.window_lists(B, Hkv, n, n_sink, n_recent, DEV)
    ro, ri = oracle.window_lists(B, Hkv, n, n_sink, n_recent)
    assert offs.cpu().numpy().tolist() == ro.tolist()
    total = int(ro[-1])
    assert idx[:total].cpu().numpy().tolist() == ri.tolist()


def test_window_lists_feed_sparse_decode():
    g = torch.Generator().manual_seed(31)
    B, Hq, Hkv, d, n = 1, 32, 8, 128, 4096
    k, v = _rand((B, Hkv, n, d), g), _rand((B, Hkv, n, d), g)
    q = _rand((B, Hq, d), g)
    offs, idx = sk.window_lists(B, Hkv, n, 4, 64, DEV)
    o, lse = sk.sparse_decode_attn(q.to(DEV), k.to(DEV), v.to(DEV), offs, idx, scale_of(d))
    ro, ri = oracle.window_lists(B, Hkv, n, 4, 64)
    o_ref, l_ref = oracle.sparse_decode(q, k, v, ro, ri)
    assert_attn_close(o, o_ref, "window decode")
    assert_lse_close(lse, l_ref, "window decode")


# --------------------------------------------------------------------------- draft lists (f4)

def test_append_drafts_exact():
    rng = np.random.default_rng(32)
    lens = [5, 0, 130, 1, 77, 1024]
    base_o = np.concatenate([[7], 7 + np.cumsum(lens)]).astype(np.int32)          # starts inside the array
    base_i = np.concatenate([rng.integers(0, 10000, 7)] +
                            [np.sort(rng.choice(12000, L, replace=False)) for L in lens]).astype(np.int32)
    bo, bi = torch.tensor(base_o, device=DEV), torch.tensor(base_i, device=DEV)
    for n_new in (0, 1, 5):
        offs, idx = sk.append_drafts(bo, bi, int(sum(lens)), 12000, n_new)
        ro, ri = oracle.append_drafts(base_o, base_i, 12000, n_new)
        assert offs.cpu().numpy().tolist() == ro.tolist()
        assert idx[: int(ro[-1])].cpu().numpy().tolist() == ri.tolist()


def test_draft_lists_equal_appends():
    rng = np.random.default_rng(35)
    lens = [5, 0, 130, 1, 77, 1024]
    base_o = np.concatenate([[3], 3 + np.cumsum(lens)]).astype(np.int32)
    base_i = np.concatenate([rng.integers(0, 10000, 3)] +
                            [np.sort(rng.choice(12000, L, replace=False)) for L in lens]).astype(np.int32)
    bo, bi = torch.tensor(base_o, device=DEV), torch.tensor(base_i, device=DEV)
    gamma = 5
    offs, idx = sk.draft_lists(bo, bi, int(sum(lens)), 12000, gamma)
    for t in range(gamma):
        ro, ri = oracle.append_drafts(base_o, base_i, 12000, t + 1)
        assert offs[t].cpu().numpy().tolist() == ro.tolist()
        assert idx[t, : int(ro[-1])].cpu().numpy().tolist() == ri.tolist()


# --------------------------------------------------------------------------- compaction + decode (f1)

def _lists(B, Hkv, n, lens, seed, lead=0):
    rng = np.random.default_rng(seed)
    offs = np.concatenate([[lead], lead + np.cumsum(lens)]).astype(np.int32)
    parts = [rng.integers(0, n, lead)] + [np.sort(rng.choice(n, L, replace=False)) for L in lens]
    return offs, np.concatenate(parts).astype(np.int32)


@pytest.mark.parametrize("B,Hkv,n,d,lens,lead", [
    (1, 8, 4096, 128, [1229] * 8, 0),
    (2, 4, 3000, 128, [0, 1, 2, 63, 64, 65, 500, 2999], 3),
    (1, 4, 1024, 64, [128, 0, 97, 1024], 0),
])
def test_compact_kv_exact(B, Hkv, n, d, lens, lead):
    g = torch.Generator().manual_seed(n + d)
    k, v = _rand((B, Hkv, n, d), g), _rand((B, Hkv, n, d), g)
    offs, idx = _lists(B, Hkv, n, lens, n, lead)
    total = int(sum(lens))
    ws = sk.new_workspace(sk.workspace_size(sk.OP_COMPACT, B, 0, Hkv, d, 0, 0), DEV)
    k_c, v_c = sk.compact_kv(k.to(DEV), v.to(DEV), torch.tensor(offs, device=DEV), torch.tensor(idx, device=DEV),
                             total, ws=ws)
    rk, rv = oracle.compact_kv(k, v, offs, idx)
    assert np.array_equal(f64(k_c[:total]), rk) and np.array_equal(f64(v_c[:total]), rv)
    assert sk.workspace_status(ws) == 0


def test_compact_kv_flags_bad_index():
    g = torch.Generator().manual_seed(33)
    k, v = _rand((1, 2, 64, 64), g), _rand((1, 2, 64, 64), g)
    offs = torch.tensor([0, 2, 4], dtype=torch.int32, device=DEV)
    idx = torch.tensor([3, 64, -1, 5], dtype=torch.int32, device=DEV)
    ws = sk.new_workspace(sk.workspace_size(sk.OP_COMPACT, 1, 0, 2, 64, 0, 0), DEV)
    sk.compact_kv(k.to(DEV), v.to(DEV), offs, idx, 4, ws=ws)
    assert sk.workspace_status(ws) == sk._lib.SDKV_DEV_BAD_INDEX


@pytest.mark.parametrize("B,Hq,Hkv,d,n,lens", [
    (1, 4, 4, 64, 1024, [128, 128, 128, 128]),
    (1, 32, 8, 128, 8192, [2458] * 8),
    (2, 4, 4, 128, 3000, [0, 1, 2, 63, 64, 65, 500, 2999]),
    (1, 28, 4, 128, 2000, [1024, 1025, 1026, 1027]),
    (2, 32, 32, 128, 1024, list(np.random.default_rng(34).integers(0, 1025, 64))),
])
def test_sparse_decode_compact_matches_oracle(B, Hq, Hkv, d, n, lens):
    g = torch.Generator().manual_seed(n + Hq + 1)
    k, v = _rand((B, Hkv, n, d), g), _rand((B, Hkv, n, d), g)
    q = _rand((B, Hq, d), g, 1.5)
    offs, idx = _lists(B, Hkv, n, lens, n + 1)
    total = int(sum(lens))
    od, idd = torch.tensor(offs, device=DEV), torch.tensor(idx, device=DEV)
    k_c, v_c = sk.compact_kv(k.to(DEV), v.to(DEV), od, idd, total)
    ws = sk.new_workspace(sk.workspace_size(sk.OP_SPARSE_DECODE, B, Hq, Hkv, d, 0, 0), DEV)
    for _ in range(2):
        o, lse = sk.sparse_decode_compact(q.to(DEV), k_c, v_c, od, Hkv, scale_of(d), ws=ws)
        o_ref, l_ref = oracle.sparse_decode(q, k, v, offs, idx)
        assert_attn_close(o, o_ref, "compact decode")
        assert_lse_close(lse, l_ref, "compact decode")
    # the same lists gathered directly give the same attention
    o_g, l_g = sk.sparse_decode_attn(q.to(DEV), k.to(DEV), v.to(DEV), od, idd, scale_of(d))
    assert (f64(o) - f64(o_g)).__abs__().max() <= 1e-2
    assert sk.workspace_status(ws) == 0


# --------------------------------------------------------------------------- SpecVLM selection (f3)

def _spec_case(B, units, n, v_lo, v_hi, keep_lo, keep_hi, lam, r, seed):
    g = torch.Generator().manual_seed(seed)
    # attention-like scores: non-negative, a few tokens carrying more mass
    s = torch.rand((B, units, n), generator=g) ** 4
    hot = torch.randint(0, n, (B, max(n // 50, 1)), generator=g)
    for b in range(B):
        s[b, :, hot[b]] *= 30
    imp, idx, cnt = sk.specvlm_select(s.to(DEV), v_lo, v_hi, lam, r, keep_lo, keep_hi)
    imp_ref = np.stack([oracle.specvlm_importance(s[b]) for b in range(B)])
    assert np.abs(f64(imp) - imp_ref).max() <= 1e-5 * max(1.0, np.abs(imp_ref).max())
    imp_gpu = imp.cpu().numpy()
    for b in range(B):
        want = oracle.specvlm_select(imp_gpu[b], v_lo, v_hi, lam, r, keep_lo, keep_hi)
        got = idx[b, : int(cnt[b])].cpu().numpy()
        assert np.array_equal(got, want), (b, len(got), len(want))
    return cnt


@pytest.mark.parametrize("B,units,n,v_lo,v_hi,keep_lo,keep_hi,lam,r", [
    (1, 112, 12800, 0, 12544, 12544, 12800, 0.5, 0.9),      # the video workload: 28 layers x 4 KV heads
    (1, 112, 12800, 0, 12544, 12544, 12800, 0.4, 0.9),
    (2, 8, 3000, 100, 2900, 0, 100, 0.7, 0.8),              # kept range before the video tokens
    (1, 4, 20000, 0, 20000, 0, 0, 0.5, 0.9),                # more tokens than sort in shared memory
    (1, 4, 777, 0, 777, 777, 777, 0.0, 0.9),                # no Stage I: every tenth token
    (1, 4, 777, 0, 777, 777, 777, 1.0, 0.5),
    (1, 4, 300, 0, 300, 0, 0, 0.3, 0.0),                    # r = 0 keeps everything
    (1, 3, 40, 10, 10, 0, 40, 0.5, 0.9),                    # no video tokens
])
def test_specvlm_select_exact(B, units, n, v_lo, v_hi, keep_lo, keep_hi, lam, r):
    _spec_case(B, units, n, v_lo, v_hi, keep_lo, keep_hi, lam, r, seed=n + units)


def test_specvlm_ties_take_lower_tokens():
    # all video tokens equal: Stage I takes the lowest indices first
    s = torch.ones((1, 2, 64), dtype=torch.float32)
    imp, idx, cnt = sk.specvlm_select(s.to(DEV), 0, 64, 0.25, 0.999, 64, 64)
    want = oracle.specvlm_select(imp.cpu().numpy()[0], 0, 64, 0.25, 0.999, 64, 64)
    assert idx[0, : int(cnt[0])].cpu().numpy().tolist() == want.tolist()
    assert want[:16].tolist() == list(range(16))
