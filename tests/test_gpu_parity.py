"""GPU parity: every hot-path kernel, called through the C ABI, against the fp64
oracle on the same seeded inputs.  Small cases span several tiles with ragged
tails; edge cases cover empty and single-entry lists, gamma > 1, odd group
sizes, both head dims and non-contiguous caches."""
import math

import numpy as np
import pytest
import torch

import oracle
import sparse_kv_decode_gb300 as sk
import workloads
from gpu_common import (LSE_MAX_ABS, assert_attn_close, assert_lse_close, assert_scores_close,
                        check_selection_gap_rule, csr, f64, scale_of)

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


def _status_ok(ws):
    assert sk.workspace_status(ws) == 0


# ---------------------------------------------------------------------------
# a5 dense verify / decode
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("B,Hq,Hkv,d,n_prefix,gamma", [
    (1, 4, 4, 64, 1023, 1),       # tiny workload, dense decode
    (1, 4, 4, 64, 1020, 4),       # tiny workload, gamma = 4 verify
    (2, 8, 2, 128, 3000, 1),      # GQA 4, ragged tail
    (1, 32, 8, 128, 5000, 8),     # 32 rows per KV head (two row tiles)
    (1, 28, 4, 128, 2000, 5),     # video shape: 35 rows (three row tiles)
    (1, 4, 1, 128, 700, 16),      # 64 rows (four row tiles)
    (1, 64, 32, 128, 3000, 9),    # 18 rows, clusters of two
    (8, 32, 8, 128, 600, 5),      # 20 rows, several chunks a head, no cluster
    (2, 8, 2, 128, 40, 5),        # 20 rows, one chunk a head
    (3, 6, 3, 64, 77, 3),         # short cache, fewer keys than a tile per split
    (1, 2, 2, 128, 0, 1),         # a single key
    (1, 16, 2, 64, 900, 4),       # d = 64 with 32 rows (the mma.sync path's row tiles)
    (1, 17, 1, 128, 2500, 1),     # 17 rows: a one-query decode on the tensor-core verify
    (1, 22, 2, 128, 1800, 3),     # 33 rows: the smallest case with two row groups
])
def test_dense_verify_matches_oracle(B, Hq, Hkv, d, n_prefix, gamma):
    g = torch.Generator().manual_seed(B * 1000 + Hq * 10 + gamma)
    rows = n_prefix + gamma
    k = _rand((B, Hkv, rows, d), g)
    v = _rand((B, Hkv, rows, d), g)
    q = _rand((B, Hq, gamma, d), g, 1.5)
    ws = sk.new_workspace(sk.workspace_size(sk.OP_DENSE_VERIFY, B, Hq, Hkv, d, rows, gamma), DEV)
    o, lse = sk.dense_verify_attn(q.to(DEV), k.to(DEV), v.to(DEV), n_prefix, scale_of(d), ws=ws)
    o_ref, l_ref = oracle.dense_verify(q, k, v, n_prefix)
    assert_attn_close(o, o_ref, "dense")
    assert_lse_close(lse, l_ref, "dense")
    _status_ok(ws)


@pytest.mark.parametrize("B,Hq,Hkv,n_prefix,gamma", [(1, 32, 8, 6000, 8), (40, 32, 8, 300, 5), (40, 28, 4, 300, 5)])
def test_dense_verify_rising_scores(B, Hq, Hkv, n_prefix, gamma):
    # keys whose norm grows along the cache: a row's running max rises by many
    # binades inside a chunk, so the output accumulated so far must be rescaled.
    # Such rows put nearly all weight on one or two keys, so an output is about
    # one value row; values are scaled to stay below 2, where rounding the bf16
    # output costs at most 2^-8 (a randn row can reach 4, where it costs 2^-7,
    # past the 1e-2 bound whatever the kernel does).
    g = torch.Generator().manual_seed(77 + B)
    d = 128
    rows = n_prefix + gamma
    ramp = torch.linspace(0.2, 6.0, rows, dtype=torch.float64).view(1, 1, rows, 1)
    k = (_rand((B, Hkv, rows, d), g).double() * ramp).to(torch.bfloat16)
    v = _rand((B, Hkv, rows, d), g, 0.4)
    q = _rand((B, Hq, gamma, d), g, 1.5)
    o, lse = sk.dense_verify_attn(q.to(DEV), k.to(DEV), v.to(DEV), n_prefix, scale_of(d))
    o_ref, l_ref = oracle.dense_verify(q, k, v, n_prefix)
    assert_attn_close(o, o_ref, "dense")
    assert_lse_close(lse, l_ref, "dense")


@pytest.mark.parametrize("Hq,gamma", [(8, 3), (16, 5), (28, 5)])
def test_dense_verify_strided_cache_and_repeat_calls(Hq, gamma):
    # the cache has spare capacity rows (n_cap > n) and heads interleaved with
    # batch: strides differ from a packed layout; the same workspace is reused,
    # so the per-head counters must be back at zero after every call.  6, 20
    # and 35 query rows per KV head: the mma.sync verify and both row-group
    # counts of the tensor-core one
    g = torch.Generator().manual_seed(5 + Hq)
    B, Hkv, d, n_prefix, n_cap = 2, 4, 128, 1500, 1600
    big = _rand((Hkv, B, n_cap, d), g)
    k = big.permute(1, 0, 2, 3)
    v = _rand((Hkv, B, n_cap, d), g).permute(1, 0, 2, 3)
    q = _rand((B, Hq, gamma, d), g)
    ws = sk.new_workspace(sk.workspace_size(sk.OP_DENSE_VERIFY, B, Hq, Hkv, d, n_prefix + gamma, gamma), DEV)
    kd, vd, qd = k.to(DEV), v.to(DEV), q.to(DEV)
    assert kd.stride() == k.stride()
    o_ref, l_ref = oracle.dense_verify(q, k, v, n_prefix)
    for _ in range(3):
        o, lse = sk.dense_verify_attn(qd, kd, vd, n_prefix, scale_of(d), ws=ws)
        assert_attn_close(o, o_ref, "dense strided")
        assert_lse_close(lse, l_ref, "dense strided")
    _status_ok(ws)


def test_verify_equals_sequential_single_decodes_on_gpu():
    # StD 3.1: the one-pass verify of gamma drafts equals gamma single-token decodes
    g = torch.Generator().manual_seed(11)
    B, Hq, Hkv, d, n_prefix, gamma = 1, 32, 8, 128, 4096, 8
    k = _rand((B, Hkv, n_prefix + gamma, d), g).to(DEV)
    v = _rand((B, Hkv, n_prefix + gamma, d), g).to(DEV)
    q = _rand((B, Hq, gamma, d), g).to(DEV)
    o, lse = sk.dense_verify_attn(q, k, v, n_prefix, scale_of(d))
    for t in range(gamma):
        o1, l1 = sk.dense_verify_attn(q[:, :, t:t + 1].contiguous(), k, v, n_prefix + t, scale_of(d))
        assert (f64(o[:, :, t]) - f64(o1[:, :, 0])).__abs__().max() <= 1e-2
        # the verify sums its bf16-rounded weights (several row tiles), the decode
        # its fp32 ones: they agree within the lse tolerance both keep to the oracle
        assert (f64(lse[:, :, t]) - f64(l1[:, :, 0])).__abs__().max() <= LSE_MAX_ABS


# ---------------------------------------------------------------------------
# a4 sparse decode
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("B,Hq,Hkv,d,n,lens", [
    (1, 4, 4, 64, 1024, [128, 128, 128, 128]),
    (1, 32, 8, 128, 4096, [1229] * 8),
    (2, 4, 4, 128, 3000, [0, 1, 2, 63, 64, 65, 500, 2999]),   # empty, single, tile edges, ragged
    (1, 28, 4, 128, 2000, [1024, 1025, 1026, 1027]),
    (1, 64, 2, 128, 1500, [700, 900]),                        # group 32: two row tiles
    (1, 8, 8, 128, 6000, [3, 5000, 17, 1, 4096, 64, 0, 2048]),
])
def test_sparse_decode_matches_oracle(B, Hq, Hkv, d, n, lens):
    g = torch.Generator().manual_seed(n + Hq)
    k = _rand((B, Hkv, n, d), g)
    v = _rand((B, Hkv, n, d), g)
    q = _rand((B, Hq, d), g, 1.5)
    offs_d, offs = csr(lens, DEV)
    _, idx = workloads.random_lists(B, Hkv, n, lens, seed=n)
    ws = sk.new_workspace(sk.workspace_size(sk.OP_SPARSE_DECODE, B, Hq, Hkv, d, 0, 0), DEV)
    o, lse = sk.sparse_decode_attn(q.to(DEV), k.to(DEV), v.to(DEV), offs_d, idx.to(DEV), scale_of(d), ws=ws)
    o_ref, l_ref = oracle.sparse_decode(q, k, v, offs, idx.numpy())
    assert_attn_close(o, o_ref, "sparse")
    assert_lse_close(lse, l_ref, "sparse")
    _status_ok(ws)


def test_sparse_many_short_lists():
    # 20,480 (sequence, KV head) lists of 0..2 entries: the CTA ranges cross more
    # than a hundred heads each (offsets read on the fly), and the range plan
    # reads the offsets in several rounds
    g = torch.Generator().manual_seed(21)
    B, Hq, Hkv, d, n = 80, 256, 256, 64, 16
    k = _rand((B, Hkv, n, d), g)
    v = _rand((B, Hkv, n, d), g, 0.5)   # |o| < 4: a bf16 output then rounds by less than 1e-2
    q = _rand((B, Hq, d), g)
    rng = np.random.default_rng(21)
    lens = rng.integers(0, 3, size=B * Hkv).tolist()
    offs_d, offs = csr(lens, DEV)
    _, idx = workloads.random_lists(B, Hkv, n, lens, seed=21)
    ws = sk.new_workspace(sk.workspace_size(sk.OP_SPARSE_DECODE, B, Hq, Hkv, d, 0, 0), DEV)
    o, lse = sk.sparse_decode_attn(q.to(DEV), k.to(DEV), v.to(DEV), offs_d, idx.to(DEV), scale_of(d), ws=ws)
    o_ref, l_ref = oracle.sparse_decode(q, k, v, offs, idx.numpy())
    assert_attn_close(o, o_ref, "sparse short lists")
    assert_lse_close(lse, l_ref, "sparse short lists")
    _status_ok(ws)


@pytest.mark.parametrize("Hkv", [31, 32, 33])
def test_sparse_head_count_around_one_warp(Hkv):
    # up to 32 (sequence, KV head) lists one warp plans the chunks, beyond that
    # the whole block does: both sides of the switch, ragged lengths incl. empty
    g = torch.Generator().manual_seed(40 + Hkv)
    B, d, n = 1, 64, 1500
    Hq = Hkv
    k = _rand((B, Hkv, n, d), g)
    v = _rand((B, Hkv, n, d), g)
    q = _rand((B, Hq, d), g)
    rng = np.random.default_rng(40 + Hkv)
    lens = rng.integers(0, n + 1, size=B * Hkv).tolist()
    lens[0], lens[-1] = 0, n
    offs_d, offs = csr(lens, DEV)
    _, idx = workloads.random_lists(B, Hkv, n, lens, seed=40 + Hkv)
    ws = sk.new_workspace(sk.workspace_size(sk.OP_SPARSE_DECODE, B, Hq, Hkv, d, 0, 0), DEV)
    o, lse = sk.sparse_decode_attn(q.to(DEV), k.to(DEV), v.to(DEV), offs_d, idx.to(DEV), scale_of(d), ws=ws)
    o_ref, l_ref = oracle.sparse_decode(q, k, v, offs, idx.numpy())
    assert_attn_close(o, o_ref, "sparse %d heads" % Hkv)
    assert_lse_close(lse, l_ref, "sparse %d heads" % Hkv)
    _status_ok(ws)


def test_sparse_ragged_mha_lists_cross_ranges():
    # SparseMM-like: one query row per KV head, lengths from 0 to the whole cache,
    # so CTA ranges start and end inside lists and span several lists
    g = torch.Generator().manual_seed(22)
    B, Hq, Hkv, d, n = 2, 32, 32, 128, 2048
    k = _rand((B, Hkv, n, d), g)
    v = _rand((B, Hkv, n, d), g)
    q = _rand((B, Hq, d), g, 1.5)
    rng = np.random.default_rng(22)
    lens = rng.integers(0, n + 1, size=B * Hkv).tolist()
    lens[3] = 0
    lens[4] = n
    offs_d, offs = csr(lens, DEV)
    _, idx = workloads.random_lists(B, Hkv, n, lens, seed=22)
    ws = sk.new_workspace(sk.workspace_size(sk.OP_SPARSE_DECODE, B, Hq, Hkv, d, 0, 0), DEV)
    for _ in range(2):   # the per-head tickets are back at zero after a call
        o, lse = sk.sparse_decode_attn(q.to(DEV), k.to(DEV), v.to(DEV), offs_d, idx.to(DEV), scale_of(d), ws=ws)
        o_ref, l_ref = oracle.sparse_decode(q, k, v, offs, idx.numpy())
        assert_attn_close(o, o_ref, "sparse ragged mha")
        assert_lse_close(lse, l_ref, "sparse ragged mha")
    _status_ok(ws)


def _packed_lens(kind, BH, n, rng):
    if kind == "sparsemm":     # most lists 50..250 entries, one in ten 1000..n, a few empty
        lens = np.where(rng.random(BH) < 0.1, rng.integers(1000, n + 1, BH), rng.integers(50, 251, BH))
        lens[rng.integers(0, BH, 3)] = 0
    elif kind == "uniform":
        lens = rng.integers(0, 401, BH)
    elif kind == "tiny":       # 0..3 entries: spans hold tens of lists, several passes of 16 / R
        lens = rng.integers(0, 4, BH)
    elif kind == "empty":
        lens = np.zeros(BH, np.int64)
    elif kind == "one_long":   # one list over the whole cache among empty ones: cut by many spans
        lens = np.zeros(BH, np.int64)
        lens[BH // 3] = n
    return [int(x) for x in lens]


@pytest.mark.parametrize("B,Hq,Hkv,d,n,kind", [
    (8, 32, 32, 128, 4000, "sparsemm"),   # MHA, 256 lists: one query row per list, 16 lists a pass
    (4, 64, 32, 64, 900, "uniform"),      # 2 rows per list, head dim 64
    (16, 32, 8, 128, 1500, "uniform"),    # GQA 4: 4 lists a pass
    (25, 12, 4, 64, 700, "uniform"),      # 3 rows per list: 5 lists a pass, one padding row
    (80, 16, 1, 128, 600, "uniform"),     # 16 rows per list: one list a pass
    (12, 64, 8, 64, 1200, "sparsemm"),    # GQA 8 at d = 64: 2 lists a pass
    (20, 20, 4, 128, 900, "uniform"),     # 5 rows per list: 3 lists a pass, one padding row
    (32, 32, 32, 64, 64, "tiny"),         # 1024 lists of 0..3 entries
    (4, 25, 25, 128, 300, "empty"),       # every list empty
    (2, 50, 50, 128, 9000, "one_long"),   # one list cut by ~70 spans, merged by the last of them
])
def test_sparse_packed_lists_match_oracle(B, Hq, Hkv, d, n, kind):
    # more lists than the clusters of one wave cover: the CTAs take equal spans of
    # the concatenated lists, several short lists per pass; lists cut by span ends
    # are merged through the per-list tickets, which are back at zero after a call
    seed = 60 + B + Hkv + d
    g = torch.Generator().manual_seed(seed)
    k = _rand((B, Hkv, n, d), g)
    v = _rand((B, Hkv, n, d), g, 0.5)   # |o| < 4 even for lists of a few entries: bf16 output rounds < 1e-2
    q = _rand((B, Hq, d), g, 1.5)
    rng = np.random.default_rng(seed)
    lens = _packed_lens(kind, B * Hkv, n, rng)
    offs_d, offs = csr(lens, DEV)
    _, idx = workloads.random_lists(B, Hkv, n, lens, seed=seed)
    if idx.numel() == 0:
        idx = torch.zeros(1, dtype=torch.int32)   # the index array must exist even when no list has entries
    ws = sk.new_workspace(sk.workspace_size(sk.OP_SPARSE_DECODE, B, Hq, Hkv, d, 0, 0), DEV)
    o_ref, l_ref = oracle.sparse_decode(q, k, v, offs, idx.numpy())
    qd, kd, vd, idxd = q.to(DEV), k.to(DEV), v.to(DEV), idx.to(DEV)
    for _ in range(2):
        o, lse = sk.sparse_decode_attn(qd, kd, vd, offs_d, idxd, scale_of(d), ws=ws)
        assert_attn_close(o, o_ref, "packed %s" % kind)
        assert_lse_close(lse, l_ref, "packed %s" % kind)
    _status_ok(ws)


def test_sparse_packed_lists_with_an_offset_base():
    # offsets[0] > 0: the lists sit at the end of a longer index array
    seed = 71
    g = torch.Generator().manual_seed(seed)
    B, Hq, Hkv, d, n, base = 4, 32, 32, 128, 1000, 37
    k = _rand((B, Hkv, n, d), g)
    v = _rand((B, Hkv, n, d), g, 0.5)
    q = _rand((B, Hq, d), g, 1.5)
    rng = np.random.default_rng(seed)
    lens = _packed_lens("sparsemm", B * Hkv, n, rng)
    _, offs = csr(lens, "cpu")
    _, idx = workloads.random_lists(B, Hkv, n, lens, seed=seed)
    junk = torch.full((base,), n + 5, dtype=torch.int32)   # never read: outside every list
    idx_all = torch.cat([junk, idx])
    offs_d = torch.tensor((offs + base).astype(np.int32), device=DEV)
    ws = sk.new_workspace(sk.workspace_size(sk.OP_SPARSE_DECODE, B, Hq, Hkv, d, 0, 0), DEV)
    o, lse = sk.sparse_decode_attn(q.to(DEV), k.to(DEV), v.to(DEV), offs_d, idx_all.to(DEV), scale_of(d), ws=ws)
    o_ref, l_ref = oracle.sparse_decode(q, k, v, offs, idx.numpy())
    assert_attn_close(o, o_ref, "packed offset base")
    assert_lse_close(lse, l_ref, "packed offset base")
    _status_ok(ws)


def test_dense_many_heads_per_range():
    # 256 KV heads of 302 rows: CTA ranges hold parts of two or three heads
    g = torch.Generator().manual_seed(23)
    B, Hq, Hkv, d, n_prefix, gamma = 4, 64, 64, 128, 300, 2
    k = _rand((B, Hkv, n_prefix + gamma, d), g)
    v = _rand((B, Hkv, n_prefix + gamma, d), g)
    q = _rand((B, Hq, gamma, d), g, 1.5)
    ws = sk.new_workspace(sk.workspace_size(sk.OP_DENSE_VERIFY, B, Hq, Hkv, d, n_prefix + gamma, gamma), DEV)
    o, lse = sk.dense_verify_attn(q.to(DEV), k.to(DEV), v.to(DEV), n_prefix, scale_of(d), ws=ws)
    o_ref, l_ref = oracle.dense_verify(q, k, v, n_prefix)
    assert_attn_close(o, o_ref, "dense many heads")
    assert_lse_close(lse, l_ref, "dense many heads")
    _status_ok(ws)


def test_sparse_keep_all_equals_dense_on_gpu():
    g = torch.Generator().manual_seed(3)
    B, Hq, Hkv, d, n = 1, 32, 8, 128, 5000
    k = _rand((B, Hkv, n, d), g).to(DEV)
    v = _rand((B, Hkv, n, d), g).to(DEV)
    q = _rand((B, Hq, d), g).to(DEV)
    offs_d, _ = csr([n] * (B * Hkv), DEV)
    idx = torch.arange(n, dtype=torch.int32).repeat(B * Hkv).to(DEV)
    o_s, l_s = sk.sparse_decode_attn(q, k, v, offs_d, idx, scale_of(d))
    o_d, l_d = sk.dense_verify_attn(q[:, :, None].contiguous(), k, v, n - 1, scale_of(d))
    assert (f64(o_s) - f64(o_d[:, :, 0])).__abs__().max() <= 1e-2
    assert (f64(l_s) - f64(l_d[:, :, 0])).__abs__().max() <= 1e-4


def test_sparse_bad_index_is_flagged_not_faulted():
    g = torch.Generator().manual_seed(9)
    B, Hq, Hkv, d, n = 1, 4, 2, 128, 256
    k = _rand((B, Hkv, n, d), g).to(DEV)
    v = _rand((B, Hkv, n, d), g).to(DEV)
    q = _rand((B, Hq, d), g).to(DEV)
    offs_d, _ = csr([3, 3], DEV)
    idx = torch.tensor([0, 5, n + 7, 1, 2, -4], dtype=torch.int32, device=DEV)
    ws = sk.new_workspace(sk.workspace_size(sk.OP_SPARSE_DECODE, B, Hq, Hkv, d, 0, 0), DEV)
    sk.sparse_decode_attn(q, k, v, offs_d, idx, scale_of(d), ws=ws)
    assert sk.workspace_status(ws) == 2      # SDKV_DEV_BAD_INDEX
    assert sk.workspace_status(ws) == 0      # cleared by the read


@pytest.mark.parametrize("B,Hq", [(4, 32), (2, 64)])
def test_sparse_strided_cache_chunked_and_packed(B, Hq):
    # heads interleaved with batch and spare rows: the gathers use the caller's
    # strides (128 one-row lists: the packed decode; 64 lists of GQA 2: the chunked one)
    g = torch.Generator().manual_seed(31 + Hq)
    Hkv, d, n_cap = 32, 128, 700
    k = _rand((Hkv, B, n_cap, d), g).permute(1, 0, 2, 3)
    v = _rand((Hkv, B, n_cap, d), g, 0.5).permute(1, 0, 2, 3)
    q = _rand((B, Hq, d), g)
    rng = np.random.default_rng(31 + Hq)
    lens = rng.integers(0, 400, B * Hkv).tolist()
    offs_d, offs = csr(lens, DEV)
    _, idx = workloads.random_lists(B, Hkv, n_cap, lens, seed=31 + Hq)
    kd, vd = k.to(DEV), v.to(DEV)
    assert kd.stride() == k.stride()
    ws = sk.new_workspace(sk.workspace_size(sk.OP_SPARSE_DECODE, B, Hq, Hkv, d, 0, 0), DEV)
    o, lse = sk.sparse_decode_attn(q.to(DEV), kd, vd, offs_d, idx.to(DEV), scale_of(d), ws=ws)
    o_ref, l_ref = oracle.sparse_decode(q, k, v, offs, idx.numpy())
    assert_attn_close(o, o_ref, "sparse strided")
    assert_lse_close(lse, l_ref, "sparse strided")
    _status_ok(ws)


def test_sparse_packed_bad_index_and_bad_list_are_flagged_not_faulted():
    # 128 lists (the packed decode): an entry outside [0, n_cap) is flagged and
    # read as row 0; decreasing offsets are flagged before any per-list ticket is
    # taken, so the same workspace then serves a valid call correctly
    g = torch.Generator().manual_seed(19)
    B, Hq, Hkv, d, n = 4, 32, 32, 128, 300
    k = _rand((B, Hkv, n, d), g)
    v = _rand((B, Hkv, n, d), g, 0.5)
    q = _rand((B, Hq, d), g)
    lens = [3 + (i % 200) for i in range(B * Hkv)]
    offs_d, offs = csr(lens, DEV)
    _, idx = workloads.random_lists(B, Hkv, n, lens, seed=19)
    ws = sk.new_workspace(sk.workspace_size(sk.OP_SPARSE_DECODE, B, Hq, Hkv, d, 0, 0), DEV)
    kd, vd, qd = k.to(DEV), v.to(DEV), q.to(DEV)
    bad_idx = idx.clone()
    bad_idx[5] = n + 7
    bad_idx[int(offs[40]) + 1] = -4
    sk.sparse_decode_attn(qd, kd, vd, offs_d, bad_idx.to(DEV), scale_of(d), ws=ws)
    assert sk.workspace_status(ws) == 2      # SDKV_DEV_BAD_INDEX
    bad_offs = offs.copy()
    bad_offs[10] = bad_offs[11] + 5          # list 9 runs past list 10's start: list 10 has negative length
    assert bad_offs[10] <= offs[-1]
    sk.sparse_decode_attn(qd, kd, vd, torch.tensor(bad_offs.astype(np.int32), device=DEV), idx.to(DEV),
                          scale_of(d), ws=ws)
    assert sk.workspace_status(ws) == 3      # SDKV_DEV_BAD_LIST
    o, lse = sk.sparse_decode_attn(qd, kd, vd, offs_d, idx.to(DEV), scale_of(d), ws=ws)
    o_ref, l_ref = oracle.sparse_decode(q, k, v, offs, idx.numpy())
    assert_attn_close(o, o_ref, "packed after bad calls")
    assert_lse_close(lse, l_ref, "packed after bad calls")
    _status_ok(ws)


# ---------------------------------------------------------------------------
# a2 window scoring
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("B,Hq,Hkv,d,n,W,q_pos0", [
    (1, 4, 4, 64, 1024, 32, 992),        # tiny workload
    (1, 32, 8, 128, 3000, 32, 2968),     # Llama GQA shape, ragged key tail
    (2, 8, 4, 128, 777, 16, 700),        # window not at the end: later keys unseen
    (1, 28, 4, 128, 1300, 40, 1260),     # group 7 x window 40 = 280 rows: three row blocks
    (1, 4, 1, 64, 200, 64, 136),         # 256 rows: two full row blocks
    (1, 8, 2, 64, 1001, 48, 950),        # 192 rows: two row blocks, odd key count (unaligned rows)
    (4, 16, 16, 128, 9000, 32, 8968),    # 64 heads, two splits of 36 tiles: five-stage pass 1
    (8, 20, 20, 128, 4200, 32, 4100),    # 160 heads, one split of 33 tiles, window before the end
])
def test_score_matches_oracle(B, Hq, Hkv, d, n, W, q_pos0):
    g = torch.Generator().manual_seed(n + W)
    q_obs = _rand((B, Hq, W, d), g, 1.5)
    k = _rand((B, Hkv, n, d), g)
    ws = sk.new_workspace(sk.workspace_size(sk.OP_SCORE, B, Hq, Hkv, d, n, W), DEV)
    sc = sk.score_obs_window(q_obs.to(DEV), k.to(DEV), n, q_pos0, scale_of(d), ws=ws)
    ref = oracle.score_obs_window(q_obs, k, n, q_pos0)
    assert_scores_close(sc, ref, "score")
    # every window row sums to one, so each KV head's scores sum to G
    sums = f64(sc).sum(axis=2)
    assert np.allclose(sums, Hq // Hkv, rtol=1e-4)
    # deterministic: a second call gives identical bits
    sc2 = sk.score_obs_window(q_obs.to(DEV), k.to(DEV), n, q_pos0, scale_of(d), ws=ws)
    assert torch.equal(sc, sc2)
    _status_ok(ws)


# ---------------------------------------------------------------------------
# a3 selection: on identical fp32 scores the lists must be bit-exact
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("n,cand_lo,cand_hi,n_sink,n_recent,K", [
    (1024, 4, 992, 4, 32, 92),
    (5000, 4, 4936, 4, 64, 1000),
    (300, 0, 300, 0, 0, 299),
    (300, 0, 300, 0, 0, 1),
    (300, 2, 290, 2, 10, 0),
    (300, 2, 290, 2, 10, 288),
    (20000, 0, 19968, 0, 32, 4000),
    (70000, 0, 69968, 0, 32, 21000),   # long candidate range: 16 CTAs per head
])
def test_select_exact_on_same_scores(n, cand_lo, cand_hi, n_sink, n_recent, K):
    rng = np.random.default_rng(n + K)
    B, Hkv = 2, 3
    sc = rng.lognormal(0, 2, (B, Hkv, n)).astype(np.float32)
    sc[0, 0] = np.round(sc[0, 0] * 4) / 4            # many exact ties
    sc[0, 1, ::7] = 0.0
    sc[0, 1, 1::7] = -0.0                             # -0.0 equals +0.0
    sc[1, 2, ::5] = np.nan                            # NaN ranks last
    sc[1, 1, :] = 0.5                                 # all equal
    kh = n_sink + K + n_recent
    offs_d, offs = csr([kh] * (B * Hkv), DEV)
    scd = torch.from_numpy(sc).to(DEV)
    idx = sk.select_topk(scd, n, cand_lo, cand_hi, n_sink, n_recent, offs_d, int(offs[-1]))
    want = oracle.select_topk(sc, n, cand_lo, cand_hi, n_sink, n_recent, offs)
    assert np.array_equal(idx.cpu().numpy()[: len(want)], want)


@pytest.mark.parametrize("B,Hkv", [(4, 8), (8, 8), (16, 8)])
def test_select_many_heads(B, Hkv):
    # 32, 64 and 128 heads: fewer CTAs per head (4, 2, 1) so that all heads run at once
    rng = np.random.default_rng(B * Hkv)
    n, cand_lo, n_recent = 3000, 4, 64
    cand_hi = n - n_recent
    sc = rng.lognormal(0, 2, (B, Hkv, n)).astype(np.float32)
    sc[0, 0] = np.round(sc[0, 0] * 2) / 2            # ties
    sc[1, 3, ::3] = 0.0
    sc[B - 1, Hkv - 1, ::11] = np.nan
    lens = [4 + int(k) + n_recent for k in rng.integers(0, cand_hi - cand_lo + 1, B * Hkv)]
    offs_d, offs = csr(lens, DEV)
    idx = sk.select_topk(torch.from_numpy(sc).to(DEV), n, cand_lo, cand_hi, 4, n_recent, offs_d, int(offs[-1]))
    want = oracle.select_topk(sc, n, cand_lo, cand_hi, 4, n_recent, offs)
    assert np.array_equal(idx.cpu().numpy(), want)


@pytest.mark.parametrize("B,Hkv,n", [(1, 2, 70000), (4, 8, 40000), (8, 8, 20000), (16, 8, 12000)])
def test_select_large_ctas(B, Hkv, n):
    # more than 8192 candidates per CTA at 8, 4, 2 and 1 CTAs per head: the 1024-thread CTAs
    rng = np.random.default_rng(n + B)
    cand_lo, n_recent = 4, 64
    cand_hi = n - n_recent
    sc = rng.lognormal(0, 2, (B, Hkv, n)).astype(np.float32)
    sc[0, 0] = np.round(sc[0, 0] * 4) / 4            # many ties
    sc[0, 1, ::5] = 0.0
    sc[B - 1, Hkv - 1, ::13] = np.nan
    lens = [4 + int(k) + n_recent for k in rng.integers(0, cand_hi - cand_lo + 1, B * Hkv)]
    offs_d, offs = csr(lens, DEV)
    idx = sk.select_topk(torch.from_numpy(sc).to(DEV), n, cand_lo, cand_hi, 4, n_recent, offs_d, int(offs[-1]))
    want = oracle.select_topk(sc, n, cand_lo, cand_hi, 4, n_recent, offs)
    assert np.array_equal(idx.cpu().numpy(), want)


def test_select_ragged_budgets_and_bad_list():
    rng = np.random.default_rng(1)
    B, Hkv, n = 1, 5, 4000
    sc = rng.lognormal(0, 1, (B, Hkv, n)).astype(np.float32)
    lens = [32, 33, 3968, 100, 2000]
    offs_d, offs = csr(lens, DEV)
    idx = sk.select_topk(torch.from_numpy(sc).to(DEV), n, 0, n - 32, 0, 32, offs_d, int(offs[-1]))
    want = oracle.select_topk(sc, n, 0, n - 32, 0, 32, offs)
    assert np.array_equal(idx.cpu().numpy(), want)
    ws = sk.new_workspace(256, DEV)
    offs_bad, _ = csr([10, 32, 32, 32, 32], DEV)    # 10 < n_recent: does not fit
    sk.select_topk(torch.from_numpy(sc).to(DEV), n, 0, n - 32, 0, 32, offs_bad, 138, ws=ws)
    assert sk.workspace_status(ws) == 3             # SDKV_DEV_BAD_LIST


# ---------------------------------------------------------------------------
# the whole path on the tiny and video-shaped workloads (small enough for the oracle)
# ---------------------------------------------------------------------------

def test_pipeline_tiny_workload():
    w = workloads.WORKLOADS[1]
    t = workloads.make_layer(w, 0)
    gd = {k: v.to(DEV) for k, v in t.items()}
    n, d, B, Hkv = w.n, w.d, w.batch, w.hkv
    b = sk.head_budgets(np.ones(B * Hkv, np.float32), B * Hkv * w.keep[0], 0, 1.0)
    offs_d, offs = csr(b, DEV)
    sc = sk.score_obs_window(gd["q_obs"], gd["k"], n, w.q_pos0, scale_of(d))
    idx = sk.select_topk(sc, n, w.cand_lo, w.cand_hi, w.n_sink, w.n_recent, offs_d, int(offs[-1]))
    o, lse = sk.sparse_decode_attn(gd["q"], gd["k"], gd["v"], offs_d, idx, scale_of(d))
    s_ref = oracle.score_obs_window(t["q_obs"], t["k"], n, w.q_pos0)
    assert_scores_close(sc, s_ref, "tiny score")
    exact = check_selection_gap_rule(idx.cpu().numpy(), offs, s_ref, n, w.cand_lo, w.cand_hi,
                                     w.n_sink, w.n_recent)
    assert exact >= 1
    # attention over the GPU's own lists
    o_ref, l_ref = oracle.sparse_decode(t["q"], t["k"], t["v"], offs, idx.cpu().numpy())
    assert_attn_close(o, o_ref, "tiny sparse")
    assert_lse_close(lse, l_ref, "tiny sparse")


def test_pipeline_video_workload_reduced():
    # video shape (group 7, 256 text window queries over visual frames), one
    # layer at a reduced frame count so the oracle stays quick
    w = workloads.WORKLOADS[3]
    n = 8 * w.frame_tokens + w.text_tokens       # 8 frames + 256 text
    t = workloads.make_layer(w, 0, n=n)
    t["q_obs"] = t["q_obs"][:, :, : w.text_tokens].contiguous()
    gd = {k: v.to(DEV) for k, v in t.items()}
    m_v = n - w.text_tokens
    sc = sk.score_obs_window(gd["q_obs"], gd["k"], n, m_v, scale_of(w.d))
    s_ref = oracle.score_obs_window(t["q_obs"], t["k"], n, m_v)
    assert_scores_close(sc, s_ref, "video score")
    kh = w.text_tokens + 768
    offs_d, offs = csr([kh] * w.hkv, DEV)
    idx = sk.select_topk(sc, n, 0, m_v, 0, w.text_tokens, offs_d, int(offs[-1]))
    check_selection_gap_rule(idx.cpu().numpy(), offs, s_ref, n, 0, m_v, 0, w.text_tokens)
    o, lse = sk.sparse_decode_attn(gd["q"], gd["k"], gd["v"], offs_d, idx, scale_of(w.d))
    o_ref, l_ref = oracle.sparse_decode(t["q"], t["k"], t["v"], offs, idx.cpu().numpy())
    assert_attn_close(o, o_ref, "video sparse")
    # StD verify of gamma = 5 drafts over the whole cache
    ov, lv = sk.dense_verify_attn(gd["q_ver"], gd["k"], gd["v"], n - w.gamma, scale_of(w.d))
    ov_ref, lv_ref = oracle.dense_verify(t["q_ver"], t["k"], t["v"], n - w.gamma)
    assert_attn_close(ov, ov_ref, "video verify")
    assert_lse_close(lv, lv_ref, "video verify")
