"""The dense verify entry point that allocates nothing.

Some callers cannot give the library a workspace: their device memory belongs
to a pool they may not draw from at that moment, or an allocation (with its
implicit synchronisation) is not allowed in their loop.  For them
sdkv_dense_verify_attn_noalloc keeps its scratch in a fixed array inside the
library.  This test calls it through the C ABI, twice in a row (the second call
sees the first call's leftovers in the shared array), and checks each result
against sdkv_dense_verify_attn with a workspace, within the tolerances of the
other GPU tests; one small case is also checked against the fp64 oracle, with
the array's status word read after each call.  It also checks that a shape
needing more scratch than the array holds is refused with an error.  The file
sorts last on purpose.
"""
import ctypes
import math

import pytest
import torch

import sparse_kv_decode_gb300 as sk
from sparse_kv_decode_gb300 import _lib

pytestmark = pytest.mark.gpu

DEV = "cuda"
MAX_ABS = 1e-2      # same bar as the attention parity tests
MEAN_ABS = 1e-3
LSE_ABS = 2e-3


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from sparse_kv_decode_gb300 import build
    build.build()
    sk.lib()


def _noalloc(q, k, v, n_prefix, scale, o, lse):
    L = sk.lib()
    st = _lib._I64x3(k.stride(0), k.stride(1), k.stride(2))
    B, Hq, gamma, d = q.shape
    return L.sdkv_dense_verify_attn_noalloc(q.data_ptr(), k.data_ptr(), v.data_ptr(), st, B, Hq, k.shape[1], d,
                                            n_prefix, gamma, ctypes.c_float(scale), o.data_ptr(),
                                            lse.data_ptr() if lse is not None else None,
                                            torch.cuda.current_stream().cuda_stream)


@pytest.mark.parametrize("B,Hq,Hkv,d,n_prefix,gamma", [
    (1, 32, 8, 128, 32767, 1),    # dense decode of the Llama-shaped 32K workload
    (1, 32, 8, 128, 6000, 8),     # verify of 8 drafts, two row tiles
    (2, 4, 4, 64, 1020, 4),
])
def test_noalloc_matches_workspace_call_twice(B, Hq, Hkv, d, n_prefix, gamma):
    g = torch.Generator().manual_seed(n_prefix + gamma)
    rows = n_prefix + gamma
    k = torch.randn((B, Hkv, rows, d), generator=g).to(torch.bfloat16).to(DEV)
    v = torch.randn((B, Hkv, rows, d), generator=g).to(torch.bfloat16).to(DEV)
    scale = 1.0 / math.sqrt(d)
    for call in range(2):
        q = torch.randn((B, Hq, gamma, d), generator=torch.Generator().manual_seed(1 + call)).to(torch.bfloat16)
        q = q.to(DEV)
        o_ref, l_ref = sk.dense_verify_attn(q, k, v, n_prefix, scale)
        o = torch.full_like(q, float("nan"))
        lse = torch.full((B, Hq, gamma), float("nan"), device=DEV)
        assert _noalloc(q, k, v, n_prefix, scale, o, lse) == 0, sk.lib().sdkv_last_error()
        torch.cuda.synchronize()
        diff = (o.double() - o_ref.double()).abs()
        assert torch.isfinite(o).all()
        assert diff.max().item() <= MAX_ABS and diff.mean().item() <= MEAN_ABS, (call, diff.max().item())
        assert (lse - l_ref).abs().max().item() <= LSE_ABS


def _status():
    st = ctypes.c_int32(-1)
    rc = sk.lib().sdkv_dense_verify_attn_noalloc_status(ctypes.byref(st), torch.cuda.current_stream().cuda_stream)
    assert rc == 0, sk.lib().sdkv_last_error()
    return st.value


def test_noalloc_matches_oracle_and_reports_a_clean_status():
    # the tiny workload's gamma = 4 verify, checked against the fp64 oracle itself
    # (not only against the workspace call), twice, reading the status word after each
    import numpy as np
    import oracle
    import workloads
    w = workloads.by_name("tiny")
    t = workloads.make_layer(w, 0, device="cpu")
    k, v = t["k"].to(DEV), t["v"].to(DEV)
    n_prefix, scale = w.n - w.gamma, 1.0 / math.sqrt(w.d)
    o_ref, l_ref = oracle.dense_verify(t["q_ver"], t["k"], t["v"], n_prefix, scale)
    for _ in range(2):
        q = t["q_ver"].to(DEV)
        o = torch.full_like(q, float("nan"))
        lse = torch.full(q.shape[:3], float("nan"), device=DEV)
        assert _noalloc(q, k, v, n_prefix, scale, o, lse) == 0, sk.lib().sdkv_last_error()
        assert _status() == 0
        diff = np.abs(o.cpu().double().numpy() - o_ref)
        assert diff.max() <= MAX_ABS and diff.mean() <= MEAN_ABS
        assert np.abs(lse.cpu().double().numpy() - l_ref).max() <= LSE_ABS


def test_noalloc_refuses_shapes_beyond_its_scratch():
    # 512 (sequence, KV head) pairs x 64 query rows of partials need about
    # 17 MB of scratch, more than the fixed array holds: a clear error, no launch
    B, Hq, Hkv, d, gamma = 64, 64, 8, 128, 8
    need = sk.workspace_size(sk.OP_DENSE_VERIFY, B, Hq, Hkv, d, 64 + gamma, gamma)
    assert need > (8 << 20)
    q = torch.zeros((B, Hq, gamma, d), dtype=torch.bfloat16, device=DEV)
    k = torch.zeros((B, Hkv, 64 + gamma, d), dtype=torch.bfloat16, device=DEV)
    o = torch.zeros_like(q)
    rc = _noalloc(q, k, k, 64, 0.1, o, None)
    assert rc == _lib.SDKV_ERR_UNSUPPORTED
    assert b"scratch" in sk.lib().sdkv_last_error()
