"""Host-side checks of the C-ABI library that need no GPU: it loads, exports
every entry point include/sdkv.h declares, computes head budgets on the host
exactly as the oracle does, and rejects bad arguments before any launch."""
import ctypes
import os
import re

import numpy as np
import pytest

import oracle
import sparse_kv_decode_gb300 as sk
from sparse_kv_decode_gb300 import _lib

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    from sparse_kv_decode_gb300 import build
    build.build()
    return sk.lib()


def _declared():
    with open(os.path.join(ROOT, "include", "sdkv.h")) as f:
        text = f.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(sdkv_[a-z_]+)\s*\(", text)))


def test_exports_every_declared_symbol(L):
    names = _declared()
    assert len(names) == 17, names
    for name in names:
        assert hasattr(L, name), name
    assert sk.version() == 102


def test_budgets_match_oracle_exactly(L):
    rng = np.random.default_rng(7)
    cases = [
        (np.ones(8, np.float32), 8 * 128, 0, 1.0, 0),
        (np.array([1, 2, 3, 4], np.float32), 400, 32, 0.1, 0),
        (np.array([3, 2, 1], np.float32), 300, 0, 0.0, 120),
        (np.array([3, 2, 1], np.float32), 300, 0, 0.0, 110),
        (np.zeros(5, np.float32), 5 * 40 + 3, 32, 0.25, 0),
    ]
    for _ in range(25):
        N = int(rng.integers(1, 1025))
        s = rng.lognormal(0, 0.5, N).astype(np.float32)
        s[rng.uniform(size=N) < 0.05] *= 20
        w = int(rng.integers(0, 33))
        B = N * w + int(rng.integers(0, 300 * N))
        cases.append((s, B, w, float(rng.uniform(0, 1)), 0))
    # the sparsemm workload: 32 x 32 heads, B = 256 N, w = 32, rho = 0.1, cap = 32768
    import workloads
    wl = workloads.WORKLOADS[5]
    cases.append((workloads.head_scores(wl).numpy(), 256 * 1024, 32, 0.1, 32768))
    for s, B, w, rho, cap in cases:
        got = sk.head_budgets(s, B, w, rho, cap)
        want = oracle.head_budgets(s, B, w, rho, cap if cap > 0 else None)
        assert np.array_equal(got, want.astype(np.int32)), (len(s), B, w, rho, cap)


def test_budget_errors(L):
    with pytest.raises(sk.SdkvError) as e:
        sk.head_budgets(np.ones(4, np.float32), 10, 8, 0.1)
    assert e.value.code == _lib.SDKV_ERR_INVALID_ARG
    with pytest.raises(sk.SdkvError):
        sk.head_budgets(np.array([1, -1], np.float32), 100, 8, 0.1)
    with pytest.raises(sk.SdkvError):
        sk.head_budgets(np.ones(2, np.float32), 100, 8, 1.5)
    with pytest.raises(sk.SdkvError):
        sk.head_budgets(np.ones(2, np.float32), 100, 8, 0.1, cap=40)


def _strides(*s):
    return _lib._I64x3(*s)


def test_gpu_calls_reject_bad_arguments_without_launching(L):
    P = ctypes.c_void_p(256)   # a 16-byte aligned dummy, never dereferenced on these paths
    st = (1 << 20, 1 << 16, 128)
    # unsupported head dim
    assert L.sdkv_dense_verify_attn(P, P, P, _strides(*st), 1, 4, 4, 96, 10, 1, 0.1, P, None, P, 1 << 20,
                                    None) == _lib.SDKV_ERR_UNSUPPORTED
    # Hq not a multiple of Hkv
    assert L.sdkv_sparse_decode_attn(P, P, P, _strides(*st), 64, P, P, 0, 1, 6, 4, 128, 0.1, P, None, P,
                                     1 << 20, None) == _lib.SDKV_ERR_INVALID_ARG
    # negative index-array length
    assert L.sdkv_sparse_decode_attn(P, P, P, _strides(*st), 64, P, P, -1, 1, 8, 4, 128, 0.1, P, None, P,
                                     1 << 20, None) == _lib.SDKV_ERR_INVALID_ARG
    # null q
    assert L.sdkv_dense_verify_attn(None, P, P, _strides(*st), 1, 4, 4, 128, 10, 1, 0.1, P, None, P,
                                    1 << 20, None) == _lib.SDKV_ERR_INVALID_ARG
    # misaligned K
    assert L.sdkv_dense_verify_attn(P, ctypes.c_void_p(258), P, _strides(*st), 1, 4, 4, 128, 10, 1, 0.1, P,
                                    None, P, 1 << 20, None) == _lib.SDKV_ERR_INVALID_ARG
    # stride not a multiple of 8 elements
    assert L.sdkv_dense_verify_attn(P, P, P, _strides(1 << 20, 1 << 16, 130), 1, 4, 4, 128, 10, 1, 0.1, P,
                                    None, P, 1 << 20, None) == _lib.SDKV_ERR_INVALID_ARG
    # group * gamma above 64
    assert L.sdkv_dense_verify_attn(P, P, P, _strides(*st), 1, 32, 2, 128, 10, 5, 0.1, P, None, P, 1 << 20,
                                    None) == _lib.SDKV_ERR_UNSUPPORTED
    # negative n_prefix / zero gamma
    assert L.sdkv_dense_verify_attn(P, P, P, _strides(*st), 1, 4, 4, 128, -1, 1, 0.1, P, None, P, 1 << 20,
                                    None) == _lib.SDKV_ERR_INVALID_ARG
    # window outside the cache
    assert L.sdkv_score_obs_window(P, P, _strides(*st), 1, 4, 4, 128, 100, 32, 80, 0.1, P, P, 1 << 20,
                                   None) == _lib.SDKV_ERR_INVALID_ARG
    # window too large for the row blocks
    assert L.sdkv_score_obs_window(P, P, _strides(*st), 1, 64, 1, 128, 100000, 100, 0, 0.1, P, P, 1 << 20,
                                   None) == _lib.SDKV_ERR_UNSUPPORTED
    # overlapping sinks / candidates / recent window
    assert L.sdkv_select_topk(P, 1, 4, 100, 2, 99, 4, 8, P, P, P, 1 << 20, None) == _lib.SDKV_ERR_INVALID_ARG
    assert L.sdkv_select_topk(None, 1, 4, 100, 4, 90, 4, 8, P, P, P, 1 << 20, None) == _lib.SDKV_ERR_INVALID_ARG
    assert b"n_sink" in L.sdkv_last_error() or b"null" in L.sdkv_last_error()
    # draft lists: zero gamma, outputs aliasing the base lists
    assert L.sdkv_draft_lists(P, P, 4, 100, 0, 1000, ctypes.c_void_p(512), ctypes.c_void_p(768), None) == \
        _lib.SDKV_ERR_INVALID_ARG
    assert L.sdkv_draft_lists(P, ctypes.c_void_p(512), 4, 100, 2, 1000, P, ctypes.c_void_p(768), None) == \
        _lib.SDKV_ERR_INVALID_ARG


def test_product_path_fails_loudly_without_library(tmp_path, monkeypatch):
    # a missing library is an ImportError, never a silent fallback
    monkeypatch.setattr(_lib, "_lib", None)
    monkeypatch.setattr(_lib, "LIB_PATH", str(tmp_path / "missing.so"))
    with pytest.raises(ImportError):
        _lib.lib()
