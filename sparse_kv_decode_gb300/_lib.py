"""ctypes binding of libsdkv.so: argument marshalling only.

Every function mirrors one C entry point of include/sdkv.h (same name without
the `sdkv_` prefix).  Tensors are torch tensors: PyTorch supplies device memory
and the current CUDA stream; all computation runs in the library's kernels.
There is no fallback: if the library is missing or a call fails, an exception
is raised.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np
import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libsdkv.so")

SDKV_OK = 0
SDKV_ERR_INVALID_ARG = -1
SDKV_ERR_UNSUPPORTED = -2
SDKV_ERR_CUDA = -3
SDKV_ERR_WORKSPACE = -4

SDKV_DEV_OK = 0
SDKV_DEV_TIMEOUT = 1
SDKV_DEV_BAD_INDEX = 2
SDKV_DEV_BAD_LIST = 3

OP_SCORE = 1
OP_SELECT = 2
OP_SPARSE_DECODE = 3
OP_DENSE_VERIFY = 4
OP_COMPACT = 5
OP_SPECVLM = 6

_c_i32 = ctypes.c_int32
_c_i64 = ctypes.c_int64
_c_vp = ctypes.c_void_p
_c_sz = ctypes.c_size_t
_c_f = ctypes.c_float
_I64x3 = ctypes.c_int64 * 3


class SdkvError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__("sdkv error %d: %s" % (code, msg))
        self.code = code


_lib = None


def lib() -> ctypes.CDLL:
    """Load libsdkv.so (raises if it was not built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise ImportError("libsdkv.so not built: run `python -m sparse_kv_decode_gb300.build` "
                          "(or __graft_entry__.build())")
    L = ctypes.CDLL(LIB_PATH)
    L.sdkv_version.restype = _c_i32
    L.sdkv_last_error.restype = ctypes.c_char_p
    L.sdkv_head_budgets.argtypes = [ctypes.POINTER(ctypes.c_float), _c_i32, _c_i64, _c_i32,
                                    ctypes.c_double, _c_i32, ctypes.POINTER(_c_i32)]
    L.sdkv_head_budgets.restype = ctypes.c_int
    L.sdkv_workspace_size.argtypes = [_c_i32] * 7
    L.sdkv_workspace_size.restype = _c_sz
    L.sdkv_score_obs_window.argtypes = [_c_vp, _c_vp, _I64x3, _c_i32, _c_i32, _c_i32, _c_i32, _c_i32,
                                        _c_i32, _c_i32, _c_f, _c_vp, _c_vp, _c_sz, _c_vp]
    L.sdkv_score_obs_window.restype = ctypes.c_int
    L.sdkv_select_topk.argtypes = [_c_vp, _c_i32, _c_i32, _c_i32, _c_i32, _c_i32, _c_i32, _c_i32,
                                   _c_vp, _c_vp, _c_vp, _c_sz, _c_vp]
    L.sdkv_select_topk.restype = ctypes.c_int
    L.sdkv_sparse_decode_attn.argtypes = [_c_vp, _c_vp, _c_vp, _I64x3, _c_i32, _c_vp, _c_vp, _c_i64, _c_i32,
                                          _c_i32, _c_i32, _c_i32, _c_f, _c_vp, _c_vp, _c_vp, _c_sz, _c_vp]
    L.sdkv_sparse_decode_attn.restype = ctypes.c_int
    L.sdkv_dense_verify_attn.argtypes = [_c_vp, _c_vp, _c_vp, _I64x3, _c_i32, _c_i32, _c_i32, _c_i32,
                                         _c_i32, _c_i32, _c_f, _c_vp, _c_vp, _c_vp, _c_sz, _c_vp]
    L.sdkv_dense_verify_attn.restype = ctypes.c_int
    L.sdkv_dense_verify_attn_noalloc.argtypes = [_c_vp, _c_vp, _c_vp, _I64x3, _c_i32, _c_i32, _c_i32, _c_i32,
                                                 _c_i32, _c_i32, _c_f, _c_vp, _c_vp, _c_vp]
    L.sdkv_dense_verify_attn_noalloc.restype = ctypes.c_int
    L.sdkv_dense_verify_attn_noalloc_status.argtypes = [ctypes.POINTER(_c_i32), _c_vp]
    L.sdkv_dense_verify_attn_noalloc_status.restype = ctypes.c_int
    L.sdkv_workspace_status.argtypes = [_c_vp, ctypes.POINTER(_c_i32), _c_vp]
    L.sdkv_workspace_status.restype = ctypes.c_int
    L.sdkv_window_lists.argtypes = [_c_i32, _c_i32, _c_i32, _c_i32, _c_i32, _c_vp, _c_vp, _c_vp]
    L.sdkv_window_lists.restype = ctypes.c_int
    L.sdkv_append_drafts.argtypes = [_c_vp, _c_vp, _c_i32, _c_i32, _c_i32, _c_vp, _c_vp, _c_vp]
    L.sdkv_append_drafts.restype = ctypes.c_int
    L.sdkv_draft_lists.argtypes = [_c_vp, _c_vp, _c_i32, _c_i32, _c_i32, _c_i64, _c_vp, _c_vp, _c_vp]
    L.sdkv_draft_lists.restype = ctypes.c_int
    L.sdkv_compact_kv.argtypes = [_c_vp, _c_vp, _I64x3, _c_i32, _c_vp, _c_vp, _c_i32, _c_i32, _c_i32, _c_i64,
                                  _c_vp, _c_vp, _c_vp, _c_sz, _c_vp]
    L.sdkv_compact_kv.restype = ctypes.c_int
    L.sdkv_sparse_decode_compact.argtypes = [_c_vp, _c_vp, _c_vp, _c_i64, _c_vp, _c_i32, _c_i32, _c_i32, _c_i32,
                                             _c_f, _c_vp, _c_vp, _c_vp, _c_sz, _c_vp]
    L.sdkv_sparse_decode_compact.restype = ctypes.c_int
    L.sdkv_specvlm_select.argtypes = [_c_vp, _c_i32, _c_i32, _c_i32, _c_i32, _c_i32, ctypes.c_double,
                                      ctypes.c_double, _c_i32, _c_i32, _c_vp, _c_vp, _c_vp, _c_vp, _c_sz, _c_vp]
    L.sdkv_specvlm_select.restype = ctypes.c_int
    _lib = L
    return L


def _check(rc: int):
    if rc != SDKV_OK:
        raise SdkvError(rc, lib().sdkv_last_error().decode())


def _ptr(t) -> int:
    return 0 if t is None else t.data_ptr()


def _stream(t=None) -> int:
    dev = t.device if t is not None else None
    return torch.cuda.current_stream(dev).cuda_stream


def _need(t: torch.Tensor, name: str, dtype, cuda=True):
    if t.dtype != dtype:
        raise TypeError("%s must be %s, got %s" % (name, dtype, t.dtype))
    if cuda and not t.is_cuda:
        raise TypeError("%s must be a CUDA tensor" % name)


def _kv_strides(k: torch.Tensor):
    if k.dim() != 4 or k.stride(3) != 1:
        raise ValueError("K/V must be [B][Hkv][rows][d] with d contiguous")
    return _I64x3(k.stride(0), k.stride(1), k.stride(2))


def version() -> int:
    return int(lib().sdkv_version())


def workspace_size(op: int, B: int, Hq: int, Hkv: int, d: int, n: int, gamma_or_w: int) -> int:
    return int(lib().sdkv_workspace_size(op, B, Hq, Hkv, d, n, gamma_or_w))


def new_workspace(nbytes: int, device) -> torch.Tensor:
    """A zeroed workspace buffer (uint8) of at least `nbytes`, 256-byte rounded."""
    nbytes = max(256, (int(nbytes) + 255) // 256 * 256)
    return torch.zeros(nbytes, dtype=torch.uint8, device=device)


def workspace_status(ws: torch.Tensor) -> int:
    st = _c_i32(0)
    _check(lib().sdkv_workspace_status(ctypes.c_void_p(ws.data_ptr()), ctypes.byref(st),
                                       ctypes.c_void_p(_stream(ws))))
    return int(st.value)


def head_budgets(s, total_B: int, w: int, rho: float, cap: int = 0) -> np.ndarray:
    """sdkv_head_budgets on host arrays; returns int32 budgets."""
    s = np.ascontiguousarray(np.asarray(s, dtype=np.float32).ravel())
    out = np.zeros(s.size, dtype=np.int32)
    _check(lib().sdkv_head_budgets(s.ctypes.data_as(ctypes.POINTER(ctypes.c_float)), s.size,
                                   int(total_B), int(w), float(rho), int(cap),
                                   out.ctypes.data_as(ctypes.POINTER(_c_i32))))
    return out


def score_obs_window(q_obs: torch.Tensor, k: torch.Tensor, n: int, q_pos0: int, scale: float,
                     scores: torch.Tensor | None = None, ws: torch.Tensor | None = None) -> torch.Tensor:
    _need(q_obs, "q_obs", torch.bfloat16)
    _need(k, "k", torch.bfloat16)
    if not q_obs.is_contiguous():
        raise ValueError("q_obs must be contiguous [B][Hq][W][d]")
    B, Hq, W, d = q_obs.shape
    Hkv = k.shape[1]
    if scores is None:
        scores = torch.empty((B, Hkv, n), dtype=torch.float32, device=q_obs.device)
    _need(scores, "scores", torch.float32)
    if ws is None:
        ws = new_workspace(workspace_size(OP_SCORE, B, Hq, Hkv, d, n, W), q_obs.device)
    _check(lib().sdkv_score_obs_window(q_obs.data_ptr(), k.data_ptr(), _kv_strides(k), B, Hq, Hkv, d, n,
                                       W, q_pos0, scale, scores.data_ptr(), ws.data_ptr(), ws.numel(),
                                       _stream(q_obs)))
    return scores


def select_topk(scores: torch.Tensor, n: int, cand_lo: int, cand_hi: int, n_sink: int, n_recent: int,
                offsets: torch.Tensor, total: int, indices: torch.Tensor | None = None,
                ws: torch.Tensor | None = None) -> torch.Tensor:
    """`total` = offsets[-1] (list entries to allocate when `indices` is None)."""
    _need(scores, "scores", torch.float32)
    _need(offsets, "offsets", torch.int32)
    if not scores.is_contiguous():
        raise ValueError("scores must be contiguous [B][Hkv][n]")
    B, Hkv = scores.shape[0], scores.shape[1]
    if indices is None:
        indices = torch.empty(max(int(total), 1), dtype=torch.int32, device=scores.device)
    _need(indices, "indices", torch.int32)
    if ws is None:
        ws = new_workspace(workspace_size(OP_SELECT, B, 0, Hkv, 0, n, 0), scores.device)
    _check(lib().sdkv_select_topk(scores.data_ptr(), B, Hkv, n, cand_lo, cand_hi, n_sink, n_recent,
                                  offsets.data_ptr(), indices.data_ptr(), ws.data_ptr(), ws.numel(),
                                  _stream(scores)))
    return indices


def sparse_decode_attn(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, offsets: torch.Tensor,
                       indices: torch.Tensor, scale: float, o: torch.Tensor | None = None,
                       lse: torch.Tensor | None = None, ws: torch.Tensor | None = None,
                       want_lse: bool = True, early: bool = True):
    """`early`: pass the length of `indices` as n_idx, so the kernel prefetches the
    lists into L2 while the previous kernel on the stream finishes."""
    for t, nm in ((q, "q"), (k, "k"), (v, "v")):
        _need(t, nm, torch.bfloat16)
    _need(offsets, "offsets", torch.int32)
    _need(indices, "indices", torch.int32)
    if not indices.is_contiguous():
        raise ValueError("indices must be contiguous")
    if not q.is_contiguous():
        raise ValueError("q must be contiguous [B][Hq][d]")
    if k.stride() != v.stride() or k.shape != v.shape:
        raise ValueError("K and V must share shape and strides")
    B, Hq, d = q.shape
    Hkv, n_cap = k.shape[1], k.shape[2]
    if o is None:
        o = torch.empty_like(q)
    if lse is None and want_lse:
        lse = torch.empty((B, Hq), dtype=torch.float32, device=q.device)
    if ws is None:
        ws = new_workspace(workspace_size(OP_SPARSE_DECODE, B, Hq, Hkv, d, 0, 0), q.device)
    _check(lib().sdkv_sparse_decode_attn(q.data_ptr(), k.data_ptr(), v.data_ptr(), _kv_strides(k), n_cap,
                                         offsets.data_ptr(), indices.data_ptr(), indices.numel() if early else 0,
                                         B, Hq, Hkv, d, scale,
                                         o.data_ptr(), _ptr(lse), ws.data_ptr(), ws.numel(), _stream(q)))
    return o, lse


def dense_verify_attn(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, n_prefix: int, scale: float,
                      o: torch.Tensor | None = None, lse: torch.Tensor | None = None,
                      ws: torch.Tensor | None = None, want_lse: bool = True):
    for t, nm in ((q, "q"), (k, "k"), (v, "v")):
        _need(t, nm, torch.bfloat16)
    if not q.is_contiguous():
        raise ValueError("q must be contiguous [B][Hq][gamma][d]")
    if k.stride() != v.stride() or k.shape != v.shape:
        raise ValueError("K and V must share shape and strides")
    B, Hq, gamma, d = q.shape
    Hkv = k.shape[1]
    if k.shape[2] < n_prefix + gamma:
        raise ValueError("cache holds fewer than n_prefix + gamma rows")
    if o is None:
        o = torch.empty_like(q)
    if lse is None and want_lse:
        lse = torch.empty((B, Hq, gamma), dtype=torch.float32, device=q.device)
    if ws is None:
        ws = new_workspace(workspace_size(OP_DENSE_VERIFY, B, Hq, Hkv, d, n_prefix + gamma, gamma), q.device)
    _check(lib().sdkv_dense_verify_attn(q.data_ptr(), k.data_ptr(), v.data_ptr(), _kv_strides(k), B, Hq, Hkv,
                                        d, n_prefix, gamma, scale, o.data_ptr(), _ptr(lse), ws.data_ptr(),
                                        ws.numel(), _stream(q)))
    return o, lse


def dense_verify_attn_noalloc(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, n_prefix: int, scale: float,
                              o: torch.Tensor, lse: torch.Tensor | None = None):
    """sdkv_dense_verify_attn_noalloc: the dense verify with the library's fixed
    scratch array instead of a workspace.  The caller passes the outputs; this
    wrapper allocates nothing either."""
    for t, nm in ((q, "q"), (k, "k"), (v, "v"), (o, "o")):
        _need(t, nm, torch.bfloat16)
    if not q.is_contiguous() or not o.is_contiguous():
        raise ValueError("q and o must be contiguous [B][Hq][gamma][d]")
    if k.stride() != v.stride() or k.shape != v.shape:
        raise ValueError("K and V must share shape and strides")
    B, Hq, gamma, d = q.shape
    Hkv = k.shape[1]
    if k.shape[2] < n_prefix + gamma:
        raise ValueError("cache holds fewer than n_prefix + gamma rows")
    _check(lib().sdkv_dense_verify_attn_noalloc(q.data_ptr(), k.data_ptr(), v.data_ptr(), _kv_strides(k), B, Hq,
                                                Hkv, d, n_prefix, gamma, scale, o.data_ptr(), _ptr(lse),
                                                _stream(q)))
    return o, lse


# --------------------------------------------------------------------------- around the hot path

def window_lists(B: int, Hkv: int, n: int, n_sink: int, n_recent: int, device,
                 offsets: torch.Tensor | None = None, indices: torch.Tensor | None = None):
    """sdkv_window_lists: sink-plus-recent lists, k = min(n, n_sink + n_recent) per head."""
    k = min(n, n_sink + n_recent)
    if offsets is None:
        offsets = torch.empty(B * Hkv + 1, dtype=torch.int32, device=device)
    if indices is None:
        indices = torch.empty(max(B * Hkv * k, 1), dtype=torch.int32, device=device)
    _need(offsets, "offsets", torch.int32)
    _need(indices, "indices", torch.int32)
    _check(lib().sdkv_window_lists(B, Hkv, n, n_sink, n_recent, offsets.data_ptr(), indices.data_ptr(),
                                   _stream(offsets)))
    return offsets, indices


def append_drafts(base_offsets: torch.Tensor, base_indices: torch.Tensor, total: int, n_pos: int, n_new: int,
                  offsets: torch.Tensor | None = None, indices: torch.Tensor | None = None):
    """sdkv_append_drafts: every base list followed by n_pos .. n_pos + n_new - 1.
    `total` = base_offsets[-1] - base_offsets[0] (host value, sizes the output)."""
    _need(base_offsets, "base_offsets", torch.int32)
    _need(base_indices, "base_indices", torch.int32)
    BH = base_offsets.numel() - 1
    if offsets is None:
        offsets = torch.empty(BH + 1, dtype=torch.int32, device=base_offsets.device)
    if indices is None:
        indices = torch.empty(max(total + BH * n_new, 1), dtype=torch.int32, device=base_offsets.device)
    _check(lib().sdkv_append_drafts(base_offsets.data_ptr(), base_indices.data_ptr(), BH, n_pos, n_new,
                                    offsets.data_ptr(), indices.data_ptr(), _stream(base_offsets)))
    return offsets, indices


def draft_lists(base_offsets: torch.Tensor, base_indices: torch.Tensor, total: int, n_pos: int, gamma: int,
                offsets: torch.Tensor | None = None, indices: torch.Tensor | None = None):
    """sdkv_draft_lists: the lists of draft steps 0 .. gamma-1 in one launch.
    Returns offsets [gamma][BH + 1] and indices [gamma][stride] (set t = base
    lists + n_pos .. n_pos + t); `total` = base_offsets[-1] - base_offsets[0]."""
    _need(base_offsets, "base_offsets", torch.int32)
    _need(base_indices, "base_indices", torch.int32)
    BH = base_offsets.numel() - 1
    stride = total + BH * gamma
    if offsets is None:
        offsets = torch.empty((gamma, BH + 1), dtype=torch.int32, device=base_offsets.device)
    if indices is None:
        indices = torch.empty((gamma, max(stride, 1)), dtype=torch.int32, device=base_offsets.device)
    if offsets.shape != (gamma, BH + 1) or indices.dim() != 2 or indices.shape[0] != gamma:
        raise ValueError("offsets must be [gamma][BH+1] and indices [gamma][stride]")
    if indices.shape[1] < stride or not (offsets.is_contiguous() and indices.is_contiguous()):
        raise ValueError("indices rows must hold total + BH * gamma entries, contiguous")
    _check(lib().sdkv_draft_lists(base_offsets.data_ptr(), base_indices.data_ptr(), BH, n_pos, gamma,
                                  indices.shape[1], offsets.data_ptr(), indices.data_ptr(), _stream(base_offsets)))
    return offsets, indices


def compact_kv(k: torch.Tensor, v: torch.Tensor, offsets: torch.Tensor, indices: torch.Tensor, total: int,
               k_out: torch.Tensor | None = None, v_out: torch.Tensor | None = None,
               ws: torch.Tensor | None = None):
    """sdkv_compact_kv: the listed rows of every head into contiguous [total][d] buffers."""
    for t, nm in ((k, "k"), (v, "v")):
        _need(t, nm, torch.bfloat16)
    _need(offsets, "offsets", torch.int32)
    _need(indices, "indices", torch.int32)
    if k.stride() != v.stride() or k.shape != v.shape:
        raise ValueError("K and V must share shape and strides")
    B, Hkv, n_cap, d = k.shape
    if k_out is None:
        k_out = torch.empty((max(total, 1), d), dtype=torch.bfloat16, device=k.device)
    if v_out is None:
        v_out = torch.empty((max(total, 1), d), dtype=torch.bfloat16, device=k.device)
    if ws is None:
        ws = new_workspace(workspace_size(OP_COMPACT, B, 0, Hkv, d, 0, 0), k.device)
    _check(lib().sdkv_compact_kv(k.data_ptr(), v.data_ptr(), _kv_strides(k), n_cap, offsets.data_ptr(),
                                 indices.data_ptr(), B, Hkv, d, k_out.shape[0], k_out.data_ptr(), v_out.data_ptr(),
                                 ws.data_ptr(), ws.numel(), _stream(k)))
    return k_out, v_out


def sparse_decode_compact(q: torch.Tensor, k_c: torch.Tensor, v_c: torch.Tensor, offsets: torch.Tensor,
                          Hkv: int, scale: float, o: torch.Tensor | None = None, lse: torch.Tensor | None = None,
                          ws: torch.Tensor | None = None, want_lse: bool = True):
    """sdkv_sparse_decode_compact: decode over rows compacted by compact_kv."""
    for t, nm in ((q, "q"), (k_c, "k_c"), (v_c, "v_c")):
        _need(t, nm, torch.bfloat16)
    _need(offsets, "offsets", torch.int32)
    if not (q.is_contiguous() and k_c.is_contiguous() and v_c.is_contiguous()):
        raise ValueError("q, k_c and v_c must be contiguous")
    B, Hq, d = q.shape
    if o is None:
        o = torch.empty_like(q)
    if lse is None and want_lse:
        lse = torch.empty((B, Hq), dtype=torch.float32, device=q.device)
    if ws is None:
        ws = new_workspace(workspace_size(OP_SPARSE_DECODE, B, Hq, Hkv, d, 0, 0), q.device)
    _check(lib().sdkv_sparse_decode_compact(q.data_ptr(), k_c.data_ptr(), v_c.data_ptr(), k_c.shape[0],
                                            offsets.data_ptr(), B, Hq, Hkv, d, scale, o.data_ptr(), _ptr(lse),
                                            ws.data_ptr(), ws.numel(), _stream(q)))
    return o, lse


def specvlm_select(scores: torch.Tensor, v_lo: int, v_hi: int, lam_r: float, r: float, keep_lo: int,
                   keep_hi: int, importance: torch.Tensor | None = None, indices: torch.Tensor | None = None,
                   counts: torch.Tensor | None = None, ws: torch.Tensor | None = None):
    """sdkv_specvlm_select: scores [B][units][n] fp32 -> (importance [B][n],
    indices [B][cap], counts [B]); row b's list is indices[b, :counts[b]]."""
    _need(scores, "scores", torch.float32)
    if not scores.is_contiguous():
        raise ValueError("scores must be contiguous [B][units][n]")
    B, units, n = scores.shape
    cap = (v_hi - v_lo) + (keep_hi - keep_lo)
    dev = scores.device
    if importance is None:
        importance = torch.empty((B, n), dtype=torch.float32, device=dev)
    if indices is None:
        indices = torch.empty((B, max(cap, 1)), dtype=torch.int32, device=dev)
    if counts is None:
        counts = torch.empty(B, dtype=torch.int32, device=dev)
    if ws is None:
        ws = new_workspace(workspace_size(OP_SPECVLM, B, 0, 0, 0, v_hi - v_lo, 0), dev)
    _check(lib().sdkv_specvlm_select(scores.data_ptr(), B, units, n, v_lo, v_hi, lam_r, r, keep_lo, keep_hi,
                                     importance.data_ptr(), indices.data_ptr(), counts.data_ptr(), ws.data_ptr(),
                                     ws.numel(), _stream(scores)))
    return importance, indices, counts
