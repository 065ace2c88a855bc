"""GPU parity at the workloads' full sizes, on sampled heads.

One layer of each workload is drawn on the GPU at its full context length and
run through the same library calls (same shapes, hence the same launch
configuration) that bench.py times; the oracle then recomputes a sample of KV
heads one by one and the outputs are compared element by element.  Selection
is checked with the gap rule against oracle scores and bit-exactly against the
oracle's selection on the GPU's own fp32 scores."""
import math

import numpy as np
import pytest
import torch

import oracle
import sparse_kv_decode_gb300 as sk
import workloads
from gpu_common import (assert_attn_close, assert_lse_close, assert_scores_close, check_selection_gap_rule,
                        csr, f64)

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from sparse_kv_decode_gb300 import build
    build.build()
    sk.lib()


def _head_slices(t, b, h, G):
    """CPU copies of one (sequence, KV head) and its G query heads."""
    return {
        "k": t["k"][b:b + 1, h:h + 1].cpu(),
        "v": t["v"][b:b + 1, h:h + 1].cpu(),
        "q": t["q"][b:b + 1, h * G:(h + 1) * G].cpu(),
        "q_obs": t["q_obs"][b:b + 1, h * G:(h + 1) * G].cpu(),
        "q_ver": t["q_ver"][b:b + 1, h * G:(h + 1) * G].cpu(),
    }


def _run_path(w, t, lens, n, gamma_ver=None):
    """score -> select -> sparse decode -> dense decode (and verify) for one layer."""
    B, Hq, Hkv, d = w.batch, w.hq, w.hkv, w.d
    scale = 1.0 / math.sqrt(d)
    offs_d, offs = csr(lens, DEV)
    sc = sk.score_obs_window(t["q_obs"], t["k"], n, w.q_pos0, scale)
    idx = sk.select_topk(sc, n, w.cand_lo, w.cand_hi, w.n_sink, w.n_recent, offs_d, int(offs[-1]))
    o_sp, l_sp = sk.sparse_decode_attn(t["q"], t["k"], t["v"], offs_d, idx, scale)
    o_de, l_de = sk.dense_verify_attn(t["q"][:, :, None].contiguous(), t["k"], t["v"], n - 1, scale)
    out = {"sc": sc, "idx": idx, "offs": offs, "o_sp": o_sp, "l_sp": l_sp, "o_de": o_de, "l_de": l_de}
    if gamma_ver:
        ov, lv = sk.dense_verify_attn(t["q_ver"], t["k"], t["v"], n - gamma_ver, scale)
        out["o_ver"], out["l_ver"] = ov, lv
    torch.cuda.synchronize()
    return out


def _check_heads(w, t, out, n, heads, gamma_ver=None):
    G = w.group
    idx_all = out["idx"].cpu().numpy()
    offs = out["offs"]
    for (b, h) in heads:
        s = _head_slices(t, b, h, G)
        i = b * w.hkv + h
        # window scores of this KV head
        s_ref = oracle.score_obs_window(s["q_obs"], s["k"], n, w.q_pos0)
        s_gpu = out["sc"][b:b + 1, h:h + 1]
        assert_scores_close(s_gpu, s_ref, "score (%d,%d)" % (b, h))
        one = np.array([0, offs[i + 1] - offs[i]])
        lst = idx_all[offs[i]:offs[i + 1]]
        # selection: exact on the GPU's own scores, gap rule against the oracle's
        want_same = oracle.select_topk(s_gpu.cpu(), n, w.cand_lo, w.cand_hi, w.n_sink, w.n_recent, one)
        assert np.array_equal(lst, want_same), "select (%d,%d) differs on identical scores" % (b, h)
        check_selection_gap_rule(lst, one, s_ref, n, w.cand_lo, w.cand_hi, w.n_sink, w.n_recent)
        # sparse decode over the GPU's lists
        o_ref, l_ref = oracle.sparse_decode(s["q"], s["k"], s["v"], one, lst)
        assert_attn_close(out["o_sp"][b:b + 1, h * G:(h + 1) * G], o_ref, "sparse (%d,%d)" % (b, h))
        assert_lse_close(out["l_sp"][b:b + 1, h * G:(h + 1) * G], l_ref, "sparse lse (%d,%d)" % (b, h))
        # dense decode over the whole cache
        od_ref, ld_ref = oracle.dense_verify(s["q"][:, :, None], s["k"], s["v"], n - 1)
        assert_attn_close(out["o_de"][b:b + 1, h * G:(h + 1) * G], od_ref, "dense (%d,%d)" % (b, h))
        assert_lse_close(out["l_de"][b:b + 1, h * G:(h + 1) * G], ld_ref, "dense lse (%d,%d)" % (b, h))
        if gamma_ver:
            ov_ref, lv_ref = oracle.dense_verify(s["q_ver"], s["k"], s["v"], n - gamma_ver)
            assert_attn_close(out["o_ver"][b:b + 1, h * G:(h + 1) * G], ov_ref, "verify (%d,%d)" % (b, h))
            assert_lse_close(out["l_ver"][b:b + 1, h * G:(h + 1) * G], lv_ref, "verify lse (%d,%d)" % (b, h))


def test_llama8b_32k_full_layer():
    w = workloads.WORKLOADS[2]
    t = workloads.make_layer(w, 31, device=DEV)
    out = _run_path(w, t, [w.keep[0]] * (w.batch * w.hkv), w.n)
    _check_heads(w, t, out, w.n, [(0, 0), (0, 5), (0, 7)])


@pytest.mark.parametrize("keep_index", [0, 1, 2])
def test_llama8b_128k_full_layer(keep_index):
    w = workloads.WORKLOADS[4]
    t = workloads.make_layer(w, 3, device=DEV)
    gamma = w.gamma if keep_index == 1 else None   # gamma = 8 verify: 32 rows per KV head
    out = _run_path(w, t, [w.keep[keep_index]] * (w.batch * w.hkv), w.n, gamma_ver=gamma)
    _check_heads(w, t, out, w.n, [(0, 2), (0, 6)], gamma_ver=gamma)


def test_sparsemm_ragged_full_layer():
    w = workloads.WORKLOADS[5]
    t = workloads.make_layer(w, 0, device=DEV)
    s = workloads.head_scores(w).numpy()
    budgets = sk.head_budgets(s, w.avg_budget * w.layers * w.hkv, w.w_local, w.rho, w.n)
    assert budgets.sum() == w.avg_budget * w.layers * w.hkv
    layer0 = budgets[: w.hkv]
    lens = np.tile(layer0, w.batch)
    out = _run_path(w, t, lens, w.n)
    big = int(np.argmax(layer0))
    small = int(np.argmin(layer0))
    _check_heads(w, t, out, w.n, [(0, big), (3, small), (7, 5)])
    # the sparse decode of every one of the 256 lists (the packed kernel's spans cut
    # the long lists and pack the short ones), over the GPU's own lists
    G = w.group
    idx_all = out["idx"].cpu().numpy()
    offs = out["offs"]
    o_ref = np.zeros((w.batch, w.hq, w.d))
    l_ref = np.zeros((w.batch, w.hq))
    for i in range(w.batch * w.hkv):
        b, h = divmod(i, w.hkv)
        lst = idx_all[offs[i]:offs[i + 1]]
        sel = torch.as_tensor(lst.astype(np.int64), device=DEV)
        kk = t["k"][b, h].index_select(0, sel).cpu()[None, None]
        vv = t["v"][b, h].index_select(0, sel).cpu()[None, None]
        q = t["q"][b:b + 1, h * G:(h + 1) * G].cpu()
        o1, l1 = oracle.sparse_decode(q, kk, vv, np.array([0, len(lst)]), np.arange(len(lst)))
        o_ref[b, h * G:(h + 1) * G] = o1[0]
        l_ref[b, h * G:(h + 1) * G] = l1[0]
    assert_attn_close(out["o_sp"], o_ref, "sparse, every list")
    assert_lse_close(out["l_sp"], l_ref, "sparse lse, every list")


def test_video_full_layer_with_draft_steps():
    # StD: 256 text queries score the 12,544 visual tokens; 768 visual + 256
    # text kept; gamma = 5 sparse draft steps whose lists grow by the drafted
    # tokens' own entries; then one dense verify of the 5 positions
    w = workloads.WORKLOADS[3]
    gamma = w.gamma
    n = w.n
    t = workloads.make_layer(w, 7, device=DEV, n=n + gamma)      # cache holds the drafted rows too
    t["q_obs"] = t["q_obs"][:, :, : w.text_tokens].contiguous()
    d, G, Hkv = w.d, w.group, w.hkv
    scale = 1.0 / math.sqrt(d)
    kh = w.text_tokens + 768
    offs_d, offs = csr([kh] * Hkv, DEV)
    sc = sk.score_obs_window(t["q_obs"], t["k"], n, w.q_pos0, scale)
    base = sk.select_topk(sc, n, w.cand_lo, w.cand_hi, w.n_sink, w.n_recent, offs_d, int(offs[-1]))
    base_h = base.cpu().numpy().reshape(Hkv, kh)
    s_ref = oracle.score_obs_window(t["q_obs"][:, :4 * G].cpu(), t["k"][:, :4].cpu(), n, w.q_pos0)
    assert_scores_close(sc, s_ref, "video score")
    check_selection_gap_rule(base.cpu().numpy(), offs, s_ref, n, w.cand_lo, w.cand_hi, w.n_sink, w.n_recent)
    kc, vc = t["k"].cpu(), t["v"].cpu()
    for step in range(gamma):
        lists = np.concatenate([np.concatenate([base_h[h], np.arange(n, n + step + 1)]) for h in range(Hkv)])
        so_d, so = csr([kh + step + 1] * Hkv, DEV)
        q = t["q_ver"][:, :, step].contiguous()
        o, lse = sk.sparse_decode_attn(q, t["k"], t["v"], so_d, torch.tensor(lists, dtype=torch.int32, device=DEV),
                                       scale)
        o_ref, l_ref = oracle.sparse_decode(q.cpu(), kc, vc, so, lists)
        assert_attn_close(o, o_ref, "draft step %d" % step)
        assert_lse_close(lse, l_ref, "draft step %d" % step)
    ov, lv = sk.dense_verify_attn(t["q_ver"], t["k"], t["v"], n, scale)
    ov_ref, lv_ref = oracle.dense_verify(t["q_ver"].cpu(), kc, vc, n)
    assert_attn_close(ov, ov_ref, "video verify")
    assert_lse_close(lv, lv_ref, "video verify")
