"""fp64 CPU oracle: the definitions of the sparse-KV decode hot path, written out.

TEST INFRASTRUCTURE ONLY (tests, smoke check, bench CPU baseline).  No code is
shared with the CUDA library.  Inputs are bf16 tensors widened exactly to
float64; all arithmetic is float64; a library matmul is the only primitive.

Readings where the pages are silent (each listed in the design notes):
  * logit scale is 1/sqrt(d) unless the caller passes another;
  * GQA: query head hq reads KV head hq // G (contiguous groups);
  * window query t sits at position q_pos0 + t and sees keys 0..q_pos0+t;
  * integer budgets: largest-remainder apportionment, ties to the lower flat
    head index; a cap moves the excess to uncapped heads in proportion to s;
  * top-K order: score descending, then index ascending; -0.0 equals +0.0;
    NaN ranks below every number, -inf included;
  * an empty selected list gives o = 0 and lse = -inf;
  * lse is the natural-log log-sum-exp of the scaled logits.
"""
from __future__ import annotations

import math

import numpy as np


def to_f64(t) -> np.ndarray:
    """Exact widening of a (bf16 / fp32) torch tensor or array to float64."""
    if hasattr(t, "detach"):
        import torch
        return t.detach().to("cpu").to(torch.float64).numpy()
    return np.asarray(t, dtype=np.float64)


# ---------------------------------------------------------------------------
# a1  head budgets  (SparseMM post, methodology: the three cache parts)
# ---------------------------------------------------------------------------

def budget_terms(n_heads: int, total_B: int, w: int, rho: float):
    """The uniform share r and the score-preferred pool B_remain.

    r        = rho * (B - N w) / N
    B_remain = B - N w - rho * (B - N w)
    """
    base = float(total_B) - float(n_heads) * float(w)
    r = rho * base / n_heads
    b_remain = base - rho * base
    return r, b_remain


def head_budgets_real(s, total_B: int, w: int, rho: float, cap: int | None = None) -> list:
    """Real-valued budgets b*_i = w + r + B_remain * s_i / sum(s) (SparseMM
    methodology), with an optional cap: heads whose b* exceed it are fixed at
    the cap and their excess is shared among the other heads in proportion to
    s, repeated until no head exceeds it.  sum(s) is a plain float64 sum in
    index order; all-zero scores count as uniform."""
    s = [float(x) for x in np.asarray(s, dtype=np.float64).ravel()]
    N = len(s)
    if N == 0:
        raise ValueError("no heads")
    if total_B < N * w:
        raise ValueError("total budget below N * w")
    if not (0.0 <= rho <= 1.0):
        raise ValueError("rho outside [0, 1]")
    if cap is not None and cap * N < total_B:
        raise ValueError("cap * N below total budget")

    ssum = 0.0
    for x in s:                       # plain sum in index order
        if x < 0 or not math.isfinite(x):
            raise ValueError("head scores must be finite and >= 0")
        ssum += x
    if ssum == 0.0:
        s = [1.0] * N
        ssum = float(N)

    r, b_remain = budget_terms(N, total_B, w, rho)
    b_star = [w + r + b_remain * s[i] / ssum for i in range(N)]

    if cap is not None:
        capped = [False] * N
        while True:
            over = [i for i in range(N) if not capped[i] and b_star[i] > cap]
            if not over:
                break
            excess = 0.0
            for i in over:
                excess += b_star[i] - cap
                b_star[i] = float(cap)
                capped[i] = True
            free = [i for i in range(N) if not capped[i]]
            if not free:
                break
            free_s = 0.0
            for i in free:
                free_s += s[i]
            for i in free:
                share = s[i] / free_s if free_s > 0 else 1.0 / len(free)
                b_star[i] += excess * share
    return b_star


def head_budgets(s, total_B: int, w: int, rho: float, cap: int | None = None) -> np.ndarray:
    """Integer per-head budgets b_i (flat index i = layer * H + head).

    Floor every real budget b*_i, then hand the missing units one each to the
    heads with the largest fractional parts (ties: lower index), so that the
    budgets sum to B exactly (largest-remainder apportionment).
    """
    b_star = head_budgets_real(s, total_B, w, rho, cap)
    N = len(b_star)
    total_real = 0.0
    for x in b_star:
        total_real += x
    if abs(total_real - total_B) > 1e-6 * max(1.0, total_B):
        raise AssertionError("real budgets do not sum to B")
    floors = [int(math.floor(x)) for x in b_star]
    missing = total_B - sum(floors)
    if not (0 <= missing <= N):
        raise AssertionError("apportionment out of range")
    order = sorted(range(N), key=lambda i: (-(b_star[i] - floors[i]), i))
    b = list(floors)
    for i in order[:missing]:
        b[i] += 1
    return np.asarray(b, dtype=np.int64)


# ---------------------------------------------------------------------------
# a2  observation-window scoring
#     (StD 3.2: mean over the text queries of the attention to each key,
#      summed over the GQA group; SparseMM: last 32 queries as the window)
# ---------------------------------------------------------------------------

def score_obs_window(q_obs, k, n: int, q_pos0: int, scale: float | None = None) -> np.ndarray:
    """score[b, h, j] = (1/W) * sum_{g in group(h)} sum_t softmax_j(scale q_{g,t} . k_j)

    q_obs: [B][Hq][W][d]; k: [B][Hkv][>=n][d].  Window query t sits at position
    q_pos0 + t and attends keys 0 .. q_pos0 + t (causal); the softmax
    denominator runs over every key it sees.  Returns float64 [B][Hkv][n].
    """
    q_obs = to_f64(q_obs)
    k = to_f64(k)
    B, Hq, W, d = q_obs.shape
    Hkv = k.shape[1]
    G = Hq // Hkv
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    out = np.zeros((B, Hkv, n), dtype=np.float64)
    pos = q_pos0 + np.arange(W)
    visible = np.arange(n)[None, :] <= pos[:, None]          # [W][n]
    for b in range(B):
        for h in range(Hkv):
            keys = k[b, h, :n]                               # [n][d]
            acc = np.zeros(n, dtype=np.float64)
            for g in range(G):
                hq = h * G + g
                z = scale * (q_obs[b, hq] @ keys.T)          # [W][n]
                z = np.where(visible, z, -np.inf)
                z = z - z.max(axis=1, keepdims=True)
                e = np.exp(z)
                p = e / e.sum(axis=1, keepdims=True)
                acc += p.sum(axis=0)
            out[b, h] = acc / W
    return out


# ---------------------------------------------------------------------------
# a3  top-K selection and list assembly
#     (StD 3.2 argTopK; SparseMM K = r + b_score without the local window;
#      ByteCross: four sinks + highest-scoring entries)
# ---------------------------------------------------------------------------

def select_topk(scores, n: int, cand_lo: int, cand_hi: int, n_sink: int, n_recent: int,
                offsets) -> np.ndarray:
    """Per (b, h) list = sinks [0, n_sink) + top-K candidates + recent [n - n_recent, n).

    K = k_h - n_sink - n_recent with k_h = offsets[i+1] - offsets[i].  Candidates
    are [cand_lo, cand_hi); they are ranked by score descending, equal scores
    by lower index first; NaN ranks below every number (-inf included).
    The list is ascending.  Returns the flat
    int32 index array (CSR values for `offsets`).
    """
    sc = to_f64(scores)
    B, Hkv = sc.shape[0], sc.shape[1]
    offsets = np.asarray(offsets, dtype=np.int64)
    if not (0 <= n_sink <= cand_lo <= cand_hi <= n - n_recent <= n):
        raise ValueError("sinks, candidates and recent window must be disjoint and in order")
    out = np.zeros(int(offsets[-1]), dtype=np.int32)
    cand = np.arange(cand_lo, cand_hi)
    for b in range(B):
        for h in range(Hkv):
            i = b * Hkv + h
            kh = int(offsets[i + 1] - offsets[i])
            K = kh - n_sink - n_recent
            if K < 0 or K > cand_hi - cand_lo:
                raise ValueError("list length does not fit sinks + candidates + recent")
            s = sc[b, h, cand_lo:cand_hi]
            nan = np.isnan(s)
            key = np.where(nan, 0.0, -s)
            order = np.lexsort((cand, key, nan))              # numbers first, -score, then index
            top = np.sort(cand[order[:K]])
            lst = np.concatenate([np.arange(0, n_sink), top, np.arange(n - n_recent, n)])
            out[offsets[i]: offsets[i + 1]] = lst.astype(np.int32)
    return out


# ---------------------------------------------------------------------------
# a4  sparse decode over the selected lists
#     (StD 3.2: the sparse model loads only the retained KV entries;
#      ByteCross: unselected entries stay allocated but unread)
# ---------------------------------------------------------------------------

def _attend(qv, keys, vals, scale):
    """softmax(scale q.k_j) weighted sum of v_j, and the natural-log LSE."""
    if keys.shape[0] == 0:
        return np.zeros(vals.shape[1]), -np.inf
    z = scale * (keys @ qv)
    m = z.max()
    e = np.exp(z - m)
    l = e.sum()
    return (e @ vals) / l, m + math.log(l)


def sparse_decode(q, k, v, offsets, indices, scale: float | None = None):
    """o[b, hq] = sum_{j in S} softmax_j(scale q . k_j) v_j over the listed keys
    S of KV head hq // G; lse[b, hq] = log sum_{j in S} exp(scale q . k_j).
    q: [B][Hq][d]; k, v: [B][Hkv][n_cap][d]; CSR offsets/indices per (b, h)."""
    q = to_f64(q)
    k = to_f64(k)
    v = to_f64(v)
    offsets = np.asarray(offsets, dtype=np.int64)
    indices = np.asarray(indices, dtype=np.int64)
    B, Hq, d = q.shape
    Hkv = k.shape[1]
    G = Hq // Hkv
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    o = np.zeros((B, Hq, d))
    lse = np.zeros((B, Hq))
    for b in range(B):
        for hq in range(Hq):
            h = hq // G
            i = b * Hkv + h
            sel = indices[offsets[i]: offsets[i + 1]]
            o[b, hq], lse[b, hq] = _attend(q[b, hq], k[b, h, sel], v[b, h, sel], scale)
    return o, lse


# ---------------------------------------------------------------------------
# a5  dense verify / decode  (StD 3.1: the dense model checks all gamma drafts
#     in one pass over the full cache; ByteCross: the split-K dense baseline)
# ---------------------------------------------------------------------------

def dense_verify(q, k, v, n_prefix: int, scale: float | None = None):
    """Query t (t < gamma) sits at position n_prefix + t and attends keys
    0 .. n_prefix + t.  q: [B][Hq][gamma][d]; k, v: [B][Hkv][>= n_prefix+gamma][d].
    gamma = 1 with n_prefix = n - 1 is the dense decode over n keys."""
    q = to_f64(q)
    k = to_f64(k)
    v = to_f64(v)
    B, Hq, gamma, d = q.shape
    Hkv = k.shape[1]
    G = Hq // Hkv
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    o = np.zeros((B, Hq, gamma, d))
    lse = np.zeros((B, Hq, gamma))
    for b in range(B):
        for hq in range(Hq):
            h = hq // G
            for t in range(gamma):
                last = n_prefix + t
                o[b, hq, t], lse[b, hq, t] = _attend(q[b, hq, t], k[b, h, : last + 1],
                                                     v[b, h, : last + 1], scale)
    return o, lse


# ---------------------------------------------------------------------------
# Next rows beyond the hot path
# ---------------------------------------------------------------------------

# f2  StreamingLLM-style lists: attention sinks plus the recent window, no
#     scoring (StD, Baselines: the "Streaming" draft model; ByteCross, "The
#     Attention Baseline": a sink-plus-recent window timed against dense).

def window_lists(B: int, Hkv: int, n: int, n_sink: int, n_recent: int):
    """Every (b, h) keeps the first n_sink and the last n_recent of its n cache
    rows, ascending and without repeats (all n rows when they overlap).
    Returns CSR (offsets int64 [B*Hkv+1], indices int32)."""
    keep = sorted(set(range(0, min(n_sink, n))) | set(range(max(n - n_recent, 0), n)))
    BH = B * Hkv
    offsets = np.arange(BH + 1, dtype=np.int64) * len(keep)
    indices = np.tile(np.asarray(keep, dtype=np.int32), BH)
    return offsets, indices


# f1  contiguous compaction of the selected rows (ByteCross, "Speedup Across
#     Context": the selected entries are gathered into a contiguous buffer
#     that every later step reads in one kernel call).

def compact_kv(k, v, offsets, indices):
    """Row offsets[i] - offsets[0] + j of the output is row indices[offsets[i] + j]
    of KV head (b, h) = divmod(i, Hkv) of the cache: each head's selected rows in
    list order, the heads one after another.  Returns (k_c, v_c), [total][d]."""
    k = to_f64(k)
    v = to_f64(v)
    offsets = np.asarray(offsets, dtype=np.int64)
    indices = np.asarray(indices, dtype=np.int64)
    B, Hkv, _, d = k.shape
    total = int(offsets[-1] - offsets[0])
    k_c = np.zeros((total, d))
    v_c = np.zeros((total, d))
    for i in range(B * Hkv):
        b, h = divmod(i, Hkv)
        sel = indices[offsets[i]: offsets[i + 1]]
        a = int(offsets[i] - offsets[0])
        k_c[a: a + len(sel)] = k[b, h, sel]
        v_c[a: a + len(sel)] = v[b, h, sel]
    return k_c, v_c


def sparse_decode_compact(q, k_c, v_c, offsets, Hkv: int, scale: float | None = None):
    """Decode over compacted rows: query head hq of sequence b attends the rows
    [offsets[i] - offsets[0], offsets[i+1] - offsets[0]) of k_c / v_c, with
    i = b * Hkv + hq // G.  Same definition as sparse_decode, other addressing."""
    q = to_f64(q)
    k_c = to_f64(k_c)
    v_c = to_f64(v_c)
    offsets = np.asarray(offsets, dtype=np.int64)
    B, Hq, d = q.shape
    G = Hq // Hkv
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    o = np.zeros((B, Hq, d))
    lse = np.zeros((B, Hq))
    for b in range(B):
        for hq in range(Hq):
            i = b * Hkv + hq // G
            a, z = int(offsets[i] - offsets[0]), int(offsets[i + 1] - offsets[0])
            o[b, hq], lse[b, hq] = _attend(q[b, hq], k_c[a:z], v_c[a:z], scale)
    return o, lse


# f3  SpecVLM selection (SpecVLM post, "The SpecVLM Method": Stage I
#     verifier-guided top-P retention, Stage II spatially uniform reduction).

MASS_FRAC_BITS = 32   # masses are compared as exact sums of multiples of 2^-32


def specvlm_importance(scores):
    """a_j = the mean over all attention maps (layers x heads) of their score
    for token j.  scores: [units][n] -> [n] (float64)."""
    s = to_f64(scores)
    return s.reshape(-1, s.shape[-1]).mean(axis=0)


def specvlm_select(a, v_lo: int, v_hi: int, lam_r: float, r: float, keep_lo: int, keep_hi: int) -> np.ndarray:
    """Draft-side token list for the video tokens V = [v_lo, v_hi) and the
    always-kept range [keep_lo, keep_hi) (the text tokens), ascending.

    Stage I: order V by a_j descending (equal a_j: lower index first) and keep
    the shortest prefix V_R whose mass reaches lam_r times the mass of V.
    Stage II: walk the other tokens of V in index order at the interval
    I = (|V| - |V_R|) / ((1 - r) |V|) and keep the ones at positions
    floor(k I), k = 0, 1, ...  The list is V_R u V_U u [keep_lo, keep_hi).

    Readings: a_j are the fp32 scores the caller passes; each mass is a_j
    rounded to the nearest multiple of 2^-32 (exact integer sums, so the
    crossing is decided exactly); the target lam_r * S and I are float64.
    """
    a = np.asarray(a, dtype=np.float64)
    V = np.arange(v_lo, v_hi)
    nV = len(V)
    if nV == 0:
        return np.arange(keep_lo, keep_hi, dtype=np.int32)
    av = a[V]
    fx = [int(np.rint(x * 2.0 ** MASS_FRAC_BITS)) for x in av]          # exact Python ints
    order = sorted(range(nV), key=lambda j: (-av[j], j))
    S = sum(fx)
    target = lam_r * float(S)
    acc, c = 0, 0
    while c < nV and float(acc) < target:
        acc += fx[order[c]]
        c += 1
    retained = set(int(V[j]) for j in order[:c])
    left = [int(x) for x in V if int(x) not in retained]
    I = float(nV - c) / ((1.0 - r) * float(nV))
    sampled = set()
    k = 0
    while True:
        pos = math.floor(k * I) if I > 0 else len(left)
        if pos >= len(left):
            break
        sampled.add(left[pos])
        k += 1
    out = sorted(retained | sampled | set(range(keep_lo, keep_hi)))
    return np.asarray(out, dtype=np.int32)


# f4  StD draft lists (StD, 3.1 Decoding Procedures / 3.2): draft step t sees
#     the base selection plus the t + 1 drafted positions appended so far.

def append_drafts(base_offsets, base_indices, n_pos: int, n_new: int):
    """Each (b, h) list of the base CSR followed by n_pos, ..., n_pos + n_new - 1.
    Returns the new CSR (offsets int64, indices int32)."""
    bo = np.asarray(base_offsets, dtype=np.int64)
    bi = np.asarray(base_indices, dtype=np.int64)
    BH = len(bo) - 1
    offs = [0]
    parts = []
    for i in range(BH):
        parts.append(bi[bo[i]: bo[i + 1]])
        parts.append(np.arange(n_pos, n_pos + n_new))
        offs.append(offs[-1] + int(bo[i + 1] - bo[i]) + n_new)
    idx = np.concatenate(parts) if parts else np.zeros(0)
    return np.asarray(offs, dtype=np.int64), idx.astype(np.int32)
