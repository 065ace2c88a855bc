"""Seeded synthetic inputs shaped like the workloads the sparse-KV decode pages describe.

This module draws random tensors and nothing else: it holds none of the
method's arithmetic (no softmax, no budget formula, no selection).  Both the
CUDA path and the fp64 oracle are fed from here, and neither imports the other.

Workloads (sizes as the pages and the build contract give them):

  tiny        1 layer, 4 q / 4 KV heads, d=64, n=1024, batch 1, window 32,
              keep 128 = 4 sinks + 32 recent + 92 top-K, verify gamma=4.
  llama8b_32k Llama-3.1-8B attention shape: 32 layers x (32 q / 8 KV heads,
              d=128), batch 1, n=32768, keep 30% = 4 sinks + 64 recent + rest.
  video       Qwen2-7B shape: 28 layers x (28 q / 4 KV heads, d=128), batch 1,
              n = 12,544 visual (64 frames x 196) + 256 text, StD draft with
              256 text + 768 visual kept, verify gamma=5.
  llama8b_128k as llama8b_32k at n=131072, 1% planted keys, keep 10/30/50%,
              verify gamma=8.
  sparsemm    Vicuna-7B shape: 32 layers x 32 MHA heads, d=128, batch 8,
              n=32768, average budget 256 per head, w=32, rho=0.1, head
              scores LogNormal(0, 0.5) with a random 5% of heads x20.

Value recipe (one generator per (workload, layer), seed = 1000 + workload id,
offset by the layer index, so a single layer can be drawn on its own):
  * Q, K, V ~ N(0, 1), rounded to bf16 (round-to-nearest-even).
  * Sinks: keys 0..n_sink-1 of every head are scaled by 4.
  * Planted salient keys: per (sequence, KV head) a topic mu ~ N(0, 1)^d; the
    group's decode / verify / window queries are (mu + eps) / sqrt(2) (still
    N(0, 1) per component) and a seeded random subset of the history keys
    (frac x (n - n_sink - n_recent) of them) gets k += 2 sqrt(2) mu / |mu|,
    which lifts their expected logit q.k by about 2 sqrt(d), two standard
    deviations of q.k.
  * Video keys: visual key = frame mean + 0.5 N(0, 1), one frame mean
    ~ N(0, 1)^d per (layer, KV head, frame); text keys N(0, 1).
  * Head scores of the sparsemm workload: LogNormal(0, 0.5), and a random
    round(0.05 N) heads multiplied by 20.

The same seed draws different (equally distributed) values on a CPU and on a
CUDA generator; every test and the bench hand the very same tensors to both
the CUDA path and the oracle, so this does not matter.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import torch

BF16 = torch.bfloat16


@dataclasses.dataclass(frozen=True)
class Workload:
    wid: int
    name: str
    layers: int
    hq: int
    hkv: int
    d: int
    n: int
    batch: int
    window: int                  # observation-window length W
    q_pos0: int                  # position of the first window query
    n_sink: int
    n_recent: int
    cand_lo: int                 # candidate range [cand_lo, cand_hi) for top-K
    cand_hi: int
    keep: tuple                  # per-head list lengths k (total, incl. sinks+recent); () = ragged
    gamma: int                   # verify positions
    planted_frac: float = 0.0
    sink_scale: float = 4.0
    frames: int = 0
    frame_tokens: int = 0
    text_tokens: int = 0
    avg_budget: int = 0          # sparsemm: average budget per head
    w_local: int = 0             # sparsemm: local window w
    rho: float = 0.0             # sparsemm: uniform share
    heavy_frac: float = 0.0      # sparsemm: fraction of heads x20

    @property
    def group(self) -> int:
        return self.hq // self.hkv

    @property
    def seed(self) -> int:
        return 1000 + self.wid


def _keep_list(n: int, ratios) -> tuple:
    return tuple(int(math.floor(r * n)) for r in ratios)


WORKLOADS = {
    1: Workload(1, "tiny", layers=1, hq=4, hkv=4, d=64, n=1024, batch=1, window=32,
                q_pos0=1024 - 32, n_sink=4, n_recent=32, cand_lo=4, cand_hi=1024 - 32,
                keep=(128,), gamma=4, planted_frac=0.02),
    2: Workload(2, "llama8b_32k", layers=32, hq=32, hkv=8, d=128, n=32768, batch=1, window=32,
                q_pos0=32768 - 32, n_sink=4, n_recent=64, cand_lo=4, cand_hi=32768 - 64,
                keep=_keep_list(32768, (0.3,)), gamma=1, planted_frac=0.02),
    3: Workload(3, "video", layers=28, hq=28, hkv=4, d=128, n=12800, batch=1, window=256,
                q_pos0=12544, n_sink=0, n_recent=256, cand_lo=0, cand_hi=12544,
                keep=(1024,), gamma=5, frames=64, frame_tokens=196, text_tokens=256),
    4: Workload(4, "llama8b_128k", layers=32, hq=32, hkv=8, d=128, n=131072, batch=1, window=32,
                q_pos0=131072 - 32, n_sink=4, n_recent=64, cand_lo=4, cand_hi=131072 - 64,
                keep=_keep_list(131072, (0.1, 0.3, 0.5)), gamma=8, planted_frac=0.01),
    5: Workload(5, "sparsemm", layers=32, hq=32, hkv=32, d=128, n=32768, batch=8, window=32,
                q_pos0=32768 - 32, n_sink=0, n_recent=32, cand_lo=0, cand_hi=32768 - 32,
                keep=(), gamma=1, avg_budget=256, w_local=32, rho=0.1, heavy_frac=0.05),
}


def by_name(name: str) -> Workload:
    for w in WORKLOADS.values():
        if w.name == name:
            return w
    raise KeyError(name)


def _gen(device, seed: int) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def _randn(shape, g, device):
    return torch.randn(shape, generator=g, device=device, dtype=torch.float32)


def make_layer(w: Workload, layer: int, device="cpu", n: Optional[int] = None,
               n_cap: Optional[int] = None) -> dict:
    """Draw one layer's tensors for workload `w`.

    Returns a dict of bf16 tensors on `device`:
      q_obs   [B][Hq][W][d]   window queries (positions q_pos0 .. q_pos0+W-1)
      q       [B][Hq][d]      decode query
      q_ver   [B][Hq][gamma][d] verify queries
      k, v    [B][Hkv][n_cap][d] caches; rows >= n are zero padding
    `n` overrides the context length (smaller test cases keep the structure).
    """
    n = w.n if n is None else n
    n_cap = n if n_cap is None else n_cap
    B, Hq, Hkv, d, G = w.batch, w.hq, w.hkv, w.d, w.group
    W = min(w.window, n)
    g = _gen(device, w.seed * 1000 + layer)
    k = _randn((B, Hkv, n, d), g, device)
    v = _randn((B, Hkv, n, d), g, device)
    q = _randn((B, Hq, d), g, device)
    q_obs = _randn((B, Hq, W, d), g, device)
    q_ver = _randn((B, Hq, w.gamma, d), g, device)

    if w.frames:
        # video: visual keys clustered per frame, text keys plain N(0,1)
        m_v = w.frames * w.frame_tokens
        m_v = min(m_v, n)
        nf = (m_v + w.frame_tokens - 1) // w.frame_tokens
        mu = _randn((B, Hkv, nf, d), g, device)
        frame_of = torch.arange(m_v, device=device) // w.frame_tokens
        k[:, :, :m_v] = mu[:, :, frame_of] + 0.5 * k[:, :, :m_v]

    if w.planted_frac > 0:
        mu = _randn((B, Hkv, d), g, device)
        mu_hat = mu / mu.norm(dim=-1, keepdim=True)
        topic_q = mu.repeat_interleave(G, dim=1)                    # [B][Hq][d]
        q = (topic_q + q) / math.sqrt(2.0)
        q_obs = (topic_q[:, :, None, :] + q_obs) / math.sqrt(2.0)
        q_ver = (topic_q[:, :, None, :] + q_ver) / math.sqrt(2.0)
        lo, hi = w.n_sink, n - w.n_recent
        n_plant = int(math.floor(w.planted_frac * max(0, hi - lo)))
        if n_plant > 0:
            for b in range(B):
                for h in range(Hkv):
                    pick = torch.randperm(hi - lo, generator=g, device=device)[:n_plant] + lo
                    k[b, h, pick] += 2.0 * math.sqrt(2.0) * mu_hat[b, h]

    if w.n_sink > 0:
        k[:, :, : w.n_sink] *= w.sink_scale

    if n_cap > n:
        pad = torch.zeros((B, Hkv, n_cap - n, d), device=device)
        k = torch.cat([k, pad], dim=2)
        v = torch.cat([v, pad], dim=2)

    return {
        "q_obs": q_obs.to(BF16).contiguous(),
        "q": q.to(BF16).contiguous(),
        "q_ver": q_ver.to(BF16).contiguous(),
        "k": k.to(BF16).contiguous(),
        "v": v.to(BF16).contiguous(),
    }


def head_scores(w: Workload, seed_offset: int = 0) -> torch.Tensor:
    """Per-head visual scores s (float32, flat index = layer * H + head) for the
    head-budget step: LogNormal(0, 0.5) with a random 5% of heads x20.  For a
    workload with a uniform keep ratio every head gets the same score."""
    N = w.layers * w.hkv
    if w.heavy_frac <= 0:
        return torch.ones(N, dtype=torch.float32)
    g = _gen("cpu", w.seed * 7919 + seed_offset)
    s = torch.exp(0.5 * torch.randn(N, generator=g, dtype=torch.float32))
    n_heavy = int(round(w.heavy_frac * N))
    heavy = torch.randperm(N, generator=g)[:n_heavy]
    s[heavy] *= 20.0
    return s


def random_lists(B: int, Hkv: int, n: int, lengths, seed: int, device="cpu"):
    """Random ascending per-(b, h) index lists into [0, n) with the given
    lengths (one length per flat (b, h) or a single int).  Returns CSR
    (offsets int32 [B*Hkv+1], indices int32 [total])."""
    g = _gen("cpu", seed)
    BH = B * Hkv
    if isinstance(lengths, int):
        lengths = [lengths] * BH
    offs = [0]
    parts = []
    for i in range(BH):
        kk = int(lengths[i])
        sel = torch.randperm(n, generator=g)[:kk].sort().values.to(torch.int32)
        parts.append(sel)
        offs.append(offs[-1] + kk)
    idx = torch.cat(parts) if parts else torch.zeros(0, dtype=torch.int32)
    return (torch.tensor(offs, dtype=torch.int32, device=device), idx.to(device))


def offsets_from_counts(counts) -> torch.Tensor:
    """CSR offsets (int32, host) from per-(b, h) list lengths."""
    c = torch.as_tensor(counts, dtype=torch.int64)
    out = torch.zeros(c.numel() + 1, dtype=torch.int64)
    out[1:] = torch.cumsum(c, 0)
    return out.to(torch.int32)
