"""Byte account of a decode step: algorithmic HBM bytes per kernel launch.

Two parts:

1. The byte crossover model of "Where Activation Sparsity and KV-Cache Sparsity
   Cross in LLM Decoding" (ByteCross page, section "The Byte Crossover"):
   per layer the cache adds 2 * h_kv * d_h * 2 bytes per token (4096 n for
   Llama-3.1-8B), the seven projections hold P = 3 d d_ff + 2 d^2 + 2 d h_kv d_h
   parameters, and the crossover context is
       n* = P (1 - r_P) / (2 h_kv d_h (1 - r_KV)).
   The ideal bandwidth-bound speedup of removing dB of B_total bytes is
   B_total / (B_total - dB).

2. Algorithmic bytes of each hot-path kernel per launch (one layer), used as
   the numerator of achieved GB/s.  Split-K partials are real traffic but not
   algorithmic and are not counted.
"""
from __future__ import annotations

BF16 = 2


# --- the ByteCross byte model -------------------------------------------------

def projection_params(d: int, d_ff: int, h_kv: int, d_h: int) -> int:
    """Parameters of the seven projections of one layer: three feed-forward
    (3 d d_ff), query + output (2 d^2), key + value (2 d h_kv d_h)."""
    return 3 * d * d_ff + 2 * d * d + 2 * d * h_kv * d_h


def kv_bytes_per_token(h_kv: int, d_h: int, elem: int = BF16) -> int:
    """Cache bytes one token adds to one layer: K and V rows of every KV head."""
    return 2 * h_kv * d_h * elem


def crossover_tokens(P: int, h_kv: int, d_h: int, r_p: float, r_kv: float) -> float:
    """n* = P (1 - r_P) / (2 h_kv d_h (1 - r_KV)); element size and layer count cancel."""
    return P * (1.0 - r_p) / (2.0 * h_kv * d_h * (1.0 - r_kv))


def ideal_speedup(b_total: float, saved: float) -> float:
    return b_total / (b_total - saved)


# --- algorithmic bytes per launch --------------------------------------------

def dense_verify_bytes(B: int, Hq: int, Hkv: int, d: int, n_prefix: int, gamma: int) -> int:
    """Full K and V of every KV head (n_prefix + gamma rows) + q in + o out."""
    kv = B * Hkv * (n_prefix + gamma) * 2 * d * BF16
    qo = B * Hq * gamma * 2 * d * BF16
    return kv + qo


def sparse_decode_bytes(B: int, Hq: int, d: int, total_selected: int) -> int:
    """Selected K and V rows + their int32 indices + q in + o out.
    `total_selected` is the sum of list lengths over all (b, h)."""
    return total_selected * (2 * d * BF16 + 4) + B * Hq * 2 * d * BF16


def score_bytes(B: int, Hq: int, Hkv: int, d: int, n: int, W: int) -> int:
    """One read of K (the algorithmic minimum) + window queries + fp32 scores out."""
    return B * Hkv * n * d * BF16 + B * Hq * W * d * BF16 + B * Hkv * n * 4


def select_bytes(B: int, Hkv: int, n: int, total_selected: int) -> int:
    """fp32 scores in + int32 list out."""
    return B * Hkv * n * 4 + 4 * total_selected


# --- the StD I/O model (Sparse-to-Dense page, 3.3 I/O complexity) -------------
# Counted in KV entries read per decode round: the sparse draft model reads the
# K selected visual entries and all m_t text entries for each of gamma drafted
# tokens; the dense verify reads all m_v + m_t entries once.

def std_io_sparse(gamma: int, K: int, m_t: int) -> int:
    return gamma * (K + m_t)


def std_io_dense(m_v: int, m_t: int) -> int:
    return m_v + m_t


def std_io_total(gamma: int, K: int, m_t: int, m_v: int) -> int:
    return std_io_sparse(gamma, K, m_t) + std_io_dense(m_v, m_t)


def std_io_average(gamma: int, K: int, m_t: int, m_v: int, alpha: float) -> float:
    """Entries read per accepted token when a fraction alpha of the gamma drafts
    is accepted: I/O_total / (alpha gamma)."""
    return std_io_total(gamma, K, m_t, m_v) / (alpha * gamma)


def std_alpha_threshold(gamma: int, K: int, m_t: int, m_v: int) -> float:
    """Acceptance ratio above which StD reads fewer entries per token than
    vanilla decoding (m_v + m_t per token): (K + m_t) / (m_v + m_t) + 1 / gamma."""
    return (K + m_t) / (m_v + m_t) + 1.0 / gamma


# --- the speculative-decoding speed-up model (SpecVLM page, SD in 60 seconds) --

def sd_speedup(tau: float, gamma: int, td_over_tt: float, ttg_over_tt: float) -> float:
    """tau / (gamma T_d / T_t + T_t^gamma / T_t): accept length over the cost of
    gamma draft passes plus one verification of gamma tokens, in units of one
    target decode pass."""
    return tau / (gamma * td_over_tt + ttg_over_tt)
