"""The oracle: plain three-step attention, one query row at a time, in float64.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and
the CPU-baseline leg of ``bench.py`` may import this module.  The product path
(the CUDA library and its Python binding) never calls it and shares no code
with it.

What it computes is the textbook definition of scaled dot-product attention
with an optional causal mask, exactly as the pages write it before any tiling:

* "Flash Attention, tiled: exact attention without the T x T HBM matrix",
  section "Ordinary causal attention": ``S = (Q K^T) / sqrt(d)``, future keys
  set to ``-inf`` before the softmax, ``Y = att @ v``;
* "FlashAttention and Fused Kernels: Attention Without the n x n Matrix",
  section "Step 1: why standard attention is memory-bound": scores, then a
  row-wise softmax, then ``O = P V``; section "Step 2: tiling and the online
  softmax": the row maximum is subtracted before exponentiating;
* "FlashAttention: the IO-aware Attention Kernel", section 4,
  ``full_attention``: materialise the row, take its max, exponentiate, divide
  by the sum, weight the values.

The log-sum-exp that a FlashAttention forward pass also writes ("the output
and limited softmax state", page "Flash Attention, tiled", section "From the
example to tiled GPU work"; "the log-sum-exp of the attention values", page
"FlashAttention and Fused Kernels", section "Flash-Decoding") is not defined
on the pages.  The reading used here: the natural log of the softmax
denominator of the scaled, masked scores, ``LSE_i = m_i + ln l_i``.

The steps are separate module-level functions so that a test can plant a
mistake in one of them and check that the pins catch it.  Query rows are
independent (each row has its own softmax), so rows are processed in groups
only to bound memory; no reduction is split or reordered.  There is no online
recurrence here.
"""
from __future__ import annotations

import numpy as np


def scores(q_rows: np.ndarray, k: np.ndarray, scale: float) -> np.ndarray:
    """Scaled scores ``s_ij = scale * sum_c q_ic k_jc`` (rows of ``S = Q K^T / sqrt(d)``)."""
    return scale * (q_rows @ k.T)


def causal_mask(S: np.ndarray, row_index: np.ndarray) -> np.ndarray:
    """Query ``i`` may use only keys ``j <= i``; the others get ``-inf``."""
    j = np.arange(S.shape[1])
    out = S.copy()
    out[j[None, :] > np.asarray(row_index)[:, None]] = -np.inf
    return out


def softmax_rows(S: np.ndarray):
    """Safe softmax of every row: ``p = exp(s - m) / l`` with ``m = max s``, ``l = sum exp(s - m)``.

    Returns ``(P, m, l)``.
    """
    m = S.max(axis=1)
    e = np.exp(S - m[:, None])
    l = e.sum(axis=1)
    return e / l[:, None], m, l


def weighted_values(P: np.ndarray, v: np.ndarray) -> np.ndarray:
    """``O = P V``: each output row is the probability-weighted sum of value rows."""
    return P @ v


def log_sum_exp(m: np.ndarray, l: np.ndarray) -> np.ndarray:
    """Natural-log LSE of a row from its max and shifted sum: ``ln sum_j e^(s_j) = m + ln l``."""
    return m + np.log(l)


def attention_head(q: np.ndarray, k: np.ndarray, v: np.ndarray, causal: bool,
                   scale: float, rows=None, row_group: int = 512):
    """One (batch, head): q, k, v are (T, d) float64.  Returns (O[rows], LSE[rows])."""
    T = q.shape[0]
    rows = np.arange(T) if rows is None else np.asarray(rows, dtype=np.int64)
    O = np.empty((rows.shape[0], v.shape[1]), dtype=np.float64)
    lse = np.empty(rows.shape[0], dtype=np.float64)
    for g0 in range(0, rows.shape[0], row_group):
        r = rows[g0:g0 + row_group]
        S = scores(q[r], k, scale)
        if causal:
            S = causal_mask(S, r)
        P, m, l = softmax_rows(S)
        O[g0:g0 + r.shape[0]] = weighted_values(P, v)
        lse[g0:g0 + r.shape[0]] = log_sum_exp(m, l)
    return O, lse


def attention_fwd(q: np.ndarray, k: np.ndarray, v: np.ndarray, causal: bool,
                  scale: float, rows=None):
    """Attention for (B, H, T, d) float64 tensors.

    ``rows``: optional 1-D array of query positions to evaluate in every
    (batch, head); ``None`` means all ``T`` rows.  Returns ``O`` of shape
    (B, H, R, d) and ``LSE`` of shape (B, H, R), both float64.
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    B, H, T, d = q.shape
    R = T if rows is None else len(rows)
    O = np.empty((B, H, R, v.shape[3]), dtype=np.float64)
    lse = np.empty((B, H, R), dtype=np.float64)
    for b in range(B):
        for h in range(H):
            O[b, h], lse[b, h] = attention_head(q[b, h], k[b, h], v[b, h], causal, scale, rows)
    return O, lse


def attention_fwd_gqa(q: np.ndarray, k: np.ndarray, v: np.ndarray, causal: bool,
                      scale: float, rows=None):
    """Attention with grouped K/V heads ("FlashAttention and Fused Kernels",
    section "Step 4: decoding is a different problem": Llama 3.1 8B lets every
    K/V head serve 4 query heads).

    q is (B, H, T, d); k and v are (B, Hkv, T, d) with H a multiple of Hkv.
    Query head h attends with K/V head h // (H // Hkv): per query head this is
    exactly ``attention_head`` on that head's keys and values.  Returns O
    (B, H, R, d) and LSE (B, H, R) as ``attention_fwd`` does.
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    B, H, T, d = q.shape
    Hkv = k.shape[1]
    if H % Hkv != 0:
        raise ValueError("the number of query heads must be a multiple of the K/V heads")
    R = T if rows is None else len(rows)
    O = np.empty((B, H, R, v.shape[3]), dtype=np.float64)
    lse = np.empty((B, H, R), dtype=np.float64)
    for b in range(B):
        for h in range(H):
            g = kv_head(h, H, Hkv)
            O[b, h], lse[b, h] = attention_head(q[b, h], k[b, g], v[b, g], causal, scale, rows)
    return O, lse


def kv_head(h: int, H: int, Hkv: int) -> int:
    """The K/V head that query head ``h`` reads: consecutive groups of H / Hkv query heads share one."""
    return h // (H // Hkv)


def probabilities(q: np.ndarray, k: np.ndarray, causal: bool, scale: float) -> np.ndarray:
    """The full probability matrix P of one head (T x T).  Small inputs only."""
    S = scores(np.asarray(q, np.float64), np.asarray(k, np.float64), scale)
    if causal:
        S = causal_mask(S, np.arange(S.shape[0]))
    P, _, _ = softmax_rows(S)
    return P
