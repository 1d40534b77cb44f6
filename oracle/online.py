"""The online-softmax recurrence and the split combine, in float64, one row at a time.

TEST INFRASTRUCTURE ONLY (same import rule as ``oracle.attention``).

These routines restate the streaming recurrence the pages derive, so that the
tests can show it equals the plain three-step definition in
``oracle.attention`` (the equivalence every FlashAttention kernel rests on):

* "FlashAttention: the IO-aware Attention Kernel", section 3.2 "Online
  softmax - the key trick": ``m_new = max(m, m~)``,
  ``l_new = e^(m - m_new) l + sum_j e^(s_j - m_new)``,
  ``O_new = e^(m - m_new) O + sum_j e^(s_j - m_new) v_j``, output ``O / l``;
* "Flash Attention, tiled", section "What happens when the maximum changes":
  ``m' = max(m, max(s))``, ``r = exp(m - m')``, ``p = exp(s - m')``,
  ``l = r l + sum(p)``, ``o = r o + p^T V``;
* "FlashAttention and Fused Kernels", section "Flash-Decoding": each split
  yields a partial output and one log-sum-exp per row, and the partials are
  combined by rescaling every split to the largest maximum.

Reading where the pages leave a step open: with the running max still at
``-inf`` the rescale factor is 0 (the guard in the lesson's
``online_attention``); a block whose scores are all ``-inf`` adds nothing.
"""
from __future__ import annotations

import math

import numpy as np


def online_softmax_row(s: np.ndarray, V: np.ndarray, block: int, trace: list | None = None):
    """Stream one query row's scores ``s`` (n,) and value rows ``V`` (n, dv) in blocks.

    Returns ``(y, m, l)`` with ``y = o / l``.  If ``trace`` is a list, the state
    ``(m, l, o)`` after every block is appended to it.
    """
    s = np.asarray(s, dtype=np.float64)
    V = np.asarray(V, dtype=np.float64)
    m, l = -math.inf, 0.0
    o = np.zeros(V.shape[1], dtype=np.float64)
    for start in range(0, s.shape[0], block):
        sb = s[start:start + block]
        Vb = V[start:start + block]
        m_new = max(m, float(sb.max()))
        if m_new != -math.inf:
            r = math.exp(m - m_new) if m != -math.inf else 0.0
            p = np.exp(sb - m_new)
            l = r * l + float(p.sum())
            o = r * o + p @ Vb
            m = m_new
        if trace is not None:
            trace.append((m, l, o.copy()))
    return o / l, m, l


def online_attention_row(q_row: np.ndarray, k: np.ndarray, v: np.ndarray, scale: float,
                         block: int, visible: int | None = None):
    """One query row against keys ``k[:visible]``, scores formed block by block."""
    n = k.shape[0] if visible is None else visible
    s = scale * (np.asarray(k[:n], np.float64) @ np.asarray(q_row, np.float64))
    y, m, l = online_softmax_row(s, v[:n], block)
    return y, m + math.log(l)


def combine_partials(m_parts, l_parts, y_parts):
    """Merge per-split states of one row: maxima ``m_k``, sums ``l_k``, normalised outputs ``y_k``.

    Every split is rescaled to the largest maximum ``M``:
    ``l = sum_k e^(m_k - M) l_k``, ``acc = sum_k e^(m_k - M) l_k y_k``, output
    ``acc / l``.  Returns ``(y, lse)`` with ``lse = M + ln l``.
    """
    m_parts = np.asarray(m_parts, dtype=np.float64)
    l_parts = np.asarray(l_parts, dtype=np.float64)
    y_parts = np.asarray(y_parts, dtype=np.float64)
    M = float(m_parts.max())
    w = np.exp(m_parts - M)
    l = float((w * l_parts).sum())
    acc = ((w * l_parts)[:, None] * y_parts).sum(axis=0)
    return acc / l, M + math.log(l)


def combine_by_lse(lse_parts, y_parts):
    """The same merge written with one log-sum-exp per split: ``y = sum_k e^(lse_k - LSE) y_k``."""
    lse_parts = np.asarray(lse_parts, dtype=np.float64)
    y_parts = np.asarray(y_parts, dtype=np.float64)
    M = float(lse_parts.max())
    lse = M + math.log(float(np.exp(lse_parts - M).sum()))
    w = np.exp(lse_parts - lse)
    return (w[:, None] * y_parts).sum(axis=0), lse
