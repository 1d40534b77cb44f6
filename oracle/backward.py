"""The oracle for the backward pass of attention, in float64.

TEST INFRASTRUCTURE ONLY.  Only ``tests/`` and ``bench.py``'s CPU legs may
import this module; the CUDA library never calls it and shares no code with it.

"FlashAttention and Fused Kernels: Attention Without the n x n Matrix",
section "Training: recompute instead of store": the backward pass keeps only O
and the per-row softmax statistics from the forward pass and recomputes the
scores and probabilities block by block; "Flash Attention, tiled", section
"More arithmetic can still be faster", says the same.  What it computes is the
gradient of the forward output with respect to Q, K and V, which the pages do
not write out; the plain definition is the chain rule through the three steps
of the forward pass (scores, row softmax, weighted values), for an upstream
gradient dO:

* ``O = P V``                      gives ``dV = P^T dO`` and ``dP = dO V^T``;
* ``P_i = softmax(S_i)`` (per row) gives ``dS_ij = P_ij (dP_ij - sum_k P_ik dP_ik)``;
* ``S = scale * Q K^T`` (masked)   gives ``dQ = scale * dS K`` and ``dK = scale * dS^T Q``;
  masked scores have ``P = 0`` and so ``dS = 0``.

``sum_k P_ik dP_ik`` equals ``sum_c dO_ic O_ic`` (``dP_i . P_i = dO_i . (P V)_i``),
the per-row quantity a FlashAttention backward pass computes first from O and
dO; ``row_dot`` computes it that way and the pins check that the two agree.

P is formed here from the plain softmax of the forward oracle, not from a
stored log-sum-exp, so the backward oracle does not depend on any shortcut the
kernels take.  The steps are module-level functions so that a test can plant a
mistake in one of them.
"""
from __future__ import annotations

import numpy as np

from .attention import causal_mask, scores, softmax_rows


def probabilities_head(q: np.ndarray, k: np.ndarray, causal: bool, scale: float) -> np.ndarray:
    """P (T, T) of one head from the forward oracle's own steps."""
    T = q.shape[0]
    S = scores(q, k, scale)
    if causal:
        S = causal_mask(S, np.arange(T))
    P, _, _ = softmax_rows(S)
    return P


def grad_values(P: np.ndarray, do: np.ndarray) -> np.ndarray:
    """``dV = P^T dO``."""
    return P.T @ do


def grad_probabilities(do: np.ndarray, v: np.ndarray) -> np.ndarray:
    """``dP = dO V^T``."""
    return do @ v.T


def row_dot(do: np.ndarray, o: np.ndarray) -> np.ndarray:
    """``D_i = sum_c dO_ic O_ic``."""
    return (do * o).sum(axis=1)


def grad_scores(P: np.ndarray, dP: np.ndarray, D: np.ndarray) -> np.ndarray:
    """Softmax backward per row: ``dS = P * (dP - D)`` with ``D_i = sum_k P_ik dP_ik``."""
    return P * (dP - D[:, None])


def grad_queries(dS: np.ndarray, k: np.ndarray, scale: float) -> np.ndarray:
    """``dQ = scale * dS K``."""
    return scale * (dS @ k)


def grad_keys(dS: np.ndarray, q: np.ndarray, scale: float) -> np.ndarray:
    """``dK = scale * dS^T Q``."""
    return scale * (dS.T @ q)


def attention_bwd_head(q, k, v, do, causal: bool, scale: float):
    """One (batch, head): q, k, v, do are (T, d) float64.  Returns (dQ, dK, dV)."""
    P = probabilities_head(q, k, causal, scale)
    O = P @ v
    dV = grad_values(P, do)
    dP = grad_probabilities(do, v)
    dS = grad_scores(P, dP, row_dot(do, O))
    return grad_queries(dS, k, scale), grad_keys(dS, q, scale), dV


def attention_bwd(q, k, v, do, causal: bool, scale: float):
    """Gradients of ``sum(dO * O)`` for (B, H, T, d) inputs; returns (dQ, dK, dV), float64."""
    q, k, v, do = (np.asarray(x, dtype=np.float64) for x in (q, k, v, do))
    dq, dk, dv = np.empty_like(q), np.empty_like(k), np.empty_like(v)
    B, H = q.shape[:2]
    for b in range(B):
        for h in range(H):
            dq[b, h], dk[b, h], dv[b, h] = attention_bwd_head(q[b, h], k[b, h], v[b, h], do[b, h], causal, scale)
    return dq, dk, dv


def attention_bwd_parts(q, k, v, do, causal: bool, scale: float):
    """One head's P and dS as well (for error bounds in the tests): (dQ, dK, dV, P, dS)."""
    P = probabilities_head(q, k, causal, scale)
    O = P @ v
    dV = grad_values(P, do)
    dS = grad_scores(P, grad_probabilities(do, v), row_dot(do, O))
    return grad_queries(dS, k, scale), grad_keys(dS, q, scale), dV, P, dS
