"""Plant plausible mistakes in the oracle (on the CPU) and check that the pins catch every one.

Each mutation replaces one step of ``oracle.attention`` or ``oracle.online``
with a wrong variant: a dropped term, a wrong sign or index, a transposed
operand, a wrong base.  The pin suite must fail for each of them; a mutation
that survives means the oracle is not pinned where that step could go wrong.
"""
import math
import warnings

import numpy as np
import pytest

import oracle.attention as A
import oracle.backward as BW
import oracle.online as ON
from oracle_pins import ALL_PINS


def _online_variant(kind):
    def row(s, V, block, trace=None):
        s = np.asarray(s, dtype=np.float64)
        V = np.asarray(V, dtype=np.float64)
        m, l = -math.inf, 0.0
        o = np.zeros(V.shape[1])
        for start in range(0, s.shape[0], block):
            sb, Vb = s[start:start + block], V[start:start + block]
            m_new = max(m, float(sb.max()))
            if m_new == -math.inf:
                continue
            r = math.exp(m - m_new) if m != -math.inf else 0.0
            if kind == "wrong_sign_rescale" and m != -math.inf:
                r = math.exp(m_new - m)
            p = np.exp(sb - m_new)
            l = (l if kind == "no_rescale_l" else r * l) + float(p.sum())
            o = (o if kind == "no_rescale_o" else r * o) + p @ Vb
            if kind != "stale_max":
                m = m_new
            if trace is not None:
                trace.append((m, l, o.copy()))
        return o / l, m, l
    return row


def _combine_without_sums(m_parts, l_parts, y_parts):
    m_parts, y_parts = np.asarray(m_parts, float), np.asarray(y_parts, float)
    M = m_parts.max()
    w = np.exp(m_parts - M)
    return (w[:, None] * y_parts).sum(0) / w.sum(), M + math.log(float(np.sum(l_parts)))


MUTATIONS = {
    # scores
    "scores_no_scale": (A, "scores", lambda q, k, s: q @ k.T),
    "scores_divide_scale": (A, "scores", lambda q, k, s: (q @ k.T) / s),
    "scores_scale_squared": (A, "scores", lambda q, k, s: s * s * (q @ k.T)),
    "scores_transposed": (A, "scores", lambda q, k, s: s * (k @ q.T)),
    # causal mask
    "mask_hides_diagonal": (A, "causal_mask", lambda S, r: np.where(
        np.arange(S.shape[1])[None, :] >= np.asarray(r)[:, None], -np.inf, S)),
    "mask_one_future_key": (A, "causal_mask", lambda S, r: np.where(
        np.arange(S.shape[1])[None, :] > np.asarray(r)[:, None] + 1, -np.inf, S)),
    "mask_missing": (A, "causal_mask", lambda S, r: S),
    "mask_reversed": (A, "causal_mask", lambda S, r: np.where(
        np.arange(S.shape[1])[None, :] < np.asarray(r)[:, None], -np.inf, S)),
    # softmax
    "softmax_no_max_shift": (A, "softmax_rows", lambda S: (
        np.exp(S) / np.exp(S).sum(1, keepdims=True), np.zeros(S.shape[0]), np.exp(S).sum(1))),
    "softmax_divide_by_max_term": (A, "softmax_rows", lambda S: (
        np.exp(S - S.max(1, keepdims=True)), S.max(1), np.exp(S - S.max(1, keepdims=True)).sum(1))),
    "softmax_base2": (A, "softmax_rows", lambda S: (
        np.exp2(S - S.max(1, keepdims=True)) / np.exp2(S - S.max(1, keepdims=True)).sum(1, keepdims=True),
        S.max(1), np.exp2(S - S.max(1, keepdims=True)).sum(1))),
    "softmax_reports_zero_max": (A, "softmax_rows", lambda S: (
        np.exp(S - S.max(1, keepdims=True)) / np.exp(S - S.max(1, keepdims=True)).sum(1, keepdims=True),
        np.zeros(S.shape[0]), np.exp(S - S.max(1, keepdims=True)).sum(1))),
    # weighted values
    "values_transposed_probabilities": (A, "weighted_values", lambda P, v: P.T @ v),
    "values_drop_last_key": (A, "weighted_values", lambda P, v: P[:, :-1] @ v[:-1]),
    # grouped K/V heads
    "gqa_heads_interleaved": (A, "kv_head", lambda h, H, Hkv: h % Hkv),
    "gqa_group_off_by_one": (A, "kv_head", lambda h, H, Hkv: min((h + 1) // (H // Hkv), Hkv - 1)),
    # backward pass
    "bwd_dv_untransposed": (BW, "grad_values", lambda P, do: P @ do),
    "bwd_dp_rescaled": (BW, "grad_probabilities", lambda do, v: (do @ v.T) * 1.0001),
    "bwd_ds_drops_row_dot": (BW, "grad_scores", lambda P, dP, D: P * dP),
    "bwd_ds_row_dot_sign": (BW, "grad_scores", lambda P, dP, D: P * (dP + D[:, None])),
    "bwd_dq_no_scale": (BW, "grad_queries", lambda dS, k, s: dS @ k),
    "bwd_dq_transposed": (BW, "grad_queries", lambda dS, k, s: s * (dS.T @ k)),
    "bwd_dk_untransposed": (BW, "grad_keys", lambda dS, q, s: s * (dS @ q)),
    "bwd_row_dot_squared": (BW, "row_dot", lambda do, o: (do * o * o).sum(axis=1)),
    # LSE
    "lse_drops_max": (A, "log_sum_exp", lambda m, l: np.log(l)),
    "lse_base2": (A, "log_sum_exp", lambda m, l: m + np.log2(l)),
    "lse_wrong_sign": (A, "log_sum_exp", lambda m, l: m - np.log(l)),
    # online recurrence and split combine (test-only routines)
    "online_no_rescale_o": (ON, "online_softmax_row", _online_variant("no_rescale_o")),
    "online_no_rescale_l": (ON, "online_softmax_row", _online_variant("no_rescale_l")),
    "online_wrong_sign_rescale": (ON, "online_softmax_row", _online_variant("wrong_sign_rescale")),
    "online_stale_max": (ON, "online_softmax_row", _online_variant("stale_max")),
    "combine_without_sums": (ON, "combine_partials", _combine_without_sums),
}


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_mutation_is_caught(name, monkeypatch):
    module, attr, bad = MUTATIONS[name]
    monkeypatch.setattr(module, attr, bad)
    caught = []
    with warnings.catch_warnings():
        warnings.simplefilter("ignore")
        with np.errstate(all="ignore"):
            for pin in ALL_PINS:
                try:
                    pin()
                except Exception as e:  # an assertion, or a shape error the mistake causes
                    caught.append((pin.__name__, type(e).__name__))
    assert caught, f"mutation {name} passed every pin"
