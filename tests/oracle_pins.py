"""Pins for the float64 oracle: each check ties it to something other than itself.

The checks use values the pages print (fixtures under ``tests/golden/``),
closed forms, invariants, a textbook special case and brute force in plain
Python on tiny inputs.  Each is a function that raises ``AssertionError``
when the oracle disagrees; ``test_oracle_pins.py`` runs them one by one and
``test_oracle_mutations.py`` plants mistakes in the oracle and checks that at
least one of them fails.
"""
from __future__ import annotations

import json
import math
import os

import numpy as np

import oracle.attention as A
import oracle.backward as BW
import oracle.online as ON

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _g(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def _t(x):
    """(T, d) -> (1, 1, T, d) float64."""
    return np.asarray(x, dtype=np.float64)[None, None]


def _rng(seed):
    return np.random.default_rng(seed)


def _brute_row(q, k, v, scale, visible):
    """Plain-Python attention of one row over keys 0..visible-1 (no numpy)."""
    s = [scale * math.fsum(q[c] * k[j][c] for c in range(len(q))) for j in range(visible)]
    m = max(s)
    e = [math.exp(x - m) for x in s]
    l = math.fsum(e)
    out = [math.fsum(e[j] * v[j][c] for j in range(visible)) / l for c in range(len(v[0]))]
    return out, m + math.log(l)


# ---------------------------------------------------------------- printed values

def pin_f1_three_token_causal():
    g = _g("f1_three_token_causal.json")
    O, lse = A.attention_fwd(_t(g["q"]), _t(g["k"]), _t(g["v"]), True, g["d"] ** -0.5)
    dec = g["output_printed_decimals"]
    assert np.allclose(np.round(O[0, 0], dec), g["output_printed"], atol=0, rtol=0), O
    # exact values behind the printed ones: row 2 is (V0 + V1 + V2) / 3
    assert abs(O[0, 0, 2, 0] - 40.0 / 3.0) < 1e-12 and abs(O[0, 0, 2, 1] - 50.0 / 3.0) < 1e-12
    P = A.probabilities(np.asarray(g["q"]), np.asarray(g["k"]), True, g["d"] ** -0.5)
    assert np.allclose(P, g["probabilities"], atol=1e-15)
    # every visible score is 0, so LSE_i = ln(number of visible keys)
    assert np.allclose(lse[0, 0], np.log([1.0, 2.0, 3.0]), atol=1e-15)


def pin_f2_four_scores():
    g = _g("f2_four_score_stream.json")
    s = np.asarray(g["scores"])
    # one query q = 1 (d = 1) against keys k_j = s_j with scale 1 gives scores s_j
    T = s.shape[0]
    q = np.ones((T, 1))
    k = s[:, None]
    v = np.asarray(g["values"])[:, None]
    O, lse = A.attention_fwd(_t(q), _t(k), _t(v), False, 1.0)
    assert round(float(O[0, 0, 0, 0]), g["output_decimals"]) == g["output_printed"], O[0, 0, 0]
    P = A.probabilities(q, k, False, 1.0)
    assert np.array_equal(np.round(P[0], g["weights_decimals"]), g["weights_printed"]), P[0]
    # the page's combined denominator 1.553 is sum_j exp(s_j - 4), so LSE = 4 + ln(1.553)
    f3 = _g("f3_split_combine.json")
    lo = 4.0 + math.log(f3["combined_denominator"] - 0.0005)
    hi = 4.0 + math.log(f3["combined_denominator"] + 0.0005)
    assert lo <= lse[0, 0, 0] <= hi, lse[0, 0, 0]


def pin_f4_lesson_fixture():
    g = _g("f4_online_softmax_lesson.json")
    K = np.asarray(g["k"])
    Q = np.tile(np.asarray(g["q"]), (K.shape[0], 1))  # the one query, repeated for every row
    O, _ = A.attention_fwd(_t(Q), _t(K), _t(g["v"]), False, g["scale"])
    assert np.allclose(np.round(O[0, 0], g["output_decimals"]), np.asarray(g["output_printed"])[None, :],
                       atol=0, rtol=0), O[0, 0, 0]


# ---------------------------------------------------------------- closed forms

def pin_zero_queries_average_values():
    rng = _rng(11)
    T, d = 37, 8
    k = rng.standard_normal((T, d))
    v = rng.standard_normal((T, d))
    q = np.zeros((T, d))
    O, lse = A.attention_fwd(_t(q), _t(k), _t(v), True, 0.7)
    running = np.cumsum(v, axis=0) / np.arange(1, T + 1)[:, None]
    assert np.allclose(O[0, 0], running, atol=1e-13)
    assert np.allclose(lse[0, 0], np.log(np.arange(1, T + 1)), atol=1e-13)
    O, lse = A.attention_fwd(_t(q), _t(k), _t(v), False, 0.7)
    assert np.allclose(O[0, 0], v.mean(axis=0)[None, :], atol=1e-13)
    assert np.allclose(lse[0, 0], math.log(T), atol=1e-13)


def pin_constant_values():
    rng = _rng(12)
    T, d = 29, 4
    q, k = rng.standard_normal((T, d)), rng.standard_normal((T, d))
    v = np.full((T, d), -2.5)
    for causal in (False, True):
        O, _ = A.attention_fwd(_t(q), _t(k), _t(v), causal, 0.5)
        assert np.allclose(O, -2.5, atol=1e-13)


def pin_identity_values_give_probabilities():
    # V = I (d = T): O = P.  Rows of P sum to 1 and P_ij / P_ik = exp(s_ij - s_ik).
    rng = _rng(13)
    T = 9
    q, k = rng.standard_normal((T, T)), rng.standard_normal((T, T))
    scale = 0.4
    for causal in (False, True):
        O, _ = A.attention_fwd(_t(q), _t(k), _t(np.eye(T)), causal, scale)
        P = O[0, 0]
        assert np.allclose(P.sum(axis=1), 1.0, atol=1e-13)
        for i in range(T):
            vis = i + 1 if causal else T
            assert np.all(P[i, vis:] == 0.0)
            for j in range(vis):
                sij = scale * math.fsum(q[i, c] * k[j, c] for c in range(T))
                si0 = scale * math.fsum(q[i, c] * k[0, c] for c in range(T))
                assert abs(P[i, j] / P[i, 0] - math.exp(sij - si0)) < 1e-11 * math.exp(sij - si0)


def pin_score_shift_moves_lse_only():
    # an extra dimension with k_extra = 1 and q_extra = c / scale adds c to every score of row i
    rng = _rng(14)
    T, d = 23, 6
    q, k, v = (rng.standard_normal((T, d)) for _ in range(3))
    scale = 0.3
    c = rng.uniform(-3, 3, size=T)
    q2 = np.concatenate([q, (c / scale)[:, None]], axis=1)
    k2 = np.concatenate([k, np.ones((T, 1))], axis=1)
    for causal in (False, True):
        O1, l1 = A.attention_fwd(_t(q), _t(k), _t(v), causal, scale)
        O2, l2 = A.attention_fwd(_t(q2), _t(k2), _t(v), causal, scale)
        assert np.allclose(O1, O2, atol=1e-12)
        assert np.allclose(l2[0, 0] - l1[0, 0], c, atol=1e-12)


def pin_single_key():
    rng = _rng(15)
    q, k, v = rng.standard_normal((1, 5)), rng.standard_normal((1, 5)), rng.standard_normal((1, 5))
    for causal in (False, True):
        O, lse = A.attention_fwd(_t(q), _t(k), _t(v), causal, 0.9)
        assert np.array_equal(O[0, 0, 0], v[0])
        assert abs(lse[0, 0, 0] - 0.9 * math.fsum(q[0] * k[0])) < 1e-14


def pin_two_keys_logistic():
    # T = 2, d = 1, no mask: O = sigma(s0 - s1) v0 + sigma(s1 - s0) v1, sigma the logistic function
    q = np.array([[1.5], [-0.25]])
    k = np.array([[0.8], [-1.2]])
    v = np.array([[3.0], [-7.0]])
    scale = 0.5
    O, lse = A.attention_fwd(_t(q), _t(k), _t(v), False, scale)
    for i in range(2):
        s0, s1 = scale * q[i, 0] * k[0, 0], scale * q[i, 0] * k[1, 0]
        sig = 1.0 / (1.0 + math.exp(-(s0 - s1)))
        assert abs(O[0, 0, i, 0] - (sig * 3.0 + (1.0 - sig) * -7.0)) < 1e-14
        assert abs(lse[0, 0, i] - (max(s0, s1) + math.log1p(math.exp(-abs(s0 - s1))))) < 1e-14


# ---------------------------------------------------------------- invariants

def pin_causal_row0_is_v0():
    rng = _rng(16)
    T, d = 17, 8
    q, k, v = (rng.standard_normal((T, d)) for _ in range(3))
    O, lse = A.attention_fwd(_t(q), _t(k), _t(v), True, 0.35)
    assert np.array_equal(O[0, 0, 0], v[0])
    assert abs(lse[0, 0, 0] - 0.35 * math.fsum(q[0] * k[0])) < 1e-14


def pin_causal_ignores_future():
    rng = _rng(17)
    T, d = 20, 4
    q, k, v = (rng.standard_normal((T, d)) for _ in range(3))
    O1, l1 = A.attention_fwd(_t(q), _t(k), _t(v), True, 0.5)
    for i in (0, 7, 18):
        k2, v2 = k.copy(), v.copy()
        k2[i + 1:] = rng.standard_normal(k2[i + 1:].shape) * 5
        v2[i + 1:] = rng.standard_normal(v2[i + 1:].shape) * 5
        O2, l2 = A.attention_fwd(_t(q), _t(k2), _t(v2), True, 0.5)
        assert np.array_equal(O1[0, 0, :i + 1], O2[0, 0, :i + 1])
        assert np.array_equal(l1[0, 0, :i + 1], l2[0, 0, :i + 1])
        # and a change at or before i does change row i
        k3 = k.copy()
        k3[i] += 1.0
        O3, _ = A.attention_fwd(_t(q), _t(k3), _t(v), True, 0.5)
        assert not np.array_equal(O1[0, 0, i], O3[0, 0, i]) or i == 0


def pin_key_permutation_invariance():
    rng = _rng(18)
    T, d = 31, 8
    q, k, v = (rng.standard_normal((T, d)) for _ in range(3))
    perm = rng.permutation(T)
    O1, l1 = A.attention_fwd(_t(q), _t(k), _t(v), False, 0.6)
    O2, l2 = A.attention_fwd(_t(q), _t(k[perm]), _t(v[perm]), False, 0.6)
    assert np.allclose(O1, O2, atol=1e-13) and np.allclose(l1, l2, atol=1e-13)


def pin_large_scores_stay_finite():
    # scores near +-1000 overflow exp() unless the row max is subtracted first
    rng = _rng(19)
    T, d = 16, 4
    q, k, v = (rng.standard_normal((T, d)) for _ in range(3))
    big = 60.0
    O1, l1 = A.attention_fwd(_t(q * big), _t(k * big), _t(v), True, 1.0)
    assert np.all(np.isfinite(O1)) and np.all(np.isfinite(l1))
    for i in range(T):
        ref, ref_lse = _brute_row(list(q[i] * big), [list(r) for r in k * big], [list(r) for r in v], 1.0, i + 1)
        assert np.allclose(O1[0, 0, i], ref, atol=1e-12)
        assert abs(l1[0, 0, i] - ref_lse) < 1e-9 * max(1.0, abs(ref_lse))


def pin_brute_force_tiny():
    rng = _rng(20)
    for T, d, causal, scale in ((5, 3, True, 0.8), (7, 2, False, 1.3), (4, 6, True, 0.2), (6, 4, False, 0.5)):
        q, k, v = (rng.standard_normal((T, d)) * 2 for _ in range(3))
        O, lse = A.attention_fwd(_t(q), _t(k), _t(v), causal, scale)
        for i in range(T):
            ref, ref_lse = _brute_row(list(q[i]), [list(r) for r in k], [list(r) for r in v], scale,
                                      i + 1 if causal else T)
            assert np.allclose(O[0, 0, i], ref, rtol=0, atol=1e-13), (T, d, causal, i)
            assert abs(lse[0, 0, i] - ref_lse) < 1e-13


def pin_row_subset_matches_full():
    rng = _rng(21)
    T, d = 40, 8
    q, k, v = (rng.standard_normal((2, 3, T, d)) for _ in range(3))
    rows = np.array([0, 5, 39, 17])
    for causal in (False, True):
        O, lse = A.attention_fwd(q, k, v, causal, 0.5)
        Os, lses = A.attention_fwd(q, k, v, causal, 0.5, rows=rows)
        assert np.array_equal(O[:, :, rows], Os) and np.array_equal(lse[:, :, rows], lses)


def pin_gqa_brute_force_tiny():
    """Grouped K/V heads: every query head equals plain-Python attention with K/V head h // (H / Hkv)."""
    rng = _rng(22)
    B, H, Hkv, T, d = 2, 6, 2, 5, 3
    q = rng.standard_normal((B, H, T, d)) * 1.5
    k, v = (rng.standard_normal((B, Hkv, T, d)) * 1.5 for _ in range(2))
    for causal in (False, True):
        O, lse = A.attention_fwd_gqa(q, k, v, causal, 0.7)
        for b in range(B):
            for h in range(H):
                g = h // 3  # heads 0-2 read K/V head 0, heads 3-5 read K/V head 1
                for i in range(T):
                    ref, ref_lse = _brute_row(list(q[b, h, i]), [list(r) for r in k[b, g]], [list(r) for r in v[b, g]],
                                              0.7, i + 1 if causal else T)
                    assert np.allclose(O[b, h, i], ref, rtol=0, atol=1e-13), (b, h, i, causal)
                    assert abs(lse[b, h, i] - ref_lse) < 1e-13


def pin_gqa_one_group_per_head_is_mha():
    """With as many K/V heads as query heads the grouped form is the ordinary one."""
    rng = _rng(23)
    q, k, v = (rng.standard_normal((2, 3, 9, 4)) for _ in range(3))
    for causal in (False, True):
        O1, l1 = A.attention_fwd_gqa(q, k, v, causal, 0.4)
        O2, l2 = A.attention_fwd(q, k, v, causal, 0.4)
        assert np.array_equal(O1, O2) and np.array_equal(l1, l2)


# ---------------------------------------------------------------- online recurrence (test-only)

def pin_online_f2_two_blocks():
    g = _g("f2_four_score_stream.json")
    s, v = np.asarray(g["scores"]), np.asarray(g["values"])[:, None]
    y, m, l = ON.online_softmax_row(s, v, g["block"])
    assert round(float(y[0]), g["output_decimals"]) == g["output_printed"]
    y1, _, _ = ON.online_softmax_row(s[:2], v[:2], 2)
    assert round(float(y1[0]), g["block1_partial_decimals"]) == g["block1_partial_output"]


def pin_online_f4_block_sizes():
    g = _g("f4_online_softmax_lesson.json")
    for b in g["blocks"]:
        y, _ = ON.online_attention_row(np.asarray(g["q"]), np.asarray(g["k"]), np.asarray(g["v"]),
                                       g["scale"], b)
        assert np.array_equal(np.round(y, g["output_decimals"]), g["output_printed"]), (b, y)


def pin_online_f5_max_change():
    g = _g("f5_max_change.json")
    s = np.asarray(g["scores"])
    trace = []
    y, m, l = ON.online_softmax_row(s, np.eye(3), 2, trace)
    (m1, l1, o1), (m2, l2, o2) = trace
    assert m1 == g["m_after"][0] and m2 == g["m_after"][1]
    e = math.exp
    assert abs(l1 - (e(-1) + 1)) < 1e-15
    assert np.allclose(o1, [e(-1), 1.0, 0.0], atol=1e-15)
    r = e(g["r_at_tile2_exponent"])
    assert abs(l2 - (r * (e(-1) + 1) + 1)) < 1e-15
    assert np.allclose(o2, [r * e(-1), r, 1.0], atol=1e-15)


def pin_online_f1_row2_two_tiles():
    g = _g("f1_three_token_causal.json")
    v = np.asarray(g["v"])
    trace = []
    y, _, _ = ON.online_softmax_row(np.zeros(3), v, 2, trace)
    for (m, l, o), want in zip(trace, g["row2_tile_states"]["after_tile"]):
        assert m == want["m"] and l == want["l"] and np.array_equal(o, want["o"])
    assert np.allclose(y, [40 / 3, 50 / 3], atol=1e-14)


def pin_online_equals_three_step():
    rng = _rng(22)
    for T, d, spread in ((9, 4, 1.0), (12, 3, 8.0), (16, 5, 30.0)):
        q, k, v = rng.standard_normal((T, d)), rng.standard_normal((T, d)) * spread, rng.standard_normal((T, d))
        # ascending keys along q make the running max change at every block
        order = np.argsort(k @ q[0])
        k, v = k[order], v[order]
        for causal in (False, True):
            O, lse = A.attention_fwd(_t(q), _t(k), _t(v), causal, 0.5)
            for i in range(T):
                vis = i + 1 if causal else T
                for b in range(1, vis + 1):
                    y, l_ = ON.online_attention_row(q[i], k, v, 0.5, b, vis)
                    assert np.allclose(y, O[0, 0, i], rtol=1e-12, atol=1e-13), (T, causal, i, b)
                    assert abs(l_ - lse[0, 0, i]) <= 1e-12 * max(1.0, abs(l_))


def pin_split_combine_f3():
    g = _g("f3_split_combine.json")
    s, v = np.asarray(g["scores"]), np.asarray(g["values"])[:, None]
    ms, ls, ys = [], [], []
    for (a, b), m_want, l_want, y_want, acc_want in zip(g["splits"], g["split_max"], g["split_sum"],
                                                         g["split_output"], g["split_acc"]):
        y, m, l = ON.online_softmax_row(s[a:b], v[a:b], b - a)
        assert m == m_want
        assert round(l, g["split_sum_decimals"]) == l_want
        assert round(float(y[0]), g["split_output_decimals"]) == y_want
        assert round(float(y[0]) * l, g["split_acc_decimals"]) == acc_want
        ms.append(m), ls.append(l), ys.append(y)
    assert round(math.exp(ms[0] - ms[1]), g["rescale_decimals"]) == g["rescale_factor"]
    y, lse = ON.combine_partials(ms, ls, ys)
    assert round(float(y[0]), g["combined_decimals"]) == g["combined_output"]
    num = math.exp(ms[0] - ms[1]) * ls[0] * ys[0][0] + ls[1] * ys[1][0]
    den = math.exp(ms[0] - ms[1]) * ls[0] + ls[1]
    assert round(num, 2) == g["combined_numerator"] and round(den, 3) == g["combined_denominator"]
    y2, lse2 = ON.combine_by_lse([m + math.log(l) for m, l in zip(ms, ls)], ys)
    assert np.allclose(y, y2, atol=1e-14) and abs(lse - lse2) < 1e-14


def pin_split_combine_matches_oracle():
    rng = _rng(23)
    T, d = 50, 6
    q, k, v = rng.standard_normal((T, d)), rng.standard_normal((T, d)) * 3, rng.standard_normal((T, d))
    O, lse = A.attention_fwd(_t(q), _t(k), _t(v), False, 0.5)
    for bounds in ((0, 50), (0, 7, 50), (0, 13, 14, 40, 50)):
        for i in (0, 25, 49):
            ms, ls, ys, lses = [], [], [], []
            for a, b in zip(bounds[:-1], bounds[1:]):
                s = 0.5 * (k[a:b] @ q[i])
                y, m, l = ON.online_softmax_row(s, v[a:b], b - a)
                ms.append(m), ls.append(l), ys.append(y), lses.append(m + math.log(l))
            y, l_ = ON.combine_partials(ms, ls, ys)
            assert np.allclose(y, O[0, 0, i], atol=1e-13) and abs(l_ - lse[0, 0, i]) < 1e-12
            y2, l2 = ON.combine_by_lse(lses, ys)
            assert np.allclose(y2, O[0, 0, i], atol=1e-13) and abs(l2 - lse[0, 0, i]) < 1e-12


# ---------------------------------------------------------------- backward pass

def _loss(q, k, v, do, causal, scale):
    """sum(dO * O) with O from the forward oracle: its gradient is what the backward pass returns."""
    O, _ = A.attention_fwd(q[None, None], k[None, None], v[None, None], causal, scale)
    return float((do * O[0, 0]).sum())


def pin_bwd_finite_differences():
    """Central differences of sum(dO * O) through the forward oracle agree with the backward oracle."""
    rng = _rng(30)
    h = 1e-6
    for T, d, causal, scale in ((4, 3, False, 0.7), (5, 2, True, 1.1), (3, 4, True, 0.4)):
        q, k, v, do = (rng.standard_normal((T, d)) for _ in range(4))
        dq, dk, dv = BW.attention_bwd(q[None, None], k[None, None], v[None, None], do[None, None], causal, scale)
        for name, x, g in (("q", q, dq), ("k", k, dk), ("v", v, dv)):
            num = np.zeros_like(x)
            for idx in np.ndindex(x.shape):
                xp, xm = x.copy(), x.copy()
                xp[idx] += h
                xm[idx] -= h
                args_p = {"q": q, "k": k, "v": v}
                args_m = dict(args_p)
                args_p[name], args_m[name] = xp, xm
                num[idx] = (_loss(args_p["q"], args_p["k"], args_p["v"], do, causal, scale)
                            - _loss(args_m["q"], args_m["k"], args_m["v"], do, causal, scale)) / (2 * h)
            assert np.allclose(g[0, 0], num, rtol=0, atol=2e-8), (name, T, causal, np.abs(g[0, 0] - num).max())


def pin_bwd_constant_values():
    """If every value row is the same, O does not depend on Q or K: dQ = dK = 0 and dV = P^T dO."""
    rng = _rng(31)
    T, d = 6, 4
    q, k, do = (rng.standard_normal((T, d)) for _ in range(3))
    v = np.tile(rng.standard_normal(d), (T, 1))
    for causal in (False, True):
        dq, dk, dv = BW.attention_bwd(q[None, None], k[None, None], v[None, None], do[None, None], causal, 0.5)
        assert np.abs(dq).max() < 1e-13 and np.abs(dk).max() < 1e-13
        P = A.probabilities(q, k, causal, 0.5)
        assert np.allclose(dv[0, 0], P.T @ do, atol=1e-14)


def pin_bwd_sums():
    """Each row of P sums to 1, so the dV rows sum to the dO rows; a common shift of every key
    leaves the softmax unchanged, so the dK rows sum to zero."""
    rng = _rng(32)
    q, k, v, do = (rng.standard_normal((2, 3, 11, 5)) for _ in range(4))
    for causal in (False, True):
        dq, dk, dv = BW.attention_bwd(q, k, v, do, causal, 0.3)
        assert np.allclose(dv.sum(axis=2), do.sum(axis=2), atol=1e-12)
        assert np.abs(dk.sum(axis=2)).max() < 1e-12


def pin_bwd_row_dot():
    """sum_k P_ik dP_ik equals sum_c dO_ic O_ic."""
    rng = _rng(33)
    T, d = 9, 4
    q, k, v, do = (rng.standard_normal((T, d)) for _ in range(4))
    P = BW.probabilities_head(q, k, True, 0.6)
    dP = BW.grad_probabilities(do, v)
    assert np.allclose((P * dP).sum(axis=1), BW.row_dot(do, P @ v), atol=1e-13)


BACKWARD_PINS = [pin_bwd_finite_differences, pin_bwd_constant_values, pin_bwd_sums, pin_bwd_row_dot]


ATTENTION_PINS = [
    pin_f1_three_token_causal, pin_f2_four_scores, pin_f4_lesson_fixture,
    pin_zero_queries_average_values, pin_constant_values, pin_identity_values_give_probabilities,
    pin_score_shift_moves_lse_only, pin_single_key, pin_two_keys_logistic, pin_causal_row0_is_v0,
    pin_causal_ignores_future, pin_key_permutation_invariance, pin_large_scores_stay_finite,
    pin_brute_force_tiny, pin_row_subset_matches_full, pin_gqa_brute_force_tiny, pin_gqa_one_group_per_head_is_mha,
]
ONLINE_PINS = [
    pin_online_f2_two_blocks, pin_online_f4_block_sizes, pin_online_f5_max_change,
    pin_online_f1_row2_two_tiles, pin_online_equals_three_step, pin_split_combine_f3,
    pin_split_combine_matches_oracle,
]
ALL_PINS = ATTENTION_PINS + ONLINE_PINS + BACKWARD_PINS
