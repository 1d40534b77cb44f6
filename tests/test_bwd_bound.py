"""The backward tolerance is tight enough to catch plausible kernel mistakes (CPU only).

The GPU test accepts a gradient element when it is within ``bwd_bounds`` of the
exact value.  Here the inputs are bf16 values, the forward output is the exact O
rounded to bf16, and each check applies a mistake a kernel could make (a wrong
scale, a dropped row term, a transposed product, an off-by-one mask) to the
exact gradients: every one must land outside the bound somewhere, while the
exact gradients themselves, and the same with P and dS rounded to bf16, stay
inside.
"""
import numpy as np

import fa_inputs as fi
import oracle.backward as BW
from parity import bwd_bounds


def _bf16(x):
    return fi.bf16_bits_to_f64(fi.f32_to_bf16_bits(np.asarray(x, dtype=np.float32)))


def _case(T, d, causal, seed):
    x = fi.make_qkv(1, 1, T, d, seed=seed)
    q, k, v = x.f64("q")[0, 0], x.f64("k")[0, 0], x.f64("v")[0, 0]
    do = fi.bf16_bits_to_f64(fi.make_grad_out(1, 1, T, d, seed=seed))[0, 0]
    scale = d ** -0.5
    P = BW.probabilities_head(q, k, causal, scale)
    o = _bf16(P @ v)
    return q, k, v, do, o, causal, scale


def _inside(got, ref, bound):
    return bool(np.all(np.abs(got - ref) <= bound))


def test_rounded_products_stay_inside():
    for T, d, causal in ((200, 64, True), (130, 128, False)):
        q, k, v, do, o, causal, scale = _case(T, d, causal, 61)
        (dq, dk, dv), (bq, bk, bv) = bwd_bounds(q, k, v, do, o, causal, scale)
        P = BW.probabilities_head(q, k, causal, scale)
        D = (do * o).sum(axis=1)  # from the rounded O, as the kernels do
        dS = _bf16(P * (do @ v.T - D[:, None]))
        assert _inside(_bf16(_bf16(P).T @ do), dv, bv)
        assert _inside(_bf16(scale * dS.T @ q), dk, bk)
        assert _inside(_bf16(scale * dS @ k), dq, bq)


def test_mistakes_land_outside():
    for T, d, causal in ((200, 64, True), (130, 128, False)):
        q, k, v, do, o, causal, scale = _case(T, d, causal, 62)
        (dq, dk, dv), (bq, bk, bv) = bwd_bounds(q, k, v, do, o, causal, scale)
        P = BW.probabilities_head(q, k, causal, scale)
        dP = do @ v.T
        D = (do * (P @ v)).sum(axis=1)
        dS = P * (dP - D[:, None])
        mistakes = {
            "dK without the scale": (dk / scale, dk, bk),
            "dQ without the scale": (dq / scale, dq, bq),
            "dS without the row term": (scale * (P * dP).T @ q, dk, bk),
            "dV from P, not P^T": (P @ do, dv, bv),
            "dQ from dS^T": (scale * dS.T @ k, dq, bq),
            "dV missing the last key's row": (np.vstack([dv[:-1], 0 * dv[-1:]]), dv, bv),
        }
        if causal:
            Pm = BW.probabilities_head(q, k, False, scale)  # mask dropped
            mistakes["mask dropped in dV"] = (Pm.T @ do, dv, bv)
        for name, (got, ref, bound) in mistakes.items():
            assert not _inside(got, ref, bound), name
