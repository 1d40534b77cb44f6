"""The O tolerance reading, pinned on the CPU.

The contract prescribes bf16 P for the P V product and a bf16 O, and asks for
max |O - O_ref| <= 1e-2.  An idealised computation of that method (every
step in float64 except the two prescribed roundings: each softmax weight to
bf16, with O divided by the sum of the same rounded weights, and O to bf16)
already exceeds 1e-2 on a few elements of the stress input (Q, K ~ N(0, 3^2)),
so no kernel of this method can meet 1e-2 flat.  The parity tests therefore
accept an element beyond 1e-2 only within the derived rounding bound of
``parity.rounding_bound``; this test shows the idealised method needs exactly
that allowance and stays inside it.
"""
import numpy as np

import fa_inputs as fi
import oracle.attention as A
from parity import O_MAX_ABS, compare, rounding_bound


def _bf16(x):
    return fi.bf16_bits_to_f64(fi.f32_to_bf16_bits(np.asarray(x, dtype=np.float32)))


def _idealised_method(q, k, v, causal, scale):
    """Float64 attention with only the method's roundings: weights and output to bf16."""
    S = A.scores(q, k, scale)
    if causal:
        S = A.causal_mask(S, np.arange(S.shape[0]))
    p = np.exp(S - S.max(axis=1)[:, None])
    pt = _bf16(p)
    return _bf16((pt @ v) / pt.sum(axis=1)[:, None])


def test_flat_tolerance_is_infeasible_and_the_bound_holds():
    qkv = fi.make_qkv(1, 16, 1024, 64, seed=0, sigma_qk=3.0)  # the stress workload's first batch entry
    heads = [5, 12]
    q, k, v = (qkv.f64(n)[:, heads] for n in "qkv")
    scale = 0.125
    O_ref, lse_ref = A.attention_fwd(q, k, v, False, scale)
    O = np.stack([np.stack([_idealised_method(q[0, h], k[0, h], v[0, h], False, scale) for h in range(2)])])
    err = np.abs(O - O_ref)
    assert (err > O_MAX_ABS).sum() >= 1  # the method itself goes past 1e-2 here
    rec = compare(O, lse_ref, O_ref, lse_ref, label="idealised bf16-P method", bound=rounding_bound(q, k, v, False, scale),
                  record=False)
    assert rec["o_beyond_1e-2"] >= 1 and rec["o_beyond_worst_err_over_bound"] <= 1.0


def test_bound_rejects_a_real_mistake():
    """A kernel that drops one key from a row is caught although the row's values are large."""
    qkv = fi.make_qkv(1, 1, 200, 64, seed=4, sigma_qk=3.0)
    q, k, v = (qkv.f64(n) for n in "qkv")
    O_ref, lse_ref = A.attention_fwd(q, k, v, True, 0.125)
    S = A.causal_mask(A.scores(q[0, 0], k[0, 0], 0.125), np.arange(200))
    S[:, 0] = -np.inf  # the planted mistake: key 0 never seen (row 0 keeps it, or it would be empty)
    S[0, 0] = 0.0
    W, _, _ = A.softmax_rows(S)
    O = _bf16(W @ v[0, 0])[None, None]
    try:
        compare(O, lse_ref, O_ref, lse_ref, label="dropped key", bound=rounding_bound(q, k, v, True, 0.125),
                record=False)
    except AssertionError:
        return
    raise AssertionError("a dropped key passed the O tolerance")
