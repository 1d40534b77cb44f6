"""Shared helpers for the GPU parity tests: seeded inputs -> CUDA path and oracle -> comparison.

Tolerances (from the attention forward contract): on O (bf16), every element
within max(1e-2, one bf16 ulp of the oracle value) and a mean absolute error
<= 1e-3; on LSE (fp32), every element within 1e-3.  The ulp term covers
|O| >= 4, where correct bf16 rounding alone can differ from the float64 value
by up to 2^-6: there the fp32 accumulation may round to the neighbouring bf16
value, and such elements are counted separately.
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


def compare(o_gpu, lse_gpu, o_ref, lse_ref, label=""):
    """Asserts the tolerances; returns a dict of the observed errors."""
    assert np.all(np.isfinite(o_gpu)), f"{label}: non-finite O"
    assert np.all(np.isfinite(lse_gpu)), f"{label}: non-finite LSE"
    err = np.abs(o_gpu - o_ref)
    tol = np.maximum(O_MAX_ABS, bf16_ulp(o_ref))
    bad = err > tol
    assert not bad.any(), (f"{label}: {int(bad.sum())} O elements out of tolerance, worst err "
                           f"{float(err.max()):.3e} at |O|={float(np.abs(o_ref).flat[int(err.argmax())]):.3f}")
    mean_err = float(err.mean())
    assert mean_err <= O_MEAN_ABS, f"{label}: mean |O err| {mean_err:.3e}"
    lerr = np.abs(lse_gpu - lse_ref)
    assert float(lerr.max()) <= LSE_MAX_ABS, f"{label}: max |LSE err| {float(lerr.max()):.3e}"
    return {
        "o_max_abs": float(err.max()),
        "o_mean_abs": mean_err,
        "o_ulp_only": int(((err > O_MAX_ABS) & ~bad).sum()),
        "lse_max_abs": float(lerr.max()),
    }


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
