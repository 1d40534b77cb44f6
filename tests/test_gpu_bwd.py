"""GPU parity of the backward pass (dQ, dK, dV) against the float64 oracle.

The bound each element must meet comes from the arithmetic:

* the kernels round P and dS to bf16 before the products that use them (dV =
  P^T dO; dQ = scale dS K; dK = scale dS^T Q), and every other step is exact
  or fp32; so a gradient element can be off by 2^-9 times the sum of the
  magnitudes of the terms it adds up (``mag``), allowed four times over;
* D = sum_c dO_c O_c is formed from the forward pass's bf16 O, whose elements
  differ from the exact O by up to 2^-8 sum_k P_k |v_k| (the bf16 weights of
  P V, in numerator and denominator) plus 2^-9 |O| (the bf16 output); an error
  e_D in D moves dS by P e_D, so dQ and dK may also be off by
  scale (P e_D) |K| and scale (P e_D)^T |Q| (``mag_d``, with e_D taken twice);
* the outputs are bf16: 2^-9 |ref|, allowed twice.
"""
import numpy as np
import pytest

import fa_inputs as fi
from parity import bf16_to_f64, bwd_bounds, default_scale, record, to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _library():
    import torch

    import exact_io_aware_07_gb300 as fa

    assert torch.cuda.is_available(), "the GPU tests need a CUDA device"
    fa.build()
    fa.load_library()


def _inputs(B, H, T, d, seed):
    x = fi.make_qkv(B, H, T, d, seed=seed)
    do_bits = fi.make_grad_out(B, H, T, d, seed=seed)
    return x, do_bits


def _run(x, do_bits, causal, scale):
    import torch

    import exact_io_aware_07_gb300 as fa

    q, k, v = (to_device(None, b) for b in (x.q_bits, x.k_bits, x.v_bits))
    do = to_device(None, do_bits)
    o, lse = fa.attention(q, k, v, causal=bool(causal), scale=scale)
    dq, dk, dv = (torch.full_like(q, float("nan")) for _ in range(3))
    ws = torch.full((fa.fa_bwd_workspace_bytes(*q.shape[:3]),), 0xFF, dtype=torch.uint8, device="cuda")
    fa.fa_bwd(q, k, v, o, lse, do, dq, dk, dv, causal, scale, ws)
    torch.cuda.synchronize()
    assert fa.fa_device_status() == 0
    return (q, k, v, o, lse, do), (bf16_to_f64(dq), bf16_to_f64(dk), bf16_to_f64(dv)), bf16_to_f64(o)


def _compare(x, do_bits, grads, o_gpu, causal, scale, label):
    q, k, v = x.f64("q"), x.f64("k"), x.f64("v")
    do = fi.bf16_bits_to_f64(do_bits).reshape(q.shape)
    B, H = q.shape[:2]
    worst = {n: [0.0, 0.0] for n in ("dQ", "dK", "dV")}  # max |err|, max |err| / bound
    for b in range(B):
        for h in range(H):
            refs, bounds = bwd_bounds(q[b, h], k[b, h], v[b, h], do[b, h], o_gpu[b, h], bool(causal), scale)
            for name, got, ref, bound in zip(("dQ", "dK", "dV"), grads, refs, bounds):
                err = np.abs(got[b, h] - ref)
                bad = ~(err <= bound)  # NaN counts as bad
                assert not bad.any(), (f"{label} {name} b{b} h{h}: {int(bad.sum())} of {bad.size} elements outside "
                                       f"the bound; max err {float(np.nanmax(err)):.3g}")
                worst[name][0] = max(worst[name][0], float(err.max()))
                worst[name][1] = max(worst[name][1], float((err / bound).max()))
    record(f"backward {label}", {f"max|{n}| err": w[0] for n, w in worst.items()}
           | {f"{n} err/bound": w[1] for n, w in worst.items()})


@pytest.mark.parametrize("B,H,T,d,causal", [
    (1, 2, 128, 64, 0), (1, 2, 300, 64, 1), (2, 3, 257, 128, 0), (1, 2, 513, 128, 1), (1, 4, 1, 64, 1),
    (1, 2, 1000, 64, 1), (1, 2, 2, 128, 0), (1, 4, 1024, 128, 1), (2, 2, 640, 64, 0),
])
def test_backward_matches_oracle(B, H, T, d, causal):
    x, do_bits = _inputs(B, H, T, d, seed=51)
    scale = default_scale(d)
    _, grads, o = _run(x, do_bits, causal, scale)
    _compare(x, do_bits, grads, o, causal, scale, f"T{T} d{d} causal{causal}")


@pytest.mark.parametrize("B,H,T,d,causal", [(20, 16, 256, 64, 1), (10, 16, 384, 128, 0), (8, 16, 512, 128, 1)])
def test_backward_many_units_per_cta(B, H, T, d, causal):
    # 640 / 480 / 512 units for 152 persistent CTAs: every CTA runs several units (of
    # different lengths when causal), so the per-step vector buffers, barrier phases and the
    # output warps' hand-over (and the next unit's dO at d = 128) carry over between units
    x, do_bits = _inputs(B, H, T, d, seed=53)
    scale = default_scale(d)
    _, grads, o = _run(x, do_bits, causal, scale)
    _compare(x, do_bits, grads, o, causal, scale, f"B{B} H{H} T{T} d{d} causal{causal}")


@pytest.mark.parametrize("causal", [1, 0])
def test_backward_llama8b_size(causal):
    # the size the backward is timed at: Llama-3.1-8B attention, 32 heads, T = 4096, d = 128
    # (1,024 units per kernel); the float64 oracle runs one head at a time
    B, H, T, d = 1, 32, 4096, 128
    x, do_bits = _inputs(B, H, T, d, seed=0)
    scale = default_scale(d)
    _, grads, o = _run(x, do_bits, causal, scale)
    _compare(x, do_bits, grads, o, causal, scale, f"llama8b B1 H32 T4096 d128 causal{causal}")


def test_backward_outputs_exactly_covered():
    """Every element of dQ, dK and dV is written, and nothing past them."""
    import torch

    import exact_io_aware_07_gb300 as fa

    B, H, T, d = 2, 3, 333, 128
    x, do_bits = _inputs(B, H, T, d, seed=54)
    q, k, v = (to_device(None, b) for b in (x.q_bits, x.k_bits, x.v_bits))
    do = to_device(None, do_bits)
    o, lse = fa.attention(q, k, v, causal=True, scale=default_scale(d))
    n = B * H * T * d
    bufs = [torch.full((n + 4096,), float("nan"), dtype=torch.bfloat16, device="cuda") for _ in range(3)]
    for b in bufs:
        b[n:] = 7.0
    dq, dk, dv = (b[:n].view(B, H, T, d) for b in bufs)
    ws = torch.empty(fa.fa_bwd_workspace_bytes(B, H, T), dtype=torch.uint8, device="cuda")
    fa.fa_bwd(q, k, v, o, lse, do, dq, dk, dv, True, default_scale(d), ws)
    torch.cuda.synchronize()
    assert fa.fa_device_status() == 0
    for b in bufs:
        assert not torch.isnan(b[:n]).any()
        assert torch.all(b[n:] == 7.0)


def test_backward_deterministic():
    import torch

    import exact_io_aware_07_gb300 as fa

    x, do_bits = _inputs(2, 4, 700, 64, seed=52)
    (q, k, v, o, lse, do), grads, _ = _run(x, do_bits, 1, 0.125)
    for _ in range(2):
        dq, dk, dv = fa.attention_bwd(q, k, v, o, lse, do, causal=True, scale=0.125)
        torch.cuda.synchronize()
        for a, g in zip((dq, dk, dv), grads):
            assert np.array_equal(bf16_to_f64(a), g)


def test_backward_rejects_bad_arguments():
    import ctypes

    import torch

    import exact_io_aware_07_gb300 as fa

    lib = fa.load_library()
    B, H, T, d = 1, 2, 256, 64
    t = [torch.zeros(B, H, T, d, dtype=torch.bfloat16, device="cuda") for _ in range(8)]
    lse = torch.zeros(B, H, T, device="cuda")
    need = fa.fa_bwd_workspace_bytes(B, H, T)
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    st = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)

    def call(dq_ptr, wsp, nb):
        return lib.fa_bwd(t[0].data_ptr(), t[1].data_ptr(), t[2].data_ptr(), t[3].data_ptr(), lse.data_ptr(),
                          t[4].data_ptr(), dq_ptr, t[6].data_ptr(), t[7].data_ptr(), B, H, T, d, 1,
                          ctypes.c_float(0.125), wsp, nb, st)

    assert call(t[5].data_ptr(), 0, need) == 13                    # no workspace
    assert call(t[5].data_ptr(), ws.data_ptr(), need - 256) == 13  # too small
    assert call(0, ws.data_ptr(), need) == 1                       # NULL output
    assert call(t[0].data_ptr(), ws.data_ptr(), need) == 11        # dQ over Q
    assert call(t[5].data_ptr(), ws.data_ptr(), need) == 0
    torch.cuda.synchronize()
    assert fa.fa_device_status() == 0
