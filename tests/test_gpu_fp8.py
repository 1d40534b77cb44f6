"""GPU parity of the e4m3 forward pass (fa_fwd_fp8) against the float64 oracle.

The oracle is plain attention on the real values the e4m3 inputs stand for
(byte value times its tensor's scale).  The only rounding the kernel adds on
top of bf16-free arithmetic is P to e4m3 before the P V product, whose sum of
rounded weights also divides O; so the bound per output element is derived
from the format:

* a weight p >= 2^-6 (normal) is rounded with relative error <= 2^-4; the
  normalisation then moves the normalised weight w by at most 2 * 2^-4 * w;
* a weight below 2^-6 (subnormal) is off by <= 2^-10 absolute; in the kernel
  every weight is 2^(s - m) with the row maximum s_max >= m, so the weights
  sum to at least l = sum_k e^(S_k - S_max), and such a weight can only occur
  where e^(S_k - S_max) < 2^-6;
* O is rounded to bf16: 2^-9 |O|.

  |O - O_ref| <= 2 * (2 * 2^-4 * sum_k w_k |v_k| + 2 * 2^-10 / l * sum_{k small} |v_k|) + 2 * 2^-9 |O_ref|

with twice the derived amount allowed.  The mean error must also stay below
2^-6 of the mean of sum_k w_k |v_k|, so a wrong-but-bounded result is caught.
The LSE uses the fp32 weights and keeps the bf16 path's 1e-3.
"""
import numpy as np
import pytest

import fa_inputs as fi
import oracle.attention as A
from parity import bf16_to_f64, record

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _library():
    import torch

    import exact_io_aware_07_gb300 as fa

    assert torch.cuda.is_available(), "the GPU tests need a CUDA device"
    fa.build()
    fa.load_library()


def _run(x, causal, scale):
    import torch

    import exact_io_aware_07_gb300 as fa

    q, k, v = (torch.from_numpy(np.ascontiguousarray(getattr(x, n + "8"))).cuda() for n in "qkv")
    o = torch.full((x.B, x.H, x.T, x.d), float("nan"), dtype=torch.bfloat16, device="cuda")
    lse = torch.full((x.B, x.H, x.T), float("nan"), dtype=torch.float32, device="cuda")
    ws = torch.full((fa.fa_fwd_fp8_workspace_bytes(x.B, x.H, x.T, x.d),), 0x7F, dtype=torch.uint8, device="cuda")
    fa.fa_fwd_fp8(q, k, v, o, lse, causal, scale, x.descale, ws)
    torch.cuda.synchronize()
    assert fa.fa_device_status() == 0
    return bf16_to_f64(o), lse.cpu().numpy().astype(np.float64)


def _check(x, o, lse, causal, scale, label):
    q, k, v = x.f64("q"), x.f64("k"), x.f64("v")
    worst_mean = 0.0
    worst_ratio = worst_abs = worst_lse = 0.0
    for b in range(x.B):
        for h in range(x.H):
            S = A.scores(q[b, h], k[b, h], scale)
            if causal:
                S = A.causal_mask(S, np.arange(x.T))
            W, m, l = A.softmax_rows(S)
            O_ref = W @ v[b, h]
            lse_ref = m + np.log(l)
            u = np.exp(S - m[:, None])  # e^(S_k - S_max), 0 where masked
            small = (u < 2.0 ** -6) & (u > 0)
            wv = W @ np.abs(v[b, h])
            bound = 2 * (2 * 2.0 ** -4 * wv + 2 * 2.0 ** -10 / l[:, None] * (small @ np.abs(v[b, h]))) \
                + 2 * 2.0 ** -9 * np.abs(O_ref) + 1e-6
            err = np.abs(o[b, h] - O_ref)
            bad = ~(err <= bound)
            assert not bad.any(), f"{label} b{b} h{h}: {int(bad.sum())} elements outside the bound, max {np.nanmax(err):.3g}"
            lerr = float(np.abs(lse[b, h] - lse_ref).max())
            assert lerr <= 1e-3, f"{label} b{b} h{h}: LSE"
            worst_mean = max(worst_mean, float(err.mean() / wv.mean()))
            worst_ratio = max(worst_ratio, float((err / bound).max()))
            worst_abs = max(worst_abs, float(err.max()))
            worst_lse = max(worst_lse, lerr)
    assert worst_mean <= 2.0 ** -6, f"{label}: mean error {worst_mean:.3g} of the mean weighted |v|"
    record(label, {"max|dO|": worst_abs, "max err/bound": worst_ratio, "mean err / mean sum w|v|": worst_mean,
                   "max|dLSE|": worst_lse})


@pytest.mark.parametrize("B,H,T,causal", [(1, 2, 128, 0), (1, 2, 300, 1), (2, 2, 1000, 0), (1, 3, 17, 1),
                                          (1, 2, 1, 1), (1, 4, 1024, 1), (1, 2, 2053, 0)])
def test_fp8_matches_oracle(B, H, T, causal):
    x = fi.make_qkv_e4m3(B, H, T, 128, seed=71)
    scale = 128 ** -0.5
    o, lse = _run(x, causal, scale)
    _check(x, o, lse, causal, scale, f"fp8 T{T} causal{causal}")


@pytest.mark.parametrize("causal", [1, 0])
def test_fp8_llama8b_size(causal):
    # the size the e4m3 forward is timed at: 32 heads, T = 4096, d = 128
    x = fi.make_qkv_e4m3(1, 32, 4096, 128, seed=0)
    scale = 128 ** -0.5
    o, lse = _run(x, causal, scale)
    _check(x, o, lse, causal, scale, f"fp8 llama8b B1 H32 T4096 causal{causal}")


def test_fp8_scales():
    x = fi.make_qkv_e4m3(1, 2, 640, 128, seed=72, descale=(0.5, 0.03125, 4.0))
    o, lse = _run(x, 1, 0.1)
    _check(x, o, lse, 1, 0.1, "fp8 scaled")


def test_fp8_rejects_bad_arguments():
    import ctypes

    import torch

    import exact_io_aware_07_gb300 as fa

    lib = fa.load_library()
    B, H, T = 1, 2, 256
    q = torch.zeros(B, H, T, 128, dtype=torch.uint8, device="cuda")
    o = torch.empty(B, H, T, 128, dtype=torch.bfloat16, device="cuda")
    lse = torch.empty(B, H, T, device="cuda")
    need = fa.fa_fwd_fp8_workspace_bytes(B, H, T, 128)
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    st = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    f = ctypes.c_float

    def call(d=128, qs=1.0, wsp=None, nb=need):
        return lib.fa_fwd_fp8(q.data_ptr(), q.data_ptr(), q.data_ptr(), o.data_ptr(), lse.data_ptr(), B, H, T, d,
                              0, f(0.1), f(qs), f(1.0), f(1.0), ws.data_ptr() if wsp is None else wsp, nb, st)

    assert fa.fa_fwd_fp8_workspace_bytes(B, H, T, 64) == 0
    assert call(d=64) == 4           # FA_ERR_UNSUPPORTED_HEAD_DIM
    assert call(qs=0.0) == 5         # FA_ERR_BAD_SCALE
    assert call(qs=float("inf")) == 5
    assert call(wsp=0) == 13         # FA_ERR_WORKSPACE
    assert call(nb=need - 256) == 13
    assert call(wsp=q.data_ptr()) == 11  # the workspace over an input
    assert call() == 0
    torch.cuda.synchronize()
    assert fa.fa_device_status() == 0


def test_fp8_last_round_in_single_tiles():
    """Non-causal e4m3 launches whose last round of units would leave SMs idle work it in single
    query tiles (B1 H20 T2048: 160 units on 152 SMs, the last 8 as 16 one-tile items; B1 H4: its 32
    units as 64 items; B1 H16: 128 whole units).  Each row's arithmetic does not depend on the
    split, so H20 must equal H16 and H4 on the same heads bit for bit; the oracle checks H4."""
    import torch

    import exact_io_aware_07_gb300 as fa

    B, H, T, d = 1, 20, 2048, 128
    x = fi.make_qkv_e4m3(B, H, T, d, seed=73)
    scale = d ** -0.5

    def run(heads):
        q, k, v = (torch.from_numpy(np.ascontiguousarray(getattr(x, n + "8")[:, heads])).cuda() for n in "qkv")
        h = q.shape[1]
        o = torch.full((B, h, T, d), float("nan"), dtype=torch.bfloat16, device="cuda")
        lse = torch.full((B, h, T), float("nan"), dtype=torch.float32, device="cuda")
        ws = torch.empty(fa.fa_fwd_fp8_workspace_bytes(B, h, T, d), dtype=torch.uint8, device="cuda")
        fa.fa_fwd_fp8(q, k, v, o, lse, False, scale, x.descale, ws)
        return o, lse

    o, lse = run(slice(0, 20))
    o16, l16 = run(slice(0, 16))
    o4, l4 = run(slice(16, 20))
    torch.cuda.synchronize()
    assert fa.fa_device_status() == 0
    assert torch.equal(o.view(torch.int16), torch.cat([o16, o4], 1).view(torch.int16))
    assert torch.equal(lse, torch.cat([l16, l4], 1))
    sub = fi.QKV8(B, 4, T, d, x.q8[:, 16:20], x.k8[:, 16:20], x.v8[:, 16:20], x.descale)
    _check(sub, bf16_to_f64(o4), l4.cpu().numpy().astype(np.float64), False, scale, "fp8 one-tile last round H4 T2048")
