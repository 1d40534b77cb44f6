"""GPU parity: the sm_103a kernel through the C ABI against the float64 oracle.

Inputs are the seeded bf16 tensors of ``fa_inputs``; the oracle runs on the
same values.  Tolerances are in ``parity.py``.
"""
import math

import numpy as np
import pytest

import fa_inputs as fi
import oracle
from parity import bf16_to_f64, compare, default_scale, rounding_bound, run_gpu, sampled_rows, to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _library():
    import torch

    import exact_io_aware_07_gb300 as fa

    assert torch.cuda.is_available(), "the GPU tests need a CUDA device"
    fa.build()
    fa.load_library()


def _check(B, H, T, d, causal, seed=1, sigma_qk=1.0, scale=None, rows=None, label=None):
    qkv = fi.make_qkv(B, H, T, d, seed=seed, sigma_qk=sigma_qk)
    scale = default_scale(d) if scale is None else scale
    o, lse = run_gpu(qkv, causal, scale)
    if rows is not None:
        o, lse = o[:, :, rows], lse[:, :, rows]
    q64, k64, v64 = qkv.f64("q"), qkv.f64("k"), qkv.f64("v")
    O_ref, lse_ref = oracle.attention_fwd(q64, k64, v64, causal, scale, rows=rows)
    label = label or f"B{B} H{H} T{T} d{d} causal{causal} seed{seed}"
    return compare(o, lse, O_ref, lse_ref, label=label, bound=rounding_bound(q64, k64, v64, causal, scale, rows))


# ragged and tiny sequence lengths: one tile, several tiles, a ragged tail, a lone
# second query tile, a 256-row unit whose second tile lies past T
SMALL_T = [1, 2, 3, 17, 64, 100, 127, 128, 129, 200, 255, 256, 257, 300, 384, 511, 640, 1000]


@pytest.mark.parametrize("causal", [0, 1])
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("T", SMALL_T)
def test_small_and_ragged(T, d, causal):
    _check(1, 2, T, d, causal)


def test_three_token_example_padded():
    # "Flash Attention, tiled", section "A three-token example", with d padded to 64:
    # Q = K = 0 and V rows [10,0], [0,20], [30,30] -> O rows [10,0], [5,10], [13.333,16.667]
    import torch

    import exact_io_aware_07_gb300 as fa

    q = torch.zeros(1, 1, 3, 64, dtype=torch.bfloat16, device="cuda")
    k = torch.zeros_like(q)
    v = torch.zeros_like(q)
    v[0, 0, :, :2] = torch.tensor([[10.0, 0.0], [0.0, 20.0], [30.0, 30.0]])
    o, lse = fa.attention(q, k, v, causal=True)
    torch.cuda.synchronize()
    got = o[0, 0, :, :2].float().cpu().numpy()
    want = np.array([[10.0, 0.0], [5.0, 10.0], [40 / 3, 50 / 3]])
    # bf16 keeps 8 significant bits: 40/3 and 50/3 round to 13.3125 and 16.625
    assert np.all(np.abs(got - want) <= np.maximum(1e-2, 2.0 ** (np.floor(np.log2(np.abs(want) + 1e-30)) - 7)))
    assert np.all(o[0, 0, :, 2:].float().cpu().numpy() == 0.0)
    assert np.allclose(lse[0, 0].cpu().numpy(), np.log([1.0, 2.0, 3.0]), atol=1e-6)


@pytest.mark.parametrize("name", [
    "tiny_causal_b1h4t256d64",
    "gpt2s_causal_b8h12t1024d64",
    "gpt2m_b16h16t1024d64",
    "gpt2m_stress_b16h16t1024d64",
    "llama8b_causal_b1h32t4096d128",
    "llama8b_b1h32t4096d128",
])
@pytest.mark.parametrize("seed", [0, 1, 2])
def test_workload_full(name, seed):
    w = fi.WORKLOADS[name]
    _check(w["B"], w["H"], w["T"], w["d"], w["causal"], seed=seed, sigma_qk=w["sigma_qk"],
           label=f"{name} seed{seed}")


def test_long_context_sampled_rows():
    w = fi.WORKLOADS["long_causal_b1h32t32768d128"]
    rows = sampled_rows(w["T"], seed=7)
    _check(w["B"], w["H"], w["T"], w["d"], w["causal"], seed=0, rows=rows,
           label=f"long_causal_b1h32t32768d128 seed0 ({rows.size} sampled rows per head)")


def test_many_units_per_cta():
    # 64 * 16 heads x 4 units each: every persistent CTA runs many work units
    _check(64, 16, 1000, 64, 1, seed=3)
    _check(16, 16, 512, 128, 0, seed=4)


def test_other_scales():
    _check(1, 3, 777, 64, 1, seed=5, scale=0.5)
    _check(1, 3, 777, 128, 0, seed=6, scale=0.01)


def test_outputs_exactly_covered():
    """Every element of O and LSE is written, and nothing past them."""
    import torch

    import exact_io_aware_07_gb300 as fa

    B, H, T, d = 2, 3, 333, 128
    qkv = fi.make_qkv(B, H, T, d, seed=9)
    q, k, v = (to_device(None, b) for b in (qkv.q_bits, qkv.k_bits, qkv.v_bits))
    n = B * H * T * d
    o_buf = torch.full((n + 4096,), float("nan"), dtype=torch.bfloat16, device="cuda")
    o_buf[n:] = 7.0
    l_buf = torch.full((B * H * T + 1024,), float("nan"), dtype=torch.float32, device="cuda")
    l_buf[B * H * T:] = -3.0
    o = o_buf[:n].view(B, H, T, d)
    lse = l_buf[:B * H * T].view(B, H, T)
    fa.fa_fwd(q, k, v, o, lse, True, default_scale(d))
    torch.cuda.synchronize()
    assert not torch.isnan(o).any() and not torch.isnan(lse).any()
    assert torch.all(o_buf[n:] == 7.0) and torch.all(l_buf[B * H * T:] == -3.0)


def test_deterministic_and_stream():
    import torch

    import exact_io_aware_07_gb300 as fa

    qkv = fi.make_qkv(2, 4, 1500, 128, seed=11)
    q, k, v = (to_device(None, b) for b in (qkv.q_bits, qkv.k_bits, qkv.v_bits))
    o1, l1 = fa.attention(q, k, v, causal=True)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        o2, l2 = fa.attention(q, k, v, causal=True)
    torch.cuda.synchronize()
    assert torch.equal(o1.view(torch.int16), o2.view(torch.int16)) and torch.equal(l1, l2)


def test_rejects_bad_pointers():
    import ctypes

    import torch

    import exact_io_aware_07_gb300 as fa

    lib = fa.load_library()
    B, H, T, d = 1, 2, 256, 64
    q = torch.randn(B, H, T, d, device="cuda").to(torch.bfloat16)
    o = torch.empty_like(q)
    lse = torch.empty(B, H, T, device="cuda")
    host = torch.empty_like(q, device="cpu").pin_memory()
    st = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    call = lambda qq, oo, ll, TT=T: lib.fa_fwd(qq, q.data_ptr(), q.data_ptr(), oo, ll, B, H, TT, d, 1,
                                                ctypes.c_float(0.125), st)
    assert call(host.data_ptr(), o.data_ptr(), lse.data_ptr()) == 10           # host memory
    small = torch.empty(64, dtype=torch.bfloat16, device="cuda")
    assert call(q.data_ptr(), small.data_ptr(), lse.data_ptr(), TT=1 << 20) == 10  # allocation too small
    assert call(q.data_ptr(), q.data_ptr(), lse.data_ptr()) == 11              # O aliases Q
    assert call(q.data_ptr(), o.data_ptr(), o.data_ptr()) == 11                # LSE aliases O
    torch.cuda.synchronize()
    assert fa.fa_device_status() == 0


def test_ex2_rate_probe():
    import exact_io_aware_07_gb300 as fa

    rate = fa.fa_ex2_rate()
    # one GB300: 152 SMs at 1-2.1 GHz issuing at most one ex2 per lane per cycle
    assert 1e12 < rate < 152 * 128 * 2.2e9
    assert fa.fa_device_status() == 0


@pytest.mark.parametrize("B,H,T,reps", [(1, 6, 16384, 70), (2, 5, 19999, 3)])
def test_claimed_order_long_causal(B, H, T, reps):
    """Causal d = 128 launches whose K and V exceed 96 MB list their units by groups of heads and
    claim them at run time (B1 H6 T16384: 101 MB, two heads per group; B2 H5 T19999: 102 MB, two
    heads per group, a ragged last band).  The result must be the statically ordered launch's bit
    for bit (a one-range split launch keeps the static order), over more launches than there are
    counter pairs in the first case (so every pair is reused after its reset), and must match the
    oracle on sampled rows."""
    import torch

    import exact_io_aware_07_gb300 as fa

    d = 128
    qkv = fi.make_qkv(B, H, T, d, seed=12)
    q, k, v = (to_device(None, b) for b in (qkv.q_bits, qkv.k_bits, qkv.v_bits))
    scale = default_scale(d)
    ws = torch.empty(fa.fa_fwd_splitkv_workspace_bytes(B, H, T, d, 1), dtype=torch.uint8, device="cuda")
    o_st = torch.empty_like(q)
    l_st = torch.empty(B, H, T, device="cuda")
    fa.fa_fwd_splitkv(q, k, v, o_st, l_st, True, scale, 1, ws)
    o = torch.full_like(q, float("nan"))
    lse = torch.full((B, H, T), float("nan"), device="cuda")
    for it in range(reps):
        fa.fa_fwd(q, k, v, o, lse, True, scale)
        if it in (0, reps - 1):
            torch.cuda.synchronize()
            assert fa.fa_device_status() == 0
            assert torch.equal(o.view(torch.int16), o_st.view(torch.int16)) and torch.equal(lse, l_st), f"call {it}"
    rows = sampled_rows(T, seed=8, first=128, last=128, random=256)
    o_s = bf16_to_f64(o[:, :, rows])
    l_s = lse[:, :, rows].cpu().numpy().astype(np.float64)
    q64, k64, v64 = qkv.f64("q"), qkv.f64("k"), qkv.f64("v")
    O_ref, lse_ref = oracle.attention_fwd(q64, k64, v64, True, scale, rows=rows)
    compare(o_s, l_s, O_ref, lse_ref, label=f"claimed order B{B} H{H} T{T} d{d} causal ({rows.size} rows per head)",
            bound=rounding_bound(q64, k64, v64, True, scale, rows))

