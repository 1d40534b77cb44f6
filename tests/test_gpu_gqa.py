"""GPU parity of attention with grouped K/V heads (query head h reads K/V head h // (H / Hkv)).

Each case runs ``fa_fwd_gqa`` through the C ABI and compares it with the oracle
element by element.  The kernel does the same arithmetic for a query head
whether its K/V head is shared or not, so the grouped call must also be
bit-identical to ``fa_fwd`` on K and V with every head repeated per group.
"""
import numpy as np
import pytest

import fa_inputs as fi
import oracle
from parity import bf16_to_f64, compare, default_scale, rounding_bound, to_device

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

    q, k, v = (to_device(None, b) for b in (x.q_bits, x.k_bits, x.v_bits))
    o = torch.full_like(q, float("nan"))
    lse = torch.full(q.shape[:3], float("nan"), dtype=torch.float32, device="cuda")
    fa.fa_fwd_gqa(q, k, v, o, lse, causal, scale)
    torch.cuda.synchronize()
    assert fa.fa_device_status() == 0
    return q, k, v, o, lse


@pytest.mark.parametrize("B,H,Hkv,T,d,causal", [
    (1, 8, 2, 300, 64, 0), (1, 8, 2, 300, 64, 1), (2, 4, 1, 129, 128, 1), (2, 6, 3, 777, 64, 0),
    (1, 8, 8, 200, 128, 1), (1, 4, 2, 1, 64, 1), (1, 32, 8, 1024, 128, 1),
])
def test_gqa_matches_oracle(B, H, Hkv, T, d, causal):
    x = fi.make_grouped_qkv(B, H, Hkv, T, d, seed=41)
    scale = default_scale(d)
    _, _, _, o, lse = _run(x, causal, scale)
    q64, k64, v64 = x.f64("q"), x.f64("k"), x.f64("v")
    O_ref, lse_ref = oracle.attention_fwd_gqa(q64, k64, v64, causal, scale)
    compare(bf16_to_f64(o), lse.cpu().numpy().astype(np.float64), O_ref, lse_ref,
            label=f"gqa B{B} H{H} Hkv{Hkv} T{T} d{d} causal{causal}",
            bound=rounding_bound(q64, k64, v64, causal, scale))


@pytest.mark.parametrize("d,causal", [(64, 1), (128, 0)])
def test_gqa_equals_repeated_heads(d, causal):
    import torch

    import exact_io_aware_07_gb300 as fa

    x = fi.make_grouped_qkv(2, 8, 2, 513, d, seed=42)
    scale = default_scale(d)
    q, k, v, o, lse = _run(x, causal, scale)
    o2, lse2 = fa.attention(q, k.repeat_interleave(4, dim=1).contiguous(), v.repeat_interleave(4, dim=1).contiguous(),
                            causal=bool(causal), scale=scale)
    torch.cuda.synchronize()
    assert torch.equal(o.view(torch.int16), o2.view(torch.int16))
    assert torch.equal(lse, lse2)


def test_gqa_rejects_bad_head_counts():
    import ctypes

    import torch

    import exact_io_aware_07_gb300 as fa

    lib = fa.load_library()
    q = torch.zeros(1, 8, 128, 64, dtype=torch.bfloat16, device="cuda")
    kv = torch.zeros(1, 8, 128, 64, dtype=torch.bfloat16, device="cuda")
    o = torch.empty_like(q)
    lse = torch.empty(1, 8, 128, device="cuda")
    st = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    call = lambda H, Hkv: lib.fa_fwd_gqa(q.data_ptr(), kv.data_ptr(), kv.data_ptr(), o.data_ptr(), lse.data_ptr(),
                                         1, H, Hkv, 128, 64, 0, ctypes.c_float(0.125), st)
    assert call(8, 3) == 3    # FA_ERR_BAD_SHAPE: 3 does not divide 8
    assert call(8, 0) == 3
    assert call(4, 8) == 3    # more K/V heads than query heads
    assert call(8, 4) == 0
    torch.cuda.synchronize()
    assert fa.fa_device_status() == 0
