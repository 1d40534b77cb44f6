"""GPU parity of the split-KV forward (per-split partials merged by log-sum-exp) against the oracle.

The workspace is filled with NaN before every call, so a merge that read a
partial no unit wrote would poison O.
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


def _run_split(qkv, causal, scale, num_splits):
    import torch

    import exact_io_aware_07_gb300 as fa

    q, k, v = (to_device(None, b) for b in (qkv.q_bits, qkv.k_bits, qkv.v_bits))
    o = torch.full_like(q, float("nan"))
    lse = torch.full(q.shape[:3], float("nan"), dtype=torch.float32, device="cuda")
    B, H, T, d = q.shape
    ws = torch.full((fa.fa_fwd_splitkv_workspace_bytes(B, H, T, d, num_splits),), 0xFF, dtype=torch.uint8,
                    device="cuda")
    fa.fa_fwd_splitkv(q, k, v, o, lse, causal, scale, num_splits, ws)
    torch.cuda.synchronize()
    assert fa.fa_device_status() == 0
    return bf16_to_f64(o), lse.cpu().numpy().astype(np.float64)


@pytest.mark.parametrize("causal", [0, 1])
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("T,num_splits", [(1, 1), (1, 4), (129, 2), (300, 3), (700, 2), (1000, 8), (2048, 3),
                                          (2048, 64), (640, 5)])
def test_splitkv_matches_oracle(T, num_splits, d, causal):
    qkv = fi.make_qkv(1, 3, T, d, seed=21)
    scale = default_scale(d)
    o, lse = _run_split(qkv, causal, scale, num_splits)
    q64, k64, v64 = qkv.f64("q"), qkv.f64("k"), qkv.f64("v")
    O_ref, lse_ref = oracle.attention_fwd(q64, k64, v64, causal, scale)
    compare(o, lse, O_ref, lse_ref, label=f"split{num_splits} T{T} d{d} causal{causal}",
            bound=rounding_bound(q64, k64, v64, causal, scale))


@pytest.mark.parametrize("name,num_splits", [("tiny_causal_b1h4t256d64", 2), ("gpt2s_causal_b8h12t1024d64", 4),
                                             ("gpt2m_stress_b16h16t1024d64", 3)])
def test_splitkv_workloads(name, num_splits):
    w = fi.WORKLOADS[name]
    qkv = fi.make_qkv(w["B"], w["H"], w["T"], w["d"], seed=0, sigma_qk=w["sigma_qk"])
    scale = default_scale(w["d"])
    o, lse = _run_split(qkv, w["causal"], scale, num_splits)
    q64, k64, v64 = qkv.f64("q"), qkv.f64("k"), qkv.f64("v")
    O_ref, lse_ref = oracle.attention_fwd(q64, k64, v64, w["causal"], scale)
    compare(o, lse, O_ref, lse_ref, label=f"{name} split{num_splits}",
            bound=rounding_bound(q64, k64, v64, w["causal"], scale))


@pytest.mark.parametrize("B,H,T,d,causal", [(1, 4, 8192, 128, 1), (1, 4, 256, 64, 1), (1, 2, 3000, 64, 0)])
def test_splitkv_automatic_count(B, H, T, d, causal):
    """num_splits = 0: the library picks the count (few work units, long rows: more than one split)."""
    import torch

    import exact_io_aware_07_gb300 as fa

    qkv = fi.make_qkv(B, H, T, d, seed=23)
    scale = default_scale(d)
    o, lse = _run_split(qkv, causal, scale, 0)
    q64, k64, v64 = qkv.f64("q"), qkv.f64("k"), qkv.f64("v")
    O_ref, lse_ref = oracle.attention_fwd(q64, k64, v64, causal, scale)
    compare(o, lse, O_ref, lse_ref, label=f"split-auto B{B} H{H} T{T} d{d} causal{causal}",
            bound=rounding_bound(q64, k64, v64, causal, scale))
    nk = (T + 127) // 128
    assert fa.fa_fwd_splitkv_workspace_bytes(B, H, T, d, 0) >= fa.fa_fwd_splitkv_workspace_bytes(B, H, T, d, 1)
    if (B, H, T) == (1, 4, 8192):  # 128 units of work for 152 SMs, the longest 64 key tiles long
        assert fa.fa_fwd_splitkv_workspace_bytes(B, H, T, d, 0) > fa.fa_fwd_splitkv_workspace_bytes(B, H, T, d, 1)
    assert nk >= 1 and torch.cuda.is_available()


def test_splitkv_reused_workspace_and_repeatable():
    """The counters are cleared by every call: a workspace reused across calls (and shapes) gives the same bits."""
    import torch

    import exact_io_aware_07_gb300 as fa

    ws = torch.full((fa.fa_fwd_splitkv_workspace_bytes(2, 3, 1000, 128, 4),), 0x7F, dtype=torch.uint8, device="cuda")
    outs = []
    for T, seed in ((1000, 24), (700, 25), (1000, 24)):
        qkv = fi.make_qkv(2, 3, T, 128, seed=seed)
        q, k, v = (to_device(None, b) for b in (qkv.q_bits, qkv.k_bits, qkv.v_bits))
        o = torch.full_like(q, float("nan"))
        lse = torch.full(q.shape[:3], float("nan"), dtype=torch.float32, device="cuda")
        fa.fa_fwd_splitkv(q, k, v, o, lse, True, default_scale(128), 4, ws)
        outs.append((o, lse))
    torch.cuda.synchronize()
    assert fa.fa_device_status() == 0
    assert torch.equal(outs[0][0].view(torch.int16), outs[2][0].view(torch.int16)) and torch.equal(outs[0][1], outs[2][1])


def test_splitkv_rejects_bad_workspace():
    import ctypes

    import torch

    import exact_io_aware_07_gb300 as fa

    lib = fa.load_library()
    B, H, T, d = 1, 2, 512, 64
    q = torch.randn(B, H, T, d, device="cuda").to(torch.bfloat16)
    o = torch.empty_like(q)
    lse = torch.empty(B, H, T, device="cuda")
    need = fa.fa_fwd_splitkv_workspace_bytes(B, H, T, d, 2)
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    st = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    call = lambda wsp, nb: lib.fa_fwd_splitkv(q.data_ptr(), q.data_ptr(), q.data_ptr(), o.data_ptr(),
                                              lse.data_ptr(), B, H, T, d, 1, ctypes.c_float(0.125), 2, wsp, nb, st)
    assert call(0, need) == 13                      # no workspace
    assert call(ws.data_ptr(), need - 256) == 13    # too small
    assert call(o.data_ptr(), need) in (10, 11)     # over O (also too small an allocation for it)
    host = torch.empty(need, dtype=torch.uint8).pin_memory()
    assert call(host.data_ptr(), need) == 10        # host memory
    assert call(ws.data_ptr(), need) == 0
    torch.cuda.synchronize()
    assert fa.fa_device_status() == 0


@pytest.mark.parametrize("T,num_splits,causal", [(1000, 1, 1), (100, 4, 0), (200, 1, 0)])
def test_one_key_range_is_the_plain_kernel(T, num_splits, causal):
    """A count that comes to one key range (num_splits 1, or T within one tile) runs fa_fwd itself:
    the same bits, and the workspace is left as it was."""
    import torch

    import exact_io_aware_07_gb300 as fa

    qkv = fi.make_qkv(2, 3, T, 128, seed=26)
    q, k, v = (to_device(None, b) for b in (qkv.q_bits, qkv.k_bits, qkv.v_bits))
    scale = default_scale(128)
    ws = torch.full((fa.fa_fwd_splitkv_workspace_bytes(2, 3, T, 128, num_splits),), 0x5A, dtype=torch.uint8,
                    device="cuda")
    o = torch.empty_like(q)
    lse = torch.empty(q.shape[:3], dtype=torch.float32, device="cuda")
    fa.fa_fwd_splitkv(q, k, v, o, lse, causal, scale, num_splits, ws)
    o_ref = torch.empty_like(q)
    lse_ref = torch.empty_like(lse)
    fa.fa_fwd(q, k, v, o_ref, lse_ref, causal, scale)
    torch.cuda.synchronize()
    assert fa.fa_device_status() == 0
    assert torch.equal(o.view(torch.int16), o_ref.view(torch.int16)) and torch.equal(lse, lse_ref)
    assert bool((ws == 0x5A).all())
