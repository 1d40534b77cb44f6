"""The allocation-free split-KV entry point, through the C ABI.

fa_fwd_splitkv_noalloc is for callers that cannot allocate device memory while
they run (their memory belongs to a framework pool or a fixed budget, or the
allocator must not be called at that point).  It keeps its split partials in a
fixed scratch array the library holds on each device, so it takes only inputs
and outputs.

This test issues two calls back to back on one stream, on different inputs and
shapes, and synchronises once: the second call reuses the scratch the first
one wrote, so stream order alone must keep them apart.  Each output must equal
fa_fwd_splitkv's (same kernels, same split count, a caller-provided workspace)
bit for bit, and must match the float64 oracle within the parity tolerances
used for every GPU result here.  A problem whose partials would not fit the
fixed scratch is refused before anything is launched.

The file name sorts last so that a run stopping at the first failure has
already run every other test; it also passes on its own in a fresh process.
"""
import ctypes

import numpy as np
import pytest

import fa_inputs as fi
import oracle
from parity import bf16_to_f64, compare, default_scale, rounding_bound, to_device

pytestmark = pytest.mark.gpu


def _noalloc(lib, q, k, v, o, lse, causal, scale, num_splits):
    import torch

    B, H, T, d = q.shape
    st = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return lib.fa_fwd_splitkv_noalloc(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
                                      B, H, T, d, int(causal), ctypes.c_float(scale), num_splits, st)


def test_noalloc_two_calls_in_a_row():
    import torch

    import exact_io_aware_07_gb300 as fa

    assert torch.cuda.is_available(), "the GPU tests need a CUDA device"
    fa.build()
    lib = fa.load_library()
    cases = [  # two calls in a row on different inputs and shapes
        (fi.make_qkv(2, 3, 1000, 128, seed=31), True, 3),
        (fi.make_qkv(1, 4, 777, 64, seed=32, sigma_qk=2.0), False, 2),
    ]
    runs = []
    for qkv, causal, ns in cases:
        q, k, v = (to_device(None, b) for b in (qkv.q_bits, qkv.k_bits, qkv.v_bits))
        B, H, T, d = q.shape
        assert fa.fa_fwd_splitkv_workspace_bytes(B, H, T, d, ns) <= fa.FA_NOALLOC_SCRATCH_BYTES
        o = torch.full_like(q, float("nan"))
        lse = torch.full((B, H, T), float("nan"), dtype=torch.float32, device="cuda")
        runs.append((qkv, causal, ns, q, k, v, o, lse))
    torch.cuda.synchronize()
    for qkv, causal, ns, q, k, v, o, lse in runs:  # no synchronisation between the calls
        assert _noalloc(lib, q, k, v, o, lse, causal, default_scale(q.shape[3]), ns) == 0
    torch.cuda.synchronize()
    assert fa.fa_device_status() == 0
    for qkv, causal, ns, q, k, v, o, lse in runs:
        B, H, T, d = q.shape
        scale = default_scale(d)
        o_ws, lse_ws = fa.attention_splitkv(q, k, v, causal=causal, num_splits=ns, scale=scale)
        torch.cuda.synchronize()
        assert torch.equal(o.view(torch.int16), o_ws.view(torch.int16)), f"T{T} d{d}: O differs from fa_fwd_splitkv"
        assert torch.equal(lse, lse_ws), f"T{T} d{d}: LSE differs from fa_fwd_splitkv"
        q64, k64, v64 = qkv.f64("q"), qkv.f64("k"), qkv.f64("v")
        O_ref, lse_ref = oracle.attention_fwd(q64, k64, v64, causal, scale)
        compare(bf16_to_f64(o), lse.cpu().numpy().astype(np.float64), O_ref, lse_ref,
                label=f"noalloc split{ns} B{B} H{H} T{T} d{d} causal{int(causal)}",
                bound=rounding_bound(q64, k64, v64, causal, scale))


def test_noalloc_refuses_problems_beyond_the_fixed_scratch():
    import torch

    import exact_io_aware_07_gb300 as fa

    fa.build()
    lib = fa.load_library()
    B, H, T, d, ns = 1, 8, 4096, 128, 4  # 4 splits x 32768 rows x 129 x 4 bytes = 67.6 MB > 32 MiB
    assert fa.fa_fwd_splitkv_workspace_bytes(B, H, T, d, ns) > fa.FA_NOALLOC_SCRATCH_BYTES
    q = torch.zeros(B, H, T, d, dtype=torch.bfloat16, device="cuda")
    o = torch.empty_like(q)
    lse = torch.empty(B, H, T, device="cuda")
    assert _noalloc(lib, q, q, q, o, lse, False, 0.1, ns) == 13  # FA_ERR_WORKSPACE, nothing launched
    torch.cuda.synchronize()
    assert fa.fa_device_status() == 0
