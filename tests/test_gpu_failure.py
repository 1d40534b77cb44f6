"""Failure detection on the GPU without a fault: a bounded in-kernel wait runs out.

The self-test kernel waits, through the same bounded-wait code the attention
kernel uses, on a barrier that nothing completes.  The wait must give up after
the requested time, record FA_ERR_DEVICE_TIMEOUT in the device status word and
return; afterwards the context must still run attention correctly.
"""
import time

import pytest

import fa_inputs as fi
from parity import compare, default_scale, rounding_bound, run_gpu

pytestmark = pytest.mark.gpu


def test_bounded_wait_times_out_and_reports():
    import torch

    import exact_io_aware_07_gb300 as fa

    fa.build()
    assert fa.fa_device_status() == 0
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    fa.fa_selftest_wait_timeout(20_000)  # 20 ms
    status = fa.fa_device_status()       # synchronises the stream
    dt = time.perf_counter() - t0
    assert status == 8, fa.STATUS.get(status)
    assert 0.015 <= dt < 2.0, dt
    assert fa.fa_device_status() == 0    # reading clears the word

    # the context is intact: an attention launch still matches the oracle
    import oracle

    qkv = fi.make_qkv(1, 2, 300, 64, seed=12)
    o, lse = run_gpu(qkv, True, default_scale(64))
    q64, k64, v64 = qkv.f64("q"), qkv.f64("k"), qkv.f64("v")
    O_ref, lse_ref = oracle.attention_fwd(q64, k64, v64, True, default_scale(64))
    compare(o, lse, O_ref, lse_ref, label="after timeout", bound=rounding_bound(q64, k64, v64, True, default_scale(64)))
