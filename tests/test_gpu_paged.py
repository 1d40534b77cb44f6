"""GPU parity of the paged-K/V forward pass (fa_fwd_paged).

K and V are scattered into a pool of 128-key pages in a random order, with
finite filler in the last page's rows past T and in the unused pages; the
result must equal the oracle on the contiguous K and V, and be bit-identical
to fa_fwd_gqa on them (the kernel does the same arithmetic, only the addresses
of the K/V tiles differ).  A block-table entry outside the pool must read as
zeros and be reported by fa_device_status.
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


def _paged(x, seed, extra_pages=3):
    """Pools (num_pages, Hkv, 128, d) bf16 bits and a (B, max_pages) table, pages in a random order."""
    rng = np.random.default_rng(seed)
    B, Hkv, T, d = x.B, x.Hkv, x.T, x.d
    nk = (T + 127) // 128
    max_pages = nk + 1
    num_pages = B * nk + extra_pages
    perm = rng.permutation(num_pages)
    table = np.full((B, max_pages), -7, dtype=np.int32)  # entries past nk are never read
    filler = fi.f32_to_bf16_bits(np.float32(7.0))
    kp = np.full((num_pages, Hkv, 128, d), filler, dtype=np.uint16)
    vp = np.full((num_pages, Hkv, 128, d), filler, dtype=np.uint16)
    for b in range(B):
        for lp in range(nk):
            pg = perm[b * nk + lp]
            table[b, lp] = pg
            rows = min(128, T - lp * 128)
            kp[pg, :, :rows] = x.k_bits[b, :, lp * 128:lp * 128 + rows]
            vp[pg, :, :rows] = x.v_bits[b, :, lp * 128:lp * 128 + rows]
    return kp, vp, table, num_pages


def _run(x, kp, vp, table, causal, scale):
    import torch

    import exact_io_aware_07_gb300 as fa

    q = to_device(None, x.q_bits)
    k_pages, v_pages = to_device(None, kp), to_device(None, vp)
    bt = torch.from_numpy(table).cuda()
    o = torch.full_like(q, float("nan"))
    lse = torch.full(q.shape[:3], float("nan"), dtype=torch.float32, device="cuda")
    fa.fa_fwd_paged(q, k_pages, v_pages, bt, o, lse, causal, scale)
    torch.cuda.synchronize()
    return q, o, lse


@pytest.mark.parametrize("B,H,Hkv,T,d,causal", [
    (2, 8, 2, 300, 64, 1), (2, 4, 4, 1000, 128, 0), (1, 8, 1, 129, 128, 1), (3, 2, 2, 640, 64, 0), (1, 2, 2, 1, 64, 1),
])
def test_paged_matches_contiguous(B, H, Hkv, T, d, causal):
    import torch

    import exact_io_aware_07_gb300 as fa

    x = fi.make_grouped_qkv(B, H, Hkv, T, d, seed=81)
    kp, vp, table, _ = _paged(x, seed=82)
    scale = default_scale(d)
    q, o, lse = _run(x, kp, vp, table, causal, scale)
    assert fa.fa_device_status() == 0
    q64, k64, v64 = x.f64("q"), x.f64("k"), x.f64("v")
    O_ref, lse_ref = oracle.attention_fwd_gqa(q64, k64, v64, causal, scale)
    compare(bf16_to_f64(o), lse.cpu().numpy().astype(np.float64), O_ref, lse_ref, label=f"paged T{T} d{d}",
            bound=rounding_bound(q64, k64, v64, causal, scale))
    k, v = to_device(None, x.k_bits), to_device(None, x.v_bits)
    o2, lse2 = fa.attention_gqa(q, k, v, causal=bool(causal), scale=scale)
    torch.cuda.synchronize()
    assert torch.equal(o.view(torch.int16), o2.view(torch.int16)) and torch.equal(lse, lse2)


def test_paged_reports_a_page_outside_the_pool():
    import exact_io_aware_07_gb300 as fa

    x = fi.make_grouped_qkv(1, 2, 2, 256, 64, seed=83)
    kp, vp, table, num_pages = _paged(x, seed=84)
    table[0, 1] = num_pages + 5
    _run(x, kp, vp, table, 0, 0.125)
    assert fa.fa_device_status() == 14  # FA_ERR_BAD_PAGE, then cleared
    assert fa.fa_device_status() == 0
