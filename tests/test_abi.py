"""The C-ABI library: it builds, loads, exports every declared symbol, and validates on the host.

No test here launches a kernel; they run without a GPU.
"""
import ctypes
import os
import re

import pytest

import exact_io_aware_07_gb300 as fa

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "fa.h")


@pytest.fixture(scope="module")
def lib():
    fa.build()
    return fa.load_library()


def _declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?[A-Za-z_]+\s*\*?\s*(fa_[a-z_0-9]+)\s*\(", text, flags=re.M)))


def _declared_status_codes():
    text = open(HEADER).read()
    return {int(v): k for k, v in re.findall(r"(FA_[A-Z_]+)\s*=\s*(\d+)", text)}


def test_header_declares_the_entry_points():
    assert _declared_functions() == sorted(fa.EXPORTED)


def test_library_exports_every_declared_symbol(lib):
    for name in _declared_functions():
        assert hasattr(lib, name), name
    # exported with C linkage (no C++ mangling) in the dynamic symbol table
    out = os.popen(f"nm -D --defined-only {fa.lib_path()}").read()
    for name in _declared_functions():
        assert re.search(rf"\bT {name}$", out, flags=re.M), name


def test_status_codes_match_header(lib):
    assert _declared_status_codes() == fa.STATUS
    for code in fa.STATUS:
        assert fa.fa_status_string(code) and "unknown" not in fa.fa_status_string(code)
    assert "unknown" in fa.fa_status_string(99)


def test_version(lib):
    assert re.match(r"^\d+\.\d+\.\d+$", fa.fa_version())


A = 0x10000  # fake, 16-byte-aligned addresses: validation fails before any is touched


def _call(lib, q=A, k=A + 0x1000, v=A + 0x2000, o=A + 0x3000, lse=A + 0x4000,
          B=1, H=2, T=128, d=64, causal=0, scale=0.125):
    return lib.fa_fwd(q, k, v, o, lse, B, H, T, d, causal, ctypes.c_float(scale), None)


@pytest.mark.parametrize("kw,code", [
    (dict(q=0), 1), (dict(k=0), 1), (dict(v=0), 1), (dict(o=0), 1), (dict(lse=0), 1),
    (dict(B=0), 3), (dict(H=0), 3), (dict(T=0), 3), (dict(T=-5), 3), (dict(T=(1 << 30) + 1), 3),
    (dict(B=1 << 16, H=1 << 16), 3),
    (dict(d=96), 4), (dict(d=0), 4), (dict(d=256), 4),
    (dict(scale=0.0), 5), (dict(scale=-1.0), 5), (dict(scale=float("nan")), 5), (dict(scale=float("inf")), 5),
    (dict(causal=2), 9), (dict(causal=-1), 9),
    (dict(q=A + 8), 2), (dict(o=A + 0x3004), 2), (dict(lse=A + 0x4002), 2),
])
def test_host_validation(lib, kw, code):
    assert _call(lib, **kw) == code


def test_valid_arguments_reach_the_device_checks(lib):
    # every host check passes; without a GPU the device check refuses, with one the
    # fake addresses are refused as non-device memory; nothing is launched either way
    assert _call(lib) in (6, 10)


def test_launch_shape(lib):
    assert fa.fa_fwd_launch_shape(1, 4, 256, 64, True, 152)[0] == 4       # 4 units of 256 rows
    assert fa.fa_fwd_launch_shape(8, 12, 1024, 64, True, 152)[0] == 152   # 384 units, capped at the SMs
    g, t, s = fa.fa_fwd_launch_shape(1, 32, 4096, 128, False, 152)
    assert (g, t) == (152, 320) and 128 * 1024 < s <= 232_448   # d = 128: one MMA-issuing warp
    g, t, s = fa.fa_fwd_launch_shape(1, 1, 1, 64, False, 152)
    assert (g, t) == (1, 384) and s <= 232_448   # d = 64: one MMA-issuing warp per query tile
    with pytest.raises(fa.FAError):
        fa.fa_fwd_launch_shape(1, 1, 128, 80, False, 152)


def test_selftest_rejects_bad_timeout(lib):
    assert lib.fa_selftest_wait_timeout(0, None) == 9
    assert lib.fa_selftest_wait_timeout(2_000_001, None) == 9


def test_splitkv_workspace_size(lib):
    # partial outputs and LSE of every split, then one counter per 32 query rows of every head
    assert fa.fa_fwd_splitkv_workspace_bytes(1, 4, 256, 64, 2) == (2 * 4 * 256 * 65 * 4 + 4 * 8 * 4 + 255) // 256 * 256
    assert fa.fa_fwd_splitkv_workspace_bytes(2, 3, 1000, 128, 7) == \
        (7 * 6 * 1000 * 129 * 4 + 6 * 32 * 4 + 255) // 256 * 256
    for bad in ((0, 1, 1, 64, 1), (1, 1, 1, 96, 1), (1, 1, 1, 64, -1), (1, 1, 1, 64, fa.FA_MAX_SPLITS + 1)):
        assert fa.fa_fwd_splitkv_workspace_bytes(*bad) == 0


def test_splitkv_count(lib):
    # explicit counts: ceil(tiles / ceil(tiles / num_splits)) key ranges of equal tile count
    assert fa.fa_fwd_splitkv_count(1, 4, 8192, 128, True, 1) == 1
    assert fa.fa_fwd_splitkv_count(1, 4, 8192, 128, True, 3) == 3      # 64 tiles: 3 ranges of 22
    assert fa.fa_fwd_splitkv_count(1, 4, 1000, 64, False, 5) == 4      # 8 tiles: ranges of 2
    assert fa.fa_fwd_splitkv_count(1, 4, 100, 64, False, 4) == 1       # one tile
    assert fa.fa_fwd_splitkv_count(2, 3, 1000, 128, True, 8) == 8
    for bad in ((0, 1, 1, 64, 0, 1), (1, 1, 1, 96, 0, 1), (1, 1, 1, 64, 2, 1), (1, 1, 1, 64, 0, -1),
                (1, 1, 1, 64, 0, fa.FA_MAX_SPLITS + 1)):
        assert lib.fa_fwd_splitkv_count(*bad) == -1


@pytest.mark.parametrize("ns,ws,code", [(-1, A + 0x5000, 9), (fa.FA_MAX_SPLITS + 1, A + 0x5000, 9)])
def test_splitkv_host_validation(lib, ns, ws, code):
    rc = lib.fa_fwd_splitkv(A, A + 0x1000, A + 0x2000, A + 0x3000, A + 0x4000, 1, 2, 128, 64, 0,
                            ctypes.c_float(0.125), ns, ws, 1 << 20, None)
    assert rc == code


def test_splitkv_checks_inputs_first(lib):
    # the shared checks run before the workspace is looked at
    rc = lib.fa_fwd_splitkv(0, A, A, A, A, 1, 2, 128, 64, 0, ctypes.c_float(0.125), 2, A, 1 << 20, None)
    assert rc == 1


def test_bwd_workspace_size(lib):
    # D and LSE * log2 e for every row, each head's rows padded to a multiple of 128
    assert fa.fa_bwd_workspace_bytes(1, 4, 1000) == (2 * 4 * 1024 * 4 + 255) // 256 * 256
    assert fa.fa_bwd_workspace_bytes(2, 3, 128) == 2 * 6 * 128 * 4
    for bad in ((0, 1, 1), (1, 0, 1), (1, 1, 0)):
        assert fa.fa_bwd_workspace_bytes(*bad) == 0
