"""FlashAttention forward on one GB300: Python binding of the C-ABI library ``libfa_gb300.so``.

The binding only marshals arguments: it checks tensor dtypes, shapes and
devices, then passes raw device pointers and the current CUDA stream to the
C entry points declared in ``include/fa.h``.  Every step of the attention
computation runs in the library's sm_103a kernel; there is no other path.  If
the library has not been built, importing works but the first call raises.

Entry points (same names as the C ABI):
    fa_fwd(q, k, v, o, lse, causal, scale, stream=None)
    fa_fwd_gqa(q, k, v, o, lse, causal, scale, stream=None)
    fa_fwd_paged(q, k_pages, v_pages, block_table, o, lse, causal, scale, stream=None)
    fa_fwd_fp8(q8, k8, v8, o, lse, causal, scale, descales, workspace, stream=None)
    fa_fwd_splitkv(q, k, v, o, lse, causal, scale, num_splits, workspace, stream=None)
    fa_fwd_splitkv_noalloc(q, k, v, o, lse, causal, scale, num_splits, stream=None)
    fa_bwd(q, k, v, o, lse, dout, dq, dk, dv, causal, scale, workspace, stream=None)
    fa_fwd_splitkv_workspace_bytes, fa_fwd_splitkv_count, fa_fwd_fp8_workspace_bytes, fa_bwd_workspace_bytes
    fa_status_string(code), fa_device_status(stream=None), fa_selftest_wait_timeout(us, stream=None)
    fa_fwd_launch_shape(B, H, T, d, causal, num_sms), fa_ex2_rate(stream=None), fa_version()
and the convenience wrappers ``attention``, ``attention_gqa``, ``attention_splitkv``
and ``attention_bwd`` that allocate their outputs (and workspaces) with PyTorch.
"""
from __future__ import annotations

import ctypes
import math
import os

from ._build import build, lib_path  # noqa: F401

__all__ = [
    "FAError", "fa_fwd", "fa_fwd_splitkv", "fa_fwd_splitkv_noalloc", "fa_fwd_splitkv_workspace_bytes",
    "fa_fwd_splitkv_count", "fa_status_string", "fa_device_status", "FA_NOALLOC_SCRATCH_BYTES",
    "fa_fwd_launch_shape", "fa_selftest_wait_timeout", "fa_ex2_rate", "fa_version",
    "attention", "attention_splitkv", "load_library", "STATUS", "FA_MAX_SPLITS",
]

STATUS = {
    0: "FA_OK", 1: "FA_ERR_NULL_PTR", 2: "FA_ERR_MISALIGNED", 3: "FA_ERR_BAD_SHAPE",
    4: "FA_ERR_UNSUPPORTED_HEAD_DIM", 5: "FA_ERR_BAD_SCALE", 6: "FA_ERR_NO_DEVICE_SUPPORT",
    7: "FA_ERR_LAUNCH", 8: "FA_ERR_DEVICE_TIMEOUT", 9: "FA_ERR_BAD_ARG", 10: "FA_ERR_BAD_POINTER",
    11: "FA_ERR_ALIAS", 12: "FA_ERR_CUDA", 13: "FA_ERR_WORKSPACE", 14: "FA_ERR_BAD_PAGE",
}
FA_MAX_SPLITS = 256
EXPORTED = ["fa_fwd", "fa_fwd_gqa", "fa_fwd_paged", "fa_fwd_fp8", "fa_fwd_fp8_workspace_bytes", "fa_bwd",
            "fa_bwd_workspace_bytes", "fa_fwd_splitkv", "fa_fwd_splitkv_noalloc", "fa_fwd_splitkv_workspace_bytes",
            "fa_fwd_splitkv_count", "fa_status_string", "fa_device_status", "fa_fwd_launch_shape", "fa_selftest_wait_timeout", "fa_ex2_rate",
            "fa_version"]
FA_NOALLOC_SCRATCH_BYTES = 32 << 20


class FAError(RuntimeError):
    """A non-zero status from the library."""

    def __init__(self, code: int, where: str):
        self.code = code
        self.name = STATUS.get(code, str(code))
        super().__init__(f"{where}: {self.name} ({fa_status_string(code)})")


_LIB = None


def load_library(path: str | None = None) -> ctypes.CDLL:
    """Loads the built library (once).  Raises if it is missing: there is no fallback."""
    global _LIB
    if _LIB is not None and path is None:
        return _LIB
    path = path or lib_path()
    if not os.path.exists(path):
        raise RuntimeError(f"attention library not built ({path}); run exact_io_aware_07_gb300.build()")
    lib = ctypes.CDLL(path)
    vp, i, f = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
    lib.fa_fwd.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, f, vp]
    lib.fa_fwd.restype = i
    lib.fa_fwd_gqa.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, i, f, vp]
    lib.fa_fwd_gqa.restype = i
    lib.fa_fwd_paged.argtypes = [vp, vp, vp, vp, vp, vp, i, i, i, i, i, i, f, i, i, vp]
    lib.fa_fwd_paged.restype = i
    lib.fa_fwd_fp8.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, f, f, f, f, vp, ctypes.c_size_t, vp]
    lib.fa_fwd_fp8.restype = i
    lib.fa_fwd_fp8_workspace_bytes.argtypes = [i, i, i, i]
    lib.fa_fwd_fp8_workspace_bytes.restype = ctypes.c_size_t
    lib.fa_bwd.argtypes = [vp] * 9 + [i, i, i, i, i, f, vp, ctypes.c_size_t, vp]
    lib.fa_bwd.restype = i
    lib.fa_bwd_workspace_bytes.argtypes = [i, i, i]
    lib.fa_bwd_workspace_bytes.restype = ctypes.c_size_t
    lib.fa_status_string.argtypes = [i]
    lib.fa_status_string.restype = ctypes.c_char_p
    lib.fa_device_status.argtypes = [vp, ctypes.POINTER(i)]
    lib.fa_device_status.restype = i
    lib.fa_fwd_launch_shape.argtypes = [i, i, i, i, i, i] + [ctypes.POINTER(i)] * 3
    lib.fa_fwd_launch_shape.restype = i
    lib.fa_fwd_splitkv.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, f, i, vp, ctypes.c_size_t, vp]
    lib.fa_fwd_splitkv.restype = i
    lib.fa_fwd_splitkv_noalloc.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, f, i, vp]
    lib.fa_fwd_splitkv_noalloc.restype = i
    lib.fa_fwd_splitkv_workspace_bytes.argtypes = [i, i, i, i, i]
    lib.fa_fwd_splitkv_workspace_bytes.restype = ctypes.c_size_t
    lib.fa_fwd_splitkv_count.argtypes = [i, i, i, i, i, i]
    lib.fa_fwd_splitkv_count.restype = i
    lib.fa_selftest_wait_timeout.argtypes = [ctypes.c_uint, vp]
    lib.fa_selftest_wait_timeout.restype = i
    lib.fa_ex2_rate.argtypes = [ctypes.POINTER(ctypes.c_double), vp]
    lib.fa_ex2_rate.restype = i
    lib.fa_version.argtypes = []
    lib.fa_version.restype = ctypes.c_char_p
    if path == lib_path():
        _LIB = lib
    return lib


def fa_status_string(code: int) -> str:
    return load_library().fa_status_string(int(code)).decode()


def fa_version() -> str:
    return load_library().fa_version().decode()


def fa_fwd_launch_shape(B: int, H: int, T: int, d: int, causal: bool, num_sms: int):
    """(grid, threads, dynamic smem bytes) of the launch ``fa_fwd`` makes for these sizes."""
    g, t, s = ctypes.c_int(), ctypes.c_int(), ctypes.c_int()
    code = load_library().fa_fwd_launch_shape(B, H, T, d, int(causal), num_sms,
                                              ctypes.byref(g), ctypes.byref(t), ctypes.byref(s))
    if code:
        raise FAError(code, "fa_fwd_launch_shape")
    return g.value, t.value, s.value


def _stream_handle(stream):
    import torch

    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def fa_device_status(stream=None) -> int:
    """Reads and clears the device status word (0 = FA_OK, 8 = a wait ran out)."""
    out = ctypes.c_int()
    code = load_library().fa_device_status(ctypes.c_void_p(_stream_handle(stream)), ctypes.byref(out))
    if code:
        raise FAError(code, "fa_device_status")
    return out.value


def fa_selftest_wait_timeout(timeout_us: int, stream=None) -> None:
    """Enqueues the bounded-wait self-test kernel (see include/fa.h); read the outcome with fa_device_status."""
    code = load_library().fa_selftest_wait_timeout(int(timeout_us), ctypes.c_void_p(_stream_handle(stream)))
    if code:
        raise FAError(code, "fa_selftest_wait_timeout")


def fa_ex2_rate(stream=None) -> float:
    """ex2.approx operations per second of the current device (a short probe; synchronous)."""
    out = ctypes.c_double(0.0)
    code = load_library().fa_ex2_rate(ctypes.byref(out), ctypes.c_void_p(_stream_handle(stream)))
    if code:
        raise FAError(code, "fa_ex2_rate")
    return float(out.value)


def fa_fwd(q, k, v, o, lse, causal: bool, scale: float, stream=None) -> None:
    """O, LSE = attention(Q, K, V) into caller-owned tensors.

    q, k, v, o: bf16 CUDA tensors (B, H, T, d), contiguous; lse: fp32 (B, H, T).
    Enqueued on ``stream`` (default: PyTorch's current stream); not synchronised.
    """
    import torch

    for name, t in (("q", q), ("k", k), ("v", v), ("o", o)):
        if t.dtype != torch.bfloat16 or t.dim() != 4 or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous bf16 (B, H, T, d) tensor")
    if not (q.shape == k.shape == v.shape == o.shape):
        raise ValueError("q, k, v and o must have the same shape")
    B, H, T, d = q.shape
    if lse.dtype != torch.float32 or tuple(lse.shape) != (B, H, T) or not lse.is_contiguous():
        raise ValueError("lse must be a contiguous fp32 (B, H, T) tensor")
    lib = load_library()
    code = lib.fa_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
                      B, H, T, d, int(bool(causal)), float(scale), ctypes.c_void_p(_stream_handle(stream)))
    if code:
        raise FAError(code, "fa_fwd")


def fa_fwd_gqa(q, k, v, o, lse, causal: bool, scale: float, stream=None) -> None:
    """Grouped K/V heads: q, o (B, H, T, d) and k, v (B, Hkv, T, d) bf16, H a multiple of Hkv;
    query head h reads K/V head h // (H // Hkv).  lse: fp32 (B, H, T)."""
    import torch

    for name, t in (("q", q), ("k", k), ("v", v), ("o", o)):
        if t.dtype != torch.bfloat16 or t.dim() != 4 or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous bf16 4-D tensor")
    B, H, T, d = q.shape
    Hkv = k.shape[1]
    if tuple(o.shape) != (B, H, T, d) or tuple(k.shape) != (B, Hkv, T, d) or k.shape != v.shape:
        raise ValueError("q, o must be (B, H, T, d) and k, v (B, Hkv, T, d)")
    if lse.dtype != torch.float32 or tuple(lse.shape) != (B, H, T) or not lse.is_contiguous():
        raise ValueError("lse must be a contiguous fp32 (B, H, T) tensor")
    code = load_library().fa_fwd_gqa(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
                                     B, H, Hkv, T, d, int(bool(causal)), float(scale),
                                     ctypes.c_void_p(_stream_handle(stream)))
    if code:
        raise FAError(code, "fa_fwd_gqa")


def attention_gqa(q, k, v, causal: bool = False, scale: float | None = None, stream=None):
    """Allocates O and LSE and runs ``fa_fwd_gqa``; ``scale`` defaults to 1/sqrt(d)."""
    import torch

    B, H, T, d = q.shape
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    o = torch.empty_like(q)
    lse = torch.empty((B, H, T), dtype=torch.float32, device=q.device)
    fa_fwd_gqa(q, k, v, o, lse, causal, scale, stream)
    return o, lse


def fa_fwd_paged(q, k_pages, v_pages, block_table, o, lse, causal: bool, scale: float, stream=None) -> None:
    """Paged K/V: k_pages, v_pages (num_pages, Hkv, 128, d) bf16; block_table (B, max_pages) int32 on the
    device; q, o (B, H, T, d) bf16; lse (B, H, T) fp32.  Key t of batch entry b is row t % 128 of page
    block_table[b, t // 128]."""
    import torch

    for name, t in (("q", q), ("k_pages", k_pages), ("v_pages", v_pages), ("o", o)):
        if t.dtype != torch.bfloat16 or t.dim() != 4 or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous bf16 4-D tensor")
    B, H, T, d = q.shape
    num_pages, Hkv, page, dk = k_pages.shape
    if page != 128 or dk != d or v_pages.shape != k_pages.shape or tuple(o.shape) != (B, H, T, d):
        raise ValueError("pages must be (num_pages, Hkv, 128, d), like q's d")
    if block_table.dtype != torch.int32 or block_table.dim() != 2 or block_table.shape[0] != B \
            or not block_table.is_contiguous():
        raise ValueError("block_table must be a contiguous int32 (B, max_pages) tensor")
    if lse.dtype != torch.float32 or tuple(lse.shape) != (B, H, T) or not lse.is_contiguous():
        raise ValueError("lse must be a contiguous fp32 (B, H, T) tensor")
    code = load_library().fa_fwd_paged(q.data_ptr(), k_pages.data_ptr(), v_pages.data_ptr(), block_table.data_ptr(),
                                       o.data_ptr(), lse.data_ptr(), B, H, Hkv, T, d, int(bool(causal)),
                                       float(scale), num_pages, block_table.shape[1],
                                       ctypes.c_void_p(_stream_handle(stream)))
    if code:
        raise FAError(code, "fa_fwd_paged")


def fa_fwd_fp8_workspace_bytes(B: int, H: int, T: int, d: int) -> int:
    return int(load_library().fa_fwd_fp8_workspace_bytes(B, H, T, d))


def fa_fwd_fp8(q, k, v, o, lse, causal: bool, scale: float, descales=(1.0, 1.0, 1.0), workspace=None,
               stream=None) -> None:
    """e4m3 Q, K, V (uint8 CUDA tensors (B, H, T, 128) holding the bytes) with per-tensor scales
    ``descales`` = (q, k, v); O bf16 (B, H, T, 128), LSE fp32 (B, H, T).  ``workspace``: a CUDA tensor
    of at least ``fa_fwd_fp8_workspace_bytes`` bytes (allocated here when None)."""
    import torch

    for name, t in (("q", q), ("k", k), ("v", v)):
        if t.dtype != torch.uint8 or t.dim() != 4 or not t.is_contiguous() or t.shape != q.shape:
            raise ValueError(f"{name} must be a contiguous uint8 (B, H, T, d) tensor of e4m3 bytes")
    B, H, T, d = q.shape
    if o.dtype != torch.bfloat16 or tuple(o.shape) != (B, H, T, d) or not o.is_contiguous():
        raise ValueError("o must be a contiguous bf16 (B, H, T, d) tensor")
    if lse.dtype != torch.float32 or tuple(lse.shape) != (B, H, T) or not lse.is_contiguous():
        raise ValueError("lse must be a contiguous fp32 (B, H, T) tensor")
    if workspace is None:
        workspace = torch.empty(max(1, fa_fwd_fp8_workspace_bytes(B, H, T, d)), dtype=torch.uint8, device=q.device)
    nbytes = workspace.numel() * workspace.element_size()
    qs, ks, vs = (float(x) for x in descales)
    code = load_library().fa_fwd_fp8(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
                                     B, H, T, d, int(bool(causal)), float(scale), qs, ks, vs,
                                     workspace.data_ptr(), nbytes, ctypes.c_void_p(_stream_handle(stream)))
    if code:
        raise FAError(code, "fa_fwd_fp8")


def fa_bwd_workspace_bytes(B: int, H: int, T: int) -> int:
    return int(load_library().fa_bwd_workspace_bytes(B, H, T))


def fa_bwd(q, k, v, o, lse, dout, dq, dk, dv, causal: bool, scale: float, workspace, stream=None) -> None:
    """dQ, dK, dV of sum(dO * O) into caller-owned bf16 tensors (all (B, H, T, d), contiguous).

    ``o`` and ``lse`` are what ``fa_fwd`` returned for (q, k, v, causal, scale);
    ``workspace`` is a CUDA tensor of at least ``fa_bwd_workspace_bytes(B, H, T)`` bytes.
    """
    import torch

    for name, t in (("q", q), ("k", k), ("v", v), ("o", o), ("dout", dout), ("dq", dq), ("dk", dk), ("dv", dv)):
        if t.dtype != torch.bfloat16 or t.dim() != 4 or not t.is_contiguous() or t.shape != q.shape:
            raise ValueError(f"{name} must be a contiguous bf16 tensor shaped like q")
    B, H, T, d = q.shape
    if lse.dtype != torch.float32 or tuple(lse.shape) != (B, H, T) or not lse.is_contiguous():
        raise ValueError("lse must be a contiguous fp32 (B, H, T) tensor")
    nbytes = workspace.numel() * workspace.element_size()
    code = load_library().fa_bwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
                                 dout.data_ptr(), dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), B, H, T, d,
                                 int(bool(causal)), float(scale), workspace.data_ptr(), nbytes,
                                 ctypes.c_void_p(_stream_handle(stream)))
    if code:
        raise FAError(code, "fa_bwd")


def attention_bwd(q, k, v, o, lse, dout, causal: bool = False, scale: float | None = None, stream=None):
    """Allocates dQ, dK, dV and the workspace and runs ``fa_bwd``; ``scale`` defaults to 1/sqrt(d)."""
    import torch

    B, H, T, d = q.shape
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    ws = torch.empty(fa_bwd_workspace_bytes(B, H, T), dtype=torch.uint8, device=q.device)
    fa_bwd(q, k, v, o, lse, dout, dq, dk, dv, causal, scale, ws, stream)
    return dq, dk, dv


def attention(q, k, v, causal: bool = False, scale: float | None = None, stream=None):
    """Allocates O (bf16) and LSE (fp32) and runs ``fa_fwd``; ``scale`` defaults to 1/sqrt(d)."""
    import torch

    B, H, T, d = q.shape
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    o = torch.empty_like(q)
    lse = torch.empty((B, H, T), dtype=torch.float32, device=q.device)
    fa_fwd(q, k, v, o, lse, causal, scale, stream)
    return o, lse


def fa_fwd_splitkv_count(B: int, H: int, T: int, d: int, causal: bool, num_splits: int) -> int:
    """Key ranges ``fa_fwd_splitkv`` would use (``num_splits`` 0: the library's choice); -1 if invalid."""
    return int(load_library().fa_fwd_splitkv_count(B, H, T, d, int(bool(causal)), num_splits))


def fa_fwd_splitkv_workspace_bytes(B: int, H: int, T: int, d: int, num_splits: int) -> int:
    """Bytes of scratch ``fa_fwd_splitkv`` needs (0 for invalid sizes; ``num_splits`` 0: the automatic choice)."""
    return int(load_library().fa_fwd_splitkv_workspace_bytes(B, H, T, d, num_splits))


def _check_qkv_o_lse(q, k, v, o, lse):
    import torch

    for name, t in (("q", q), ("k", k), ("v", v), ("o", o)):
        if t.dtype != torch.bfloat16 or t.dim() != 4 or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous bf16 (B, H, T, d) tensor")
    if not (q.shape == k.shape == v.shape == o.shape):
        raise ValueError("q, k, v and o must have the same shape")
    B, H, T, d = q.shape
    if lse.dtype != torch.float32 or tuple(lse.shape) != (B, H, T) or not lse.is_contiguous():
        raise ValueError("lse must be a contiguous fp32 (B, H, T) tensor")
    return B, H, T, d


def fa_fwd_splitkv(q, k, v, o, lse, causal: bool, scale: float, num_splits: int, workspace, stream=None) -> None:
    """Split-KV attention into caller-owned tensors; ``workspace`` is a CUDA tensor used as scratch."""
    B, H, T, d = _check_qkv_o_lse(q, k, v, o, lse)
    if not workspace.is_cuda or not workspace.is_contiguous():
        raise ValueError("workspace must be a contiguous CUDA tensor")
    nbytes = workspace.numel() * workspace.element_size()
    code = load_library().fa_fwd_splitkv(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
                                         B, H, T, d, int(bool(causal)), float(scale), int(num_splits),
                                         workspace.data_ptr(), nbytes, ctypes.c_void_p(_stream_handle(stream)))
    if code:
        raise FAError(code, "fa_fwd_splitkv")


def attention_splitkv(q, k, v, causal: bool = False, num_splits: int = 0, scale: float | None = None, stream=None):
    """Allocates O, LSE and the split workspace and runs ``fa_fwd_splitkv`` (``num_splits`` 0: chosen by the library)."""
    import torch

    B, H, T, d = q.shape
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    o = torch.empty_like(q)
    lse = torch.empty((B, H, T), dtype=torch.float32, device=q.device)
    ws = torch.empty(fa_fwd_splitkv_workspace_bytes(B, H, T, d, num_splits), dtype=torch.uint8, device=q.device)
    fa_fwd_splitkv(q, k, v, o, lse, causal, scale, num_splits, ws, stream)
    return o, lse


def fa_fwd_splitkv_noalloc(q, k, v, o, lse, causal: bool, scale: float, num_splits: int, stream=None) -> None:
    """Split-KV attention with the library's fixed device scratch (no workspace, no allocation).

    For callers that cannot allocate device memory while running; see the
    declaration in include/fa.h for the size limit and the sharing rules.
    """
    B, H, T, d = _check_qkv_o_lse(q, k, v, o, lse)
    code = load_library().fa_fwd_splitkv_noalloc(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                                                 lse.data_ptr(), B, H, T, d, int(bool(causal)), float(scale),
                                                 int(num_splits), ctypes.c_void_p(_stream_handle(stream)))
    if code:
        raise FAError(code, "fa_fwd_splitkv_noalloc")
