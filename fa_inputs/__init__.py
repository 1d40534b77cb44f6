"""Seeded synthetic inputs for attention: Q, K, V tensors of shape (B, H, T, d).

This module is shared by the CPU oracle, the GPU tests and the bench. It holds
no attention arithmetic, only a random-number recipe:

* counter-based splitmix64 (Steele, Lea and Flood, "Fast splittable
  pseudorandom number generators", 2014): output i of a stream is the
  splitmix64 finaliser applied to ``key + (i + 1) * 0x9E3779B97F4A7C15``;
* Box-Muller (1958) turns two 24-bit uniforms into two standard normals;
* the normal is multiplied by ``sigma``, rounded to fp32 and then to bf16
  with round-to-nearest-even.

Every tensor is its own stream, keyed by ``(seed, tensor_id)``.  The values
are returned both as raw bf16 bit patterns (``uint16``) and as the exact
float64 numbers those patterns denote, so the GPU path and the oracle see the
same inputs bit for bit.
"""
from __future__ import annotations

import math
from dataclasses import dataclass

import numpy as np

_GOLDEN = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)
_CHUNK = 1 << 20  # value pairs generated per numpy pass (bounds temporary memory)

TENSOR_IDS = {"q": 1, "k": 2, "v": 3, "do": 4}


def _mix(z: np.ndarray) -> np.ndarray:
    """splitmix64 finaliser on a uint64 array (wrapping arithmetic)."""
    z = (z ^ (z >> np.uint64(30))) * _M1
    z = (z ^ (z >> np.uint64(27))) * _M2
    return z ^ (z >> np.uint64(31))


def stream_key(seed: int, tensor_id: int) -> np.uint64:
    """Key of the stream for one tensor: the finaliser of a packed (seed, id)."""
    packed = np.array([((seed & 0xFFFFFFFF) << 32) | (tensor_id & 0xFFFFFFFF)],
                      dtype=np.uint64)
    with np.errstate(over="ignore"):
        return _mix(packed + _GOLDEN)[0]


def splitmix64(key: np.uint64, start: int, count: int) -> np.ndarray:
    """Outputs ``start .. start+count-1`` of the counter-based stream ``key``."""
    idx = np.arange(start + 1, start + count + 1, dtype=np.uint64)
    with np.errstate(over="ignore"):
        return _mix(key + idx * _GOLDEN)


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round fp32 values to bf16 (round to nearest, ties to even); finite inputs."""
    b = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    b = b + np.uint32(0x7FFF) + ((b >> np.uint32(16)) & np.uint32(1))
    return (b >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """Exact float64 value of bf16 bit patterns."""
    u = bits.astype(np.uint32) << np.uint32(16)
    return u.view(np.float32).astype(np.float64)


def normal_bf16_bits(seed: int, tensor_id: int, n: int, sigma: float = 1.0) -> np.ndarray:
    """``n`` values of N(0, sigma^2), rounded to bf16, as uint16 bit patterns."""
    key = stream_key(seed, tensor_id)
    out = np.empty(n, dtype=np.uint16)
    npairs = (n + 1) // 2
    c = min(_CHUNK, npairs)
    # work buffers reused across chunks (fresh allocations are the slow part)
    z = np.empty(2 * c, dtype=np.uint64)
    t = np.empty(2 * c, dtype=np.uint64)
    top = np.empty(2 * c, dtype=np.float64)
    r = np.empty(c, dtype=np.float64)
    ang = np.empty(c, dtype=np.float64)
    val = np.empty(2 * c, dtype=np.float64)
    f32 = np.empty(2 * c, dtype=np.float32)
    u32 = np.empty(2 * c, dtype=np.uint32)
    base = np.arange(1, 2 * c + 1, dtype=np.uint64)
    with np.errstate(over="ignore"):
        for p0 in range(0, npairs, c):
            m = 2 * min(c, npairs - p0)
            zz, tt = z[:m], t[:m]
            # counter-based splitmix64: finaliser of key + (i + 1) * golden
            np.add(base[:m], np.uint64(2 * p0), out=zz)
            np.multiply(zz, _GOLDEN, out=zz)
            np.add(zz, key, out=zz)
            for sh, mul in ((30, _M1), (27, _M2)):
                np.right_shift(zz, np.uint64(sh), out=tt)
                np.bitwise_xor(zz, tt, out=zz)
                np.multiply(zz, mul, out=zz)
            np.right_shift(zz, np.uint64(31), out=tt)
            np.bitwise_xor(zz, tt, out=zz)
            # Box-Muller on the top 24 bits of each pair of outputs
            np.right_shift(zz, np.uint64(40), out=tt)
            tp = top[:m]
            tp[:] = tt
            h = m // 2
            rr, aa = r[:h], ang[:h]
            np.add(tp[0::2], 1.0, out=rr)
            np.multiply(rr, 1.0 / 16777216.0, out=rr)          # u1 in (0, 1]
            np.log(rr, out=rr)
            np.multiply(rr, -2.0, out=rr)
            np.sqrt(rr, out=rr)
            np.multiply(rr, sigma, out=rr)
            np.multiply(tp[1::2], 2.0 * math.pi / 16777216.0, out=aa)  # 2 pi u2
            vv = val[:m]
            np.cos(aa, out=vv[0::2])
            np.sin(aa, out=vv[1::2])
            vv[0::2] *= rr
            vv[1::2] *= rr
            # fp64 -> fp32 -> bf16 (round to nearest even)
            ff = f32[:m]
            ff[:] = vv
            uu = u32[:m]
            bits = ff.view(np.uint32)
            np.right_shift(bits, np.uint32(16), out=uu)
            np.bitwise_and(uu, np.uint32(1), out=uu)
            np.add(uu, np.uint32(0x7FFF), out=uu)
            np.add(uu, bits, out=uu)
            np.right_shift(uu, np.uint32(16), out=uu)
            lo = 2 * p0
            hi = min(n, lo + m)
            out[lo:hi] = uu[: hi - lo]
    return out


@dataclass
class QKV:
    """One seeded attention input: bf16 bit patterns plus their float64 values."""

    B: int
    H: int
    T: int
    d: int
    q_bits: np.ndarray
    k_bits: np.ndarray
    v_bits: np.ndarray

    def f64(self, name: str) -> np.ndarray:
        return bf16_bits_to_f64(getattr(self, name + "_bits")).reshape(self.B, self.H, self.T, self.d)


def make_qkv(B: int, H: int, T: int, d: int, seed: int = 0,
             sigma_qk: float = 1.0, sigma_v: float = 1.0) -> QKV:
    """Q, K ~ N(0, sigma_qk^2) and V ~ N(0, sigma_v^2), i.i.d., bf16, shape (B,H,T,d)."""
    n = B * H * T * d
    q = normal_bf16_bits(seed, TENSOR_IDS["q"], n, sigma_qk).reshape(B, H, T, d)
    k = normal_bf16_bits(seed, TENSOR_IDS["k"], n, sigma_qk).reshape(B, H, T, d)
    v = normal_bf16_bits(seed, TENSOR_IDS["v"], n, sigma_v).reshape(B, H, T, d)
    return QKV(B, H, T, d, q, k, v)


@dataclass
class GroupedQKV:
    """Seeded inputs with grouped K/V heads: q (B, H, T, d), k and v (B, Hkv, T, d), bf16 bits."""

    B: int
    H: int
    Hkv: int
    T: int
    d: int
    q_bits: np.ndarray
    k_bits: np.ndarray
    v_bits: np.ndarray

    def f64(self, name: str) -> np.ndarray:
        heads = self.H if name == "q" else self.Hkv
        return bf16_bits_to_f64(getattr(self, name + "_bits")).reshape(self.B, heads, self.T, self.d)


def make_grouped_qkv(B: int, H: int, Hkv: int, T: int, d: int, seed: int = 0,
                     sigma_qk: float = 1.0, sigma_v: float = 1.0) -> GroupedQKV:
    """Q ~ N(0, sigma_qk^2) with H heads; K ~ N(0, sigma_qk^2) and V ~ N(0, sigma_v^2) with Hkv heads."""
    q = normal_bf16_bits(seed, TENSOR_IDS["q"], B * H * T * d, sigma_qk).reshape(B, H, T, d)
    k = normal_bf16_bits(seed, TENSOR_IDS["k"], B * Hkv * T * d, sigma_qk).reshape(B, Hkv, T, d)
    v = normal_bf16_bits(seed, TENSOR_IDS["v"], B * Hkv * T * d, sigma_v).reshape(B, Hkv, T, d)
    return GroupedQKV(B, H, Hkv, T, d, q, k, v)


def make_grad_out(B: int, H: int, T: int, d: int, seed: int = 0, sigma: float = 1.0) -> np.ndarray:
    """The upstream gradient dO ~ N(0, sigma^2), bf16 bits (B, H, T, d), for the backward pass."""
    return normal_bf16_bits(seed, TENSOR_IDS["do"], B * H * T * d, sigma).reshape(B, H, T, d)


# ---------------------------------------------------------------- e4m3 (OCP FP8) inputs

def _e4m3_table() -> np.ndarray:
    """Values of the 256 e4m3 codes: sign, 4 exponent bits (bias 7), 3 mantissa bits; no
    infinities; 0x7F and 0xFF are NaN.  Subnormals (exponent 0) are m / 8 * 2^-6."""
    vals = np.empty(256, dtype=np.float64)
    for code in range(256):
        s, e, m = code >> 7, (code >> 3) & 0xF, code & 0x7
        if e == 0xF and m == 0x7:
            v = np.nan
        elif e == 0:
            v = m / 8.0 * 2.0 ** -6
        else:
            v = (1.0 + m / 8.0) * 2.0 ** (e - 7)
        vals[code] = -v if s else v
    return vals


E4M3_VALUES = _e4m3_table()
E4M3_MAX = 448.0


def e4m3_to_f64(codes: np.ndarray) -> np.ndarray:
    """Exact float64 values of e4m3 bytes."""
    return E4M3_VALUES[np.asarray(codes, dtype=np.uint8)]


def f64_to_e4m3(x: np.ndarray) -> np.ndarray:
    """Nearest e4m3 code (ties to the even code), magnitudes above 448 saturated to 448."""
    x = np.asarray(x, dtype=np.float64)
    pos = E4M3_VALUES[:0x7F]  # 0x00 .. 0x7E: the non-negative finite values, increasing
    a = np.minimum(np.abs(x), E4M3_MAX)
    hi = np.clip(np.searchsorted(pos, a, side="left"), 0, 0x7E)
    lo = np.maximum(hi - 1, 0)
    d_lo, d_hi = a - pos[lo], pos[hi] - a
    pick_hi = (d_hi < d_lo) | ((d_hi == d_lo) & (hi % 2 == 0))
    code = np.where(pick_hi, hi, lo).astype(np.uint8)
    return np.where(np.signbit(x) & (code != 0), code | 0x80, code).astype(np.uint8)


@dataclass
class QKV8:
    """Seeded e4m3 inputs: bytes (B, H, T, d) and one scale per tensor (real value = byte value * scale)."""

    B: int
    H: int
    T: int
    d: int
    q8: np.ndarray
    k8: np.ndarray
    v8: np.ndarray
    descale: tuple

    def f64(self, name: str) -> np.ndarray:
        i = "qkv".index(name)
        return e4m3_to_f64(getattr(self, name + "8")) * self.descale[i]


def make_qkv_e4m3(B: int, H: int, T: int, d: int, seed: int = 0, descale=(1.0, 1.0, 1.0)) -> QKV8:
    """Q, K, V ~ N(0, 1) in real value: each tensor's N(0, 1) draw divided by its scale,
    rounded to e4m3 (so the bytes use the format's range whatever the scale)."""
    out = []
    for name, sc in zip("qkv", descale):
        z = bf16_bits_to_f64(normal_bf16_bits(seed, TENSOR_IDS[name], B * H * T * d))
        out.append(f64_to_e4m3(z / sc).reshape(B, H, T, d))
    return QKV8(B, H, T, d, out[0], out[1], out[2], tuple(float(x) for x in descale))


# The attention workloads: shapes, masks and value distributions.
WORKLOADS = {
    "tiny_causal_b1h4t256d64": dict(B=1, H=4, T=256, d=64, causal=True, sigma_qk=1.0),
    "gpt2s_causal_b8h12t1024d64": dict(B=8, H=12, T=1024, d=64, causal=True, sigma_qk=1.0),
    "gpt2m_b16h16t1024d64": dict(B=16, H=16, T=1024, d=64, causal=False, sigma_qk=1.0),
    "gpt2m_stress_b16h16t1024d64": dict(B=16, H=16, T=1024, d=64, causal=False, sigma_qk=3.0),
    "llama8b_causal_b1h32t4096d128": dict(B=1, H=32, T=4096, d=128, causal=True, sigma_qk=1.0),
    "llama8b_b1h32t4096d128": dict(B=1, H=32, T=4096, d=128, causal=False, sigma_qk=1.0),
    "long_causal_b1h32t32768d128": dict(B=1, H=32, T=32768, d=128, causal=True, sigma_qk=1.0),
}


def workload_qkv(name: str, seed: int = 0) -> QKV:
    w = WORKLOADS[name]
    return make_qkv(w["B"], w["H"], w["T"], w["d"], seed=seed, sigma_qk=w["sigma_qk"])
