"""Seeded synthetic inputs for the packed trellis-coded weight matmul.

This module only draws numbers: it holds none of the method's arithmetic
(no window extraction, no decoding, no contraction).  Both the oracle checks
and the CUDA path are fed from here.

Generator: counter-based SplitMix64 (Steele, Lea and Flood, "Fast splittable
pseudorandom number generators", OOPSLA 2014; the finaliser constants of
Vigna's public-domain splitmix64.c).  Element ``i`` of stream ``tag`` under
``seed`` is ``mix(base + (i + 1) * GAMMA)`` with
``base = mix(seed XOR tag * 0xD1B54A32D192ED03)``.

Recipes (all on bf16 carried as uint16 bit patterns):
  codes   uint32: the high 32 bits of each draw, uniform
  lut     f32:    N(0, 1) by Box-Muller on pairs of uniforms
  scales  bf16:   U[0.01, 0.03] rounded to bf16 (to nearest, ties to even)
  x       bf16:   N(0, 1) rounded to bf16
  kv_cache: the TurboQuant K/V cache (recipe in its docstring)
The bf16 rounding of drawn inputs uses PyTorch's CPU conversion, a library
routine that neither the oracle nor the CUDA path uses.
"""
from __future__ import annotations

import numpy as np

GAMMA = 0x9E3779B97F4A7C15
_M1 = 0xBF58476D1CE4E5B9
_M2 = 0x94D049BB133111EB
_TAG = 0xD1B54A32D192ED03

TAG_CODES, TAG_LUT, TAG_SCALES, TAG_X = 1, 2, 3, 4

BT = 256
L = 12


def _mix(z: np.ndarray) -> np.ndarray:
    z = z.copy()
    z ^= z >> np.uint64(30)
    z *= np.uint64(_M1)
    z ^= z >> np.uint64(27)
    z *= np.uint64(_M2)
    z ^= z >> np.uint64(31)
    return z


def stream_u64(seed: int, tag: int, n: int, offset: int = 0) -> np.ndarray:
    """``n`` draws of stream ``tag`` starting at counter ``offset``."""
    with np.errstate(over="ignore"):
        s = np.array([(int(seed) ^ (int(tag) * _TAG)) & 0xFFFFFFFFFFFFFFFF], np.uint64)
        base = _mix(s)[0]
        out = np.empty(n, np.uint64)
        chunk = 1 << 22
        for lo in range(0, n, chunk):
            hi = min(n, lo + chunk)
            i = np.arange(offset + lo + 1, offset + hi + 1, dtype=np.uint64)
            out[lo:hi] = _mix(base + i * np.uint64(GAMMA))
    return out


def uniform(seed: int, tag: int, n: int, offset: int = 0) -> np.ndarray:
    """Uniform doubles in [0, 1): the top 53 bits of each draw times 2^-53."""
    return (stream_u64(seed, tag, n, offset) >> np.uint64(11)).astype(np.float64) * (2.0 ** -53)


def normal(seed: int, tag: int, n: int) -> np.ndarray:
    """N(0, 1) doubles, Box-Muller cosine branch on draws (2i, 2i+1)."""
    u = uniform(seed, tag, 2 * n)
    u1 = 1.0 - u[0::2]          # (0, 1]
    u2 = u[1::2]
    return np.sqrt(-2.0 * np.log(u1)) * np.cos(2.0 * np.pi * u2)


def to_bf16_bits(v: np.ndarray) -> np.ndarray:
    """float32 -> bf16 bits by PyTorch's CPU conversion (nearest, ties to even)."""
    import torch
    t = torch.from_numpy(np.ascontiguousarray(v, np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16).copy()


def words_per_row(cols: int, k: int, bt: int = BT) -> int:
    return (cols // bt) * (bt * k // 32)


def codes(seed: int, rows: int, cols: int, k: int, bt: int = BT) -> np.ndarray:
    """Uniform uint32 code words [rows, (cols/bt)*wpb] (contiguous block layout)."""
    w = words_per_row(cols, k, bt)
    z = stream_u64(seed, TAG_CODES, rows * w)
    return (z >> np.uint64(32)).astype(np.uint32).reshape(rows, w)


def lut(seed: int, l: int = L) -> np.ndarray:
    return normal(seed, TAG_LUT, 1 << l).astype(np.float32)


def scales(seed: int, rows: int) -> np.ndarray:
    v = (0.01 + 0.02 * uniform(seed, TAG_SCALES, rows)).astype(np.float32)
    return to_bf16_bits(v)


def activations(seed: int, m: int, k: int) -> np.ndarray:
    return to_bf16_bits(normal(seed, TAG_X, m * k).astype(np.float32)).reshape(m, k)


def problem(axis: int, m: int, rows: int, cols: int, k: int, seed: int = 0) -> dict:
    """One packed matmul: codes, scales, lut and activations x.

    Axis 1: rows are output features and x is [m, cols].
    Axis 0: rows are input features and x is [m, rows].
    """
    kin = cols if axis == 1 else rows
    return {
        "axis": axis, "m": m, "rows": rows, "cols": cols, "k": k, "seed": seed,
        "codes": codes(seed, rows, cols, k),
        "scales": scales(seed, rows),
        "lut": lut(seed),
        "x": activations(seed, m, kin),
    }


# ----------------------------------------------------------------------------
# TurboQuant packed K/V cache (the second workload)
# ----------------------------------------------------------------------------

TAG_KV_K, TAG_KV_V, TAG_KV_KS, TAG_KV_KZ, TAG_KV_VS, TAG_KV_C, TAG_KV_SIGN = 11, 12, 13, 14, 15, 16, 17


def _bytes(seed: int, tag: int, n: int) -> np.ndarray:
    return (stream_u64(seed, tag, n) >> np.uint64(56)).astype(np.uint8)


def _as_dtype(v: np.ndarray, dtype: str) -> np.ndarray:
    """f32 draws stored as f32, f16 (numpy's conversion) or bf16 bit patterns."""
    if dtype == "f32":
        return v.astype(np.float32)
    if dtype == "f16":
        return v.astype(np.float16)
    return to_bf16_bits(v.astype(np.float32))


def kv_cache(seed: int, rows: int, D: int, key_bits: int, value_bits: int, key_group: int = 32,
             value_group: int = 32, dtypes=("f16", "f16", "f16")) -> dict:
    """A packed K/V cache of `rows` positions: uniform code bytes; key scales
    U[0.005, 0.05]; key zeros U[-2^(b-1) - 1, -2^(b-1) + 1] for b-bit
    unsigned codes, U[-1, 1] for signed 8-bit ones; value scales
    U[0.5, 1.5]; sorted N(0, 1) centroids (f32); signs +-1 (f32)."""
    kdt, zdt, vdt = dtypes
    gk, gv = D // key_group, D // value_group
    kz_mid = 0.0 if key_bits == 8 else -float(1 << (key_bits - 1))
    return {
        "rows": rows, "D": D, "key_bits": key_bits, "value_bits": value_bits,
        "key_group": key_group, "value_group": value_group, "dtypes": tuple(dtypes),
        "kp": _bytes(seed, TAG_KV_K, rows * D * key_bits // 8).reshape(rows, -1),
        "vp": _bytes(seed, TAG_KV_V, rows * D * value_bits // 8).reshape(rows, -1),
        "ks": _as_dtype(0.005 + 0.045 * uniform(seed, TAG_KV_KS, rows * gk), kdt).reshape(rows, gk),
        "kz": _as_dtype(kz_mid - 1.0 + 2.0 * uniform(seed, TAG_KV_KZ, rows * gk), zdt).reshape(rows, gk),
        "vs": _as_dtype(0.5 + uniform(seed, TAG_KV_VS, rows * gv), vdt).reshape(rows, gv),
        "centroids": np.sort(normal(seed, TAG_KV_C, 1 << value_bits)).astype(np.float32),
        "signs": np.where(uniform(seed, TAG_KV_SIGN, D) < 0.5, -1.0, 1.0).astype(np.float32),
    }


# ----------------------------------------------------------------------------
# the same codes drawn on a torch device (for multi-GB inputs)
# ----------------------------------------------------------------------------

def _s64(v: int) -> int:
    """A 64-bit pattern as a signed int64 constant."""
    v &= 0xFFFFFFFFFFFFFFFF
    return v - (1 << 64) if v >= (1 << 63) else v


def _mix_t(z):
    import torch
    z = z ^ ((z >> 30) & ((1 << 34) - 1))
    z = z * _s64(_M1)
    z = z ^ ((z >> 27) & ((1 << 37) - 1))
    z = z * _s64(_M2)
    z = z ^ ((z >> 31) & ((1 << 33) - 1))
    return z


def codes_torch(seed: int, rows: int, cols: int, k: int, device, bt: int = BT):
    """``codes(seed, rows, cols, k)`` computed with int64 tensor arithmetic
    (wrapping multiply, masked logical shifts) on ``device``; int32 storage."""
    import torch
    w = words_per_row(cols, k, bt)
    n = rows * w
    s = np.array([(int(seed) ^ (TAG_CODES * _TAG)) & 0xFFFFFFFFFFFFFFFF], np.uint64)
    base = _s64(int(_mix(s)[0]))
    out = torch.empty(n, dtype=torch.int32, device=device)
    chunk = 1 << 24
    for lo in range(0, n, chunk):
        hi = min(n, lo + chunk)
        i = torch.arange(lo + 1, hi + 1, dtype=torch.int64, device=device)
        z = _mix_t(i * _s64(GAMMA) + base)
        out[lo:hi] = ((z >> 32) & 0xFFFFFFFF).to(torch.int32)
    return out.view(rows, w)
