"""CPU oracle for the TurboQuant packed K/V decode (the second workload).

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the
CPU legs of ``bench.py`` may import this module; the product path
(``trellis_coded_quantized_gb300`` and ``libtrellis``) never does.

It restates two kernels of @mlx-bun/inference 1.0.0 in plain numpy:

- kernels/turboquant/decode.ts, the joint K/V decode kernel: every position
  of a [B, H, N, D] cache holds D keys packed at KBITS bits and D values
  packed at VBITS bits, each code at bit offset col * BITS of the row's byte
  string, low bits first, reaching into the next byte when it straddles one.
  An 8-bit key code is a signed byte.  Keys and values have one scale (and
  the keys one zero) per group of KG or VG consecutive columns:
      K[col] = bf16( (f32(code) + f32(zero[col // KG])) * f32(scale[col // KG]) )
  with the addition done first in f32 (the page insists on that order), and
      V[col] = f32(centroid[code]) * f32(vscale[col // VG])
  returned as f32, or rounded to bf16 when the rotation is deferred.
- kernels/turboquant/inverse.ts, the same decode at D = 256, KBITS = 8,
  VBITS = 3, groups of 32, followed by the inverse rotation of each value
  row: the 256-point Walsh-Hadamard transform (the page runs it as two
  radix-16 butterfly passes), times 1/16, times a per-column sign, rounded to
  bf16.  The oracle writes the transform as its definition,
      y[c] = (1/16) * sign[c] * sum_j (-1)^popcount(c & j) * v[j],
  in float64 and rounds once at the end.

The pages fix the precision of the decode itself (f32 add, f32 multiply), so
those steps are computed in numpy float32 and match a correct kernel bit for
bit; only the rotation is computed in float64.  bf16 values are carried as
uint16 bit patterns; scale/zero arrays may be float32, float16 or bf16
(uint16 patterns with ``dtype="bf16"``).
"""
from __future__ import annotations

import numpy as np

KEY_BITS = (2, 4, 5, 8)
VALUE_BITS = (2, 3, 4, 5, 8)
HEAD_DIMS = (64, 128, 256, 512)
GROUPS = (32, 64)


def bf16_rne(x) -> np.ndarray:
    """float32 -> bf16 bit patterns, round to nearest even (NaN kept quiet)."""
    f = np.ascontiguousarray(x, dtype=np.float32)
    u = f.view(np.uint32).astype(np.uint64)
    r = ((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint16)
    nan = np.isnan(f)
    if nan.any():
        r = np.where(nan, ((u >> 16) | 0x40).astype(np.uint16), r)
    return r


def bf16_to_f32(b) -> np.ndarray:
    return (np.asarray(b, dtype=np.uint32) << 16).view(np.float32)


def to_f32(a, dtype: str) -> np.ndarray:
    """A scale/zero array given as float32, float16 or bf16 bit patterns."""
    if dtype == "f32":
        return np.asarray(a, dtype=np.float32)
    if dtype == "f16":
        return np.asarray(a, dtype=np.float16).astype(np.float32)
    if dtype == "bf16":
        return bf16_to_f32(np.asarray(a, dtype=np.uint16))
    raise ValueError(dtype)


def unpack_codes(packed, bits: int, D: int) -> np.ndarray:
    """Codes of columns 0..D-1 of every row of ``packed`` [..., D*bits/8]
    (uint8): bit offset col*bits, the low bits in the lower byte, a second
    byte joined above the first when the code straddles them."""
    p = np.asarray(packed, dtype=np.uint8)
    assert p.shape[-1] * 8 == D * bits
    out = np.empty(p.shape[:-1] + (D,), dtype=np.int64)
    mask = (1 << bits) - 1
    for col in range(D):
        bit = col * bits
        byte, shift = bit // 8, bit % 8
        word = p[..., byte].astype(np.int64)
        if shift + bits > 8:
            word = word | (p[..., byte + 1].astype(np.int64) << 8)
        out[..., col] = (word >> shift) & mask
    return out


def key_codes(kp, kbits: int, D: int) -> np.ndarray:
    """Key codes: an 8-bit code is the signed byte, narrower codes unsigned."""
    if kbits == 8:
        return np.asarray(kp, dtype=np.uint8).view(np.int8).astype(np.int64)
    return unpack_codes(kp, kbits, D)


def decode_keys(kp, ks, kz, kbits: int, D: int, kgroup: int, ks_dtype: str = "f32",
                kz_dtype: str = "f32") -> np.ndarray:
    """bf16 keys [..., D]: (code + zero) * scale in f32, then bf16."""
    code = key_codes(kp, kbits, D).astype(np.float32)
    g = np.arange(D) // kgroup
    zero = to_f32(kz, kz_dtype)[..., g]
    scale = to_f32(ks, ks_dtype)[..., g]
    shifted = (code + zero).astype(np.float32)          # the f32 addition first
    return bf16_rne((shifted * scale).astype(np.float32))


def decode_values(vp, vs, centroids, vbits: int, D: int, vgroup: int, vs_dtype: str = "f32") -> np.ndarray:
    """f32 values [..., D]: centroid[code] * scale."""
    code = unpack_codes(vp, vbits, D)
    c = np.asarray(centroids, dtype=np.float32)
    assert c.shape == (1 << vbits,)
    g = np.arange(D) // vgroup
    return (c[code] * to_f32(vs, vs_dtype)[..., g]).astype(np.float32)


def hadamard_matrix(n: int) -> np.ndarray:
    """Entries (-1)^popcount(i & j), i, j < n (n a power of two)."""
    i = np.arange(n)
    bits = np.bitwise_and.outer(i, i)
    pop = np.zeros_like(bits)
    while bits.any():
        pop += bits & 1
        bits >>= 1
    return np.where(pop % 2 == 0, 1.0, -1.0)


def inverse_rotation(v, signs) -> np.ndarray:
    """float64 (1/16) * signs * (H_256 v) of each row of v [..., 256]."""
    v = np.asarray(v, dtype=np.float64)
    assert v.shape[-1] == 256
    H = hadamard_matrix(256)
    return (v @ H.T) * (1.0 / 16.0) * np.asarray(signs, dtype=np.float64)


def decode_inverse256(kp, ks, kz, vp, vs, centroids, signs, dtype: str = "f16"):
    """The inverse.ts regime: D = 256, 8-bit keys, 3-bit values, groups of
    32.  Returns (bf16 keys, float64 rotated values before rounding)."""
    k = decode_keys(kp, ks, kz, 8, 256, 32, dtype, dtype)
    v = decode_values(vp, vs, centroids, 3, 256, 32, dtype)
    return k, inverse_rotation(v, signs)


def rotation_error_bound(v, signs) -> np.ndarray:
    """Bound on |f32 result - exact| of one rotated value before its bf16
    rounding.  Each of the 8 butterfly stages rounds every partial sum once
    (relative error <= 2^-24 of a value bounded by the sum of |v_j| that
    reach it); the scaling by 1/16 is exact and the sign multiply rounds
    once more: |err| <= 9 * 2^-24 * (sum_j |v_j|) / 16 * |sign[c]|."""
    a = np.abs(np.asarray(v, dtype=np.float64)).sum(axis=-1, keepdims=True)
    return 9.0 * 2.0 ** -24 * a / 16.0 * np.abs(np.asarray(signs, dtype=np.float64))


def bf16_ulp(x) -> np.ndarray:
    """Spacing of bf16 numbers at |x| (the normal range; 2^-133 below it)."""
    ax = np.abs(np.asarray(x, dtype=np.float64))
    e = np.floor(np.log2(np.where(ax > 0, ax, 1.0)))
    return np.where(ax >= 2.0 ** -126, 2.0 ** (e - 7), 2.0 ** -133)


def rotated_within_bound(got_bf16, exact, bound) -> np.ndarray:
    """A correct kernel rounds to bf16 an f32 value within ``bound`` of the
    exact one: the result is within half a bf16 unit (at the larger of the
    two magnitudes) plus ``bound`` of the exact value."""
    e = np.asarray(exact, dtype=np.float64)
    g = bf16_to_f32(got_bf16).astype(np.float64)
    b = np.broadcast_to(np.asarray(bound, dtype=np.float64), e.shape)
    return np.abs(g - e) <= 0.5 * bf16_ulp(np.abs(e) + b) + b
