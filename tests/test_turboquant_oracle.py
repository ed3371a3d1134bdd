"""Pins of the TurboQuant K/V decode oracle (oracle/turboquant.py), on the CPU.

Each pin ties the oracle to something other than itself (@mlx-bun/inference
1.0.0, kernels/turboquant/decode.ts, joint K/V decode kernel, and
kernels/turboquant/inverse.ts, inverse-256 kernel):
  - the bit layout: a code stream packed by hand from the page's rule, and
    an independent bit-by-bit packer on random codes of every width;
  - the keys: small integers through unit scale and zero come out exact;
    the 8-bit code is the signed byte; the group of a column is col / KG;
    one input where adding the zero before scaling (the page's order) and
    scaling both terms give different bf16 keys, derived with exact
    double-precision intermediates;
  - the values: centroid times scale, exact in f32;
  - the rotation: the Hadamard matrix equals scipy's Sylvester construction,
    H H = 256 I, and two closed forms (a unit vector, a constant row);
  - planted mistakes (bit order, unsigned 8-bit keys, column modulo instead
    of group division, scaling before the zero, a missing 1/16) each fail a
    pin.
"""
import numpy as np
import pytest

from oracle import turboquant as tq


def _pack_bits(codes, bits):
    """Independent packer: write each code's bits one at a time, least
    significant first, at bit offset col * bits of a zeroed byte string."""
    codes = np.asarray(codes, dtype=np.int64)
    D = codes.shape[-1]
    out = np.zeros(codes.shape[:-1] + (D * bits // 8,), dtype=np.uint8)
    flat_c = codes.reshape(-1, D)
    flat_o = out.reshape(-1, D * bits // 8)
    for r in range(flat_c.shape[0]):
        for col in range(D):
            for b in range(bits):
                if (int(flat_c[r, col]) >> b) & 1:
                    pos = col * bits + b
                    flat_o[r, pos // 8] |= np.uint8(1 << (pos % 8))
    return out


def test_hand_packed_three_bit_codes():
    # codes 5 1 7 0 2 6 3 4 at 3 bits, least significant bit first:
    # bits 0..7   = 1 0 1 | 1 0 0 | 1 1      -> 0b11001101 = 0xCD
    # bits 8..15  = 1 | 0 0 0 | 0 1 0 | 0    -> 0b00100001 = 0x21
    # bits 16..23 = 1 1 | 1 1 0 | 0 0 1      -> 0b10001111 = 0x8F
    got = tq.unpack_codes(np.array([0xCD, 0x21, 0x8F], np.uint8), 3, 8)
    assert got.tolist() == [5, 1, 7, 0, 2, 6, 3, 4]


@pytest.mark.parametrize("bits", [2, 3, 4, 5, 8])
@pytest.mark.parametrize("D", [64, 256])
def test_unpack_inverts_an_independent_packer(bits, D):
    rng = np.random.default_rng(bits * 1000 + D)
    codes = rng.integers(0, 1 << bits, size=(3, D))
    assert np.array_equal(tq.unpack_codes(_pack_bits(codes, bits), bits, D), codes)


def test_keys_exact_small_integers_and_signed_bytes():
    D = 64
    raw = np.arange(64, dtype=np.int64) * 4 - 128          # -128 .. 124
    kp = raw.astype(np.int8).view(np.uint8)[None, :]
    k = tq.decode_keys(kp, np.ones((1, 2), np.float32), np.zeros((1, 2), np.float32), 8, D, 32)
    assert np.array_equal(tq.bf16_to_f32(k)[0], raw.astype(np.float32))
    # 4-bit codes are unsigned: 15 stays 15
    kp4 = _pack_bits(np.full((1, D), 15), 4)
    k4 = tq.decode_keys(kp4, np.ones((1, 2), np.float32), np.zeros((1, 2), np.float32), 4, D, 32)
    assert np.all(tq.bf16_to_f32(k4) == 15.0)


def test_key_groups_divide_columns():
    D = 128
    kp = _pack_bits(np.ones((1, D), np.int64), 2)
    scales = np.array([[1.0, 2.0, 4.0, 8.0]], np.float32)       # KG = 32: 4 groups
    zeros = np.array([[0.0, 1.0, 2.0, 3.0]], np.float32)
    k = tq.bf16_to_f32(tq.decode_keys(kp, scales, zeros, 2, D, 32))[0]
    want = np.repeat([(1 + 0) * 1.0, (1 + 1) * 2.0, (1 + 2) * 4.0, (1 + 3) * 8.0], 32)
    assert np.array_equal(k, want)
    k64 = tq.bf16_to_f32(tq.decode_keys(kp, scales[:, :2], zeros[:, :2], 2, D, 64))[0]
    assert np.array_equal(k64, np.repeat([1.0, 4.0], 64))


def _f32(x):
    return float(np.float32(x))


def _bf16_from_double(x):
    """RNE of a double that is already an f32 value, to bf16 bits."""
    u = int(np.float32(x).view(np.uint32))
    return (u + 0x7FFF + ((u >> 16) & 1)) >> 16


def test_zero_is_added_before_scaling():
    # code 65, zero and scale given as f32 bit patterns; the page adds the
    # zero first (one rounding), then scales (one rounding); scaling both
    # terms first rounds differently here.
    z = float(np.uint32(3248102409).view(np.float32))
    s = float(np.uint32(1059282700).view(np.float32))
    add_first = _bf16_from_double(_f32(_f32(65 + z) * s))       # 65 + z and the product are exact in double
    distributed = _bf16_from_double(_f32(_f32(65 * s) + _f32(z * s)))
    assert add_first != distributed
    kp = np.full((1, 64), 65, np.uint8)
    k = tq.decode_keys(kp, np.full((1, 2), s, np.float32), np.full((1, 2), z, np.float32), 8, 64, 32)
    assert int(k[0, 0]) == add_first == 0x41EA


def test_scale_dtypes():
    D = 64
    kp = np.full((1, D), 3, np.uint8)
    h = np.array([[0.5, 0.25]], np.float16)
    kh = tq.decode_keys(kp, h, np.zeros((1, 2), np.float16), 8, D, 32, "f16", "f16")
    bf = np.array([[0x3F00, 0x3E80]], np.uint16)                 # 0.5 and 0.25 as bf16
    kb = tq.decode_keys(kp, bf, np.zeros((1, 2), np.uint16), 8, D, 32, "bf16", "bf16")
    want = np.repeat([1.5, 0.75], 32).astype(np.float32)
    assert np.array_equal(tq.bf16_to_f32(kh)[0], want) and np.array_equal(tq.bf16_to_f32(kb)[0], want)


def test_values_are_centroid_times_scale():
    D, vbits = 64, 3
    codes = np.arange(D) % 8
    vp = _pack_bits(codes[None, :], vbits)
    cent = np.array([-1.5, -0.75, -0.25, -0.0625, 0.0625, 0.25, 0.75, 1.5], np.float32)
    vs = np.array([[2.0, 0.5]], np.float32)
    v = tq.decode_values(vp, vs, cent, vbits, D, 32)[0]
    assert np.array_equal(v, (cent[codes] * np.repeat([2.0, 0.5], 32)).astype(np.float32))


def test_hadamard_is_sylvester():
    scipy_linalg = pytest.importorskip("scipy.linalg")
    H = tq.hadamard_matrix(256)
    assert np.array_equal(H, scipy_linalg.hadamard(256).astype(np.float64))
    assert np.array_equal(H @ H, 256.0 * np.eye(256))


def test_rotation_closed_forms():
    signs = np.where(np.arange(256) % 3 == 0, -1.0, 1.0)
    e0 = np.zeros(256)
    e0[0] = 1.0
    assert np.allclose(tq.inverse_rotation(e0, signs), signs / 16.0, rtol=0, atol=0)
    ones = np.ones(256)
    y = tq.inverse_rotation(ones, signs)
    want = np.zeros(256)
    want[0] = 16.0 * signs[0]
    assert np.array_equal(y, want)
    # the transform is its own inverse up to 256: applying it twice (signs
    # one) gives the input back
    rng = np.random.default_rng(5)
    v = rng.standard_normal(256)
    back = tq.inverse_rotation(tq.inverse_rotation(v, np.ones(256)), np.ones(256))
    assert np.allclose(back, v, rtol=0, atol=1e-12)


# ---------------------------------------------------------------- planted mistakes

def _pins_pass():
    """True when every pin above holds for the module as it stands."""
    checks = [test_hand_packed_three_bit_codes, test_keys_exact_small_integers_and_signed_bytes,
              test_key_groups_divide_columns, test_zero_is_added_before_scaling, test_values_are_centroid_times_scale,
              test_rotation_closed_forms]
    try:
        for c in checks:
            c()
        for bits in (2, 3, 5):
            test_unpack_inverts_an_independent_packer(bits, 64)
    except AssertionError:
        return False
    return True


def test_the_pins_catch_planted_mistakes(monkeypatch):
    assert _pins_pass()

    def msb_first(packed, bits, D):
        p = np.asarray(packed, dtype=np.uint8)
        out = np.empty(p.shape[:-1] + (D,), dtype=np.int64)
        for col in range(D):
            v = 0
            for b in range(bits):
                pos = col * bits + b
                v = (v << 1) | ((p[..., pos // 8].astype(np.int64) >> (7 - pos % 8)) & 1)
            out[..., col] = v
        return out

    def unsigned_keys(kp, kbits, D):
        if kbits == 8:
            return np.asarray(kp, dtype=np.uint8).astype(np.int64)
        return tq.unpack_codes(kp, kbits, D)

    orig_keys = tq.decode_keys

    def modulo_groups(kp, ks, kz, kbits, D, kgroup, ks_dtype="f32", kz_dtype="f32"):
        code = tq.key_codes(kp, kbits, D).astype(np.float32)
        g = np.arange(D) % (D // kgroup)
        zero, scale = tq.to_f32(kz, kz_dtype)[..., g], tq.to_f32(ks, ks_dtype)[..., g]
        return tq.bf16_rne(((code + zero).astype(np.float32) * scale).astype(np.float32))

    def scale_first(kp, ks, kz, kbits, D, kgroup, ks_dtype="f32", kz_dtype="f32"):
        code = tq.key_codes(kp, kbits, D).astype(np.float32)
        g = np.arange(D) // kgroup
        zero, scale = tq.to_f32(kz, kz_dtype)[..., g], tq.to_f32(ks, ks_dtype)[..., g]
        return tq.bf16_rne(((code * scale).astype(np.float32) + (zero * scale).astype(np.float32)).astype(np.float32))

    orig_rot = tq.inverse_rotation

    def no_sixteenth(v, signs):
        return orig_rot(v, signs) * 16.0

    for name, fn in (("unpack_codes", msb_first), ("key_codes", unsigned_keys), ("decode_keys", modulo_groups),
                     ("decode_keys", scale_first), ("inverse_rotation", no_sixteenth)):
        with monkeypatch.context() as m:
            m.setattr(tq, name, fn)
            assert not _pins_pass(), f"planted mistake in {name} ({fn.__name__}) passed every pin"
    assert tq.decode_keys is orig_keys and _pins_pass()
