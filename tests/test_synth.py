"""Seeded input generators: determinism, the published SplitMix64 steps, and
the stated distributions (CPU only)."""
import numpy as np

from trellis_coded_quantized_gb300 import synth

MASK = (1 << 64) - 1


def splitmix64_scalar(state: int) -> int:
    z = state & MASK
    z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & MASK
    z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & MASK
    return z ^ (z >> 31)


def test_stream_matches_scalar_definition():
    for seed, tag in ((0, 1), (5, 2), (123456789, 4)):
        base = splitmix64_scalar(seed ^ (tag * 0xD1B54A32D192ED03 & MASK))
        want = [splitmix64_scalar(base + (i + 1) * synth.GAMMA) for i in range(50)]
        got = synth.stream_u64(seed, tag, 50)
        assert [int(v) for v in got] == want
        # an offset window of the same stream
        assert [int(v) for v in synth.stream_u64(seed, tag, 10, offset=20)] == want[20:30]


def test_deterministic_and_distinct_streams():
    a = synth.problem(1, 2, 8, 512, 3, seed=0)
    b = synth.problem(1, 2, 8, 512, 3, seed=0)
    c = synth.problem(1, 2, 8, 512, 3, seed=1)
    for key in ("codes", "scales", "lut", "x"):
        assert np.array_equal(a[key], b[key])
        assert not np.array_equal(a[key], c[key])
    assert a["codes"].shape == (8, 2 * 24) and a["codes"].dtype == np.uint32
    assert a["x"].shape == (2, 512) and a["x"].dtype == np.uint16
    p0 = synth.problem(0, 3, 512, 256, 2, seed=0)
    assert p0["x"].shape == (3, 512) and p0["scales"].shape == (512,)


def test_distributions():
    n = synth.normal(0, synth.TAG_LUT, 200000)
    assert abs(n.mean()) < 0.01 and abs(n.std() - 1) < 0.01
    s = synth.scales(0, 100000)
    sf = (s.astype(np.uint32) << 16).view(np.float32)
    assert sf.min() >= 0.0099 and sf.max() <= 0.0301
    codes = synth.codes(0, 64, 1024, 4)
    bits = np.unpackbits(codes.view(np.uint8))
    assert abs(bits.mean() - 0.5) < 0.01


def test_torch_generator_matches_numpy():
    for seed, rows, cols, k in ((0, 3, 256, 2), (2001, 40, 1024, 3), (7, 5, 512, 4)):
        a = synth.codes(seed, rows, cols, k)
        b = synth.codes_torch(seed, rows, cols, k, "cpu").numpy().view(np.uint32)
        assert np.array_equal(a, b)
