"""Checks that pin the oracle to facts other than itself.

Each check takes an ``oracle.Oracle`` and raises ``AssertionError`` on a
mismatch, so the same checks run against the real oracle (the pin tests) and
against copies of it with a planted mistake (the mutation tests, which expect
at least one check to fail).

What pins what:
  * hand-derived windows (tests/golden/windows_*.txt) and an independent
    string-of-bits construction pin the window of every column, the bit order,
    the position (BT-1-t)*k and the tail-biting wrap;
  * the word-level extraction printed on the pages (shift, spill into the next
    word, wrap to word 0, mask) pins the same from the pages' own formula;
  * single-bit probes and cyclic rotation pin positions in closed form;
  * PyTorch's float32 -> bf16 conversion and exact rational rounding pin the
    bf16 rounding; a searched double-rounding case pins that the weight is
    rounded to f32 first;
  * numpy's float64 matmul, exact rational brute force, unit vectors and the
    bilinear identity pin both contractions and their index maps.
"""
from __future__ import annotations

import os
from fractions import Fraction

import numpy as np

import oracle as _o

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")
BT, L = 256, 12


# ----------------------------------------------------------------------------
# independent constructions used by the checks
# ----------------------------------------------------------------------------

def pack_symbols(symbols, k: int) -> np.ndarray:
    """Pack BT k-bit symbols least significant bit first into 32-bit words."""
    bits = []
    for s in symbols:
        for b in range(k):
            bits.append((int(s) >> b) & 1)
    words = []
    for j in range(len(bits) // 32):
        w = 0
        for b in range(32):
            w |= bits[32 * j + b] << b
        words.append(w)
    return np.array(words, np.uint32)


def bitstring(words) -> str:
    """'0'/'1' characters of a block, character j = block bit j."""
    return "".join(format(int(w), "032b")[::-1] for w in words)


def window_by_string(words, k: int, t: int) -> int:
    s = bitstring(words)
    n = len(s)
    p = (BT - 1 - t) * k
    piece = "".join(s[(p + i) % n] for i in range(L))   # piece[i] = window bit i
    return int(piece[::-1], 2)


def window_by_words(words, k: int, t: int) -> int:
    """The pages' word arithmetic: shift, spill into the next word (wrapping to
    word 0 of the block), mask to L bits."""
    wpb = BT * k // 32
    pos = (BT - 1 - t) * k
    wi, off = pos >> 5, pos & 31
    win = int(words[wi]) >> off
    if off + L > 32:
        nxt = 0 if wi + 1 == wpb else wi + 1
        win |= (int(words[nxt]) << (32 - off)) & 0xFFFFFFFF
    return win & ((1 << L) - 1)


def bf16_round_fraction(q: Fraction) -> int:
    """Exact round-to-nearest-even of a rational to bf16 bits (finite range)."""
    if q == 0:
        return 0
    sign = 0x8000 if q < 0 else 0
    a = abs(q)
    # exponent e with 2^e <= a < 2^(e+1)
    e = a.numerator.bit_length() - a.denominator.bit_length()
    if Fraction(2) ** e > a:
        e -= 1
    qe = max(e - 7, -133)
    quantum = Fraction(2) ** qe
    n = a / quantum
    fl = n.numerator // n.denominator
    rem = n - fl
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and fl % 2 == 1):
        fl += 1
    v = Fraction(fl) * quantum
    f = np.float32(float(v))
    assert Fraction(float(f)) == v
    return sign | (int(f.view(np.uint32)) >> 16)


def torch_bf16(v_f32: np.ndarray) -> np.ndarray:
    import torch
    t = torch.from_numpy(np.ascontiguousarray(v_f32, np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def read_golden_windows(name: str):
    k = mod = None
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            a, b = line.split()
            if a == "k":
                k = int(b)
            elif a == "modulus":
                mod = int(b)
            else:
                rows.append((int(a), int(b, 16)))
    return k, mod, rows


# ----------------------------------------------------------------------------
# checks
# ----------------------------------------------------------------------------

def check_golden_windows(o: _o.Oracle):
    for name in ("windows_k4_mod15.txt", "windows_k3_mod7.txt", "windows_k2_mod3.txt"):
        k, mod, rows = read_golden_windows(name)
        words = pack_symbols([q % mod for q in range(BT)], k)
        for t, want in rows:
            got = o.window(words, k, t)
            assert got == want, (name, t, hex(got), hex(want))


def check_windows_random(o: _o.Oracle, seed: int = 7, blocks: int = 3):
    rng = np.random.default_rng(seed)
    for k in (2, 3, 4):
        wpb = BT * k // 32
        for _ in range(blocks):
            words = rng.integers(0, 2 ** 32, wpb, dtype=np.uint64).astype(np.uint32)
            for t in range(BT):
                got = o.window(words, k, t)
                assert got == window_by_string(words, k, t), (k, t)
                assert got == window_by_words(words, k, t), (k, t)


def check_single_bit_probes(o: _o.Oracle):
    for k in (2, 3, 4):
        n = BT * k
        wpb = n // 32
        for j in (0, 1, 31, 32, n // 2 + 5, n - 12, n - 1):
            words = np.zeros(wpb, np.uint32)
            words[j // 32] = np.uint32(1 << (j % 32))
            for t in range(BT):
                p = (BT - 1 - t) * k
                d = (j - p) % n
                want = (1 << d) if d < L else 0
                assert o.window(words, k, t) == want, (k, j, t)


def check_wrap_and_rotation(o: _o.Oracle, seed: int = 11):
    rng = np.random.default_rng(seed)
    for k in (2, 3, 4):
        n = BT * k
        wpb = n // 32
        # columns whose window runs past the end of the block read word 0:
        # exactly t < L/k - 1
        wrapped = {t for t in range(BT) if (BT - 1 - t) * k + L > n}
        assert wrapped == {t for t in range(BT) if (t + 1) * k < L}
        words = np.zeros(wpb, np.uint32)
        words[0] = np.uint32(0xFFFFFFFF)
        for t in wrapped:
            p = (BT - 1 - t) * k
            spill = p + L - n                     # bits taken from word 0
            want = ((1 << spill) - 1) << (L - spill)
            assert o.window(words, k, t) == want, (k, t)
        # rotating the block bitstring down by k bits moves win(t) to column t+1
        words = rng.integers(0, 2 ** 32, wpb, dtype=np.uint64).astype(np.uint32)
        s = bitstring(words)
        r = s[k:] + s[:k]
        rot = np.array([int(r[32 * j:32 * j + 32][::-1], 2) for j in range(wpb)], np.uint32)
        for t in range(BT):
            assert o.window(rot, k, t) == o.window(words, k, (t - 1) % BT), (k, t)


def check_special_patterns(o: _o.Oracle):
    for k in (2, 3, 4):
        wpb = BT * k // 32
        zero = np.zeros(wpb, np.uint32)
        ones = np.full(wpb, 0xFFFFFFFF, np.uint32)
        for t in (0, 1, 2, 100, 255):
            assert o.window(zero, k, t) == 0
            assert o.window(ones, k, t) == 0xFFF
    per = {2: (np.full(16, 0x55555555, np.uint32), 0x555),
           4: (np.full(32, 0x77777777, np.uint32), 0x777),
           3: (pack_symbols([1] * BT, 3), 0x249)}
    for k, (words, want) in per.items():
        for t in range(BT):
            assert o.window(words, k, t) == want, (k, t)


def check_bf16_rounding(o: _o.Oracle, seed: int = 3):
    # fixture of ties, overflow and subnormals
    with open(os.path.join(GOLDEN, "bf16_rounding.txt")) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            fb, hb = line.split()[:2]
            v = np.array([int(fb, 16)], np.uint32).view(np.float32)
            assert int(o.bf16_from_float(v)[0]) == int(hb, 16), (fb, hb)
    # against PyTorch's conversion on random patterns and on exact ties
    rng = np.random.default_rng(seed)
    bits = rng.integers(0, 2 ** 32, 200000, dtype=np.uint64).astype(np.uint32)
    ties = (bits & np.uint32(0xFFFF0000)) | np.uint32(0x8000)
    v = np.concatenate([bits, ties]).view(np.float32)
    v = v[np.isfinite(v)]
    assert np.array_equal(o.bf16_from_float(v), torch_bf16(v))
    # double -> bf16 against exact rational rounding
    d = rng.standard_normal(3000) * np.exp2(rng.integers(-140, 120, 3000))
    got = o.bf16_from_double(d)
    for i in range(d.size):
        assert int(got[i]) == bf16_round_fraction(Fraction(float(d[i]))), d[i]


def check_weight_rounds_to_f32_first(o: _o.Oracle, seed: int = 5):
    """w = bf16(f32(lut*scale)): find pairs where rounding the exact product
    straight to bf16 differs, and check the oracle takes the two-step value."""
    rng = np.random.default_rng(seed)
    lutv = rng.standard_normal(400000).astype(np.float32)
    s_bits = torch_bf16(rng.uniform(0.01, 0.03, 400000).astype(np.float32))
    s = _o.bf16_to_float(s_bits)
    prod32 = lutv * s                                   # IEEE binary32 multiply
    two_step = torch_bf16(prod32)
    exact = lutv.astype(np.float64) * s.astype(np.float64)
    # candidates: the f32 product lands on a bf16 tie
    cand = np.nonzero((prod32.view(np.uint32) & np.uint32(0xFFFF)) == np.uint32(0x8000))[0]
    hits = [i for i in cand if bf16_round_fraction(Fraction(float(exact[i]))) != int(two_step[i])]
    assert len(hits) > 0
    for i in hits[:50]:
        codes = np.zeros((1, 32), np.uint32)           # one k=4 block, window 0
        lut = np.zeros(1 << L, np.float32)
        lut[0] = lutv[i]
        w = o.weight(codes, 1, BT, 4, s_bits[i:i + 1], lut, 0, 0)
        assert w == int(two_step[i]), i
    # and the ordinary case on a whole random matrix
    rows, cols, k = 3, 512, 3
    codes = rng.integers(0, 2 ** 32, _o.code_words(rows, cols, k), dtype=np.uint64).astype(np.uint32)
    lut = rng.standard_normal(1 << L).astype(np.float32)
    sc = torch_bf16(rng.uniform(0.01, 0.03, rows).astype(np.float32))
    w, win = o.expand(codes, rows, cols, k, sc, lut)
    want = torch_bf16(lut[win.astype(np.int64)] * _o.bf16_to_float(sc)[:, None])
    assert np.array_equal(w, want)


def check_expand_layout(o: _o.Oracle, seed: int = 13):
    """Windows of the expanded matrix follow the block addressing: row r,
    block b at word r*(C/BT)*wpb + b*wpb (interleave 0), or grouped by block
    pairs (interleave 2)."""
    rng = np.random.default_rng(seed)
    rows, cols = 3, 1024
    for k in (2, 3, 4):
        wpb = BT * k // 32
        nb = cols // BT
        codes = rng.integers(0, 2 ** 32, rows * nb * wpb, dtype=np.uint64).astype(np.uint32)
        lut = np.arange(1 << L, dtype=np.float32)
        sc = np.full(rows, 0x3F80, np.uint16)
        _, win = o.expand(codes, rows, cols, k, sc, lut)
        for r in range(rows):
            for b in range(nb):
                blk = codes[r * nb * wpb + b * wpb:][:wpb]
                for t in (0, 1, 77, 255):
                    assert win[r, b * BT + t] == window_by_string(blk, k, t)
        # interleave 2 holds the same blocks at other addresses: built here by
        # array reshaping alone, without the address formula -- view the
        # row-major codes as [row][block pair][pair member, words], move the
        # block-pair axis outermost, and flatten
        inter = np.ascontiguousarray(
            codes.reshape(rows, nb // 2, 2 * wpb).transpose(1, 0, 2)).reshape(-1)
        assert inter.size == _o.code_words(rows, cols, k, 2)
        _, win2 = o.expand(inter, rows, cols, k, sc, lut, interleave=2)
        assert np.array_equal(win, win2)


def _random_matrix(rng, rows, cols, k):
    codes = rng.integers(0, 2 ** 32, _o.code_words(rows, cols, k), dtype=np.uint64).astype(np.uint32)
    lut = rng.standard_normal(1 << L).astype(np.float32)
    sc = torch_bf16(rng.uniform(0.01, 0.03, rows).astype(np.float32))
    return codes, lut, sc


def check_contraction_vs_numpy(o: _o.Oracle, seed: int = 17):
    rng = np.random.default_rng(seed)
    rows, cols, k, M = 37, 768, 4, 6
    codes, lut, sc = _random_matrix(rng, rows, cols, k)
    w, _ = o.expand(codes, rows, cols, k, sc, lut)
    wf = _o.bf16_to_float(w).astype(np.float64)
    x1 = torch_bf16(rng.standard_normal((M, cols)).astype(np.float32))
    y, a, out = o.matmul_axis1(x1, w)
    xf = _o.bf16_to_float(x1).astype(np.float64)
    assert np.allclose(y, xf @ wf.T, rtol=1e-12, atol=1e-12)
    assert np.allclose(a, np.abs(xf) @ np.abs(wf).T, rtol=1e-12, atol=1e-12)
    for idx in np.ndindex(*y.shape):
        assert int(out[idx]) == bf16_round_fraction(Fraction(float(y[idx])))
    x0 = torch_bf16(rng.standard_normal((M, rows)).astype(np.float32))
    y0, a0, out0, part = o.matmul_axis0(x0, w, splits=5)
    x0f = _o.bf16_to_float(x0).astype(np.float64)
    assert np.allclose(y0, x0f @ wf, rtol=1e-12, atol=1e-12)
    assert np.allclose(a0, np.abs(x0f) @ np.abs(wf), rtol=1e-12, atol=1e-12)
    # split ranges: rp = ceil(37/5) = 8 -> [0,8),[8,16),[16,24),[24,32),[32,37)
    rp = -(-rows // 5)
    for s in range(5):
        r0, r1 = s * rp, min(rows, (s + 1) * rp)
        assert np.allclose(part[:, s, :], x0f[:, r0:r1] @ wf[r0:r1], rtol=1e-12, atol=1e-12)
    # splits past the end of the rows are empty
    _, _, _, part2 = o.matmul_axis0(x0[:, :3], w[:3], splits=4)
    assert np.all(part2[:, 3, :] == 0.0)


def check_unit_vectors_and_bilinear(o: _o.Oracle, seed: int = 19):
    rng = np.random.default_rng(seed)
    rows, cols, k = 9, 512, 2
    codes, lut, sc = _random_matrix(rng, rows, cols, k)
    w, _ = o.expand(codes, rows, cols, k, sc, lut)
    one = 0x3F80
    for c in (0, 1, 255, 256, 511):
        e = np.zeros((1, cols), np.uint16)
        e[0, c] = one
        _, _, out = o.matmul_axis1(e, w)
        assert np.array_equal(out[0], w[:, c])
    for r in (0, 4, 8):
        e = np.zeros((1, rows), np.uint16)
        e[0, r] = one
        _, _, out, _ = o.matmul_axis0(e, w)
        assert np.array_equal(out[0], w[r, :])
    x = torch_bf16(rng.standard_normal((1, cols)).astype(np.float32))
    u = torch_bf16(rng.standard_normal((1, rows)).astype(np.float32))
    y1, _, _ = o.matmul_axis1(x, w)
    y0, _, _, _ = o.matmul_axis0(u, w)
    lhs = float(_o.bf16_to_float(u).astype(np.float64)[0] @ y1[0])
    rhs = float(y0[0] @ _o.bf16_to_float(x).astype(np.float64)[0])
    assert abs(lhs - rhs) <= 1e-12 * max(1.0, abs(lhs))


def check_reductions(o: _o.Oracle, seed: int = 23):
    """lut = 1 and scale = 1 give out = bf16(sum x); constant windows give
    out = bf16(lut[v] * s) * sum x."""
    rng = np.random.default_rng(seed)
    rows, cols = 4, 512
    x = torch_bf16(rng.standard_normal((2, cols)).astype(np.float32))
    xs = _o.bf16_to_float(x).astype(np.float64).sum(axis=1)
    for k, (word, v) in {2: (0x55555555, 0x555), 4: (0x77777777, 0x777)}.items():
        codes = np.full(_o.code_words(rows, cols, k), word, np.uint32)
        ones = np.ones(1 << L, np.float32)
        sc1 = np.full(rows, 0x3F80, np.uint16)
        w, _ = o.expand(codes, rows, cols, k, sc1, ones)
        y, _, out = o.matmul_axis1(x, w)
        assert np.allclose(y, np.repeat(xs[:, None], rows, 1), rtol=1e-13)
        lut = rng.standard_normal(1 << L).astype(np.float32)
        sc = torch_bf16(rng.uniform(0.01, 0.03, rows).astype(np.float32))
        w, _ = o.expand(codes, rows, cols, k, sc, lut)
        wv = _o.bf16_to_float(torch_bf16(lut[v] * _o.bf16_to_float(sc))).astype(np.float64)
        y, _, _ = o.matmul_axis1(x, w)
        assert np.allclose(y, xs[:, None] * wv[None, :], rtol=1e-12)


def check_lut_readback(o: _o.Oracle, seed: int = 29):
    """lut[v] = v & 255, then v >> 8 (exact in bf16), scale 1, x = e_c: the
    contraction returns the window of column c, bit for bit."""
    rng = np.random.default_rng(seed)
    rows, cols, k = 5, 512, 3
    codes = rng.integers(0, 2 ** 32, _o.code_words(rows, cols, k), dtype=np.uint64).astype(np.uint32)
    sc = np.full(rows, 0x3F80, np.uint16)
    v = np.arange(1 << L)
    lo = (v & 255).astype(np.float32)
    hi = (v >> 8).astype(np.float32)
    w_lo, win = o.expand(codes, rows, cols, k, sc, lo)
    w_hi, _ = o.expand(codes, rows, cols, k, sc, hi)
    for c in (0, 3, 200, 256, 300, 511):
        e = np.zeros((1, cols), np.uint16)
        e[0, c] = 0x3F80
        _, _, a = o.matmul_axis1(e, w_lo)
        _, _, b = o.matmul_axis1(e, w_hi)
        got = _o.bf16_to_float(a[0]).astype(np.int64) + 256 * _o.bf16_to_float(b[0]).astype(np.int64)
        blocks = [codes[r * 2 * 24 + (c // BT) * 24:][:24] for r in range(rows)]
        want = [window_by_string(blocks[r], k, c % BT) for r in range(rows)]
        assert list(got) == want


def check_brute_force_tiny(o: _o.Oracle, seed: int = 31):
    """R in {1,3}, C in {256,512}, M in {1,5}: weights by the bit-string
    construction and PyTorch rounding, products summed exactly as rationals."""
    rng = np.random.default_rng(seed)
    for rows in (1, 3):
        for cols in (256, 512):
            for M in (1, 5):
                k = int(rng.integers(2, 5))
                wpb = BT * k // 32
                nb = cols // BT
                codes, lut, sc = _random_matrix(rng, rows, cols, k)
                W = np.empty((rows, cols), np.uint16)
                for r in range(rows):
                    s = _o.bf16_to_float(sc[r:r + 1])[0]
                    for c in range(cols):
                        blk = codes[(r * nb + c // BT) * wpb:][:wpb]
                        win = window_by_string(blk, k, c % BT)
                        W[r, c] = torch_bf16(np.array([lut[win] * s], np.float32))[0]
                w, _ = o.expand(codes, rows, cols, k, sc, lut)
                assert np.array_equal(w, W)
                x = torch_bf16(rng.standard_normal((M, cols)).astype(np.float32))
                y, _, out = o.matmul_axis1(x, w)
                xf = _o.bf16_to_float(x)
                wf = _o.bf16_to_float(W)
                for m in range(M):
                    for r in range(rows):
                        ex = sum(Fraction(float(xf[m, c])) * Fraction(float(wf[r, c]))
                                 for c in range(cols))
                        assert abs(Fraction(float(y[m, r])) - ex) <= abs(ex) * Fraction(1, 10 ** 12) + Fraction(1, 10 ** 30)
                        assert int(out[m, r]) == bf16_round_fraction(Fraction(float(y[m, r])))
                # axis 0 on the same matrix: x is [M, rows]
                x0 = torch_bf16(rng.standard_normal((M, rows)).astype(np.float32))
                y0, _, _, _ = o.matmul_axis0(x0, w)
                x0f = _o.bf16_to_float(x0)
                for m in range(M):
                    for c in (0, cols // 2, cols - 1):
                        ex = sum(Fraction(float(x0f[m, r])) * Fraction(float(wf[r, c])) for r in range(rows))
                        assert abs(Fraction(float(y0[m, c])) - ex) <= abs(ex) * Fraction(1, 10 ** 12) + Fraction(1, 10 ** 30)


def check_sampled_matches_full(o: _o.Oracle, seed: int = 37):
    rng = np.random.default_rng(seed)
    rows, cols, k, M = 20, 768, 3, 3
    codes, lut, sc = _random_matrix(rng, rows, cols, k)
    w, _ = o.expand(codes, rows, cols, k, sc, lut)
    x1 = torch_bf16(rng.standard_normal((M, cols)).astype(np.float32))
    y1, a1, _ = o.matmul_axis1(x1, w)
    ms = rng.integers(0, M, 30)
    js = rng.integers(0, rows, 30)
    ys, as_ = o.sample(x1, codes, rows, cols, k, sc, lut, 1, ms, js)
    assert np.array_equal(ys, y1[ms, js]) and np.array_equal(as_, a1[ms, js])
    x0 = torch_bf16(rng.standard_normal((M, rows)).astype(np.float32))
    y0, a0, _, _ = o.matmul_axis0(x0, w)
    js = rng.integers(0, cols, 30)
    ys, as_ = o.sample(x0, codes, rows, cols, k, sc, lut, 0, ms, js)
    assert np.array_equal(ys, y0[ms, js]) and np.array_equal(as_, a0[ms, js])


def check_glue(o: _o.Oracle, seed: int = 41):
    import torch
    rng = np.random.default_rng(seed)
    x = torch_bf16(rng.standard_normal((3, 64)).astype(np.float32) * 5)
    got = o.rmsnorm(x, 1e-6)
    xf = _o.bf16_to_float(x).astype(np.float64)
    want = xf / np.sqrt(np.mean(xf * xf, axis=1, keepdims=True) + 1e-6)
    gf = _o.bf16_to_float(got).astype(np.float64)
    assert np.all(np.abs(gf - want) <= _o.bf16_ulp(want) * 0.5 + 1e-30)
    g = torch_bf16(rng.standard_normal(500).astype(np.float32) * 3)
    u = torch_bf16(rng.standard_normal(500).astype(np.float32))
    got = _o.bf16_to_float(o.silu_mul(g, u)).astype(np.float64)
    gt = torch.from_numpy(_o.bf16_to_float(g).astype(np.float64))
    want = (torch.nn.functional.silu(gt) * torch.from_numpy(_o.bf16_to_float(u).astype(np.float64))).numpy()
    assert np.all(np.abs(got - want) <= _o.bf16_ulp(want) * 0.5 + 1e-30)


def check_unrounded_contract(o: _o.Oracle, seed: int = 43):
    """f32 weights: numpy's float32 product of lut[win] and the scale; their
    bf16 rounding is the rounded contract's weight; both contractions against
    numpy's float64 matmul."""
    rng = np.random.default_rng(seed)
    rows, cols, k, M = 13, 768, 3, 4
    codes, lut, sc = _random_matrix(rng, rows, cols, k)
    w32 = o.expand_f32(codes, rows, cols, k, sc, lut)
    w, win = o.expand(codes, rows, cols, k, sc, lut)
    want = lut[win.astype(np.int64)] * _o.bf16_to_float(sc)[:, None]      # float32 multiply
    assert want.dtype == np.float32 and np.array_equal(w32, want)
    assert np.array_equal(torch_bf16(w32), w)
    x1 = torch_bf16(rng.standard_normal((M, cols)).astype(np.float32))
    y, a, _ = o.matmul_axis1_f32w(x1, w32)
    xf = _o.bf16_to_float(x1).astype(np.float64)
    assert np.allclose(y, xf @ w32.astype(np.float64).T, rtol=1e-12, atol=1e-12)
    assert np.allclose(a, np.abs(xf) @ np.abs(w32.astype(np.float64)).T, rtol=1e-12, atol=1e-12)
    x0 = torch_bf16(rng.standard_normal((M, rows)).astype(np.float32))
    S = 6                                         # rp = 3: the last split is empty
    y0, _, _, part = o.matmul_axis0_f32w(x0, w32, S)
    x0f = _o.bf16_to_float(x0).astype(np.float64)
    assert np.allclose(y0, x0f @ w32.astype(np.float64), rtol=1e-12, atol=1e-12)
    for s in range(S):
        r0, r1 = 3 * s, min(rows, 3 * s + 3)
        want = x0f[:, r0:r1] @ w32[r0:r1].astype(np.float64) if r0 < r1 else np.zeros((M, cols))
        assert np.allclose(part[:, s, :], want, rtol=1e-12, atol=1e-12), s


def read_default_splits():
    """(rows, cols, M, splits) rows of tests/golden/default_splits.txt."""
    out = []
    with open(os.path.join(GOLDEN, "default_splits.txt")) as f:
        for line in f:
            line = line.split("#", 1)[0].split()
            if line:
                out.append(tuple(int(v) for v in line))
    return out


def check_default_splits(o: _o.Oracle):
    """The default split count of the scatter against values worked by hand
    from the split-K launcher's rule (and 128 up to 4 activation rows)."""
    for rows, cols, M, want in read_default_splits():
        assert o.scatter_default_splits(rows, cols, M) == want, (rows, cols, M)


ALL_CHECKS = [
    check_golden_windows, check_windows_random, check_single_bit_probes,
    check_wrap_and_rotation, check_special_patterns, check_bf16_rounding,
    check_weight_rounds_to_f32_first, check_expand_layout,
    check_contraction_vs_numpy, check_unit_vectors_and_bilinear,
    check_reductions, check_lut_readback, check_brute_force_tiny,
    check_sampled_matches_full, check_glue, check_unrounded_contract,
    check_default_splits,
]
