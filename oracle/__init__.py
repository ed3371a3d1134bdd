"""CPU oracle for the packed trellis-coded weight matmul.

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package; the product path
(``trellis_coded_quantized_gb300`` and ``libtrellis``) never does.

This module is a thin numpy wrapper around ``tcq_oracle.c`` (plain C, double
precision), which restates the method from its definition; that file's header
lists the steps and the pages they come from.  Arrays of bf16 values are
carried as ``uint16`` bit patterns.

``Oracle(path)`` binds the wrapper to one compiled library; the module-level
functions use the default build next to this file.  Tests that plant a
mistake in the oracle compile a mutated copy of the C source into a temporary
library and bind an ``Oracle`` to it.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
SOURCE = os.path.join(_HERE, "tcq_oracle.c")
LIB_PATH = os.path.join(_HERE, "liboracle.so")

BT = 256
L = 12

GCC_FLAGS = ["-O2", "-fPIC", "-shared", "-fopenmp", "-ffp-contract=off",
             "-fno-fast-math", "-frounding-math", "-std=c11"]


def compile_library(src: str, out: str) -> str:
    """gcc ``src`` into the shared library ``out`` (atomic replace)."""
    tmp = out + f".tmp{os.getpid()}"
    subprocess.run(["gcc", *GCC_FLAGS, src, "-o", tmp, "-lm"], check=True)
    os.replace(tmp, out)
    return out


def build(force: bool = False) -> str:
    """Compile ``tcq_oracle.c`` into ``liboracle.so`` if it is missing or stale."""
    if force or not os.path.exists(LIB_PATH) or os.path.getmtime(LIB_PATH) < os.path.getmtime(SOURCE):
        compile_library(SOURCE, LIB_PATH)
    return LIB_PATH


def _c(a, dtype) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=dtype)


def _ptr(a):
    return None if a is None else ctypes.c_void_p(a.ctypes.data)


def words_per_block(k: int, bt: int = BT) -> int:
    return bt * k // 32


def code_words(rows: int, cols: int, k: int, interleave: int = 0, bt: int = BT) -> int:
    """Number of uint32 words of a packed matrix."""
    nb = cols // bt
    wpb = words_per_block(k, bt)
    if interleave == 2:
        return ((nb + 1) // 2) * rows * 2 * wpb
    return rows * nb * wpb


def bf16_to_float(h) -> np.ndarray:
    """bf16 bits -> float32 (exact: the upper half of a binary32 pattern)."""
    h = _c(h, np.uint16)
    return (h.astype(np.uint32) << np.uint32(16)).view(np.float32)


def bf16_ulp(v) -> np.ndarray:
    """Spacing of bf16 values at the magnitude of each finite value."""
    v = np.abs(np.asarray(v, np.float64))
    e = np.floor(np.log2(np.where(v > 0, v, 1.0)))
    e = np.maximum(e, -126.0)
    return np.where(v > 0, np.ldexp(1.0, (e - 7).astype(np.int64)), np.ldexp(1.0, -133))


class Oracle:
    """The oracle's entry points bound to one compiled library."""

    def __init__(self, path: str):
        lib = ctypes.CDLL(path)
        P, I64, I = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
        lib.tcq_oracle_set_threads.argtypes = [I]
        lib.tcq_oracle_max_threads.restype = I
        lib.tcq_oracle_bf16_from_double_n.argtypes = [P, I64, P]
        lib.tcq_oracle_bf16_from_float_n.argtypes = [P, I64, P]
        lib.tcq_oracle_window.argtypes = [P, I, I, I, I]
        lib.tcq_oracle_window.restype = ctypes.c_uint32
        lib.tcq_oracle_weight.argtypes = [P, I64, I64, I, I, I, I, P, P, I64, I64]
        lib.tcq_oracle_weight.restype = ctypes.c_uint16
        lib.tcq_oracle_expand.argtypes = [P, I64, I64, I, I, I, I, P, P, P, P]
        lib.tcq_oracle_matmul_axis1.argtypes = [P, I64, P, I64, I64, P, P, P]
        lib.tcq_oracle_matmul_axis0.argtypes = [P, I64, P, I64, I64, I64, P, P, P, P]
        lib.tcq_oracle_sample.argtypes = [P, I64, P, I64, I64, I, I, I, I, I, P, P, P, P, I64, P, P]
        lib.tcq_oracle_expand_f32.argtypes = [P, I64, I64, I, I, I, I, P, P, P]
        lib.tcq_oracle_matmul_axis1_f32w.argtypes = [P, I64, P, I64, I64, P, P, P]
        lib.tcq_oracle_matmul_axis0_f32w.argtypes = [P, I64, P, I64, I64, I64, P, P, P, P]
        lib.tcq_oracle_rmsnorm.argtypes = [P, I64, I64, ctypes.c_double, P]
        lib.tcq_oracle_silu_mul.argtypes = [P, P, I64, P]
        lib.tcq_oracle_scatter_default_splits.argtypes = [I64, I64, I64]
        lib.tcq_oracle_scatter_default_splits.restype = I64
        self.lib = lib
        self.path = path

    # -- threads -------------------------------------------------------------
    def set_threads(self, n: int) -> None:
        self.lib.tcq_oracle_set_threads(int(n))

    def max_threads(self) -> int:
        return int(self.lib.tcq_oracle_max_threads())

    # -- bf16 ----------------------------------------------------------------
    def bf16_from_double(self, y) -> np.ndarray:
        y = _c(y, np.float64)
        out = np.empty(y.shape, np.uint16)
        self.lib.tcq_oracle_bf16_from_double_n(_ptr(y), y.size, _ptr(out))
        return out

    def bf16_from_float(self, y) -> np.ndarray:
        y = _c(y, np.float32)
        out = np.empty(y.shape, np.uint16)
        self.lib.tcq_oracle_bf16_from_float_n(_ptr(y), y.size, _ptr(out))
        return out

    # -- windows and weights -------------------------------------------------
    def window(self, block_words, k: int, t: int, bt: int = BT, l: int = L) -> int:
        w = _c(block_words, np.uint32)
        assert w.size == words_per_block(k, bt)
        return int(self.lib.tcq_oracle_window(_ptr(w), bt, k, l, int(t)))

    def expand(self, codes, rows: int, cols: int, k: int, scales, lut, interleave: int = 0,
               bt: int = BT, l: int = L):
        """Decode the packed matrix: (w bf16 bits [rows, cols], windows u16 [rows, cols])."""
        codes = _c(codes, np.uint32)
        scales = _c(scales, np.uint16)
        lut = _c(lut, np.float32)
        assert codes.size == code_words(rows, cols, k, interleave, bt)
        assert scales.size == rows and lut.size == (1 << l)
        w = np.empty((rows, cols), np.uint16)
        win = np.empty((rows, cols), np.uint16)
        self.lib.tcq_oracle_expand(_ptr(codes), rows, cols, bt, k, l, interleave,
                                   _ptr(scales), _ptr(lut), _ptr(w), _ptr(win))
        return w, win

    def weight(self, codes, rows: int, cols: int, k: int, scales, lut, r: int, c: int,
               interleave: int = 0, bt: int = BT, l: int = L) -> int:
        codes = _c(codes, np.uint32)
        scales = _c(scales, np.uint16)
        lut = _c(lut, np.float32)
        return int(self.lib.tcq_oracle_weight(_ptr(codes), rows, cols, bt, k, l, interleave,
                                              _ptr(scales), _ptr(lut), int(r), int(c)))

    # -- contractions --------------------------------------------------------
    def matmul_axis1(self, x, w):
        """x bf16 [M, K], w bf16 [N, K] -> (y f64 [M, N], a f64 [M, N], out bf16 [M, N])."""
        x = _c(x, np.uint16)
        w = _c(w, np.uint16)
        M, K = x.shape
        N, K2 = w.shape
        assert K == K2
        y = np.empty((M, N), np.float64)
        a = np.empty((M, N), np.float64)
        out = np.empty((M, N), np.uint16)
        self.lib.tcq_oracle_matmul_axis1(_ptr(x), M, _ptr(w), N, K, _ptr(y), _ptr(a), _ptr(out))
        return y, a, out

    def matmul_axis0(self, x, w, splits: int = 0):
        """x bf16 [M, R], w bf16 [R, C] -> (y, a, out [M, C], partial f64 [M, splits, C] | None)."""
        x = _c(x, np.uint16)
        w = _c(w, np.uint16)
        M, R = x.shape
        R2, C = w.shape
        assert R == R2
        y = np.empty((M, C), np.float64)
        a = np.empty((M, C), np.float64)
        out = np.empty((M, C), np.uint16)
        part = np.empty((M, splits, C), np.float64) if splits > 0 else None
        self.lib.tcq_oracle_matmul_axis0(_ptr(x), M, _ptr(w), R, C, int(splits),
                                         _ptr(y), _ptr(a), _ptr(out), _ptr(part))
        return y, a, out, part

    def sample(self, x, codes, rows: int, cols: int, k: int, scales, lut, axis: int, ms, js,
               interleave: int = 0, bt: int = BT, l: int = L):
        """Outputs (m, j) of the packed matmul computed one by one from the codes."""
        x = _c(x, np.uint16)
        codes = _c(codes, np.uint32)
        scales = _c(scales, np.uint16)
        lut = _c(lut, np.float32)
        ms = _c(ms, np.int64)
        js = _c(js, np.int64)
        n = ms.size
        y = np.empty(n, np.float64)
        a = np.empty(n, np.float64)
        self.lib.tcq_oracle_sample(_ptr(x), x.shape[0], _ptr(codes), rows, cols, bt, k, l,
                                   interleave, axis, _ptr(scales), _ptr(lut),
                                   _ptr(ms), _ptr(js), n, _ptr(y), _ptr(a))
        return y, a

    # -- the unrounded contract ----------------------------------------------
    def expand_f32(self, codes, rows: int, cols: int, k: int, scales, lut, interleave: int = 0,
                   bt: int = BT, l: int = L):
        """Weights of the unrounded contract: f32(lut[win] * scale), float32 [rows, cols]."""
        codes = _c(codes, np.uint32)
        scales = _c(scales, np.uint16)
        lut = _c(lut, np.float32)
        assert codes.size == code_words(rows, cols, k, interleave, bt)
        w = np.empty((rows, cols), np.float32)
        self.lib.tcq_oracle_expand_f32(_ptr(codes), rows, cols, bt, k, l, interleave,
                                       _ptr(scales), _ptr(lut), _ptr(w))
        return w

    def matmul_axis1_f32w(self, x, w):
        x = _c(x, np.uint16)
        w = _c(w, np.float32)
        M, K = x.shape
        N, K2 = w.shape
        assert K == K2
        y = np.empty((M, N), np.float64)
        a = np.empty((M, N), np.float64)
        out = np.empty((M, N), np.uint16)
        self.lib.tcq_oracle_matmul_axis1_f32w(_ptr(x), M, _ptr(w), N, K, _ptr(y), _ptr(a), _ptr(out))
        return y, a, out

    def matmul_axis0_f32w(self, x, w, splits: int = 0):
        """x bf16 [M, R], w f32 [R, C] -> (y, a, out [M, C], partial f64 [M, splits, C] | None)."""
        x = _c(x, np.uint16)
        w = _c(w, np.float32)
        M, R = x.shape
        R2, C = w.shape
        assert R == R2
        y = np.empty((M, C), np.float64)
        a = np.empty((M, C), np.float64)
        out = np.empty((M, C), np.uint16)
        part = np.empty((M, splits, C), np.float64) if splits > 0 else None
        self.lib.tcq_oracle_matmul_axis0_f32w(_ptr(x), M, _ptr(w), R, C, int(splits),
                                              _ptr(y), _ptr(a), _ptr(out), _ptr(part))
        return y, a, out, part

    # -- glue of the synthetic MLP stack -------------------------------------
    def rmsnorm(self, x, eps: float = 1e-6):
        x = _c(x, np.uint16)
        M, D = x.shape
        out = np.empty_like(x)
        self.lib.tcq_oracle_rmsnorm(_ptr(x), M, D, float(eps), _ptr(out))
        return out

    def silu_mul(self, g, u):
        g = _c(g, np.uint16)
        u = _c(u, np.uint16)
        assert g.shape == u.shape
        out = np.empty_like(g)
        self.lib.tcq_oracle_silu_mul(_ptr(g), _ptr(u), g.size, _ptr(out))
        return out

    # -- split count ----------------------------------------------------------
    def scatter_default_splits(self, rows: int, cols: int, M: int) -> int:
        """Row splits of the axis-0 scatter when the caller gives none."""
        return int(self.lib.tcq_oracle_scatter_default_splits(rows, cols, M))

    # -- the tolerance of the contraction ------------------------------------
    def within_tolerance(self, got_bf16, y, a, rel: float = 4e-3):
        """|got - y| <= rel * a + 1 bf16 ulp of the oracle's rounded output."""
        got = bf16_to_float(got_bf16).astype(np.float64)
        ref = bf16_to_float(self.bf16_from_double(y)).astype(np.float64)
        bound = rel * np.asarray(a, np.float64) + bf16_ulp(ref)
        err = np.abs(got - np.asarray(y, np.float64))
        return err <= bound, err, bound


_default = None
_lock = threading.Lock()


def default() -> Oracle:
    global _default
    with _lock:
        if _default is None:
            _default = Oracle(build())
        return _default


def __getattr__(name):
    # module-level access to the default oracle's methods: oracle.expand(...)
    if name in Oracle.__dict__ and not name.startswith("_"):
        return getattr(default(), name)
    raise AttributeError(name)
