"""The C ABI on the host: the library loads, exports every entry point that
include/trellis.h declares, and rejects bad arguments with the documented
status before touching the device (CPU only: every call here returns before
any CUDA call)."""
import ctypes
import os
import re

import pytest

from trellis_coded_quantized_gb300 import _lib, geometry

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "trellis.h")

OK, NULL, GEOM, SHAPE, ALIGN, WORKSPACE = 0, 1, 2, 3, 4, 5


@pytest.fixture(scope="module")
def lib():
    from trellis_coded_quantized_gb300 import build
    build.build()
    return _lib.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(trellis_\w+)\s*\(", text)))


def test_header_and_binding_agree():
    assert declared_functions() == sorted(_lib.EXPORTS)


def test_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_strerror(lib):
    for s in range(8):
        assert lib.trellis_strerror(s)
    assert b"unknown" in lib.trellis_strerror(99)


def _p(v):
    return ctypes.c_void_p(v)


A = 0x10000     # aligned fake addresses: never dereferenced, every call below fails validation first
U = 0x10004     # 4-byte aligned only


def test_null_pointers(lib):
    g = geometry(1, 256, 512, 2)
    assert lib.trellis_matvec(None, _p(A), _p(A), _p(A), ctypes.byref(g), _p(A), None) == NULL
    assert lib.trellis_matvec(_p(A), _p(A), _p(A), _p(A), None, _p(A), None) == NULL
    assert lib.trellis_prefill(_p(A), 8, _p(A), None, _p(A), ctypes.byref(g), _p(A), None) == NULL
    g0 = geometry(0, 512, 256, 3)
    assert lib.trellis_scatter(_p(A), 1, _p(A), _p(A), _p(A), ctypes.byref(g0), 0, None, 1 << 20, _p(A), None) == NULL
    assert lib.trellis_expand(_p(A), _p(A), _p(A), ctypes.byref(g), None, None, None) == NULL
    assert lib.trellis_device_status(None) == NULL


@pytest.mark.parametrize("field,value", [("bt", 128), ("L", 11), ("k", 1), ("k", 5), ("interleave", 1),
                                         ("interleave", 3),
                                         ("cols", 300), ("cols", 0), ("rows", 0), ("axis", 2)])
def test_bad_geometry(lib, field, value):
    g = geometry(1, 256, 512, 2)
    setattr(g, field, value)
    st = lib.trellis_matvec(_p(A), _p(A), _p(A), _p(A), ctypes.byref(g), _p(A), None)
    assert st == GEOM
    assert lib.trellis_expand(_p(A), _p(A), _p(A), ctypes.byref(g), _p(A), None, None) == GEOM


def test_axis_must_match_entry_point(lib):
    g1 = geometry(1, 256, 512, 2)
    g0 = geometry(0, 256, 512, 2)
    assert lib.trellis_matvec(_p(A), _p(A), _p(A), _p(A), ctypes.byref(g0), _p(A), None) == SHAPE
    assert lib.trellis_prefill(_p(A), 8, _p(A), _p(A), _p(A), ctypes.byref(g0), _p(A), None) == SHAPE
    assert lib.trellis_scatter(_p(A), 1, _p(A), _p(A), _p(A), ctypes.byref(g1), 0, _p(A), 1 << 30, _p(A), None) == SHAPE


def test_sizes_out_of_range(lib):
    g1 = geometry(1, 256, 512, 2)
    for M in (0, 33, -1):
        assert lib.trellis_prefill(_p(A), M, _p(A), _p(A), _p(A), ctypes.byref(g1), _p(A), None) == SHAPE
    wide = geometry(1, 256, 20480 + 256, 4)
    assert lib.trellis_matvec(_p(A), _p(A), _p(A), _p(A), ctypes.byref(wide), _p(A), None) == SHAPE
    g0 = geometry(0, 512, 256, 3)
    for M, s in ((0, 0), (33, 0), (1, -1), (1, 1025)):
        assert lib.trellis_scatter(_p(A), M, _p(A), _p(A), _p(A), ctypes.byref(g0), s, _p(A), 1 << 30, _p(A), None) == SHAPE


def test_misaligned(lib):
    g1 = geometry(1, 256, 512, 2)
    assert lib.trellis_matvec(_p(U), _p(A), _p(A), _p(A), ctypes.byref(g1), _p(A), None) == ALIGN
    assert lib.trellis_matvec(_p(A), _p(U), _p(A), _p(A), ctypes.byref(g1), _p(A), None) == ALIGN
    assert lib.trellis_prefill(_p(A), 5, _p(U), _p(A), _p(A), ctypes.byref(g1), _p(A), None) == ALIGN
    g0 = geometry(0, 512, 256, 3)
    assert lib.trellis_scatter(_p(A), 1, _p(A), _p(A), _p(A), ctypes.byref(g0), 0, _p(U), 1 << 30, _p(A), None) == ALIGN


def _fix(M, unrounded=False):
    """Bytes of the tensor-core scatter's fix-up slots (3+ rows, rounded)."""
    return 160 * M * 256 * 4 if M >= 3 and not unrounded else 0


def test_workspace_size(lib):
    g0 = geometry(0, 17408, 5120, 3)
    assert lib.trellis_scatter_workspace_bytes(ctypes.byref(g0), 1, 0) == 1 * 128 * 5120 * 4
    assert lib.trellis_scatter_workspace_bytes(ctypes.byref(g0), 2, 0) == 2 * 128 * 5120 * 4
    assert lib.trellis_scatter_workspace_bytes(ctypes.byref(g0), 4, 64) == 4 * 64 * 5120 * 4 + _fix(4)
    gu = geometry(0, 17408, 5120, 3, unrounded=True)
    assert lib.trellis_scatter_workspace_bytes(ctypes.byref(gu), 4, 64) == 4 * 64 * 5120 * 4
    assert lib.trellis_scatter_workspace_bytes(ctypes.byref(g0), 0, 0) == 0
    bad = geometry(0, 17408, 5000, 3)
    assert lib.trellis_scatter_workspace_bytes(ctypes.byref(bad), 1, 0) == 0
    need = 1 * 128 * 5120 * 4
    assert lib.trellis_scatter(_p(A), 1, _p(A), _p(A), _p(A), ctypes.byref(g0), 0, _p(A), need - 4, _p(A), None) == WORKSPACE


def test_default_split_count(lib):
    """splits = 0: 128 up to 4 activation rows, else the split-K launcher's
    rule (the hand-worked values of tests/golden/default_splits.txt); 128 at
    every M under the unrounded contract."""
    import pins
    for rows, cols, M, want in pins.read_default_splits():
        g0 = geometry(0, rows, cols, 3)
        assert lib.trellis_scatter_workspace_bytes(ctypes.byref(g0), M, 0) == M * want * cols * 4 + _fix(M), \
            (rows, cols, M)
    g0 = geometry(0, 17408, 5120, 3)
    assert lib.trellis_scatter_workspace_bytes(ctypes.byref(g0), 4, 0) == 4 * 128 * 5120 * 4 + _fix(4)
    assert lib.trellis_scatter_workspace_bytes(ctypes.byref(g0), 8, 0) == 8 * 8 * 5120 * 4 + _fix(8)
    # the unrounded contract keeps scatter.ts's 128 ranges at every M
    gu = geometry(0, 17408, 5120, 3, unrounded=True)
    for M in (1, 4, 5, 8, 32):
        assert lib.trellis_scatter_workspace_bytes(ctypes.byref(gu), M, 0) == M * 128 * 5120 * 4, M


def test_glue_validation(lib):
    assert lib.trellis_rmsnorm(None, 1, 16, ctypes.c_float(1e-6), _p(A), None) == NULL
    assert lib.trellis_rmsnorm(_p(A), 1, 70000, ctypes.c_float(1e-6), _p(A), None) == SHAPE
    assert lib.trellis_silu_mul(_p(A), _p(A), 0, _p(A), None) == SHAPE
    assert lib.trellis_gather_probe(_p(A), 0, 1, 1, _p(A), None) == SHAPE
    assert lib.trellis_gather_probe(_p(A), 1, 1, 3, _p(A), None) == SHAPE
    assert lib.trellis_gather_probe(_p(U), 1, 1, 1, _p(A), None) == ALIGN


def test_interleave_two_needs_an_even_block_count(lib):
    g = geometry(1, 256, 768, 2, interleave=2)      # 3 blocks
    assert lib.trellis_matvec(_p(A), _p(A), _p(A), _p(A), ctypes.byref(g), _p(A), None) == GEOM
    g = geometry(1, 256, 512, 2, interleave=2)      # 2 blocks: passes validation up to alignment
    assert lib.trellis_matvec(_p(U), _p(A), _p(A), _p(A), ctypes.byref(g), _p(A), None) == ALIGN


def test_unrounded_flag_only_where_the_call_takes_it(lib):
    g1 = geometry(1, 256, 512, 2, unrounded=True)
    g0 = geometry(0, 512, 256, 3, unrounded=True)
    # taken: validation goes on to the pointers (misaligned x -> ALIGN)
    assert lib.trellis_matvec(_p(U), _p(A), _p(A), _p(A), ctypes.byref(g1), _p(A), None) == ALIGN
    assert lib.trellis_scatter(_p(U), 1, _p(A), _p(A), _p(A), ctypes.byref(g0), 0, _p(A), 1 << 30, _p(A), None) == ALIGN
    assert lib.trellis_scatter_workspace_bytes(ctypes.byref(g0), 1, 0) == 128 * 256 * 4
    # refused: the tensor-core prefill and the bf16 expansion
    assert lib.trellis_prefill(_p(A), 8, _p(A), _p(A), _p(A), ctypes.byref(g1), _p(A), None) == GEOM
    assert lib.trellis_expand(_p(A), _p(A), _p(A), ctypes.byref(g1), _p(A), None, None) == GEOM
    # unknown bits
    for flags in (2, 3, 1 << 30, -1):
        g = geometry(1, 256, 512, 2)
        g.flags = flags
        assert lib.trellis_matvec(_p(A), _p(A), _p(A), _p(A), ctypes.byref(g), _p(A), None) == GEOM


def test_gate_up_validation(lib):
    g1 = geometry(1, 256, 512, 2)
    g0 = geometry(0, 256, 512, 2)
    f = lib.trellis_gate_up_matvec
    assert f(_p(A), _p(A), _p(A), None, _p(A), _p(A), ctypes.byref(g1), _p(A), None) == NULL
    assert f(_p(A), _p(A), _p(A), _p(A), _p(A), _p(A), ctypes.byref(g0), _p(A), None) == SHAPE
    assert f(_p(A), _p(A), _p(A), _p(U), _p(A), _p(A), ctypes.byref(g1), _p(A), None) == ALIGN
    wide = geometry(1, 256, 20480 + 256, 4)
    assert f(_p(A), _p(A), _p(A), _p(A), _p(A), _p(A), ctypes.byref(wide), _p(A), None) == SHAPE
    gu = geometry(1, 256, 512, 2, unrounded=True)
    assert f(_p(U), _p(A), _p(A), _p(A), _p(A), _p(A), ctypes.byref(gu), _p(A), None) == ALIGN


def test_gate_up_prefill_validation(lib):
    g1 = geometry(1, 256, 512, 2)
    g0 = geometry(0, 256, 512, 2)
    f = lib.trellis_gate_up_prefill
    assert f(_p(A), 8, _p(A), _p(A), None, _p(A), _p(A), ctypes.byref(g1), _p(A), None) == NULL
    assert f(_p(A), 8, _p(A), _p(A), _p(A), _p(A), _p(A), ctypes.byref(g0), _p(A), None) == SHAPE
    for M in (0, 33):
        assert f(_p(A), M, _p(A), _p(A), _p(A), _p(A), _p(A), ctypes.byref(g1), _p(A), None) == SHAPE
    assert f(_p(A), 8, _p(A), _p(A), _p(U), _p(A), _p(A), ctypes.byref(g1), _p(A), None) == ALIGN
    assert f(_p(U), 8, _p(A), _p(A), _p(A), _p(A), _p(A), ctypes.byref(g1), _p(A), None) == ALIGN
    gu = geometry(1, 256, 512, 2, unrounded=True)
    assert f(_p(A), 8, _p(A), _p(A), _p(A), _p(A), _p(A), ctypes.byref(gu), _p(A), None) == GEOM


def test_kv_decode_validation(lib):
    from trellis_coded_quantized_gb300 import kv_geometry
    f, fi = lib.trellis_kv_decode, lib.trellis_kv_decode_inverse256
    g = kv_geometry(8, 256, 8, 3)
    args = [_p(A)] * 6
    assert f(None, *args[1:], ctypes.byref(g), _p(A), _p(A), None) == NULL
    assert f(*args, None, _p(A), _p(A), None) == NULL
    assert fi(*args, None, ctypes.byref(g), _p(A), _p(A), None) == NULL
    for field, value in (("rows", 0), ("head_dim", 96), ("key_bits", 3), ("value_bits", 6), ("key_group", 16),
                         ("value_group", 128), ("key_scale_dtype", 3), ("value_out_bf16", 2)):
        bad = kv_geometry(8, 256, 8, 3)
        setattr(bad, field, value)
        assert f(*args, ctypes.byref(bad), _p(A), _p(A), None) == GEOM, field
    assert f(_p(U), *args[1:], ctypes.byref(g), _p(A), _p(A), None) == ALIGN
    assert f(*args, ctypes.byref(g), _p(A), _p(U), None) == ALIGN
    odd = [_p(A), _p(A + 1)] + args[2:]                       # f16 scales at an odd address
    assert f(*odd, ctypes.byref(g), _p(A), _p(A), None) == ALIGN
    # the inverse takes only the pages' regime, with bf16 values
    assert fi(*args, _p(A), ctypes.byref(g), _p(A), _p(A), None) == GEOM
    for field, value in (("head_dim", 128), ("key_bits", 4), ("value_bits", 2), ("key_group", 64)):
        bad = kv_geometry(8, 256, 8, 3, value_out_bf16=True)
        setattr(bad, field, value)
        assert fi(*args, _p(A), ctypes.byref(bad), _p(A), _p(A), None) == GEOM, field
    gb = kv_geometry(8, 256, 8, 3, value_out_bf16=True)
    assert fi(*args, _p(A + 2), ctypes.byref(gb), _p(A), _p(A), None) == ALIGN


def test_product_path_never_uses_the_oracle():
    """The package and its CUDA sources neither import, include, link nor call
    the oracle (it is test infrastructure only)."""
    pkg = os.path.join(ROOT, "trellis_coded_quantized_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if not f.endswith((".py", ".cu", ".cuh", ".h")):
                continue
            text = open(os.path.join(dirpath, f)).read()
            assert not re.search(r"^\s*(import|from)\s+oracle\b", text, re.M), f
            assert "tcq_oracle" not in text and "liboracle" not in text, f
