"""trellis_gate_up_matvec (gate and up projections plus the SiLU gate in one
launch) through the C ABI.

The fused kernel computes each row sum exactly as trellis_matvec does (same
per-thread sums, same butterfly, same warp order), so its output must equal,
bit for bit, trellis_silu_mul applied to two trellis_matvec outputs.  Those
are checked against the oracle too: the projections within the contraction
tolerance, h within one bf16 ulp of the oracle's silu(g) * u.
"""
import numpy as np
import pytest

import trellis_coded_quantized_gb300 as tcq
from trellis_coded_quantized_gb300 import synth
from gpu_util import check_close, dev, host_bf16
from conftest import has_gpu

pytestmark = [pytest.mark.gpu, pytest.mark.skipif(not has_gpu(), reason="needs a CUDA GPU")]


@pytest.fixture(scope="module", autouse=True)
def _built():
    from trellis_coded_quantized_gb300 import build
    build.build()


def _inter(codes, rows, cols, k):
    wpb = 256 * k // 32
    c = codes.reshape(rows, cols // 512, 2 * wpb)
    return np.ascontiguousarray(c.transpose(1, 0, 2)).reshape(rows, -1)


def _ulps(a, b):
    from oracle import bf16_to_float, bf16_ulp
    fa, fb = bf16_to_float(a).astype(np.float64), bf16_to_float(b).astype(np.float64)
    return np.abs(fa - fb) / bf16_ulp(np.maximum(np.abs(fa), np.abs(fb)))


@pytest.mark.parametrize("rows,cols,k,interleave,unrounded", [
    (17408, 5120, 3, 0, False),      # the MLP layer's gate/up geometry
    (17408, 5120, 4, 0, True),
    (1, 256, 2, 0, False),           # one pair
    (37, 512, 2, 0, False),          # 20 row groups per CTA
    (1000, 2304, 4, 0, False),       # 6 row groups
    (153, 20480, 3, 0, True),        # one row group; one or two row pairs per CTA
    (300, 1024, 2, 2, False),
    (611, 2560, 3, 2, True),
])
def test_gate_up_equals_matvecs_then_silu(orc, rows, cols, k, interleave, unrounded):
    pg = synth.problem(1, 1, rows, cols, k, seed=31)
    pu = synth.problem(1, 1, rows, cols, k, seed=32)
    lut = pg["lut"]                          # one codebook for both matrices
    cg, cu = pg["codes"], pu["codes"]
    if interleave == 2:
        cg, cu = _inter(cg, rows, cols, k), _inter(cu, rows, cols, k)
    g = tcq.geometry(1, rows, cols, k, interleave, unrounded=unrounded)
    x = dev(pg["x"])[0]
    dcg, dsg, dcu, dsu, dl = dev(cg), dev(pg["scales"]), dev(cu), dev(pu["scales"]), dev(lut)
    h = tcq.trellis_gate_up_matvec(x, dcg, dsg, dcu, dsu, dl, g)
    gate = tcq.trellis_matvec(x, dcg, dsg, dl, g)
    up = tcq.trellis_matvec(x, dcu, dsu, dl, g)
    h_chain = tcq.trellis_silu_mul(gate, up)
    assert np.array_equal(host_bf16(h), host_bf16(h_chain)), "fused output differs from matvec, matvec, silu_mul"
    # the chain against the oracle
    xs = pg["x"]
    for p, got in ((pg, gate), (pu, up)):
        if unrounded:
            w = orc.expand_f32(p["codes"], rows, cols, k, p["scales"], lut)
            y, a, _ = orc.matmul_axis1_f32w(xs, w)
        else:
            w, _ = orc.expand(p["codes"], rows, cols, k, p["scales"], lut)
            y, a, _ = orc.matmul_axis1(xs, w)
        check_close(orc, host_bf16(got)[None, :], y, a, f"gate/up projection {rows}x{cols} k={k}")
    ref = orc.silu_mul(host_bf16(gate)[None, :], host_bf16(up)[None, :])[0]
    assert np.all(_ulps(host_bf16(h), ref) <= 1.0)


def test_gate_up_errors():
    p = synth.problem(1, 1, 256, 512, 2, seed=33)
    g1 = tcq.geometry(1, 256, 512, 2)
    g0 = tcq.geometry(0, 256, 512, 2)
    x, c, s, l = dev(p["x"])[0], dev(p["codes"]), dev(p["scales"]), dev(p["lut"])
    with pytest.raises(tcq.TrellisError) as e:
        tcq.trellis_gate_up_matvec(x, c, s, c, s, l, g0)
    assert e.value.status == 3
    wide = tcq.geometry(1, 4, 20480 + 256, 2)
    big = dev(synth.codes(1, 4, 20480 + 256, 2))
    ws = dev(synth.scales(1, 4))
    xw = dev(synth.activations(1, 1, 20480 + 256))[0]
    with pytest.raises(tcq.TrellisError) as e:
        tcq.trellis_gate_up_matvec(xw, big, ws, big, ws, l, wide)
    assert e.value.status == 3
    assert tcq.trellis_gate_up_matvec(x, c, s, c, s, l, g1).shape == (256,)


@pytest.mark.parametrize("M,rows,cols,k,interleave", [
    (16, 17408, 5120, 3, 0),         # the MLP layer's gate/up geometry at M = 16
    (32, 17408, 5120, 4, 0),
    (5, 17408, 5120, 2, 0),
    (2, 300, 1024, 2, 2),            # two CTAs of 128 rows and a ragged one
    (17, 1000, 2304, 4, 0),          # N = 32, 9 column blocks, ragged rows
    (1, 129, 512, 3, 0),             # one row past a 128-row tile
    (32, 37, 256, 2, 0),             # one block, one partial tile
])
def test_gate_up_prefill_equals_prefills_then_silu(orc, M, rows, cols, k, interleave):
    """trellis_gate_up_prefill is bit for bit trellis_prefill twice and
    trellis_silu_mul; the chain's projections agree with the oracle."""
    pg = synth.problem(1, M, rows, cols, k, seed=41)
    pu = synth.problem(1, M, rows, cols, k, seed=42)
    lut = pg["lut"]
    cg, cu = pg["codes"], pu["codes"]
    if interleave == 2:
        cg, cu = _inter(cg, rows, cols, k), _inter(cu, rows, cols, k)
    g = tcq.geometry(1, rows, cols, k, interleave)
    x = dev(pg["x"])
    dcg, dsg, dcu, dsu, dl = dev(cg), dev(pg["scales"]), dev(cu), dev(pu["scales"]), dev(lut)
    h = tcq.trellis_gate_up_prefill(x, dcg, dsg, dcu, dsu, dl, g)
    gate = tcq.trellis_prefill(x, dcg, dsg, dl, g)
    up = tcq.trellis_prefill(x, dcu, dsu, dl, g)
    h_chain = tcq.trellis_silu_mul(gate, up)
    assert h.shape == (M, rows)
    assert np.array_equal(host_bf16(h), host_bf16(h_chain)), "fused output differs from prefill, prefill, silu_mul"
    assert tcq.trellis_device_status() == 0
    if rows * cols <= 2304 * 1000:       # the oracle on the small geometries
        for p, got in ((pg, gate), (pu, up)):
            w, _ = orc.expand(p["codes"], rows, cols, k, p["scales"], lut)
            y, a, _ = orc.matmul_axis1(pg["x"], w)
            check_close(orc, host_bf16(got), y, a, f"gate/up prefill projection {rows}x{cols} k={k} M={M}")
        ref = orc.silu_mul(host_bf16(gate), host_bf16(up))
        assert np.all(_ulps(host_bf16(h), ref) <= 1.0)


def test_gate_up_prefill_errors():
    p = synth.problem(1, 4, 256, 512, 2, seed=43)
    g0 = tcq.geometry(0, 256, 512, 2)
    gu = tcq.geometry(1, 256, 512, 2, unrounded=True)
    x, c, s, l = dev(p["x"]), dev(p["codes"]), dev(p["scales"]), dev(p["lut"])
    with pytest.raises(tcq.TrellisError) as e:
        tcq.trellis_gate_up_prefill(x, c, s, c, s, l, g0)
    assert e.value.status == 3
    with pytest.raises(tcq.TrellisError) as e:
        tcq.trellis_gate_up_prefill(x, c, s, c, s, l, gu)
    assert e.value.status == 2
