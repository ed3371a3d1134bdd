"""CUDA path (through the C ABI) against the oracle, element by element.

Decoded windows and weights must be bit-exact; contractions must satisfy
|gpu - y| <= 4e-3 * sum|x*w| + 1 bf16 ulp per element (y, sum|x*w| from the
oracle in double).  Probes with unit vectors and integer codebooks must come
back bit-exact through every fused kernel.
"""
import numpy as np
import pytest

import trellis_coded_quantized_gb300 as tcq
from trellis_coded_quantized_gb300 import synth
from gpu_util import check_close, dev, host_bf16, on_device
from conftest import has_gpu

pytestmark = [pytest.mark.gpu, pytest.mark.skipif(not has_gpu(), reason="needs a CUDA GPU")]

ONE = 0x3F80  # bf16 1.0


@pytest.fixture(scope="module", autouse=True)
def _built():
    from trellis_coded_quantized_gb300 import build
    build.build()


def _oracle_axis1(orc, p):
    W, _ = orc.expand(p["codes"], p["rows"], p["cols"], p["k"], p["scales"], p["lut"])
    y, a, _ = orc.matmul_axis1(p["x"], W)
    return W, y, a


def _oracle_axis0(orc, p, splits=0):
    W, _ = orc.expand(p["codes"], p["rows"], p["cols"], p["k"], p["scales"], p["lut"])
    y, a, _, part = orc.matmul_axis0(p["x"], W, splits)
    return W, y, a, part


# ----------------------------------------------------------------- expand

@pytest.mark.parametrize("axis,rows,cols,k", [
    (1, 256, 512, 2),        # tiny matvec geometry
    (1, 17408, 5120, 4),     # decode matvec geometry
    (1, 17408, 5120, 2),     # prefill geometries
    (1, 17408, 5120, 3),
    (0, 17408, 5120, 3),     # axis-0 scatter geometry
    (1, 1, 256, 4),          # one block, one row
    (0, 37, 768, 3),         # ragged rows, odd block count
])
def test_expand_bit_exact(orc, axis, rows, cols, k):
    p = synth.problem(axis, 1, rows, cols, k, seed=0)
    d = on_device(p)
    w, win = tcq.trellis_expand(d["codes"], d["scales"], d["lut"], d["g"], with_windows=True)
    ow, owin = orc.expand(p["codes"], rows, cols, k, p["scales"], p["lut"])
    assert np.array_equal(host_bf16(win), owin), "windows differ"
    assert np.array_equal(host_bf16(w), ow), "decoded weights differ"


# ----------------------------------------------------------------- matvec

@pytest.mark.parametrize("rows,cols,k", [
    (256, 512, 2),           # tiny axis-1 matvec, seed 0
    (17408, 5120, 4),        # decode matvec, full size
    (17408, 5120, 3),
    (17408, 5120, 2),
    (1, 256, 4), (3, 256, 3), (37, 768, 2), (1000, 1280, 3),
    (4099, 20480, 4),        # widest input the kernel takes
    (152 * 3 + 5, 2304, 2),  # rows not a multiple of the grid
])
def test_matvec(orc, rows, cols, k):
    p = synth.problem(1, 1, rows, cols, k, seed=0)
    d = on_device(p)
    out = tcq.trellis_matvec(d["x"][0], d["codes"], d["scales"], d["lut"], d["g"])
    _, y, a = _oracle_axis1(orc, p)
    check_close(orc, host_bf16(out)[None, :], y, a, f"matvec {rows}x{cols} k={k}")


@pytest.mark.parametrize("k", [2, 3, 4])
def test_matvec_unit_vectors_exact(orc, k):
    rows, cols = 300, 1024
    p = synth.problem(1, 1, rows, cols, k, seed=3)
    d = on_device(p)
    W, _ = orc.expand(p["codes"], rows, cols, k, p["scales"], p["lut"])
    for c in (0, 1, 2, 127, 255, 256, 511, 1023):
        e = np.zeros(cols, np.uint16)
        e[c] = ONE
        out = tcq.trellis_matvec(dev(e), d["codes"], d["scales"], d["lut"], d["g"])
        assert np.array_equal(host_bf16(out), W[:, c]), c


@pytest.mark.parametrize("k", [2, 3, 4])
def test_matvec_lut_readback_exact(orc, k):
    """lut[v] = v & 255 and v >> 8 with unit scales return every window."""
    rows, cols = 200, 768
    p = synth.problem(1, 1, rows, cols, k, seed=4)
    _, win = orc.expand(p["codes"], rows, cols, k, p["scales"], p["lut"])
    v = np.arange(4096)
    d = on_device(p)
    sc1 = dev(np.full(rows, ONE, np.uint16))
    lo, hi = dev((v & 255).astype(np.float32)), dev((v >> 8).astype(np.float32))
    for c in (0, 1, 4, 200, 255, 256, 767):
        e = np.zeros(cols, np.uint16)
        e[c] = ONE
        a = host_bf16(tcq.trellis_matvec(dev(e), d["codes"], sc1, lo, d["g"]))
        b = host_bf16(tcq.trellis_matvec(dev(e), d["codes"], sc1, hi, d["g"]))
        from oracle import bf16_to_float
        got = bf16_to_float(a).astype(np.int64) + 256 * bf16_to_float(b).astype(np.int64)
        assert np.array_equal(got, win[:, c].astype(np.int64)), c


# ----------------------------------------------------------------- prefill

@pytest.mark.parametrize("k", [2, 3, 4])
@pytest.mark.parametrize("M", [1, 2, 5, 8, 9, 16, 17, 31, 32])
def test_prefill_small(orc, M, k):
    rows, cols = 300, 768          # 3 CTAs with a ragged last one; 3 blocks (odd: both stages, parity flips)
    p = synth.problem(1, M, rows, cols, k, seed=5)
    d = on_device(p)
    out = tcq.trellis_prefill(d["x"], d["codes"], d["scales"], d["lut"], d["g"])
    _, y, a = _oracle_axis1(orc, p)
    check_close(orc, host_bf16(out), y, a, f"prefill M={M} k={k}")
    assert tcq.trellis_device_status() == 0


def test_prefill_rows_spread_over_sms(orc):
    """Between 64 and 128 rows per SM each CTA owns ceil(rows / SMs) rows
    (here 66 on 152 SMs, a ragged last tile); lanes past them decode nothing."""
    rows, cols, k, M = 10001, 512, 3, 9
    p = synth.problem(1, M, rows, cols, k, seed=21)
    d = on_device(p)
    out = host_bf16(tcq.trellis_prefill(d["x"], d["codes"], d["scales"], d["lut"], d["g"]))
    _, y, a = _oracle_axis1(orc, p)
    check_close(orc, out, y, a, "prefill spread tiles")
    assert tcq.trellis_device_status() == 0


@pytest.mark.parametrize("M,k", [(32, 4), (5, 2), (16, 3), (8, 4), (32, 2), (32, 3)])
def test_prefill_full_size(orc, M, k):
    rows, cols = 17408, 5120
    p = synth.problem(1, M, rows, cols, k, seed=0)
    d = on_device(p)
    out = host_bf16(tcq.trellis_prefill(d["x"], d["codes"], d["scales"], d["lut"], d["g"]))
    if (M, k) in ((32, 4), (5, 2)):
        _, y, a = _oracle_axis1(orc, p)
        check_close(orc, out, y, a, f"prefill full M={M} k={k}")
    else:
        rng = np.random.default_rng(M * 10 + k)
        ms = rng.integers(0, M, 4000)
        js = rng.integers(0, rows, 4000)
        y, a = orc.sample(p["x"], p["codes"], rows, cols, k, p["scales"], p["lut"], 1, ms, js)
        check_close(orc, out[ms, js], y, a, f"prefill full sampled M={M} k={k}")
    assert tcq.trellis_device_status() == 0


@pytest.mark.parametrize("k", [2, 3, 4])
def test_prefill_unit_vectors_exact(orc, k):
    rows, cols, M = 260, 1024, 8
    p = synth.problem(1, M, rows, cols, k, seed=6)
    d = on_device(p)
    W, _ = orc.expand(p["codes"], rows, cols, k, p["scales"], p["lut"])
    cs = [0, 1, 255, 256, 300, 511, 512, 1023]
    e = np.zeros((M, cols), np.uint16)
    for m, c in enumerate(cs):
        e[m, c] = ONE
    out = host_bf16(tcq.trellis_prefill(dev(e), d["codes"], d["scales"], d["lut"], d["g"]))
    for m, c in enumerate(cs):
        assert np.array_equal(out[m], W[:, c]), (m, c)


# ----------------------------------------------------------------- scatter

@pytest.mark.parametrize("M", [1, 4])
def test_scatter_full_size(orc, M):
    rows, cols, k = 17408, 5120, 3
    p = synth.problem(0, M, rows, cols, k, seed=0)
    d = on_device(p)
    out = tcq.trellis_scatter(d["x"], d["codes"], d["scales"], d["lut"], d["g"], splits=128)
    _, y, a, _ = _oracle_axis0(orc, p)
    check_close(orc, host_bf16(out), y, a, f"scatter full M={M}")


@pytest.mark.parametrize("rows,cols,k,M,splits", [
    (1, 256, 3, 1, 0), (7, 256, 2, 2, 0), (300, 1280, 4, 3, 7), (300, 1280, 3, 5, 1),
    (300, 768, 2, 9, 1024), (513, 2048, 3, 4, 128), (129, 256, 4, 32, 64), (64, 5120, 3, 1, 128),
    (301, 512, 3, 7, 5), (301, 512, 4, 12, 13),         # odd rows and odd split sizes on the tensor path
    (2048, 512, 3, 32, 2), (4099, 256, 2, 9, 1),        # splits too long to stage their activations in shared memory
    (1000, 768, 3, 4, 100),     # tensor path, 100 splits: reduction runs of 4 splits, the last runs empty
])
def test_scatter_small(orc, rows, cols, k, M, splits):
    p = synth.problem(0, M, rows, cols, k, seed=7)
    d = on_device(p)
    out = tcq.trellis_scatter(d["x"], d["codes"], d["scales"], d["lut"], d["g"], splits=splits)
    _, y, a, _ = _oracle_axis0(orc, p)
    check_close(orc, host_bf16(out), y, a, f"scatter {rows}x{cols} k={k} M={M} S={splits}")


def test_scatter_partials(orc):
    """The fp32 partial of every split against the oracle's split sums; empty
    splits past the last row hold zeros."""
    import torch
    rows, cols, k, M, S = 100, 512, 3, 2, 48      # rp = 3: splits 34..47 are empty
    p = synth.problem(0, M, rows, cols, k, seed=8)
    d = on_device(p)
    ws = torch.zeros(tcq.trellis_scatter_workspace_bytes(d["g"], M, S) // 4, dtype=torch.float32, device="cuda")
    ws.fill_(float("nan"))
    tcq.trellis_scatter(d["x"], d["codes"], d["scales"], d["lut"], d["g"], splits=S, workspace=ws)
    part = ws.view(M, S, cols).cpu().numpy().astype(np.float64)
    W, _, _, ref = _oracle_axis0(orc, p, S)
    from oracle import bf16_to_float
    xf = np.abs(bf16_to_float(p["x"]).astype(np.float64))
    wf = np.abs(bf16_to_float(W).astype(np.float64))
    rp = -(-rows // S)
    for s in range(S):
        r0, r1 = s * rp, min(rows, (s + 1) * rp)
        if r0 >= r1:
            assert np.all(part[:, s, :] == 0.0), s
            continue
        asum = xf[:, r0:r1] @ wf[r0:r1]
        assert np.all(np.abs(part[:, s, :] - ref[:, s, :]) <= 1e-5 * asum + 1e-30), s


@pytest.mark.parametrize("splits", [8, 128])
@pytest.mark.parametrize("M,k", [(16, 3), (5, 2), (32, 4), (3, 3), (4, 4)])
def test_scatter_tensor_path_full_size(orc, M, k, splits):
    """3 or more activation rows take a tensor-core scatter in one pass:
    tcgen05 below 128 splits, mma.sync from 128."""
    rows, cols = 17408, 5120
    p = synth.problem(0, M, rows, cols, k, seed=19)
    d = on_device(p)
    out = host_bf16(tcq.trellis_scatter(d["x"], d["codes"], d["scales"], d["lut"], d["g"], splits=splits))
    if M == 16:
        _, y, a, _ = _oracle_axis0(orc, p, splits)
        check_close(orc, out, y, a, f"scatter tensor path M={M} S={splits}")
    else:
        rng = np.random.default_rng(M)
        ms, js = rng.integers(0, M, 3000), rng.integers(0, cols, 3000)
        y, a = orc.sample(p["x"], p["codes"], rows, cols, k, p["scales"], p["lut"], 0, ms, js)
        check_close(orc, out[ms, js], y, a, f"scatter tensor path sampled M={M}")


@pytest.mark.parametrize("k", [2, 3, 4])
def test_scatter_tensor_path_unit_vectors_exact(orc, k):
    rows, cols, M = 200, 1024, 8
    p = synth.problem(0, M, rows, cols, k, seed=20)
    d = on_device(p)
    W, _ = orc.expand(p["codes"], rows, cols, k, p["scales"], p["lut"])
    rs = [0, 1, 15, 16, 17, 99, 150, 199]
    e = np.zeros((M, rows), np.uint16)
    for m, r in enumerate(rs):
        e[m, r] = ONE
    out = host_bf16(tcq.trellis_scatter(dev(e), d["codes"], d["scales"], d["lut"], d["g"], splits=7))
    for m, r in enumerate(rs):
        assert np.array_equal(out[m], W[r]), (m, r)


@pytest.mark.parametrize("k", [2, 3, 4])
def test_scatter_unit_vectors_exact(orc, k):
    rows, cols = 200, 1024
    p = synth.problem(0, 1, rows, cols, k, seed=9)
    d = on_device(p)
    W, _ = orc.expand(p["codes"], rows, cols, k, p["scales"], p["lut"])
    for r in (0, 1, 99, 199):
        e = np.zeros((1, rows), np.uint16)
        e[0, r] = ONE
        out = host_bf16(tcq.trellis_scatter(dev(e), d["codes"], d["scales"], d["lut"], d["g"]))
        assert np.array_equal(out[0], W[r]), r


# ----------------------------------------------------------------- interleave-2 layout

def _inter(p):
    p = dict(p)
    p["interleave"] = 2
    return p


@pytest.mark.parametrize("axis,rows,cols,k", [(0, 17408, 5120, 3), (1, 300, 1024, 4), (0, 37, 512, 2)])
def test_expand_interleave2_bit_exact(orc, axis, rows, cols, k):
    p = _inter(synth.problem(axis, 1, rows, cols, k, seed=14))
    d = on_device(p)
    w, win = tcq.trellis_expand(d["codes"], d["scales"], d["lut"], d["g"], with_windows=True)
    ow, owin = orc.expand(p["codes"], rows, cols, k, p["scales"], p["lut"], interleave=2)
    assert np.array_equal(host_bf16(win), owin) and np.array_equal(host_bf16(w), ow)


@pytest.mark.parametrize("splits", [8, 128])
@pytest.mark.parametrize("M", [1, 4, 16])
def test_scatter_interleave2_full_size(orc, M, splits):
    """The pages' k=3 axis-0 production layout at the full scatter geometry."""
    rows, cols, k = 17408, 5120, 3
    p = _inter(synth.problem(0, M, rows, cols, k, seed=15))
    d = on_device(p)
    out = host_bf16(tcq.trellis_scatter(d["x"], d["codes"], d["scales"], d["lut"], d["g"], splits=splits))
    W, _ = orc.expand(p["codes"], rows, cols, k, p["scales"], p["lut"], interleave=2)
    y, a, _, _ = orc.matmul_axis0(p["x"], W)
    check_close(orc, out, y, a, f"scatter interleave 2 M={M}")


@pytest.mark.parametrize("rows,cols,k,M,splits", [(301, 1024, 2, 5, 7), (300, 2048, 4, 32, 13), (129, 512, 3, 9, 1024)])
def test_scatter_tensor_path_interleave2(orc, rows, cols, k, M, splits):
    """The tensor-core scatter on the interleave-2 layout, odd split sizes."""
    p = _inter(synth.problem(0, M, rows, cols, k, seed=17))
    d = on_device(p)
    out = host_bf16(tcq.trellis_scatter(d["x"], d["codes"], d["scales"], d["lut"], d["g"], splits=splits))
    W, _ = orc.expand(p["codes"], rows, cols, k, p["scales"], p["lut"], interleave=2)
    y, a, _, _ = orc.matmul_axis0(p["x"], W)
    check_close(orc, out, y, a, f"tensor scatter interleave 2 {rows}x{cols} k={k} M={M} S={splits}")


@pytest.mark.parametrize("M,k", [(16, 3), (32, 2)])
def test_prefill_interleave2_full_size(orc, M, k):
    """Interleave 2 at 17408 x 5120: 115-row tiles, the code tiles copied as
    3-d boxes (block pair, rows, words) that read past the block's words."""
    rows, cols = 17408, 5120
    p = _inter(synth.problem(1, M, rows, cols, k, seed=M + k))
    d = on_device(p)
    out = host_bf16(tcq.trellis_prefill(d["x"], d["codes"], d["scales"], d["lut"], d["g"]))
    rng = np.random.default_rng(M * 3 + k)
    ms = rng.integers(0, M, 3000)
    js = rng.integers(0, rows, 3000)
    y, a = orc.sample(p["x"], p["codes"], rows, cols, k, p["scales"], p["lut"], 1, ms, js, interleave=2)
    check_close(orc, out[ms, js], y, a, f"prefill interleave 2 full M={M} k={k}")
    assert tcq.trellis_device_status() == 0


@pytest.mark.parametrize("k", [2, 3, 4])
def test_axis1_interleave2(orc, k):
    rows, cols = 300, 1536
    p = _inter(synth.problem(1, 8, rows, cols, k, seed=16))
    d = on_device(p)
    W, _ = orc.expand(p["codes"], rows, cols, k, p["scales"], p["lut"], interleave=2)
    y, a, _ = orc.matmul_axis1(p["x"], W)
    out = host_bf16(tcq.trellis_prefill(d["x"], d["codes"], d["scales"], d["lut"], d["g"]))
    check_close(orc, out, y, a, f"prefill interleave 2 k={k}")
    mv = host_bf16(tcq.trellis_matvec(d["x"][0].contiguous(), d["codes"], d["scales"], d["lut"], d["g"]))
    check_close(orc, mv[None, :], y[:1], a[:1], f"matvec interleave 2 k={k}")


# ----------------------------------------------------------------- wide geometries

def test_prefill_wide_k(orc):
    """K = 17408 (68 blocks: many stage and ring turns), ragged rows."""
    rows, cols, k, M = 200, 17408, 3, 16
    p = synth.problem(1, M, rows, cols, k, seed=17)
    d = on_device(p)
    out = host_bf16(tcq.trellis_prefill(d["x"], d["codes"], d["scales"], d["lut"], d["g"]))
    _, y, a = _oracle_axis1(orc, p)
    check_close(orc, out, y, a, "prefill K=17408")
    assert tcq.trellis_device_status() == 0


@pytest.mark.parametrize("M", [1, 3, 9])
def test_scatter_wide_cols(orc, M):
    """C = 17408: 17 column ranges, 4 blocks of ranges per split, the last partial."""
    rows, cols, k = 300, 17408, 4
    p = synth.problem(0, M, rows, cols, k, seed=18)
    d = on_device(p)
    out = host_bf16(tcq.trellis_scatter(d["x"], d["codes"], d["scales"], d["lut"], d["g"], splits=16))
    _, y, a, _ = _oracle_axis0(orc, p)
    check_close(orc, out, y, a, f"scatter C=17408 M={M}")


# ----------------------------------------------------------------- glue

def _ulps(a, b):
    from oracle import bf16_to_float
    fa, fb = bf16_to_float(a).astype(np.float64), bf16_to_float(b).astype(np.float64)
    from oracle import bf16_ulp
    return np.abs(fa - fb) / bf16_ulp(np.maximum(np.abs(fa), np.abs(fb)))


@pytest.mark.parametrize("M,D", [
    (16, 5120),     # the MLP's rows: the one-pass kernel (rows held in registers)
    (3, 8), (2, 8192),   # the one-pass kernel's smallest and largest rows
    (5, 1001),      # D not a multiple of 8: the two-pass kernel
    (2, 12288),     # longer than the one-pass kernel holds: the two-pass kernel
])
def test_rmsnorm(orc, M, D):
    x = synth.activations(11, M, D)
    out = host_bf16(tcq.trellis_rmsnorm(dev(x), 1e-6))
    assert np.all(_ulps(out, orc.rmsnorm(x, 1e-6)) <= 1.0)


def test_rmsnorm_unaligned_rows_take_the_two_pass_kernel(orc):
    import torch
    M, D = 4, 5120
    x = synth.activations(14, M, D)
    buf = torch.empty(M * D + 1, dtype=torch.bfloat16, device="cuda")
    xs = buf[1:].view(M, D)                         # 2-byte offset: not 16-byte aligned
    xs.copy_(dev(x))
    out = host_bf16(tcq.trellis_rmsnorm(xs, 1e-6))
    assert np.all(_ulps(out, orc.rmsnorm(x, 1e-6)) <= 1.0)


def test_silu_mul(orc):
    g = synth.activations(12, 4, 17408)
    u = synth.activations(13, 4, 17408)
    out = host_bf16(tcq.trellis_silu_mul(dev(g), dev(u)))
    assert np.all(_ulps(out, orc.silu_mul(g, u)) <= 1.0)


# ----------------------------------------------------------------- errors on a live device

def test_errors_do_not_launch():
    import torch
    p = synth.problem(1, 1, 256, 512, 2, seed=0)
    d = on_device(p)
    bad = tcq.geometry(1, 256, 512, 2)
    bad.L = 11
    with pytest.raises(tcq.TrellisError, match="GEOMETRY"):
        tcq.trellis_matvec(d["x"][0], d["codes"], d["scales"], d["lut"], bad)
    g0 = tcq.geometry(0, 256, 512, 2)
    x0 = dev(synth.activations(0, 1, 256))
    small = torch.empty(16, dtype=torch.float32, device="cuda")
    with pytest.raises(tcq.TrellisError, match="WORKSPACE"):
        tcq.trellis_scatter(x0, d["codes"], d["scales"], d["lut"], g0, workspace=small)
    torch.cuda.synchronize()
    assert tcq.trellis_device_status() == 0
