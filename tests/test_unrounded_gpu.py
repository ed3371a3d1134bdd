"""The unrounded contract (TRELLIS_FLAG_UNROUNDED) through the C ABI against
the oracle's unrounded functions: the weight is the f32 product of codebook
value and row scale, contracted without the bf16 rounding (@mlx-bun/inference
1.0.0, kernels/trellis/scatter.ts, the balanced scatter kernels).

Per case:
  - every element within the contraction tolerance of the unrounded oracle;
  - the bf16 outputs equal bf16(y) of the unrounded oracle on at least 99%
    of the elements (only f32 accumulation order separates them), while the
    rounded contract's own oracle output differs from that on at least 20%:
    the check tells the two contracts apart, which the tolerance alone,
    wide enough for both, does not;
  - scatter: every fp32 split partial within 2^-16 * sum|x*w| of the exact
    unrounded split sum, a bound that the rounded weights break.
"""
import numpy as np
import pytest

import trellis_coded_quantized_gb300 as tcq
from trellis_coded_quantized_gb300 import synth
from gpu_util import check_close, dev, host_bf16
from conftest import has_gpu

pytestmark = [pytest.mark.gpu, pytest.mark.skipif(not has_gpu(), reason="needs a CUDA GPU")]

AGREE = 0.99        # unrounded kernel vs unrounded oracle, bf16 outputs equal
DISAGREE = 0.20     # rounded oracle vs unrounded oracle, bf16 outputs differ
PART_REL = 2.0 ** -16


@pytest.fixture(scope="module", autouse=True)
def _built():
    from trellis_coded_quantized_gb300 import build
    build.build()


def _inter(p):
    """The codes of p re-laid out as interleave 2 (blocks paired across rows)."""
    rows, cols, k = p["rows"], p["cols"], p["k"]
    wpb = 256 * k // 32
    nb = cols // 256
    c = p["codes"].reshape(rows, nb // 2, 2 * wpb)
    return np.ascontiguousarray(c.transpose(1, 0, 2)).reshape(rows, -1)


def _device(p, interleave=0):
    codes = _inter(p) if interleave == 2 else p["codes"]
    return {"g": tcq.geometry(p["axis"], p["rows"], p["cols"], p["k"], interleave, unrounded=True),
            "codes": dev(codes), "scales": dev(p["scales"]), "lut": dev(p["lut"]), "x": dev(p["x"])}


def _agreement(orc, got, out_unr, out_rnd, what):
    agree = np.mean(got == out_unr)
    differ = np.mean(out_rnd != out_unr)
    assert differ >= DISAGREE, f"{what}: the contracts differ on only {differ:.3f} (test not discriminating)"
    assert agree >= AGREE, f"{what}: bf16 equal to the unrounded oracle on {agree:.4f} < {AGREE}"


def _oracle_axis1(orc, p, rows_sel=None):
    codes, scales, rows = p["codes"], p["scales"], p["rows"]
    if rows_sel is not None:            # interleave 0: the words of a row are contiguous
        codes, scales, rows = codes[rows_sel], scales[rows_sel], len(rows_sel)
    w32 = orc.expand_f32(codes, rows, p["cols"], p["k"], scales, p["lut"])
    wb, _ = orc.expand(codes, rows, p["cols"], p["k"], scales, p["lut"])
    y, a, out = orc.matmul_axis1_f32w(p["x"], w32)
    _, _, out_rnd = orc.matmul_axis1(p["x"], wb)
    return y, a, out, out_rnd


@pytest.mark.parametrize("rows,cols,k,interleave", [
    (256, 512, 2, 0), (37, 768, 2, 0), (2051, 5120, 4, 0), (2051, 5120, 3, 0), (2048, 5120, 2, 0),
    (1000, 20480, 3, 0), (300, 1024, 4, 2), (152 * 3 + 5, 2560, 2, 2),
])
def test_matvec_unrounded(orc, rows, cols, k, interleave):
    p = synth.problem(1, 1, rows, cols, k, seed=21)
    d = _device(p, interleave)
    got = host_bf16(tcq.trellis_matvec(d["x"][0], d["codes"], d["scales"], d["lut"], d["g"]))[None, :]
    y, a, out, out_rnd = _oracle_axis1(orc, p)
    what = f"unrounded matvec {rows}x{cols} k={k} il={interleave}"
    check_close(orc, got, y, a, what)
    _agreement(orc, got, out, out_rnd, what)


@pytest.mark.parametrize("k", [2, 3, 4])
def test_matvec_unrounded_full_size_sampled_rows(orc, k):
    rows, cols = 17408, 5120
    p = synth.problem(1, 1, rows, cols, k, seed=22)
    d = _device(p)
    got = host_bf16(tcq.trellis_matvec(d["x"][0], d["codes"], d["scales"], d["lut"], d["g"]))
    sel = np.sort(np.random.default_rng(k).choice(rows, 2000, replace=False))
    sel[-1] = rows - 1
    y, a, out, out_rnd = _oracle_axis1(orc, p, sel)
    what = f"unrounded matvec full k={k}"
    check_close(orc, got[sel][None, :], y, a, what)
    _agreement(orc, got[sel][None, :], out, out_rnd, what)


def _oracle_axis0(orc, p, splits):
    w32 = orc.expand_f32(p["codes"], p["rows"], p["cols"], p["k"], p["scales"], p["lut"])
    wb, _ = orc.expand(p["codes"], p["rows"], p["cols"], p["k"], p["scales"], p["lut"])
    y, a, out, part = orc.matmul_axis0_f32w(p["x"], w32, splits)
    _, _, out_rnd, part_rnd = orc.matmul_axis0(p["x"], wb, splits)
    return w32, y, a, out, part, out_rnd, part_rnd


def _check_partials(orc, p, w32, ws, part, part_rnd, splits, what):
    from oracle import bf16_to_float
    M, rows, cols = p["m"], p["rows"], p["cols"]
    got = ws[: M * splits * cols].view(M, splits, cols).cpu().numpy().astype(np.float64)
    xf = np.abs(bf16_to_float(p["x"]).astype(np.float64))
    wf = np.abs(w32.astype(np.float64))
    rp = -(-rows // splits)
    broken = 0
    total = 0
    for s in range(splits):
        r0, r1 = s * rp, min(rows, (s + 1) * rp)
        if r0 >= r1:
            assert np.all(got[:, s, :] == 0.0), f"{what}: empty split {s} not zero"
            continue
        bound = PART_REL * (xf[:, r0:r1] @ wf[r0:r1]) + 1e-30
        err = np.abs(got[:, s, :] - part[:, s, :])
        assert np.all(err <= bound), f"{what}: split {s}: max err/bound {np.max(err / bound):.3g}"
        broken += int(np.sum(np.abs(part_rnd[:, s, :] - part[:, s, :]) > bound))
        total += err.size
    assert broken >= 0.5 * total, f"{what}: rounded partials break the bound on only {broken} of {total}"


@pytest.mark.parametrize("rows,cols,k,M,splits,interleave", [
    (2048, 5120, 3, 1, 128, 0), (2048, 5120, 3, 4, 128, 0), (2048, 5120, 4, 5, 128, 0),
    (2048, 5120, 2, 16, 128, 0), (4096, 5120, 3, 4, 128, 2), (300, 1280, 3, 3, 7, 0),
    (100, 512, 3, 2, 48, 0),            # rp = 3: splits 34..47 are empty
    (129, 256, 4, 9, 1024, 0),          # more splits than rows
])
def test_scatter_unrounded(orc, rows, cols, k, M, splits, interleave):
    import torch
    p = synth.problem(0, M, rows, cols, k, seed=23)
    d = _device(p, interleave)
    ws = torch.full((tcq.trellis_scatter_workspace_bytes(d["g"], M, splits) // 4,), float("nan"),
                    dtype=torch.float32, device="cuda")
    got = host_bf16(tcq.trellis_scatter(d["x"], d["codes"], d["scales"], d["lut"], d["g"], splits=splits,
                                        workspace=ws))
    w32, y, a, out, part, out_rnd, part_rnd = _oracle_axis0(orc, p, splits)
    what = f"unrounded scatter {rows}x{cols} k={k} M={M} S={splits} il={interleave}"
    check_close(orc, got, y, a, what)
    if M * cols >= 4096:
        _agreement(orc, got, out, out_rnd, what)
    _check_partials(orc, p, w32, ws, part, part_rnd, splits, what)


def test_scatter_unrounded_full_size(orc):
    rows, cols, k, M = 17408, 5120, 3, 1
    p = synth.problem(0, M, rows, cols, k, seed=24)
    d = _device(p)
    got = host_bf16(tcq.trellis_scatter(d["x"], d["codes"], d["scales"], d["lut"], d["g"], splits=128))
    _, y, a, out, _, out_rnd, _ = _oracle_axis0(orc, p, 0)
    check_close(orc, got, y, a, "unrounded scatter full size")
    _agreement(orc, got, out, out_rnd, "unrounded scatter full size")


@pytest.mark.parametrize("M", [5, 16])
def test_scatter_unrounded_default_splits(orc, M):
    """splits = 0 under the unrounded contract is scatter.ts's 128 ranges at
    every M (not the split-K rule's 8 of the rounded contract): the default
    call equals the call with 128 splits bit for bit, leaves the 128 split
    partials in the workspace, and is within the tolerance of the oracle."""
    import torch
    rows, cols, k = 4096, 5120, 3
    p = synth.problem(0, M, rows, cols, k, seed=29)
    d = _device(p)
    need = tcq.trellis_scatter_workspace_bytes(d["g"], M, 0)
    assert need == M * 128 * cols * 4
    ws = torch.full((need // 4,), float("nan"), dtype=torch.float32, device="cuda")
    got = tcq.trellis_scatter(d["x"], d["codes"], d["scales"], d["lut"], d["g"], workspace=ws)
    want = tcq.trellis_scatter(d["x"], d["codes"], d["scales"], d["lut"], d["g"], splits=128)
    assert torch.equal(got.view(torch.int16), want.view(torch.int16))
    w32, y, a, out, part, out_rnd, part_rnd = _oracle_axis0(orc, p, 128)
    check_close(orc, host_bf16(got), y, a, f"unrounded scatter default splits M={M}")
    _check_partials(orc, p, w32, ws, part, part_rnd, 128, f"unrounded scatter default splits M={M}")


def test_rounded_paths_agree_with_their_own_oracle(orc):
    """The same agreement statistic for the default (rounded) contract on the
    FMA paths: the matvec and the M <= 2 scatter."""
    p = synth.problem(1, 1, 2051, 5120, 4, seed=21)
    g = tcq.geometry(1, 2051, 5120, 4)
    got = host_bf16(tcq.trellis_matvec(dev(p["x"])[0], dev(p["codes"]), dev(p["scales"]), dev(p["lut"]), g))
    _, _, out_unr, out_rnd = _oracle_axis1(orc, p)
    assert np.mean(got[None, :] == out_rnd) >= AGREE
    assert np.mean(out_unr != out_rnd) >= DISAGREE
    p = synth.problem(0, 2, 2048, 5120, 3, seed=23)
    g = tcq.geometry(0, 2048, 5120, 3)
    got = host_bf16(tcq.trellis_scatter(dev(p["x"]), dev(p["codes"]), dev(p["scales"]), dev(p["lut"]), g))
    _, _, _, out_unr, _, out_rnd, _ = _oracle_axis0(orc, p, 0)
    assert np.mean(got == out_rnd) >= AGREE
    assert np.mean(out_unr != out_rnd) >= DISAGREE


_FULL = {}


def _full_size(orc, axis, k, M, seed):
    """A 17408 x 5120 problem of the given axis and its rounded expansion
    (cached per axis and k: the expansion takes a while)."""
    rows, cols = 17408, 5120
    key = (axis, k)
    if key not in _FULL:
        p0 = synth.problem(axis, 1, rows, cols, k, seed=seed)
        wb, _ = orc.expand(p0["codes"], rows, cols, k, p0["scales"], p0["lut"])
        _FULL[key] = (p0, wb)
    p0, wb = _FULL[key]
    x = synth.activations(seed + 100 * M, M, cols if axis == 1 else rows)
    return p0, wb, x


@pytest.mark.parametrize("M", [8, 16, 32])
@pytest.mark.parametrize("k", [2, 3, 4])
def test_prefill_agrees_with_its_own_oracle_full_size(orc, M, k):
    """The tensor-core prefill (tcgen05, fp32 accumulation in tensor memory)
    at 17408 x 5120: every bf16 output within the tolerance and equal to
    bf16(y) of the oracle on at least 99% of the elements, where the
    unrounded contract's output differs from it on at least 20% (checked on
    1024 of the rows).  A dropped K chunk or a precision loss in the
    accumulation fails the 99% even where the tolerance would pass."""
    rows, cols = 17408, 5120
    p, wb, x = _full_size(orc, 1, k, M, seed=51)
    g = tcq.geometry(1, rows, cols, k)
    got = host_bf16(tcq.trellis_prefill(dev(x), dev(p["codes"]), dev(p["scales"]), dev(p["lut"]), g))
    y, a, out = orc.matmul_axis1(x, wb)
    check_close(orc, got, y, a, f"prefill full M={M} k={k}")
    agree = np.mean(got == out)
    assert agree >= AGREE, f"prefill M={M} k={k}: bf16 equal to the oracle on {agree:.4f}"
    sel = np.arange(0, rows, rows // 1024)[:1024]
    w32 = orc.expand_f32(p["codes"][sel], len(sel), cols, k, p["scales"][sel], p["lut"])
    _, _, out_unr = orc.matmul_axis1_f32w(x, w32)
    assert np.mean(out_unr != out[:, sel]) >= DISAGREE


@pytest.mark.parametrize("splits", [8, 128])
@pytest.mark.parametrize("M", [4, 16, 32])
def test_scatter_tensor_path_agrees_with_its_own_oracle_full_size(orc, M, splits):
    """The rounded axis-0 scatter from 3 activation rows on the tensor cores
    at 17408 x 5120, k=3 -- 8 splits (the split-K default from M = 5: the
    tcgen05 kernel) and 128 splits (the mma.sync kernel) -- held to the same
    99% agreement with the oracle's bf16(y), with the unrounded contract
    differing on >= 20% (checked on the first 2048 of the input rows)."""
    rows, cols, k = 17408, 5120, 3
    p, wb, x = _full_size(orc, 0, k, M, seed=53)
    g = tcq.geometry(0, rows, cols, k)
    got = host_bf16(tcq.trellis_scatter(dev(x), dev(p["codes"]), dev(p["scales"]), dev(p["lut"]), g,
                                        splits=splits))
    y, a, out, _ = orc.matmul_axis0(x, wb)
    check_close(orc, got, y, a, f"scatter tensor path full M={M} S={splits}")
    agree = np.mean(got == out)
    assert agree >= AGREE, f"scatter M={M} S={splits}: bf16 equal to the oracle on {agree:.4f}"
    n = 2048
    w32 = orc.expand_f32(p["codes"][:n], n, cols, k, p["scales"][:n], p["lut"])
    _, _, out_unr, _ = orc.matmul_axis0_f32w(x[:, :n], w32)
    _, _, out_rnd, _ = orc.matmul_axis0(x[:, :n], wb[:n])
    assert np.mean(out_unr != out_rnd) >= DISAGREE


def test_unrounded_refused_where_the_operands_are_bf16():
    p = synth.problem(1, 8, 256, 512, 3, seed=25)
    d = _device(p)
    with pytest.raises(tcq.TrellisError) as e:
        tcq.trellis_prefill(d["x"], d["codes"], d["scales"], d["lut"], d["g"])
    assert e.value.status == 2
    with pytest.raises(tcq.TrellisError) as e:
        tcq.trellis_expand(d["codes"], d["scales"], d["lut"], d["g"])
    assert e.value.status == 2
