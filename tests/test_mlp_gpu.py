"""The synthetic MLP stack (40 SwiGLU layers of packed k=3 weights) on the GPU.

Each stage is checked against the oracle on the GPU's own input of that stage,
so differences do not compound: RMSNorm and silu*up within 1 bf16 ulp, the
three packed matmuls within the contraction tolerance on sampled outputs.
The full 40-layer pass must stay finite.
"""
import numpy as np
import pytest

from conftest import has_gpu
from gpu_util import host_bf16

pytestmark = [pytest.mark.gpu, pytest.mark.skipif(not has_gpu(), reason="needs a CUDA GPU")]


@pytest.fixture(scope="module")
def stack():
    from trellis_coded_quantized_gb300 import build
    build.build()
    from trellis_coded_quantized_gb300.mlp import PackedMLPStack
    return PackedMLPStack(layers=40, k=3, device="cuda", m_max=16)


def _ulps(a, b):
    from oracle import bf16_to_float, bf16_ulp
    fa, fb = bf16_to_float(a).astype(np.float64), bf16_to_float(b).astype(np.float64)
    return np.abs(fa - fb) / bf16_ulp(np.maximum(np.abs(fa), np.abs(fb)))


def _sampled(orc, x, mat, lut, got, n, rng):
    g = mat["g"]
    codes = mat["codes"].cpu().numpy().view(np.uint32)
    scales = mat["scales"].view(__import__("torch").int16).cpu().numpy().view(np.uint16)
    lut = lut.cpu().numpy()
    M = x.shape[0]
    nout = g.rows if g.axis == 1 else g.cols
    ms = rng.integers(0, M, n)
    js = rng.integers(0, nout, n)
    y, a = orc.sample(x, codes, g.rows, g.cols, g.k, scales, lut, g.axis, ms, js)
    ok, err, bound = orc.within_tolerance(got[ms, js], y, a)
    assert ok.all(), (int((~ok).sum()), err[~ok][:4], bound[~ok][:4])


@pytest.mark.parametrize("M", [1, 16])
def test_stack_stages(orc, stack, M):
    import torch
    from trellis_coded_quantized_gb300 import synth
    x0 = torch.from_numpy(synth.activations(0, M, 5120).view(np.int16)).cuda().view(torch.bfloat16)
    keep = []
    out = stack.forward(x0, keep=keep)
    torch.cuda.synchronize()
    assert torch.isfinite(out.float()).all()
    rng = np.random.default_rng(M)
    for l in (0, 1, 39):
        st = {k: host_bf16(v) for k, v in keep[l].items()}
        assert np.all(_ulps(st["n"], orc.rmsnorm(st["x"], 1e-6)) <= 1.0), l
        gate, up, down = stack.layers[l].mats
        _sampled(orc, st["n"], gate, stack.lut, st["g"], 300, rng)
        _sampled(orc, st["n"], up, stack.lut, st["u"], 300, rng)
        # M = 1: h comes from the fused gate/up kernel, g and u from trellis_matvec
        assert np.all(_ulps(st["h"], orc.silu_mul(st["g"], st["u"])) <= 1.0), l
        _sampled(orc, st["h"], down, stack.lut, st["out"], 300, rng)
