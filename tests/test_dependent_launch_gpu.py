"""Kernels launched as programmatic dependents of the previous kernel (every
kernel of the library) must still see their predecessor's writes and must not
overwrite what it still reads.  A chain of RMSNorm -> fused gate/up matvec ->
axis-0 scatter -> split reduction, whose buffers are reused from layer to
layer (read-after-write and write-after-read on the same arrays), is run back
to back and again with a device synchronisation after every call; the two
results must be identical bit for bit, and the first layer must match the
oracle."""
import numpy as np
import pytest

import trellis_coded_quantized_gb300 as tcq
from trellis_coded_quantized_gb300 import synth
from gpu_util import dev, host_bf16
from conftest import has_gpu

pytestmark = [pytest.mark.gpu, pytest.mark.skipif(not has_gpu(), reason="needs a CUDA GPU")]

HID, INTER, K, LAYERS = 5120, 17408, 2, 6


@pytest.fixture(scope="module")
def chain():
    import torch
    from trellis_coded_quantized_gb300 import build
    build.build()
    lut = dev(synth.lut(77))
    mats = []
    for l in range(LAYERS):
        gate = (dev(synth.codes(100 * l, INTER, HID, K)), dev(synth.scales(100 * l, INTER)))
        up = (dev(synth.codes(100 * l + 1, INTER, HID, K)), dev(synth.scales(100 * l + 1, INTER)))
        down = (dev(synth.codes(100 * l + 2, INTER, HID, K)), dev(synth.scales(100 * l + 2, INTER)))
        mats.append((gate, up, down))
    g1 = tcq.geometry(1, INTER, HID, K)
    g0 = tcq.geometry(0, INTER, HID, K)
    bufs = {"x": torch.empty((1, HID), dtype=torch.bfloat16, device="cuda"),
            "n": torch.empty((1, HID), dtype=torch.bfloat16, device="cuda"),
            "h": torch.empty((1, INTER), dtype=torch.bfloat16, device="cuda"),
            "ws": torch.empty(tcq.trellis_scatter_workspace_bytes(g0, 1, 152) // 4, dtype=torch.float32,
                              device="cuda")}
    x0 = dev(synth.activations(5, 1, HID))
    return lut, mats, g1, g0, bufs, x0


def _run(chain, sync: bool):
    import torch
    lut, mats, g1, g0, b, x0 = chain
    b["x"].copy_(x0)
    torch.cuda.synchronize()
    for (gate, up, down) in mats:
        tcq.trellis_rmsnorm(b["x"], 1e-6, out=b["n"])
        if sync:
            torch.cuda.synchronize()
        tcq.trellis_gate_up_matvec(b["n"][0], gate[0], gate[1], up[0], up[1], lut, g1, out=b["h"][0])
        if sync:
            torch.cuda.synchronize()
        # overwrites x, which the RMSNorm of this layer read
        tcq.trellis_scatter(b["h"], down[0], down[1], lut, g0, splits=152, workspace=b["ws"], out=b["x"])
        if sync:
            torch.cuda.synchronize()
    torch.cuda.synchronize()
    return host_bf16(b["x"]).copy()


def test_back_to_back_equals_synchronised(chain):
    from oracle import bf16_to_float
    ref = _run(chain, sync=True)
    assert np.isfinite(bf16_to_float(ref)).all()
    for _ in range(3):
        assert np.array_equal(_run(chain, sync=False), ref)
    assert tcq.trellis_device_status() == 0


def test_first_layer_against_the_oracle(orc, chain):
    import torch
    from oracle import bf16_to_float, bf16_ulp
    lut, mats, g1, g0, b, x0 = chain
    (gate, up, down) = mats[0]
    tcq.trellis_rmsnorm(x0, 1e-6, out=b["n"])
    tcq.trellis_gate_up_matvec(b["n"][0], gate[0], gate[1], up[0], up[1], lut, g1, out=b["h"][0])
    tcq.trellis_scatter(b["h"], down[0], down[1], lut, g0, splits=152, workspace=b["ws"], out=b["x"])
    torch.cuda.synchronize()
    h = host_bf16(b["h"])
    lut_h = synth.lut(77)
    # the down projection on the GPU's own h, sampled
    rng = np.random.default_rng(0)
    js = rng.integers(0, HID, 400)
    y, a = orc.sample(h, synth.codes(2, INTER, HID, K), INTER, HID, K, synth.scales(2, INTER), lut_h, 0,
                      np.zeros(400, np.int64), js)
    ok, err, bound = orc.within_tolerance(host_bf16(b["x"])[0, js], y, a)
    assert ok.all(), (err[~ok][:4], bound[~ok][:4])
    # h is silu(gate) * up of the two projections on the GPU's own n, and
    # those projections agree with the oracle
    n = host_bf16(b["n"])
    g_gpu = tcq.trellis_matvec(b["n"][0], gate[0], gate[1], lut, g1)
    u_gpu = tcq.trellis_matvec(b["n"][0], up[0], up[1], lut, g1)
    assert np.array_equal(h[0], host_bf16(tcq.trellis_silu_mul(g_gpu, u_gpu)))
    for seed, got in ((0, g_gpu), (1, u_gpu)):
        w, _ = orc.expand(synth.codes(seed, INTER, HID, K), INTER, HID, K, synth.scales(seed, INTER), lut_h)
        y, a, _ = orc.matmul_axis1(n, w)
        ok, err, bound = orc.within_tolerance(host_bf16(got)[None, :], y, a)
        assert ok.all(), (seed, err[~ok][:4], bound[~ok][:4])
    ref = orc.silu_mul(host_bf16(g_gpu)[None, :], host_bf16(u_gpu)[None, :])
    fa, fb = bf16_to_float(h).astype(np.float64), bf16_to_float(ref).astype(np.float64)
    assert np.all(np.abs(fa - fb) <= bf16_ulp(np.maximum(np.abs(fa), np.abs(fb))))
