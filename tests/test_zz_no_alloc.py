"""trellis_scatter_noalloc: the axis-0 scatter for callers that cannot
allocate device memory (for example plugin interfaces that hand a kernel only
its input and output buffers, or serving loops where cudaMalloc's implicit
device synchronisation is not allowed).  Its split partials live in the
library's own 21 MiB device array instead of a caller workspace.

Checked through the C ABI against the ordinary trellis_scatter (which gets a
workspace from the caller) and against the oracle's tolerance, on two calls in
a row that reuse the shared array, and for the size limit.  This file is
collected last and builds and loads everything it needs, so it passes alone
in a fresh process as well as after the other tests.
"""
import numpy as np
import pytest

import trellis_coded_quantized_gb300 as tcq
from trellis_coded_quantized_gb300 import synth
from conftest import has_gpu
from gpu_util import host_bf16, on_device

pytestmark = [pytest.mark.gpu, pytest.mark.skipif(not has_gpu(), reason="needs a CUDA GPU")]


@pytest.fixture(scope="module", autouse=True)
def _built():
    from trellis_coded_quantized_gb300 import build
    build.build()


def test_noalloc_matches_scatter_on_two_calls_in_a_row(orc):
    import torch
    rows, cols, k = 17408, 5120, 3
    # first call M=4, second call M=1 on other inputs: the second reuses (and
    # must fully overwrite) the partials the first left in the shared array
    for M, seed in ((4, 0), (1, 21)):
        p = synth.problem(0, M, rows, cols, k, seed=seed)
        d = on_device(p)
        ref = tcq.trellis_scatter(d["x"], d["codes"], d["scales"], d["lut"], d["g"], splits=128)
        out = torch.empty((M, cols), dtype=torch.bfloat16, device="cuda")
        torch.cuda.synchronize()
        held = torch.cuda.memory_allocated()
        tcq.trellis_scatter_noalloc(d["x"], d["codes"], d["scales"], d["lut"], d["g"], splits=128, out=out)
        # (the holdings may drop when Python frees a tensor of the previous round meanwhile)
        assert torch.cuda.memory_allocated() <= held, "the call with out given took memory from the allocator"
        torch.cuda.synchronize()
        got, want = host_bf16(out), host_bf16(ref)
        W, _ = orc.expand(p["codes"], rows, cols, k, p["scales"], p["lut"])
        y, a, _, _ = orc.matmul_axis0(p["x"], W)
        ok, _, _ = orc.within_tolerance(got, y, a)
        assert ok.all(), f"M={M}: {int((~ok).sum())} outputs outside tolerance"
        ok, _, _ = orc.within_tolerance(want, y, a)
        assert ok.all()
        assert np.array_equal(got, want), f"M={M}: differs from trellis_scatter"


def test_noalloc_rejects_partials_beyond_its_array():
    import torch
    rows, cols, k = 512, 5120, 3
    p = synth.problem(0, 32, rows, cols, k, seed=3)
    d = on_device(p)
    out = torch.empty((32, cols), dtype=torch.bfloat16, device="cuda")
    # 32 * 128 * 5120 floats is more than the 4,194,304 partials the array holds
    with pytest.raises(tcq.TrellisError, match="WORKSPACE"):
        tcq.trellis_scatter_noalloc(d["x"], d["codes"], d["scales"], d["lut"], d["g"], splits=128, out=out)
    # 6 * 128 * 5120 = 3,932,160 fits
    x6 = d["x"][:6].contiguous()
    o6 = out[:6]
    tcq.trellis_scatter_noalloc(x6, d["codes"], d["scales"], d["lut"], d["g"], splits=128, out=o6)
    ref = tcq.trellis_scatter(x6, d["codes"], d["scales"], d["lut"], d["g"], splits=128)
    torch.cuda.synchronize()
    assert np.array_equal(host_bf16(o6), host_bf16(ref))


@pytest.mark.parametrize("M", [5, 16])
def test_noalloc_tensor_core_path_with_fixups(orc, M):
    """From 5 rows the default split count (8 at 17408 x 5120) takes the
    stream-K tcgen05 scatter, whose CTAs that start inside a split leave
    their share in fix-up slots; here those slots live in the library's
    array after the partials.  Equal to trellis_scatter bit for bit, and
    within the oracle's tolerance."""
    import torch
    rows, cols, k = 17408, 5120, 3
    p = synth.problem(0, M, rows, cols, k, seed=31 + M)
    d = on_device(p)
    ref = tcq.trellis_scatter(d["x"], d["codes"], d["scales"], d["lut"], d["g"])
    out = torch.empty((M, cols), dtype=torch.bfloat16, device="cuda")
    tcq.trellis_scatter_noalloc(d["x"], d["codes"], d["scales"], d["lut"], d["g"], out=out)
    torch.cuda.synchronize()
    got, want = host_bf16(out), host_bf16(ref)
    assert np.array_equal(got, want), f"M={M}: differs from trellis_scatter"
    W, _ = orc.expand(p["codes"], rows, cols, k, p["scales"], p["lut"])
    y, a, _, _ = orc.matmul_axis0(p["x"], W)
    ok, _, _ = orc.within_tolerance(got, y, a)
    assert ok.all(), f"M={M}: {int((~ok).sum())} outputs outside tolerance"
