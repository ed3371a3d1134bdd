"""Failure detection without a GPU fault: a bounded device-side wait that
runs out.

The kernels never trap or spin without a limit: every mbarrier wait gives up
after a wall-clock limit, sets the CTA's abort flag so that the other warps
leave their loops, skips the output, frees its tensor memory and records
kStatusWaitTimeout in the device status word that trellis_device_status()
reads and clears.  Here a test-only build of the library
(build.build_test_hooks: 50 ms wait limit, and an extra export that makes the
prefill's code-loader warp withhold one arrival on the first code tile of CTA
0) makes that wait run out once.  The test checks that the call returns, that
the status reports the timeout once and is then clear, and that the next
normal call on the same context is correct.

The library under test runs in a spawned child process, so that its second
copy of the CUDA runtime never shares a process with the product library.
"""
import multiprocessing as mp

import numpy as np
import pytest

from conftest import has_gpu

pytestmark = [pytest.mark.gpu, pytest.mark.skipif(not has_gpu(), reason="needs a CUDA GPU")]

ROWS, COLS, K, M = 300, 512, 3, 8


def _child(q):
    try:
        import ctypes
        import time

        import torch

        from trellis_coded_quantized_gb300 import _lib, build, geometry, synth

        lib = _lib.bind(ctypes.CDLL(build.build_test_hooks()))
        lib.trellis_test_set_withhold.argtypes = [ctypes.c_int]
        lib.trellis_test_set_withhold.restype = ctypes.c_int
        torch.cuda.set_device(0)
        p = synth.problem(1, M, ROWS, COLS, K, seed=61)
        codes = torch.from_numpy(p["codes"].view(np.int32)).cuda()
        scales = torch.from_numpy(p["scales"].view(np.int16)).cuda()
        lut = torch.from_numpy(p["lut"]).cuda()
        x = torch.from_numpy(p["x"].view(np.int16)).cuda()
        out = torch.zeros((M, ROWS), dtype=torch.int16, device="cuda")
        g = geometry(1, ROWS, COLS, K)

        def status():
            v = ctypes.c_int32(-1)
            rc = lib.trellis_device_status(ctypes.byref(v))
            return rc, int(v.value)

        def prefill():
            return lib.trellis_prefill(ctypes.c_void_p(x.data_ptr()), M, ctypes.c_void_p(codes.data_ptr()),
                                       ctypes.c_void_p(scales.data_ptr()), ctypes.c_void_p(lut.data_ptr()),
                                       ctypes.byref(g), ctypes.c_void_p(out.data_ptr()), None)

        res = {"before": status()}
        res["set"] = lib.trellis_test_set_withhold(1)
        t0 = time.perf_counter()
        res["rc_withheld"] = prefill()
        torch.cuda.synchronize()
        res["seconds"] = time.perf_counter() - t0
        res["after_withheld"] = status()
        res["after_clear"] = status()
        res["unset"] = lib.trellis_test_set_withhold(0)
        res["rc_normal"] = prefill()
        torch.cuda.synchronize()
        res["after_normal"] = status()
        res["out"] = out.cpu().numpy().view(np.uint16).copy()
        q.put(res)
    except Exception as e:          # report to the parent instead of hanging it
        q.put({"error": repr(e)})


def test_prefill_wait_runs_out_and_the_next_call_is_correct(orc):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    proc = ctx.Process(target=_child, args=(q,))
    proc.start()
    try:
        res = q.get(timeout=900)
    finally:
        proc.join(timeout=60)
    assert "error" not in res, res.get("error")
    assert proc.exitcode == 0
    assert res["before"] == (0, 0)
    assert res["set"] == 0 and res["unset"] == 0
    assert res["rc_withheld"] == 0                      # enqueued; the kernel itself gave up
    assert res["after_withheld"] == (0, 1)              # kStatusWaitTimeout, read once ...
    assert res["after_clear"] == (0, 0)                 # ... and cleared by the read
    assert 0.04 <= res["seconds"] < 10.0                # the 50 ms limit, not a hang
    assert res["rc_normal"] == 0 and res["after_normal"] == (0, 0)
    from trellis_coded_quantized_gb300 import synth
    p = synth.problem(1, M, ROWS, COLS, K, seed=61)
    W, _ = orc.expand(p["codes"], ROWS, COLS, K, p["scales"], p["lut"])
    y, a, _ = orc.matmul_axis1(p["x"], W)
    ok, _, _ = orc.within_tolerance(res["out"], y, a)
    assert ok.all(), f"{int((~ok).sum())} outputs of the call after the timeout outside tolerance"
