"""The device side of the multi-GPU split (trellis_scatter_f32,
trellis_round_bf16, parallel.axis0_forward / tp_mlp_layer) on one GPU.

Only one GPU is available, so the split runs with a single rank (NCCL,
world size 1, in a spawned child): the shard is the whole matrix and the
all-reduce is the identity, which pins the device path bit for bit against
the unsplit entry points.  The exchange itself between several ranks is
tested with gloo on the CPU (test_parallel_cpu.py).
"""
import multiprocessing as mp
import os
import socket

import numpy as np
import pytest

import trellis_coded_quantized_gb300 as tcq
from trellis_coded_quantized_gb300 import synth
from gpu_util import check_close, dev, host_bf16, on_device
from conftest import has_gpu

pytestmark = [pytest.mark.gpu, pytest.mark.skipif(not has_gpu(), reason="needs a CUDA GPU")]


@pytest.mark.parametrize("M,splits", [(1, 128), (2, 0), (4, 128), (16, 0), (32, 8)])
def test_scatter_f32_is_the_unrounded_sum(orc, M, splits):
    rows, cols, k = 2048, 5120, 3
    p = synth.problem(0, M, rows, cols, k, seed=81)
    d = on_device(p)
    y32 = tcq.trellis_scatter_f32(d["x"], d["codes"], d["scales"], d["lut"], d["g"], splits=splits)
    ref = tcq.trellis_scatter(d["x"], d["codes"], d["scales"], d["lut"], d["g"], splits=splits)
    got = y32.cpu().numpy()
    # the bf16 entry point rounds exactly this sum
    assert np.array_equal(orc.bf16_from_float(got), host_bf16(ref))
    assert np.array_equal(host_bf16(tcq.trellis_round_bf16(y32)), host_bf16(ref))
    W, _ = orc.expand(p["codes"], rows, cols, k, p["scales"], p["lut"])
    y, a, _, _ = orc.matmul_axis0(p["x"], W)
    assert np.all(np.abs(got.astype(np.float64) - y) <= 4e-3 * a + 1e-6)


def test_round_bf16_matches_the_oracle_rounding(orc):
    import torch
    rng = np.random.default_rng(82)
    v = rng.standard_normal(100003).astype(np.float32) * np.float32(3.0)
    # exact ties at the bf16 spacing, both parities, and the edges of the range
    ties = (np.arange(1, 2049, dtype=np.uint32) << 16 | 0x8000).view(np.float32)
    edge = np.array([0.0, -0.0, 1e-40, -1e-40, 3.3e38, -3.3e38, np.inf, -np.inf], np.float32)
    v = np.concatenate([v, ties, -ties, edge])
    got = host_bf16(tcq.trellis_round_bf16(torch.from_numpy(v).cuda()))
    assert np.array_equal(got, orc.bf16_from_float(v))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _single_rank(port, q):
    try:
        import torch
        import torch.distributed as dist

        from trellis_coded_quantized_gb300 import parallel
        from trellis_coded_quantized_gb300.mlp import PackedMLPStack
        os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
        torch.cuda.set_device(0)
        dist.init_process_group("nccl", rank=0, world_size=1)
        res = {}
        stack = PackedMLPStack(layers=1, k=3, device="cuda", m_max=16)
        for M in (1, 16):
            x = torch.from_numpy(synth.activations(5, M, stack.hidden).view(np.int16)).cuda().view(torch.bfloat16)
            want = stack.layer(0, x, torch.empty_like(x))
            gate, up, down = stack.layers[0].mats
            got = parallel.tp_mlp_layer(x, gate, up, down, stack.lut, splits=stack.splits_for(M))
            torch.cuda.synchronize()
            res[M] = bool(torch.equal(got.view(torch.int16), want.view(torch.int16)))
        dist.destroy_process_group()
        q.put(res)
    except Exception as e:
        q.put({"error": repr(e)})


def test_split_mlp_layer_on_one_rank_is_the_unsplit_layer():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    proc = ctx.Process(target=_single_rank, args=(_free_port(), q))
    proc.start()
    res = q.get(timeout=600)
    proc.join(timeout=60)
    assert "error" not in res, res
    assert res == {1: True, 16: True}
