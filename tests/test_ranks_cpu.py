"""The multi-rank path of bench.py on CPU: two gloo ranks, each with its own
independent problem (weak scaling, no collective on the data path), agree on
the slowest rank's time, and the whole-job throughput counts every rank."""
import os
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _rank_main(rank, world, port, q):
    sys.path.insert(0, ROOT)
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        r, lr, w = bench.env_rank()
        # rank r "took" 10 + 5 r milliseconds
        slowest = bench.max_over_ranks(torch, dist, 10.0 + 5.0 * rank, torch.device("cpu"))
        dist.barrier()
        q.put((r, lr, w, slowest))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_agree_on_the_slowest_time():
    world, port = 2, 29531
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(world))
    assert [g[0] for g in got] == [0, 1] and all(g[2] == world for g in got)
    assert all(g[3] == 15.0 for g in got)


def test_whole_job_throughput_and_single_rank():
    sys.path.insert(0, ROOT)
    import bench
    # 4 ranks each processing 1e9 bytes in 0.5 s -> 8e9 bytes/s for the job
    assert bench.job_throughput(1e9, 4, 0.5) == 8e9
    assert bench.max_over_ranks(torch, None, 3.25, torch.device("cpu")) == 3.25


def test_reference_arm_other_ranks_print_nothing(capsys, monkeypatch):
    sys.path.insert(0, ROOT)
    import bench
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")

    class Args:
        workload, M, k, splits, steps, warmup = "decode-matvec", 0, 0, 0, 1, 3
    bench.run_reference(Args())
    assert capsys.readouterr().out == ""
