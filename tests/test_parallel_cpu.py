"""The packed matmuls split over ranks (trellis_coded_quantized_gb300.parallel),
on the CPU with two gloo ranks.

Each rank takes its rows of the packed matrix with the module's row ranges
and code slicing, computes its share with the oracle, and the module's
collectives combine the shares; rank 0 compares the result element by
element with the oracle on the whole matrix:
  - axis 1 (output rows split): the gathered bf16 output equals the
    unsplit oracle output bit for bit (each output row is computed whole);
  - axis 0 (input rows split): the f32 all-reduce of the ranks' sums, rounded
    to bf16, is within the contraction tolerance of the unsplit oracle, and
    equals bf16 of the f32 sum of the two shares;
both for the interleave-0 and the interleave-2 code layouts.
"""
import multiprocessing as mp
import os
import socket

import numpy as np
import pytest

from trellis_coded_quantized_gb300 import parallel, synth


def _inter(codes, rows, cols, k):
    wpb = 256 * k // 32
    return np.ascontiguousarray(codes.reshape(rows, cols // 512, 2 * wpb).transpose(1, 0, 2)).reshape(rows, -1)


def test_row_range_covers_and_balances():
    for n in (1, 7, 17408, 5120, 301):
        for world in (1, 2, 3, 8):
            if world > n:
                continue
            rs = [parallel.row_range(n, world, r) for r in range(world)]
            assert rs[0][0] == 0 and rs[-1][1] == n
            assert all(a[1] == b[0] for a, b in zip(rs, rs[1:]))
            sizes = [b - a for a, b in rs]
            assert max(sizes) - min(sizes) <= 1
    with pytest.raises(ValueError):
        parallel.row_range(10, 2, 2)


@pytest.mark.parametrize("interleave", [0, 2])
def test_shard_codes_decode_to_the_matrix_rows(orc, interleave):
    rows, cols, k = 37, 1024, 3
    p = synth.problem(0, 1, rows, cols, k, seed=71)
    codes = p["codes"] if interleave == 0 else _inter(p["codes"], rows, cols, k)
    W, _ = orc.expand(codes, rows, cols, k, p["scales"], p["lut"], interleave=interleave)
    for r0, r1 in ((0, 37), (0, 1), (5, 19), (36, 37)):
        c = parallel.shard_codes(codes, rows, cols, k, r0, r1, interleave)
        assert c.shape == (r1 - r0, parallel.words_per_row(cols, k))
        Ws, _ = orc.expand(c, r1 - r0, cols, k, p["scales"][r0:r1], p["lut"], interleave=interleave)
        assert np.array_equal(Ws, W[r0:r1])
    import torch
    t = torch.from_numpy(codes.view(np.int32))
    c = parallel.shard_codes(t, rows, cols, k, 5, 19, interleave)
    assert np.array_equal(c.numpy().view(np.uint32), parallel.shard_codes(codes, rows, cols, k, 5, 19, interleave))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


ROWS1, COLS1 = 301, 1024         # axis 1: 301 output rows split 150 / 151
ROWS0, COLS0 = 517, 512          # axis 0: 517 input rows split 258 / 259
K, M = 3, 5


def _rank(rank, world, port, interleave, q):
    try:
        import torch
        import torch.distributed as dist

        import oracle
        os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
        dist.init_process_group("gloo", rank=rank, world_size=world)
        orc = oracle.default()
        res = {}
        # axis 1: this rank's output rows
        p = synth.problem(1, M, ROWS1, COLS1, K, seed=72)
        codes = p["codes"] if interleave == 0 else _inter(p["codes"], ROWS1, COLS1, K)
        c, sc, r0, r1 = parallel.shard_matrix(codes, p["scales"], ROWS1, COLS1, K, world, rank, interleave)
        W, _ = orc.expand(c, r1 - r0, COLS1, K, sc, p["lut"], interleave=interleave)
        _, _, out = orc.matmul_axis1(p["x"], W)
        full = parallel.all_gather_columns(torch.from_numpy(out.view(np.int16)), ROWS1)
        res["axis1"] = full.numpy().view(np.uint16)
        # axis 0: this rank's input rows, an f32 sum, one all-reduce
        p = synth.problem(0, M, ROWS0, COLS0, K, seed=73)
        codes = p["codes"] if interleave == 0 else _inter(p["codes"], ROWS0, COLS0, K)
        c, sc, r0, r1 = parallel.shard_matrix(codes, p["scales"], ROWS0, COLS0, K, world, rank, interleave)
        W, _ = orc.expand(c, r1 - r0, COLS0, K, sc, p["lut"], interleave=interleave)
        y, _, _, _ = orc.matmul_axis0(np.ascontiguousarray(p["x"][:, r0:r1]), W)
        mine = torch.from_numpy(y.astype(np.float32))
        res["axis0_share"] = mine.numpy().copy()
        parallel.all_reduce_sum(mine)
        res["axis0_sum"] = mine.numpy()
        dist.barrier()
        dist.destroy_process_group()
        q.put((rank, res))
    except Exception as e:
        q.put((rank, {"error": repr(e)}))


@pytest.mark.parametrize("interleave", [0, 2])
def test_two_gloo_ranks_match_the_unsplit_oracle(orc, interleave):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, interleave, q)) for r in range(2)]
    for pr in procs:
        pr.start()
    got = dict(q.get(timeout=300) for _ in procs)
    for pr in procs:
        pr.join(timeout=60)
    for r in (0, 1):
        assert "error" not in got[r], got[r]
    # axis 1: bit-exact against the whole matrix, on both ranks
    p = synth.problem(1, M, ROWS1, COLS1, K, seed=72)
    W, _ = orc.expand(p["codes"], ROWS1, COLS1, K, p["scales"], p["lut"])
    _, _, out = orc.matmul_axis1(p["x"], W)
    for r in (0, 1):
        assert np.array_equal(got[r]["axis1"], out)
    # axis 0: the all-reduced f32 sum is the sum of the two shares, on both
    # ranks, and rounds to within the tolerance of the unsplit oracle
    p = synth.problem(0, M, ROWS0, COLS0, K, seed=73)
    W, _ = orc.expand(p["codes"], ROWS0, COLS0, K, p["scales"], p["lut"])
    y, a, _, _ = orc.matmul_axis0(p["x"], W)
    want = got[0]["axis0_share"] + got[1]["axis0_share"]
    for r in (0, 1):
        assert np.array_equal(got[r]["axis0_sum"], want)
    rounded = orc.bf16_from_float(got[0]["axis0_sum"])
    ok, _, _ = orc.within_tolerance(rounded, y, a)
    assert ok.all()
