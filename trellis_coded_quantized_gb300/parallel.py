"""The packed matmuls split over several GPUs: one process per GPU,
torch.distributed for the exchange (NCCL between GPUs, gloo on the CPU).

Both axes split the way the method's own split-K structure does
(@mlx-bun/inference 1.0.0, kernels/trellis/scatter.ts and splitk-prefill.ts:
row ranges whose fp32 partial sums are added before the one rounding):

  axis 1 (rows are output features, gate/up): rank i holds the output rows
      row_range(N, world, i) of the codes and scales and computes its slice
      of the output with no exchange; all_gather_columns assembles the full
      output where a caller needs it;
  axis 0 (rows are input features, down): rank i holds the input rows
      row_range(R, world, i) and the matching columns of x, computes the f32
      sum over its rows (trellis_scatter_f32), all_reduce_sum adds the
      ranks' sums in f32, and trellis_round_bf16 rounds once.

A SwiGLU layer with gate/up split by intermediate rows and down split by the
same input rows therefore needs one all-reduce of [M, hidden] f32 per layer
(tp_mlp_layer).  The data plane is plain torch.distributed collectives on
device tensors; nothing here multicasts.

The host-side pieces (row ranges, slicing the packed codes, the collectives)
work on CPU tensors with the gloo backend as well, which is how they are
tested without several GPUs.
"""
from __future__ import annotations

import numpy as np

BT = 256


def row_range(n: int, world: int, rank: int) -> tuple[int, int]:
    """Contiguous, balanced rows [start, stop) of rank `rank` out of `world`:
    the first n % world ranks get one row more."""
    if world < 1 or not 0 <= rank < world:
        raise ValueError("rank out of range")
    return n * rank // world, n * (rank + 1) // world


def words_per_row(cols: int, k: int) -> int:
    return (cols // BT) * (BT * k // 32)


def shard_codes(codes, rows: int, cols: int, k: int, r0: int, r1: int, interleave: int = 0):
    """The packed codes of rows [r0, r1) of a rows x cols matrix, in the same
    block layout, shaped [r1 - r0, words per row].  Works on numpy arrays and
    torch tensors (CPU or device) alike.

    interleave 0: the blocks of a row are contiguous, so the shard is rows
    r0..r1 of the [rows, words] array.  interleave 2: block pair q of row r
    sits at ((q * rows) + r) * 2 * wpb, so the array is [pairs, rows, 2 wpb]
    and the shard takes rows r0..r1 of every pair (a gather into a new
    contiguous array)."""
    if not 0 <= r0 < r1 <= rows:
        raise ValueError("empty or out-of-range row shard")
    wpr = words_per_row(cols, k)
    if interleave == 0:
        out = codes.reshape(rows, wpr)[r0:r1]
    elif interleave == 2:
        wpb = BT * k // 32
        pairs = cols // (2 * BT)
        out = codes.reshape(pairs, rows, 2 * wpb)[:, r0:r1, :]
    else:
        raise ValueError("interleave must be 0 or 2")
    if isinstance(out, np.ndarray):
        return np.ascontiguousarray(out).reshape(r1 - r0, wpr)
    return out.contiguous().reshape(r1 - r0, wpr)


def shard_matrix(codes, scales, rows: int, cols: int, k: int, world: int, rank: int, interleave: int = 0):
    """(codes, scales, r0, r1) of this rank's rows of a packed matrix."""
    r0, r1 = row_range(rows, world, rank)
    return shard_codes(codes, rows, cols, k, r0, r1, interleave), scales[r0:r1], r0, r1


def all_reduce_sum(t, group=None):
    """In-place sum over the ranks of an f32 tensor (the axis-0 partial sums)."""
    import torch.distributed as dist
    dist.all_reduce(t, op=dist.ReduceOp.SUM, group=group)
    return t


def all_gather_columns(local, n_total: int, group=None):
    """Concatenate the ranks' column slices [M, n_i] (in rank order, n_i from
    row_range) into [M, n_total].  Slices of unequal width are padded to the
    widest for the collective and trimmed after it."""
    import torch
    import torch.distributed as dist
    world = dist.get_world_size(group)
    widths = [b - a for a, b in (row_range(n_total, world, r) for r in range(world))]
    wmax = max(widths)
    M = local.shape[0]
    dtype = local.dtype
    send = local
    # gloo has no 16-bit integer collectives: bf16 bit patterns travel as
    # int32 there (exact both ways)
    narrow = dist.get_backend(group) == "gloo" and dtype in (torch.int16, torch.bfloat16)
    if narrow:
        send = (local.view(torch.int16) if dtype == torch.bfloat16 else local).to(torch.int32)
    pad = torch.zeros((M, wmax), dtype=send.dtype, device=send.device)
    pad[:, :send.shape[1]] = send
    parts = [torch.empty_like(pad) for _ in range(world)]
    dist.all_gather(parts, pad, group=group)
    out = torch.cat([p[:, :w] for p, w in zip(parts, widths)], dim=1)
    if narrow:
        out = out.to(torch.int16)
        if dtype == torch.bfloat16:
            out = out.view(torch.bfloat16)
    return out


# ---------------------------------------------------------------------------
# device paths (each rank on its own GPU)
# ---------------------------------------------------------------------------

def axis1_forward(x, codes, scales, lut, g_local, out=None):
    """This rank's output rows of an axis-1 projection: x bf16 [M, cols] ->
    [M, rows of the shard] (matvec at M = 1, the tensor-core prefill else)."""
    import trellis_coded_quantized_gb300 as tcq
    if x.shape[0] == 1:
        y = tcq.trellis_matvec(x[0], codes, scales, lut, g_local, out=None if out is None else out[0])
        return y.reshape(1, -1)
    return tcq.trellis_prefill(x, codes, scales, lut, g_local, out=out)


def axis0_forward(x_local, codes, scales, lut, g_local, group=None, splits: int = 0, workspace=None):
    """An axis-0 projection split by input rows: x_local bf16 [M, rows of the
    shard] -> bf16 [M, cols] on every rank, through this rank's f32 partial
    sum, one f32 all-reduce and the one rounding."""
    import trellis_coded_quantized_gb300 as tcq
    y32 = tcq.trellis_scatter_f32(x_local, codes, scales, lut, g_local, splits=splits, workspace=workspace)
    all_reduce_sum(y32, group)
    return tcq.trellis_round_bf16(y32)


def tp_mlp_layer(x, gate, up, down, lut, group=None, splits: int = 0):
    """One SwiGLU layer split over the ranks by intermediate rows: RMSNorm of
    the full x (every rank), this rank's rows of gate and up, its slice of
    h = silu(g) * u, and the down projection over the same intermediate rows
    with one f32 all-reduce.  gate/up/down are dicts {codes, scales, g} of
    this rank's shard (g: the shard's geometry).  Returns bf16 [M, hidden]."""
    import trellis_coded_quantized_gb300 as tcq
    n = tcq.trellis_rmsnorm(x, 1e-6)
    gl = axis1_forward(n, gate["codes"], gate["scales"], lut, gate["g"])
    ul = axis1_forward(n, up["codes"], up["scales"], lut, up["g"])
    h = tcq.trellis_silu_mul(gl, ul)
    return axis0_forward(h, down["codes"], down["scales"], lut, down["g"], group, splits=splits)
