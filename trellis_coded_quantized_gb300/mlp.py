"""A synthetic stack of SwiGLU MLP layers whose weights are packed trellis codes.

Per layer l (the pages only say the prefill input is the RMSNorm output; the
SwiGLU chain is the plain reading of "Qwen's MLP geometry"):
    n = RMSNorm(x)                  unit gain, eps 1e-6
    g = gate(n), u = up(n)          axis 1, hidden -> intermediate
    h = bf16(silu(g) * u)
    x' = down(h)                    axis 0, intermediate -> hidden
Without a residual.  Layer l, matrix j (0 gate, 1 up, 2 down) is drawn with
seed 1000*l + j; all matrices share one codebook (the pages' codebook is one
fixed function of the window), drawn with seed CODEBOOK_SEED.  Gate, up and
silu*up run as one launch: trellis_gate_up_matvec at M = 1,
trellis_gate_up_prefill at M >= 2; down always uses trellis_scatter (split
count by M, see splits_for).  Every step runs in libtrellis kernels.
"""
from __future__ import annotations

import numpy as np

import trellis_coded_quantized_gb300 as tcq
from . import synth

HIDDEN = 5120
INTER = 17408
CODEBOOK_SEED = 7919


class Layer:
    def __init__(self, l: int, k: int, device, hidden: int, inter: int, lut):
        import torch
        self.mats = []
        for j, (axis, rows, cols) in enumerate(((1, inter, hidden), (1, inter, hidden), (0, inter, hidden))):
            seed = 1000 * l + j
            codes = synth.codes_torch(seed, rows, cols, k, device)
            scales = torch.from_numpy(synth.scales(seed, rows).view(np.int16)).to(device).view(torch.bfloat16)
            self.mats.append({"g": tcq.geometry(axis, rows, cols, k), "codes": codes,
                              "scales": scales, "lut": lut, "seed": seed})


class PackedMLPStack:
    def __init__(self, layers: int = 40, k: int = 3, device="cuda", m_max: int = 16,
                 hidden: int = HIDDEN, inter: int = INTER, splits: int | None = None):
        import torch
        self.sm_count = torch.cuda.get_device_properties(device).multi_processor_count
        self.k, self.hidden, self.inter, self.splits = k, hidden, inter, splits
        self.lut = torch.from_numpy(synth.lut(CODEBOOK_SEED)).to(device)
        self.layers = [Layer(l, k, device, hidden, inter, self.lut) for l in range(layers)]
        self.device = device
        self.m_max = m_max
        bf = torch.bfloat16
        self.n = torch.empty((m_max, hidden), dtype=bf, device=device)
        self.gate = torch.empty((m_max, inter), dtype=bf, device=device)
        self.up = torch.empty((m_max, inter), dtype=bf, device=device)
        self.h = torch.empty((m_max, inter), dtype=bf, device=device)
        self.xs = [torch.empty((m_max, hidden), dtype=bf, device=device) for _ in range(2)]
        g0 = self.layers[0].mats[2]["g"]
        most = max(self.splits_for(M) for M in range(1, m_max + 1))
        self.ws = torch.empty(tcq.trellis_scatter_workspace_bytes(g0, m_max, most) // 4,
                              dtype=torch.float32, device=device)

    def splits_for(self, M: int) -> int:
        """Row splits of the down projection: the constructor's, else one per
        SM for the FMA scatter (M <= 2), and from M = 3 the split-K
        launcher's count (the library's default from M = 5: the power of two
        at or above floor(tilesK / (tilesM * tilesN)), clamped to [2, 32];
        8 for 17408 x 5120), which keeps the call on the tcgen05 scatter and
        its stream-K schedule (at 8 splits 52-57 us at M = 4..16, against
        56-86 us at 128 or more)."""
        if self.splits:
            return self.splits
        if M <= 2:
            return self.sm_count
        tiles_m = -(-M // 32)
        tiles_n = -(-self.hidden // 32)
        ratio = max(1, (self.inter // 16) // (tiles_m * tiles_n))
        p2 = 1
        while p2 < ratio:
            p2 <<= 1
        return min(32, max(2, p2))

    @property
    def packed_bytes(self) -> int:
        return len(self.layers) * 3 * self.inter * self.hidden * self.k // 8

    def launches_per_pass(self, M: int) -> int:
        # rmsnorm; gate+up+silu fused; the scatter (one FMA pass up to 2
        # rows, one tensor-core pass from 3); the split reduction
        return len(self.layers) * (1 + 1 + 1 + 1)

    def layer(self, l: int, x, out, keep=None):
        """One layer on x [M, hidden] into out [M, hidden]."""
        M = x.shape[0]
        gate, up, down = self.layers[l].mats
        n, g, u, h = self.n[:M], self.gate[:M], self.up[:M], self.h[:M]
        tcq.trellis_rmsnorm(x, 1e-6, out=n)
        if M == 1:
            tcq.trellis_gate_up_matvec(n[0], gate["codes"], gate["scales"], up["codes"], up["scales"], self.lut,
                                       gate["g"], out=h[0])
            if keep is not None:        # the two projections on their own, for stage checks
                tcq.trellis_matvec(n[0], gate["codes"], gate["scales"], self.lut, gate["g"], out=g[0])
                tcq.trellis_matvec(n[0], up["codes"], up["scales"], self.lut, up["g"], out=u[0])
        else:
            tcq.trellis_gate_up_prefill(n, gate["codes"], gate["scales"], up["codes"], up["scales"], self.lut,
                                        gate["g"], out=h)
            if keep is not None:        # the two projections on their own, for stage checks
                tcq.trellis_prefill(n, gate["codes"], gate["scales"], self.lut, gate["g"], out=g)
                tcq.trellis_prefill(n, up["codes"], up["scales"], self.lut, up["g"], out=u)
        tcq.trellis_scatter(h, down["codes"], down["scales"], self.lut, down["g"], splits=self.splits_for(M),
                            workspace=self.ws, out=out)
        if keep is not None:
            keep.append({"x": x.clone(), "n": n.clone(), "g": g.clone(), "u": u.clone(), "h": h.clone(),
                         "out": out.clone()})
        return out

    def forward(self, x, layers: int | None = None, keep=None, check: bool = True):
        """All layers (or the first `layers`) on x [M, hidden]; returns the last output.

        With `check` the pass ends by reading the library's device status
        (which synchronises the device) and raises when a kernel's bounded
        wait gave up: that kernel skipped its output, so the rows of every
        later layer would be undefined.  Timed loops and CUDA-graph capture
        pass check=False and read the status once afterwards."""
        M = x.shape[0]
        assert 1 <= M <= self.m_max
        cur = x
        nl = len(self.layers) if layers is None else layers
        for l in range(nl):
            nxt = self.xs[l % 2][:M]
            self.layer(l, cur, nxt, keep)
            cur = nxt
        if check:
            status = tcq.trellis_device_status()
            if status != 0:
                raise RuntimeError(f"a kernel of the MLP pass gave up a bounded wait (device status {status}); "
                                   "the pass output is undefined")
        return cur
