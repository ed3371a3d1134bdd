"""Helpers of the GPU tests: move generated inputs to the device, bring
results back as bf16 bit patterns."""
from __future__ import annotations

import numpy as np

import trellis_coded_quantized_gb300 as tcq


def dev(a: np.ndarray):
    import torch
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        return torch.from_numpy(a.view(np.int16)).cuda().view(torch.bfloat16)
    if a.dtype == np.uint32:
        return torch.from_numpy(a.view(np.int32)).cuda()
    return torch.from_numpy(a).cuda()


def host_bf16(t) -> np.ndarray:
    import torch
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def on_device(p: dict) -> dict:
    g = tcq.geometry(p["axis"], p["rows"], p["cols"], p["k"], p.get("interleave", 0))
    return {"g": g, "codes": dev(p["codes"]), "scales": dev(p["scales"]), "lut": dev(p["lut"]),
            "x": dev(p["x"])}


def check_close(orc, got_bf16, y, a, what: str):
    ok, err, bound = orc.within_tolerance(got_bf16, y, a)
    if not ok.all():
        idx = np.argwhere(~ok)[:5]
        raise AssertionError(f"{what}: {int((~ok).sum())} of {ok.size} outside tolerance; "
                             f"first {idx.tolist()} err {err[~ok][:5]} bound {bound[~ok][:5]}")
