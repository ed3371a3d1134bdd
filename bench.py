#!/usr/bin/env python3
"""Benchmark of the packed trellis-coded weight matmul on GB300.

Default workload (one step = one pass of the hot path over one input):
  decode matvec, axis 1: M=1, K=5120 in, N=17408 out, k=4, BT=256, L=12,
  seeded synthetic codes/codebook/scales/activations.
Metric: packed-weight GB/s (packed code bytes / time), higher is better.

Timing: W untimed warm-up steps, then K timed steps bracketed by a barrier and
torch.cuda.synchronize(); every launch is also bracketed by CUDA events on the
stream it runs on (the kernel's average duration feeds the roofline).  Steps
rotate over weight sets totalling > 4x L2, so every step streams its codes
from HBM.  nvidia-smi samples clocks during the timed region.

`--impl reference` times the CPU oracle (the only reference there is) on a
bounded sample of the same workload.  Under torchrun each rank runs its own
independent problem (weak scaling, no collective on the data path).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

M1, K1, N1, KB1 = 1, 5120, 17408, 4          # the decode-matvec workload
PACKED_BYTES = N1 * K1 * KB1 // 8             # 44,564,480
WORKLOAD = "decode matvec axis-1: M=1, K=5120, N=17408, k=4, BT=256, L=12"
METRIC = "packed-weight GB/s & % HBM roofline (M=1); TFLOP/s & % roofline (M=5..32)"


def env_rank():
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("LOCAL_RANK", "0")),
            int(os.environ.get("WORLD_SIZE", "1")))


def measured_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return json.load(f), "measured"
    except Exception:
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, "fallback"


def profiled_traffic(kernel_file: str):
    """dram bytes per launch from profiles/<...>.md when it was captured on the
    current source of the kernel (the summary records the source's sha1)."""
    src = os.path.join(ROOT, "trellis_coded_quantized_gb300", "csrc", kernel_file)
    try:
        sha = hashlib.sha1(open(src, "rb").read()).hexdigest()[:12]
    except OSError:
        return None
    pdir = os.path.join(ROOT, "profiles")
    if not os.path.isdir(pdir):
        return None
    for name in sorted(os.listdir(pdir)):
        if not name.endswith(".md"):
            continue
        text = open(os.path.join(pdir, name)).read()
        m = re.search(r"traffic_per_launch_bytes:\s*(\d+)\s+source_sha1:\s*([0-9a-f]+)\s+kernel_file:\s*(\S+)", text)
        if m and m.group(3) == kernel_file and m.group(2) == sha:
            return int(m.group(1))
    return None


class ClockSampler:
    """nvidia-smi clock / throttle samples every 200 ms while running."""
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax.append(float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax),
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------------------
# our arm
# ---------------------------------------------------------------------------

def make_sets(torch, tcq, nsets: int, device):
    from trellis_coded_quantized_gb300 import synth
    p = synth.problem(1, M1, N1, K1, KB1, seed=0)
    codes0 = torch.from_numpy(p["codes"].view(np.int32)).to(device)
    scales = torch.from_numpy(p["scales"].view(np.int16)).to(device).view(torch.bfloat16)
    lut = torch.from_numpy(p["lut"]).to(device)
    x = torch.from_numpy(p["x"].view(np.int16)).to(device).view(torch.bfloat16)[0]
    # further weight sets: the first XOR a per-set constant (still uniform codes)
    sets = [codes0] + [codes0 ^ int(np.int32(np.uint32((0x9E3779B9 * (j + 1)) & 0xFFFFFFFF)))
                       for j in range(1, nsets)]
    return p, sets, scales, lut, x


def time_launches(torch, fn, steps, warmup, stream, barrier):
    for i in range(warmup):
        fn(i)
    torch.cuda.synchronize()
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    barrier()
    torch.cuda.synchronize()
    t0.record(stream)
    for i in range(steps):
        starts[i].record(stream)
        fn(warmup + i)
        ends[i].record(stream)
    t1.record(stream)
    torch.cuda.synchronize()
    barrier()
    total_ms = t0.elapsed_time(t1)
    per = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    return total_ms, per


def extra_configs(torch, tcq, device, stream, peaks):
    """Throughput of the other configurations (secondary figures)."""
    from trellis_coded_quantized_gb300 import synth
    out = {}
    hbm = peaks["hbm_gbs"]
    tc_peak = peaks["bf16_tflops"]
    reps = 30
    # prefill M x k (axis 1, K=5120, N=17408)
    for k in (2, 3, 4):
        p = synth.problem(1, 32, N1, K1, k, seed=0)
        codes = [torch.from_numpy(p["codes"].view(np.int32)).to(device)]
        codes += [codes[0] ^ int(np.int32(np.uint32((0x85EBCA6B * (j + 1)) & 0xFFFFFFFF))) for j in range(1, 8)]
        sc = torch.from_numpy(p["scales"].view(np.int16)).to(device).view(torch.bfloat16)
        lut = torch.from_numpy(p["lut"]).to(device)
        g = tcq.geometry(1, N1, K1, k)
        packed = N1 * K1 * k // 8
        for M in (5, 8, 16, 32):
            x = torch.from_numpy(p["x"][:M].view(np.int16)).to(device).view(torch.bfloat16)
            o = torch.empty((M, N1), dtype=torch.bfloat16, device=device)
            fn = lambda i: tcq.trellis_prefill(x, codes[i % len(codes)], sc, lut, g, out=o)
            _, per = time_launches(torch, fn, reps, 3, stream, lambda: None)
            t = statistics.median(per) * 1e-3
            flops = 2.0 * M * N1 * K1
            roof = min(hbm * 1e9 * flops / packed, tc_peak * 1e12)
            out[f"prefill_M{M}_k{k}"] = {
                "us": round(t * 1e6, 2), "tflops": round(flops / t / 1e12, 2),
                "packed_gbs": round(packed / t / 1e9, 1), "tokens_per_s": round(M / t, 1),
                "frac_of_roofline": round(flops / t / roof, 4)}
    # scatter (axis 0, R=17408, C=5120, k=3, 128 splits)
    p = synth.problem(0, 4, N1, K1, 3, seed=0)
    codes = [torch.from_numpy(p["codes"].view(np.int32)).to(device)]
    codes += [codes[0] ^ int(np.int32(np.uint32((0xC2B2AE35 * (j + 1)) & 0xFFFFFFFF))) for j in range(1, 8)]
    sc = torch.from_numpy(p["scales"].view(np.int16)).to(device).view(torch.bfloat16)
    lut = torch.from_numpy(p["lut"]).to(device)
    g = tcq.geometry(0, N1, K1, 3)
    packed = N1 * K1 * 3 // 8
    for M in (1, 4):
        x = torch.from_numpy(p["x"][:M].view(np.int16)).to(device).view(torch.bfloat16)
        ws = torch.empty(tcq.trellis_scatter_workspace_bytes(g, M, 128) // 4, dtype=torch.float32, device=device)
        o = torch.empty((M, K1), dtype=torch.bfloat16, device=device)
        fn = lambda i: tcq.trellis_scatter(x, codes[i % len(codes)], sc, lut, g, splits=128, workspace=ws, out=o)
        _, per = time_launches(torch, fn, reps, 3, stream, lambda: None)
        t = statistics.median(per) * 1e-3
        out[f"scatter_M{M}_k3_s128"] = {"us": round(t * 1e6, 2), "packed_gbs": round(packed / t / 1e9, 1),
                                        "frac_of_hbm": round(packed / t / 1e9 / hbm, 4),
                                        "tokens_per_s": round(M / t, 1)}
    # shared-memory gather rate (the decode's other roofline)
    lut = torch.randn(4096, device=device)
    sm = torch.cuda.get_device_properties(device).multi_processor_count
    iters = 2000
    fn = lambda i: tcq.trellis_gather_probe(lut, sm, iters)
    _, per = time_launches(torch, fn, 5, 2, stream, lambda: None)
    t = statistics.median(per) * 1e-3
    gathers = sm * 1024 * iters * 8
    out["smem_gather"] = {"gathers_per_s": gathers / t, "per_sm_per_clock_at_max": gathers / t / sm / 2.07e9}
    return out


def run_ours(args):
    import torch
    import trellis_coded_quantized_gb300 as tcq
    rank, local_rank, world = env_rank()
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    torch.cuda.set_device(local_rank)
    device = torch.device("cuda", local_rank)
    stream = torch.cuda.current_stream()
    barrier = (lambda: dist.barrier()) if dist else (lambda: None)
    peaks, peak_src = measured_peaks()

    l2 = torch.cuda.get_device_properties(device).L2_cache_size
    nsets = max(4, int(np.ceil(4 * l2 / PACKED_BYTES)) + 1)
    p, sets, scales, lut, x = make_sets(torch, tcq, nsets, device)
    g = tcq.geometry(1, N1, K1, KB1)
    out = torch.empty(N1, dtype=torch.bfloat16, device=device)

    def step(i):
        tcq.trellis_matvec(x, sets[i % nsets], scales, lut, g, out=out)

    with ClockSampler(local_rank) as clk:
        total_ms, per = time_launches(torch, step, args.steps, args.warmup, stream, barrier)
    ms = total_ms / args.steps
    if dist:
        t = torch.tensor([total_ms], device=device)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        total_ms = float(t.item())
        ms = total_ms / args.steps
    value = world * PACKED_BYTES * args.steps / (total_ms * 1e-3) / 1e9

    # roofline of the dominant kernel (the matvec: the only kernel of the step)
    kern_s = statistics.mean(per) * 1e-3
    alg_bytes = PACKED_BYTES + N1 * 2 + K1 * 2 + N1 * 2 + 4096 * 4
    achieved = alg_bytes / kern_s / 1e9
    roofline = {"bound": "hbm", "achieved": round(achieved, 1), "peak": peaks["hbm_gbs"],
                "unit": "GB/s", "frac": round(achieved / peaks["hbm_gbs"], 4),
                "traffic": profiled_traffic("matvec.cu"), "kernel": "matvec_kernel<4>",
                "peak_source": f"{peak_src} hbm_gbs (burst copy)",
                "kernel_us": round(kern_s * 1e6, 3)}

    # end to end: pinned host inputs -> device, matvec through the C ABI, result -> host
    e2e = None
    if rank == 0 or world > 1:
        h_codes = torch.from_numpy(p["codes"].view(np.int32)).pin_memory()
        h_scales = torch.from_numpy(p["scales"].view(np.int16)).pin_memory()
        h_lut = torch.from_numpy(p["lut"]).pin_memory()
        h_x = torch.from_numpy(p["x"][0].view(np.int16)).pin_memory()
        h_out = torch.empty(N1, dtype=torch.int16).pin_memory()
        d_codes = torch.empty_like(sets[0])
        d_scales = torch.empty(N1, dtype=torch.int16, device=device)
        d_lut = torch.empty(4096, dtype=torch.float32, device=device)
        d_x = torch.empty(K1, dtype=torch.int16, device=device)
        d_out = torch.empty(N1, dtype=torch.int16, device=device)

        def e2e_step(i):
            d_codes.copy_(h_codes, non_blocking=True)
            d_scales.copy_(h_scales, non_blocking=True)
            d_lut.copy_(h_lut, non_blocking=True)
            d_x.copy_(h_x, non_blocking=True)
            tcq.trellis_matvec(d_x, d_codes, d_scales, d_lut, g, out=d_out)
            h_out.copy_(d_out, non_blocking=True)

        e_steps = max(10, min(200, args.steps // 20))
        e_ms, _ = time_launches(torch, e2e_step, e_steps, 3, stream, barrier)
        bi = PACKED_BYTES + N1 * 2 + 4096 * 4 + K1 * 2
        bo = N1 * 2
        e2e = {"value": round(world * PACKED_BYTES * e_steps / (e_ms * 1e-3) / 1e9, 2), "unit": "GB/s",
               "h2d_bytes_per_step": bi, "d2h_bytes_per_step": bo,
               "ms_per_step": round(e_ms / e_steps, 4)}

    extras = None
    if rank == 0 and not args.no_extras:
        extras = extra_configs(torch, tcq, device, stream, peaks)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(seconds=args.cpu_seconds)

    status = tcq.trellis_device_status()
    if rank == 0:
        line = {
            "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 5),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "bf16", "data": "synthetic (seeded SplitMix64 codes, N(0,1) codebook and activations, U[0.01,0.03] scales)",
            "config": {"workload": WORKLOAD, "M": M1, "K": K1, "N": N1, "k": KB1, "BT": 256, "L": 12,
                       "weight_sets": nsets, "l2": f"inputs larger than L2: {nsets} rotating weight sets "
                                                   f"({nsets * PACKED_BYTES / 1e6:.0f} MB vs L2 {l2 / 1e6:.0f} MB)",
                       "parallelism": f"independent problem per GPU x{world}"},
            "roofline": roofline, "cpu_baseline": cpu, "e2e": e2e,
            "gpu_launches": args.steps, "clocks": clk.summary(), "device_status": status,
            "secondary": extras,
        }
        print(json.dumps(line))
    if dist:
        dist.destroy_process_group()


# ---------------------------------------------------------------------------
# the oracle as the CPU baseline / reference arm
# ---------------------------------------------------------------------------

def oracle_rows_per_second(orc, p, rows):
    """Decode + double matvec of `rows` rows of the decode-matvec problem."""
    codes = p["codes"][:rows]
    t0 = time.perf_counter()
    W, _ = orc.expand(codes, rows, K1, KB1, p["scales"][:rows], p["lut"])
    orc.matmul_axis1(p["x"], W)
    return rows / (time.perf_counter() - t0)


def cpu_baseline(seconds: float = 10.0, p=None):
    import oracle
    from trellis_coded_quantized_gb300 import synth
    orc = oracle.default()
    if p is None:
        p = synth.problem(1, M1, N1, K1, KB1, seed=0)
    rps = oracle_rows_per_second(orc, p, 512)
    rows = int(min(N1, max(512, rps * 1.0)))
    done_rows, t0 = 0, time.perf_counter()
    while time.perf_counter() - t0 < seconds:
        oracle_rows_per_second(orc, p, rows)
        done_rows += rows
    el = time.perf_counter() - t0
    value = done_rows * K1 * KB1 / 8 / el / 1e9
    return {"value": round(value, 4), "unit": "GB/s", "cores": orc.max_threads(), "kind": "oracle",
            "sample": f"{done_rows} rows of the decode-matvec matrix ({rows} per pass: expand to bf16 "
                      f"weights + double matvec), {el:.1f} s"}


def run_reference(args):
    rank, _, world = env_rank()
    if rank != 0:
        return
    import oracle
    from trellis_coded_quantized_gb300 import synth
    orc = oracle.default()
    p = synth.problem(1, M1, N1, K1, KB1, seed=0)
    rps = oracle_rows_per_second(orc, p, 512)
    budget = 60.0
    rows = int(max(8, min(N1, budget * rps / max(1, args.steps + args.warmup))))
    for _ in range(args.warmup):
        oracle_rows_per_second(orc, p, rows)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle_rows_per_second(orc, p, rows)
    el = time.perf_counter() - t0
    value = rows * K1 * KB1 / 8 * args.steps / el / 1e9
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(el / args.steps * 1e3, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (same seeded inputs)",
        "config": {"workload": WORKLOAD, "M": M1, "K": K1, "N": N1, "k": KB1,
                   "sample": f"{rows} of {N1} rows per step"},
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": orc.max_threads(), "kind": "oracle",
                         "sample": f"{rows} rows of the decode-matvec matrix per step"},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20000)
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-extras", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
