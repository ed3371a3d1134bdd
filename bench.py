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
from HBM.  NVML is polled for the SM clock and throttle reasons during the
timed region.  The shared-memory gather rate is measured first in the same
run: every decoded weight costs one codebook gather, so weights / rate is a
floor on each kernel's time, reported beside the HBM fraction.

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


def source_fingerprint(kernel_file: str):
    """sha1 (12 hex digits) of a kernel source with comments and blank lines
    removed, so that editing documentation does not void a capture."""
    src = os.path.join(ROOT, "trellis_coded_quantized_gb300", "csrc", kernel_file)
    try:
        text = open(src).read()
    except OSError:
        return None
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    lines = [re.sub(r"//.*$", "", ln).rstrip() for ln in text.splitlines()]
    code = "\n".join(ln for ln in lines if ln.strip())
    return hashlib.sha1(code.encode()).hexdigest()[:12]


def profiled_traffic(kernel_file: str, kernel: str):
    """DRAM bytes per launch of `kernel` from a summary under profiles/ when it
    was captured on the current source of the kernel (the summary records the
    source's fingerprint): a line "traffic_per_launch_bytes: B source_sha1: S
    kernel_file: F kernel: K"."""
    sha = source_fingerprint(kernel_file)
    if sha is None:
        return None
    pdir = os.path.join(ROOT, "profiles")
    if not os.path.isdir(pdir):
        return None
    pat = re.compile(r"traffic_per_launch_bytes:\s*(\d+)\s+source_sha1:\s*([0-9a-f]+)\s+"
                     r"kernel_file:\s*(\S+)\s+kernel:\s*(.+)$", re.M)
    for name in sorted(os.listdir(pdir)):
        if not name.endswith(".md"):
            continue
        for m in pat.finditer(open(os.path.join(pdir, name)).read()):
            if m.group(3) == kernel_file and m.group(2) == sha and m.group(4).strip() == kernel:
                return int(m.group(1))
    return None


class ClockSampler:
    """SM clock and throttle-reason samples while running.

    NVML (libnvidia-ml, loaded with ctypes) is polled back to back from a
    thread, about every 0.2 ms, so that even a timed region of well under a
    millisecond gets samples; each sample carries its host time, and
    `summary(t0, t1)` keeps the samples taken between t0 and t1.  Without
    NVML, nvidia-smi is sampled every 200 ms instead."""
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    # NVML clock-event reason bits
    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.samples = []        # (host time, sm MHz, sm max MHz, reason bits or None, reason names)
        self.source = None
        self._stop = threading.Event()
        self.thread = None

    def _nvml(self):
        import ctypes
        lib = None
        for name in ("libnvidia-ml.so.1", "libnvidia-ml.so"):
            try:
                lib = ctypes.CDLL(name)
                break
            except OSError:
                continue
        if lib is None or lib.nvmlInit_v2() != 0:
            return None
        h = ctypes.c_void_p()
        if lib.nvmlDeviceGetHandleByIndex_v2(ctypes.c_uint(self.gpu), ctypes.byref(h)) != 0:
            return None
        return lib, h

    def __enter__(self):
        nv = None
        try:
            nv = self._nvml()
        except Exception:
            nv = None
        if nv is not None:
            self.source = "nvml"
            self.thread = threading.Thread(target=self._poll_nvml, args=nv, daemon=True)
            self.thread.start()
            return self
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.source = "nvidia-smi"
            self.thread = threading.Thread(target=self._read_smi, daemon=True)
            self.thread.start()
        except Exception:
            self.proc = None
        return self

    def _poll_nvml(self, lib, h):
        import ctypes
        clk, cmax, rs = ctypes.c_uint(), ctypes.c_uint(), ctypes.c_ulonglong()
        get_reasons = getattr(lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            getattr(lib, "nvmlDeviceGetCurrentClocksThrottleReasons", None)
        lib.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(cmax))
        while not self._stop.is_set():
            if lib.nvmlDeviceGetClockInfo(h, 1, ctypes.byref(clk)) == 0:       # NVML_CLOCK_SM
                bits = None
                if get_reasons is not None and get_reasons(h, ctypes.byref(rs)) == 0:
                    bits = int(rs.value)
                names = [n for b, n in self.REASONS.items() if bits is not None and bits & b]
                self.samples.append((time.perf_counter(), float(clk.value), float(cmax.value), bits, names))
            time.sleep(0.0002)

    def _read_smi(self):
        for line in self.proc.stdout:
            f = [x.strip() for x in line.strip().split(",")]
            if len(f) < 9:
                continue
            try:
                sm, smax = float(f[1]), float(f[2])
            except ValueError:
                continue
            names = [n for n, v in zip(["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"],
                                       f[5:9]) if v.lower().startswith("active")]
            self.samples.append((time.perf_counter(), sm, smax, None, names))

    def __exit__(self, *exc):
        self._stop.set()
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
        if self.thread is not None:
            self.thread.join(timeout=5)

    def summary(self, t0=None, t1=None):
        """Median SM clock, the largest max clock and every active throttle
        reason of the samples taken between host times t0 and t1 (all
        samples when not given)."""
        sel = [x for x in self.samples if (t0 is None or x[0] >= t0) and (t1 is None or x[0] <= t1)]
        if not sel:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0, "source": self.source}
        reasons = sorted({n for x in sel for n in x[4]})
        return {"sm_mhz": statistics.median(x[1] for x in sel), "sm_max_mhz": max(x[2] for x in sel),
                "reasons": reasons, "samples": len(sel), "source": self.source}


# ---------------------------------------------------------------------------
# our arm
# ---------------------------------------------------------------------------

def xor_sets(torch, codes0, nsets: int, salt: int):
    """Further weight sets for L2 rotation: the first XOR a per-set constant
    (uniform codes stay uniform)."""
    return [codes0] + [codes0 ^ int(np.int32(np.uint32((salt * (j + 1)) & 0xFFFFFFFF)))
                       for j in range(1, nsets)]


def dev_problem(torch, p, device):
    return (torch.from_numpy(p["codes"].view(np.int32)).to(device),
            torch.from_numpy(p["scales"].view(np.int16)).to(device).view(torch.bfloat16),
            torch.from_numpy(p["lut"]).to(device),
            torch.from_numpy(p["x"].view(np.int16)).to(device).view(torch.bfloat16))


def workload_config(args) -> dict:
    """The workload's shape and its JSON `config` (shared by both arms)."""
    w = args.workload
    unrounded = bool(getattr(args, "unrounded", False))
    splits = None
    if w in ("decode-matvec", "tiny-matvec"):
        M, K, N, k, axis = (1, 5120, 17408, 4, 1) if w == "decode-matvec" else (1, 512, 256, 2, 1)
        desc = (f"decode matvec axis-1: M=1, K={K}, N={N}, k={k}, BT=256, L=12" if w == "decode-matvec"
                else f"tiny axis-1 matvec: M=1, K={K}, N={N}, k={k}, BT=256, L=12, seed 0")
    elif w == "prefill":
        M, K, N, k, axis = args.M or 32, 5120, 17408, args.k or 4, 1
        desc = f"tiled prefill axis-1: M={M}, K=5120, N=17408, k={k}, BT=256, L=12"
    elif w == "scatter":
        M, K, N, k, axis = args.M or 1, 17408, 5120, 3, 0
        splits = getattr(args, "splits", 0) or 128
        desc = f"axis-0 split-K scatter: M={M}, R=17408, C=5120, k=3, BT=256, L=12, {splits} splits"
    else:
        raise ValueError(w)
    if unrounded:
        desc += ", unrounded contract"
    rows, cols = (N, K) if axis == 1 else (K, N)
    return {"name": w, "M": M, "K": K, "N": N, "k": k, "axis": axis, "rows": rows, "cols": cols,
            "splits": splits, "unrounded": unrounded, "desc": desc,
            "config": {"workload": desc, "M": M, "K_in": K, "N_out": N, "k": k, "BT": 256, "L": 12, "axis": axis}}


class Workload:
    """One configuration: step(i) runs one pass of the hot path on weight set
    i mod nsets; the step's launches are timed for the roofline."""

    def __init__(self, args, torch, tcq, device, l2):
        from trellis_coded_quantized_gb300 import synth
        self.args, self.torch, self.tcq, self.device = args, torch, tcq, device
        w = args.workload
        self.name = w
        cf = workload_config(args)
        self.cfg = cf
        self.unrounded = cf["unrounded"]
        if self.unrounded and w == "prefill":
            raise ValueError("the prefill takes the rounded contract only")
        self.M, self.K, self.N, self.k, self.axis = cf["M"], cf["K"], cf["N"], cf["k"], cf["axis"]
        self.desc = cf["desc"]
        if w in ("decode-matvec", "tiny-matvec"):
            self.kernel = f"matvec_kernel<{self.k}>"
            self.kernel_file = "matvec.cu"
        elif w == "prefill":
            self.kernel = f"prefill_kernel<{self.k},{16 if self.M <= 16 else 32}>"
            self.kernel_file = "prefill.cu"
        elif w == "scatter":
            self.splits = cf["splits"]
            nt = 1 if self.M <= 8 else 2 if self.M <= 16 else 4
            if self.M <= 2:
                self.kernel = "scatter_kernel<3> + split_reduce_kernel"
            elif self.unrounded:
                self.kernel = f"scatter_mma_kernel<3,{nt}> + split_reduce_kernel"
            else:
                self.kernel = f"scatter_tc_kernel<3,{16 if self.M <= 16 else 32}> + tc_split_reduce_kernel"
            self.kernel_file = "scatter_tc.cu" if self.M >= 3 and not self.unrounded else "scatter.cu"
        else:
            raise ValueError(w)
        rows, cols = (self.N, self.K) if self.axis == 1 else (self.K, self.N)
        self.rows, self.cols = rows, cols
        self.packed = rows * cols * self.k // 8
        self.flops = 2.0 * self.M * rows * cols
        p = synth.problem(self.axis, self.M, rows, cols, self.k, seed=0)
        self.p = p
        codes0, self.scales, self.lut, self.x = dev_problem(torch, p, device)
        self.nsets = max(2, int(np.ceil(4 * l2 / self.packed)) + 1)
        self.sets = xor_sets(torch, codes0, self.nsets, 0x9E3779B9)
        self.g = tcq.geometry(self.axis, rows, cols, self.k, unrounded=self.unrounded)
        if self.unrounded and "(unrounded)" not in self.kernel:
            self.kernel += " (unrounded)"
        nout = rows if self.axis == 1 else cols
        self.out = torch.empty((self.M, nout), dtype=torch.bfloat16, device=device)
        self.ws = None
        if w == "scatter":
            self.ws = torch.empty(tcq.trellis_scatter_workspace_bytes(self.g, self.M, self.splits) // 4,
                                  dtype=torch.float32, device=device)
        # algorithmic bytes of the step: the method's inputs and output --
        # codes, scales, codebook, x, out.  The scatter's fp32 split partials
        # are the implementation's buffer (written and read back once, mostly
        # in L2) and are reported apart as partial_bytes.
        self.alg_bytes = self.packed + rows * 2 + 4096 * 4 + self.M * (cols if self.axis == 1 else rows) * 2 \
            + self.M * nout * 2
        self.partial_bytes = 2 * self.M * self.splits * cols * 4 if w == "scatter" else 0
        # decoded weights per step: one codebook gather each
        self.weights = rows * cols
        # the scatter: one FMA pass up to 2 rows, one tensor-core pass for 3
        # and more rows; then the split reduction
        if w != "scatter":
            self.launches_per_step = 1
        else:
            self.launches_per_step = 2

    def run(self, codes, x=None, out=None):
        tcq = self.tcq
        x = self.x if x is None else x
        out = self.out if out is None else out
        if self.name in ("decode-matvec", "tiny-matvec"):
            tcq.trellis_matvec(x[0], codes, self.scales, self.lut, self.g, out=out[0])
        elif self.name == "prefill":
            tcq.trellis_prefill(x, codes, self.scales, self.lut, self.g, out=out)
        else:
            tcq.trellis_scatter(x, codes, self.scales, self.lut, self.g, splits=self.splits, workspace=self.ws,
                                out=out)

    def step(self, i):
        self.run(self.sets[i % self.nsets])


def max_over_ranks(torch, dist, value: float, device) -> float:
    """The largest `value` over all ranks (the whole job ends with the
    slowest rank); `value` itself with no process group."""
    if dist is None:
        return value
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(per_rank_units: float, world: int, seconds: float) -> float:
    """Whole-job throughput under weak scaling: every rank processes
    per_rank_units in the (max over ranks) time."""
    return world * per_rank_units / seconds


def time_launches(torch, fn, steps, warmup, stream, barrier, per_launch=True):
    """Events on the launching stream around `steps` back-to-back steps
    (total ms) and, with per_launch, around each step as well (a list of ms).
    An event between two launches keeps the second from being placed while
    the first drains, so the total of the timed region is taken without them."""
    for i in range(warmup):
        fn(i)
    torch.cuda.synchronize()
    n = steps if per_launch else 0
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(n)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(n)]
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    barrier()
    torch.cuda.synchronize()
    # Hold the stream for ~0.2 ms before the start event, so that the host
    # has enqueued the first launches by the time it fires: otherwise the
    # host's latency to enqueue the first step would be timed as GPU idle.
    # The spin runs before the start event, outside the timed region.
    torch.cuda._sleep(400_000)
    t0.record(stream)
    for i in range(steps):
        if per_launch:
            starts[i].record(stream)
        fn(warmup + i)
        if per_launch:
            ends[i].record(stream)
    t1.record(stream)
    torch.cuda.synchronize()
    barrier()
    total_ms = t0.elapsed_time(t1)
    per = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    return total_ms, per


def gather_rates(torch, tcq, device, stream, clk):
    """Shared-memory gather rate, the ceiling of the decode (one random
    4-byte codebook read per weight), with 1, 4 and 8 interleaved table
    copies: gathers per second on the whole GPU, and per SM and clock at the
    SM clock sampled while the probe ran."""
    lut = torch.randn(4096, device=device)
    sm = torch.cuda.get_device_properties(device).multi_processor_count
    iters = 2000
    out = {}
    for rep in (1, 4, 8):
        h0 = time.perf_counter()
        _, per = time_launches(torch, lambda i: tcq.trellis_gather_probe(lut, sm, iters, rep), 5, 2,
                               stream, lambda: None)
        h1 = time.perf_counter()
        t = statistics.median(per) * 1e-3
        gathers = sm * 1024 * iters * 8
        mhz = clk.summary(h0, h1)["sm_mhz"] or 2070.0
        out[f"smem_gather_x{rep}"] = {"gathers_per_s": gathers / t, "sm_mhz": mhz,
                                      "per_sm_per_clock": round(gathers / t / sm / (mhz * 1e6), 3)}
    return out, sm


def gather_floor_s(weights: float, rates: dict, sm: int, sm_mhz) -> float:
    """Shortest time the decode of `weights` weights can take: one gather each
    at the measured 8-copy rate (per SM and clock) on all SMs at the sampled
    median SM clock of the run."""
    r = rates["smem_gather_x8"]
    mhz = sm_mhz or r["sm_mhz"]
    return weights / (r["per_sm_per_clock"] * sm * mhz * 1e6)


def kv_lines(torch, tcq, device, stream, hbm, only=None, steps=50, warmup=3):
    """The TurboQuant packed K/V decode (the second workload): the pages'
    measured regime (D 256, 8-bit keys, 3-bit values, f16 scales, groups of
    32) at B1 H4 N65536, joint decode (f32 values) and the inverse-256
    rotation (bf16 values), plus a D 128 4-bit/4-bit joint decode.  Inputs
    and outputs together are larger than L2.  Bytes are the arrays read and
    written once."""
    from trellis_coded_quantized_gb300 import synth
    out = {}

    def dev(a):
        a = np.ascontiguousarray(a)
        return torch.from_numpy(a.view(np.int16) if a.dtype == np.uint16 else a).to(device)
    for name, rows, D, kb, vb, inverse in (("kv_decode_D256_k8v3", 4 * 65536, 256, 8, 3, False),
                                           ("kv_inverse256_D256_k8v3", 4 * 65536, 256, 8, 3, True),
                                           ("kv_decode_D128_k4v4", 4 * 131072, 128, 4, 4, False)):
        if only is not None and name != only:
            continue
        c = synth.kv_cache(11, rows, D, kb, vb)
        g = tcq.kv_geometry(rows, D, kb, vb, value_out_bf16=inverse)
        args = [dev(c[n]) for n in ("kp", "ks", "kz", "vp", "vs", "centroids")]
        signs = dev(c["signs"])
        ko = torch.empty((rows, D), dtype=torch.bfloat16, device=device)
        vo = torch.empty((rows, D), dtype=torch.bfloat16 if inverse else torch.float32, device=device)
        if inverse:
            fn = lambda i: tcq.trellis_kv_decode_inverse256(*args, signs, g, ko, vo)
        else:
            fn = lambda i: tcq.trellis_kv_decode(*args, g, ko, vo)
        tb, _ = time_launches(torch, fn, steps, warmup, stream, lambda: None, per_launch=False)
        tb = tb * 1e-3 / steps
        nbytes = sum(a.numel() * a.element_size() for a in args) + ko.numel() * 2 + vo.numel() * vo.element_size()
        out[name] = {"us_back_to_back": round(tb * 1e6, 2), "rows": rows, "bytes": nbytes,
                     "gbs": round(nbytes / tb / 1e9, 1), "frac_of_hbm": round(nbytes / tb / 1e9 / hbm, 4)}
        del args, ko, vo
        torch.cuda.empty_cache()
    return out


def secondary(torch, tcq, device, stream, peaks, l2, rates, sm, sm_mhz):
    """Launch times of the other configurations (context figures): `us` is
    the median of launches each bracketed by events, `us_back_to_back` the
    average over 100 launches in a row.  Each line carries its fraction of
    HBM (algorithmic bytes) and of the gather floor."""
    out = {}
    hbm = peaks["hbm_gbs"]
    tc_peak = peaks["bf16_tflops"]

    class A:
        pass
    for w, M, k, S, unr in ([("prefill", M, k, 0, False) for k in (2, 3, 4) for M in (5, 8, 16, 32)] +
                            [("scatter", 1, 3, 128, False), ("scatter", 4, 3, 128, False),
                             ("scatter", 1, 3, 152, False), ("scatter", 4, 3, 152, False),
                             ("scatter", 16, 3, 128, False), ("scatter", 16, 3, 8, False),
                             ("scatter", 32, 3, 8, False), ("tiny-matvec", 1, 2, 0, False),
                             ("decode-matvec", 1, 4, 0, True), ("scatter", 1, 3, 128, True),
                             ("scatter", 4, 3, 128, True), ("scatter", 16, 3, 128, True)]):
        a = A()
        a.workload, a.M, a.k, a.splits, a.unrounded = w, M, k, S, unr
        wl = Workload(a, torch, tcq, device, l2)
        _, per = time_launches(torch, wl.step, 30, 3, stream, lambda: None)
        t = statistics.median(per) * 1e-3
        tb, _ = time_launches(torch, wl.step, 100, 3, stream, lambda: None, per_launch=False)
        tb = tb * 1e-3 / 100
        key = f"{w}_M{M}_k{k}" + (f"_s{S}" if w == "scatter" else "") + ("_unrounded" if unr else "")
        floor = gather_floor_s(wl.weights, rates, sm, sm_mhz)
        rec = {"us": round(t * 1e6, 2), "us_back_to_back": round(tb * 1e6, 2),
               "packed_gbs": round(wl.packed / tb / 1e9, 1), "tokens_per_s": round(M / tb, 1),
               "frac_of_hbm_alg": round(wl.alg_bytes / tb / 1e9 / hbm, 4),
               "gather_floor_us": round(floor * 1e6, 2), "frac_of_gather_floor": round(floor / tb, 4),
               "frac_of_gather_floor_isolated": round(floor / t, 4)}
        if w == "scatter":
            rec["partial_bytes"] = wl.partial_bytes
        if w == "prefill":
            roof = min(hbm * 1e9 * wl.flops / wl.packed, tc_peak * 1e12)
            rec["tflops"] = round(wl.flops / tb / 1e12, 2)
            rec["frac_of_roofline"] = round(wl.flops / tb / roof, 4)
        out[key] = rec
        del wl
        torch.cuda.empty_cache()
    out.update(kv_lines(torch, tcq, device, stream, hbm))
    # the 40-layer MLP stack, M = 1 and 16
    from trellis_coded_quantized_gb300.mlp import PackedMLPStack
    stack = PackedMLPStack(layers=40, k=3, device=device, m_max=16)
    from trellis_coded_quantized_gb300 import synth
    weights = len(stack.layers) * 3 * stack.inter * stack.hidden
    floor = gather_floor_s(weights, rates, sm, sm_mhz)
    for M in (1, 16):
        x0 = torch.from_numpy(synth.activations(0, M, 5120).view(np.int16)).to(device).view(torch.bfloat16)
        _, per = time_launches(torch, lambda i: stack.forward(x0, check=False), 5, 2, stream, lambda: None)
        t = statistics.median(per) * 1e-3
        rec = {"ms_per_pass": round(t * 1e3, 3), "tokens_per_s": round(M / t, 1),
               "packed_gbs": round(stack.packed_bytes / t / 1e9, 1),
               "tflops": round(2.0 * M * weights / t / 1e12, 2),
               "launches_per_pass": stack.launches_per_pass(M),
               "gather_floor_ms": round(floor * 1e3, 3), "frac_of_gather_floor": round(floor / t, 4)}
        # the same pass captured once in a CUDA graph and replayed
        try:
            graph = torch.cuda.CUDAGraph()
            side = torch.cuda.Stream()
            side.wait_stream(torch.cuda.current_stream())
            with torch.cuda.stream(side):
                stack.forward(x0, check=False)
            torch.cuda.current_stream().wait_stream(side)
            with torch.cuda.graph(graph):
                stack.forward(x0, check=False)
            _, per = time_launches(torch, lambda i: graph.replay(), 5, 2, stream, lambda: None)
            tg = statistics.median(per) * 1e-3
            rec["graph_ms_per_pass"] = round(tg * 1e3, 3)
            rec["graph_tokens_per_s"] = round(M / tg, 1)
            rec["graph_frac_of_gather_floor"] = round(floor / tg, 4)
            del graph
        except Exception as e:          # report, do not fail the bench line
            rec["graph_error"] = str(e)[:200]
        out[f"mlp40_M{M}_k3"] = rec
    del stack
    torch.cuda.empty_cache()
    out.update(rates)
    return out


def run_kv(args):
    """The TurboQuant K/V decode alone (the second workload, for profiling
    and for a stand-alone line): the pages' regime at B1 H4 N65536, W
    warm-up and K timed launches back to back; one JSON line with the
    achieved bandwidth against the measured HBM peak."""
    import torch
    import trellis_coded_quantized_gb300 as tcq
    torch.cuda.set_device(0)
    device = torch.device("cuda:0")
    peaks, peak_src = measured_peaks()
    name = "kv_inverse256_D256_k8v3" if args.workload == "kv-inverse" else "kv_decode_D256_k8v3"
    rec = kv_lines(torch, tcq, device, torch.cuda.current_stream(), peaks["hbm_gbs"], only=name,
                   steps=args.steps, warmup=args.warmup)[name]
    print(json.dumps({"metric": "TurboQuant K/V decode GB/s (inputs read + outputs written once)",
                      "value": rec["gbs"], "unit": "GB/s", "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
                      "higher_is_better": True, "data": "synthetic", "config": {"workload": name, "rows": rec["rows"]},
                      "roofline": {"bound": "hbm", "achieved": rec["gbs"], "peak": peaks["hbm_gbs"], "unit": "GB/s",
                                   "frac": rec["frac_of_hbm"], "peak_source": peak_src},
                      "us_back_to_back": rec["us_back_to_back"], "status": tcq.trellis_device_status()}))


def run_mlp(args):
    """The synthetic packed SwiGLU stack alone: `--layers` layers (40), M
    activation rows (16), W warm-up passes and K timed passes back to back;
    one JSON line in tokens/s with the pass time and its share of the gather
    ceiling.  For a stand-alone line and for launch lists of one layer's
    kernels (a few layers suffice)."""
    import torch
    import trellis_coded_quantized_gb300 as tcq
    from trellis_coded_quantized_gb300 import synth
    from trellis_coded_quantized_gb300.mlp import PackedMLPStack
    torch.cuda.set_device(0)
    device = torch.device("cuda:0")
    stream = torch.cuda.current_stream()
    M = args.M or 16
    stack = PackedMLPStack(layers=args.layers, k=3, device=device, m_max=max(16, M))
    x0 = torch.from_numpy(synth.activations(0, M, stack.hidden).view(np.int16)).to(device).view(torch.bfloat16)
    with ClockSampler(0) as clk:
        rates, sm = gather_rates(torch, tcq, device, stream, clk)
        h0 = time.perf_counter()
        total_ms, _ = time_launches(torch, lambda i: stack.forward(x0, check=False), args.steps, args.warmup,
                                    stream, lambda: None, per_launch=False)
        h1 = time.perf_counter()
    clocks = clk.summary(h0, h1)
    t = total_ms * 1e-3 / args.steps
    weights = len(stack.layers) * 3 * stack.inter * stack.hidden
    floor = gather_floor_s(weights, rates, sm, clocks["sm_mhz"])
    print(json.dumps({"metric": "tokens/s through the packed MLP stack", "value": round(M / t, 1), "unit": "tokens/s",
                      "n_gpus": 1, "steps": args.steps, "warmup": args.warmup, "higher_is_better": True,
                      "data": "synthetic", "dtype": "bf16",
                      "config": {"workload": f"mlp stack: {args.layers} layers, hidden 5120, intermediate 17408, k=3",
                                 "M": M, "layers": args.layers},
                      "ms_per_pass": round(t * 1e3, 4), "launches_per_pass": stack.launches_per_pass(M),
                      "gather_floor_ms": round(floor * 1e3, 4), "frac_of_gather_floor": round(floor / t, 4),
                      "clocks": clocks, "status": tcq.trellis_device_status()}))


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

    wl = Workload(args, torch, tcq, device, l2)
    with ClockSampler(local_rank) as clk:
        # the gather ceiling of this run, measured first on the same GPU
        rates, sm = gather_rates(torch, tcq, device, stream, clk)
        h0 = time.perf_counter()
        total_ms, _ = time_launches(torch, wl.step, args.steps, args.warmup, stream, barrier, per_launch=False)
        h1 = time.perf_counter()
        total_ms = max_over_ranks(torch, dist, total_ms, device)
        # the same launches one at a time, each between two events (context only)
        h2 = time.perf_counter()
        _, per = time_launches(torch, wl.step, min(args.steps, 2000), 3, stream, lambda: None)
        h3 = time.perf_counter()
    clocks = clk.summary(h0, h1)
    clocks_all = clk.summary(h0, h3)
    sm_mhz = clocks["sm_mhz"] or clocks_all["sm_mhz"]
    ms = total_ms / args.steps
    sec = total_ms * 1e-3
    if wl.name == "prefill":
        value, unit = job_throughput(wl.flops * args.steps, world, sec) / 1e12, "TFLOP/s"
    else:
        value, unit = job_throughput(wl.packed * args.steps, world, sec) / 1e9, "GB/s"

    # roofline of the dominant launch (the only launch of the step, or the
    # scatter with its split reduction): its average duration over the timed
    # region, where back-to-back dependent launches overlap one launch's
    # start with the previous one's tail
    kern_s = ms * 1e-3
    achieved = wl.alg_bytes / kern_s / 1e9
    iso_s = statistics.median(per) * 1e-3
    floor = gather_floor_s(wl.weights, rates, sm, sm_mhz)
    roofline = {"bound": "hbm", "achieved": round(achieved, 1), "peak": peaks["hbm_gbs"],
                "unit": "GB/s", "frac": round(achieved / peaks["hbm_gbs"], 4),
                "traffic": profiled_traffic(wl.kernel_file, wl.kernel), "kernel": wl.kernel,
                "peak_source": f"{peak_src} hbm_gbs (burst copy)", "kernel_us": round(kern_s * 1e6, 3),
                "kernel_us_isolated": round(iso_s * 1e6, 3),
                "algorithmic_bytes": wl.alg_bytes, "partial_bytes": wl.partial_bytes,
                "gather_floor_us": round(floor * 1e6, 3), "frac_of_gather_floor": round(floor / kern_s, 4),
                "frac_of_gather_floor_isolated": round(floor / iso_s, 4),
                "gather_rate_per_sm_per_clock": rates["smem_gather_x8"]["per_sm_per_clock"],
                "gather_floor_basis": f"{wl.weights} weights x 1 shared-memory gather at the measured 8-copy rate "
                                      f"on {sm} SMs at {sm_mhz} MHz"}

    # end to end: pinned host inputs -> device, the C-ABI call, result -> host
    h = {"codes": torch.from_numpy(wl.p["codes"].view(np.int32)).pin_memory(),
         "scales": torch.from_numpy(wl.p["scales"].view(np.int16)).pin_memory(),
         "lut": torch.from_numpy(wl.p["lut"]).pin_memory(),
         "x": torch.from_numpy(wl.p["x"].view(np.int16)).pin_memory()}
    # Two sets of device buffers: the copies of step i+1 run on a side stream
    # while the kernel of step i runs; every step still copies all of its
    # inputs in and its result out inside the timed region.
    h_outs = [torch.empty(tuple(wl.out.shape), dtype=torch.int16).pin_memory() for _ in range(2)]
    ds = [{k: torch.empty(v.shape, dtype=v.dtype, device=device) for k, v in h.items()} for _ in range(2)]
    d_outs = [torch.empty(tuple(wl.out.shape), dtype=torch.int16, device=device) for _ in range(2)]
    copy_stream = torch.cuda.Stream(device)
    landed = [torch.cuda.Event() for _ in range(2)]
    done = [torch.cuda.Event() for _ in range(2)]
    last = {"b": 0}
    e_warm = 3

    def e2e_step(i):
        b = i % 2
        d = ds[b]
        if i in (0, e_warm):                     # the first warm-up and the first timed step start
            copy_stream.wait_stream(stream)      # after everything before them (the start event)
        copy_stream.wait_event(done[b])          # step i-2 no longer reads these buffers
        with torch.cuda.stream(copy_stream):
            for k in d:
                d[k].copy_(h[k], non_blocking=True)
            landed[b].record(copy_stream)
        stream.wait_event(landed[b])
        sc, lt = wl.scales, wl.lut
        wl.scales, wl.lut = d["scales"].view(torch.bfloat16), d["lut"]
        wl.run(d["codes"], x=d["x"].view(torch.bfloat16), out=d_outs[b].view(torch.bfloat16))
        wl.scales, wl.lut = sc, lt
        h_outs[b].copy_(d_outs[b], non_blocking=True)
        done[b].record(stream)
        last["b"] = b

    e_steps = max(10, min(200, args.steps // 20))
    e_ms, _ = time_launches(torch, e2e_step, e_steps, e_warm, stream, barrier, per_launch=False)
    h_out, d_out = h_outs[last["b"]], d_outs[last["b"]]
    e_ms = max_over_ranks(torch, dist, e_ms, device)
    # the end-to-end result must be the device path's result, bit for bit
    torch.cuda.synchronize()
    ref_out = torch.empty_like(d_out)
    wl.run(wl.sets[0], out=ref_out.view(torch.bfloat16))
    torch.cuda.synchronize()
    e2e_same = bool(torch.equal(h_out, ref_out.cpu()))
    bi = sum(v.numel() * v.element_size() for v in h.values())
    bo = h_out.numel() * 2
    work = wl.flops / 1e12 if wl.name == "prefill" else wl.packed / 1e9
    e2e = {"value": round(world * work * e_steps / (e_ms * 1e-3), 3), "unit": unit,
           "h2d_bytes_per_step": bi, "d2h_bytes_per_step": bo, "ms_per_step": round(e_ms / e_steps, 4),
           "matches_device_path": e2e_same}

    extras = None
    if rank == 0 and not args.no_extras:
        del wl.sets
        torch.cuda.empty_cache()
        extras = secondary(torch, tcq, device, stream, peaks, l2, rates, sm, sm_mhz)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(wl, seconds=args.cpu_seconds)

    torch.cuda.synchronize()
    status = tcq.trellis_device_status()
    if rank == 0:
        line = {
            "metric": METRIC, "value": round(value, 3), "unit": unit, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 5),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "bf16", "data": "synthetic (seeded SplitMix64 codes, N(0,1) codebook and activations, U[0.01,0.03] scales)",
            "config": {**wl.cfg["config"], "weight_sets": wl.nsets,
                       "l2": f"inputs larger than L2: {wl.nsets} rotating weight sets "
                             f"({wl.nsets * wl.packed / 1e6:.0f} MB vs L2 {l2 / 1e6:.0f} MB)",
                       "parallelism": f"independent problem per GPU x{world}"},
            "roofline": roofline, "cpu_baseline": cpu, "e2e": e2e,
            "gpu_launches": args.steps * wl.launches_per_step, "clocks": clocks,
            "clocks_whole_measurement": clocks_all,
            "device_status": status, "secondary": extras,
        }
        print(json.dumps(line))
    if dist:
        dist.destroy_process_group()


# ---------------------------------------------------------------------------
# the oracle as the CPU baseline / reference arm
# ---------------------------------------------------------------------------

def oracle_parts(orc, wl, rows):
    """The oracle on the first `rows` rows of the workload's packed matrix,
    its two steps timed apart: (seconds to expand them to weights, seconds of
    the double contraction -- axis 1: those output rows; axis 0: the sum over
    those input rows)."""
    p = wl.p
    codes = p["codes"][:rows]
    unr = getattr(wl, "unrounded", False)
    t0 = time.perf_counter()
    if unr:                                     # the unrounded contract: f32 weights
        W = orc.expand_f32(codes, rows, wl.cols, wl.k, p["scales"][:rows], p["lut"])
    else:
        W, _ = orc.expand(codes, rows, wl.cols, wl.k, p["scales"][:rows], p["lut"])
    t1 = time.perf_counter()
    if wl.axis == 1:
        (orc.matmul_axis1_f32w if unr else orc.matmul_axis1)(p["x"], W)
    else:
        (orc.matmul_axis0_f32w if unr else orc.matmul_axis0)(p["x"][:, :rows], W)
    t2 = time.perf_counter()
    return t1 - t0, t2 - t1


def oracle_pass(orc, wl, rows):
    """Seconds of one oracle pass (expansion + contraction) over `rows` rows."""
    a, b = oracle_parts(orc, wl, rows)
    return a + b


def _timed_parts(orc, wl, seconds):
    """Rows, expansion seconds and contraction seconds of repeated oracle
    passes filling about `seconds` of wall-clock time."""
    t = oracle_pass(orc, wl, min(wl.rows, 16))
    rows = int(min(wl.rows, max(8, 16 * (seconds / 4) / max(t, 1e-6))))   # a pass of about a quarter of the time
    done_rows, te, tm, t0 = 0, 0.0, 0.0, time.perf_counter()
    while True:
        a, b = oracle_parts(orc, wl, rows)
        done_rows, te, tm = done_rows + rows, te + a, tm + b
        if time.perf_counter() - t0 >= seconds:
            break
    return done_rows, te, tm


def cpu_baseline(wl, seconds: float = 10.0):
    """The oracle as it stands on this host's cores: expansion (packed GB/s)
    and double contraction (GFLOP/s) timed apart, each on 1 thread and on
    all cores, on a bounded sample of the workload's rows; `value` is the
    whole pass on all cores in the metric's unit."""
    import oracle
    orc = oracle.default()
    cores = orc.max_threads()
    parts = {}
    try:
        for label, threads in (("1_thread", 1), ("all_cores", cores)):
            orc.set_threads(threads)
            n, te, tm = _timed_parts(orc, wl, seconds / 2)
            frac = n / wl.rows
            parts[label] = {"threads": threads, "rows": n,
                            "expand_gbs": round(frac * wl.packed / te / 1e9, 6),
                            "expand_weights_per_s": round(n * wl.cols / te, 1),
                            "matmul_gflops": round(frac * wl.flops / tm / 1e9, 6),
                            "expand_s": round(te, 3), "matmul_s": round(tm, 3)}
    finally:
        orc.set_threads(cores)
    a = parts["all_cores"]
    frac = a["rows"] / wl.rows
    el = a["expand_s"] + a["matmul_s"]
    if wl.name == "prefill":
        value, unit = frac * wl.flops / el / 1e12, "TFLOP/s"
    else:
        value, unit = frac * wl.packed / el / 1e9, "GB/s"
    return {"value": round(value, 6), "unit": unit, "cores": cores, "kind": "oracle",
            "sample": f"expansion to weights + double contraction of the first rows of the {wl.rows}-row matrix: "
                      f"{parts['1_thread']['rows']} rows on 1 thread, {a['rows']} rows on {cores} threads, "
                      f"about {seconds / 2:.0f} s each",
            "expand": {"unit": "GB/s packed", "1_thread": parts["1_thread"]["expand_gbs"],
                       "all_cores": a["expand_gbs"]},
            "matmul": {"unit": "GFLOP/s (double)", "1_thread": parts["1_thread"]["matmul_gflops"],
                       "all_cores": a["matmul_gflops"]},
            "parts": parts}


class _HostWorkload:
    """The workload's sizes and seeded inputs without a GPU (reference arm)."""

    def __init__(self, args):
        from trellis_coded_quantized_gb300 import synth
        cf = workload_config(args)
        self.cfg = cf
        self.name = cf["name"]
        self.M, self.k, self.axis, self.unrounded = cf["M"], cf["k"], cf["axis"], cf["unrounded"]
        rows, cols = cf["rows"], cf["cols"]
        self.rows, self.cols = rows, cols
        self.packed = rows * cols * self.k // 8
        self.flops = 2.0 * self.M * rows * cols
        self.p = synth.problem(self.axis, self.M, rows, cols, self.k, seed=0)
        self.desc = cf["desc"]


def run_reference(args):
    rank, _, world = env_rank()
    if rank != 0:
        return
    import oracle
    orc = oracle.default()
    wl = _HostWorkload(args)
    t = oracle_pass(orc, wl, min(wl.rows, 256))
    budget = 60.0
    per_row = t / min(wl.rows, 256)
    rows = int(max(8, min(wl.rows, budget / per_row / max(1, args.steps + args.warmup))))
    for _ in range(args.warmup):
        oracle_pass(orc, wl, rows)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle_pass(orc, wl, rows)
    el = time.perf_counter() - t0
    frac = rows / wl.rows * args.steps
    if wl.name == "prefill":
        value, unit = frac * wl.flops / el / 1e12, "TFLOP/s"
    else:
        value, unit = frac * wl.packed / el / 1e9, "GB/s"
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 6), "unit": unit, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(el / args.steps * 1e3, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (the same seeded inputs)",
        "config": {**wl.cfg["config"], "sample": f"{rows} of {wl.rows} rows per step"},
        "cpu_baseline": {"value": round(value, 6), "unit": unit, "cores": orc.max_threads(), "kind": "oracle",
                         "sample": f"{rows} of the {wl.rows} matrix rows per step (expand + double contraction)"},
        "e2e": {"value": round(value, 6), "unit": unit, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50000)
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=["decode-matvec", "tiny-matvec", "prefill", "scatter", "kv-decode",
                                           "kv-inverse", "mlp"],
                    default="decode-matvec")
    ap.add_argument("--M", type=int, default=0, help="activation rows (prefill: 32, scatter: 1)")
    ap.add_argument("--k", type=int, default=0, help="bits per symbol of the prefill (4)")
    ap.add_argument("--splits", type=int, default=0, help="row splits of the scatter (128)")
    ap.add_argument("--layers", type=int, default=40, help="layers of the MLP stack (--workload mlp)")
    ap.add_argument("--unrounded", action="store_true",
                    help="the contract without the bf16 rounding of the weight (matvec, scatter)")
    ap.add_argument("--no-extras", action="store_true", help="skip the secondary configurations")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    if args.impl == "reference":
        run_reference(args)
    elif args.workload in ("kv-decode", "kv-inverse"):
        run_kv(args)
    elif args.workload == "mlp":
        run_mlp(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
