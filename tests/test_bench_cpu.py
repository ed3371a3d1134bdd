"""Host logic of bench.py on the CPU: both arms describe the same workload,
and the reference arm's oracle pass runs on a bounded sample."""
import argparse
import os
import sys

import pytest

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
import bench  # noqa: E402


def _args(**kw):
    base = dict(workload="decode-matvec", M=0, k=0, splits=0, unrounded=False)
    base.update(kw)
    return argparse.Namespace(**base)


@pytest.mark.parametrize("kw,shape", [
    ({}, (1, 17408, 5120, 4, 1)),
    ({"workload": "tiny-matvec"}, (1, 256, 512, 2, 1)),
    ({"workload": "prefill"}, (32, 17408, 5120, 4, 1)),
    ({"workload": "prefill", "M": 8, "k": 3}, (8, 17408, 5120, 3, 1)),
    ({"workload": "scatter"}, (1, 17408, 5120, 3, 0)),
    ({"workload": "scatter", "M": 16, "splits": 136, "unrounded": True}, (16, 17408, 5120, 3, 0)),
])
def test_workload_config(kw, shape):
    cf = bench.workload_config(_args(**kw))
    assert (cf["M"], cf["rows"], cf["cols"], cf["k"], cf["axis"]) == shape
    assert cf["config"]["workload"] == cf["desc"]
    if kw.get("unrounded"):
        assert "unrounded" in cf["desc"]
    if kw.get("workload") == "scatter":
        assert f"{kw.get('splits') or 128} splits" in cf["desc"]


def test_reference_arm_describes_the_same_workload():
    a = _args(workload="tiny-matvec")
    host = bench._HostWorkload(a)
    assert host.cfg["config"] == bench.workload_config(a)["config"]
    assert host.packed == 256 * 512 * 2 // 8


def test_oracle_pass_on_a_sample(orc):
    host = bench._HostWorkload(_args(workload="scatter", unrounded=True))
    assert bench.oracle_pass(orc, host, 8) > 0.0
    host = bench._HostWorkload(_args(workload="tiny-matvec"))
    assert bench.oracle_pass(orc, host, 16) > 0.0


def test_cpu_baseline_times_expansion_and_contraction_apart(orc):
    host = bench._HostWorkload(_args(workload="tiny-matvec"))
    cb = bench.cpu_baseline(host, seconds=0.4)
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] > 0
    for part in ("expand", "matmul"):
        assert cb[part]["1_thread"] > 0 and cb[part]["all_cores"] > 0
    assert cb["parts"]["1_thread"]["threads"] == 1
    assert orc.max_threads() == cb["cores"]          # the thread count is restored


def test_gather_floor_arithmetic():
    rates = {"smem_gather_x8": {"per_sm_per_clock": 10.0, "sm_mhz": 2000.0}}
    # 1e9 weights / (10 per SM-clock * 100 SMs * 2e9 Hz) = 0.5 ms
    assert abs(bench.gather_floor_s(1e9, rates, 100, 2000.0) - 5e-4) < 1e-12
    # without a sampled run clock the probe's own clock is used
    assert abs(bench.gather_floor_s(1e9, rates, 100, None) - 5e-4) < 1e-12


def test_clock_summary_keeps_the_timed_window():
    c = bench.ClockSampler(0)
    c.samples = [(0.0, 1000.0, 2070.0, 0, []), (1.0, 2070.0, 2070.0, 4, ["sw_power_cap"]),
                 (1.5, 2000.0, 2070.0, 0, []), (3.0, 500.0, 2070.0, 8, ["hw_slowdown"])]
    s = c.summary(0.9, 2.0)
    assert s["samples"] == 2 and s["sm_mhz"] == 2035.0 and s["reasons"] == ["sw_power_cap"]
    assert c.summary()["samples"] == 4
    assert c.summary(5.0, 6.0)["sm_mhz"] is None
