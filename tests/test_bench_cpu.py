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
