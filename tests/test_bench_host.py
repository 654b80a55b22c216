"""bench.py's host-side logic (no GPU): session groups, the schedule each
workload runs, and the argument defaults the headline relies on."""
import argparse

import pytest

import bench
from synth import workloads as W


@pytest.mark.parametrize("sessions,layers,n", [(16, 2, 2), (16, 2, 3), (16, 2, 4), (5, 3, 2), (1, 4, 2), (7, 1, 7)])
def test_session_groups_cover_the_units_in_order(sessions, layers, n):
    g = bench.session_groups(sessions, layers, n)
    assert len(g) == min(n, sessions)
    assert g[0][0] == 0 and g[-1][1] == sessions * layers
    for (lo, hi), (lo2, _) in zip(g, g[1:]):
        assert hi == lo2                       # contiguous, in unit order
    sizes = [(hi - lo) // layers for lo, hi in g]
    assert all((hi - lo) % layers == 0 for lo, hi in g)   # whole sessions
    assert max(sizes) - min(sizes) <= 1 and min(sizes) >= 1


def _args(**kw):
    d = dict(no_pipeline=False, schedule=None, path=None)
    d.update(kw)
    return argparse.Namespace(**d)


def test_schedules_by_workload():
    cap, single = W.WORKLOADS[4], W.WORKLOADS[1]
    assert bench.use_pipeline(_args(), cap) == "partition"
    assert bench.use_pipeline(_args(path="fused"), cap) == "partition"
    assert bench.use_pipeline(_args(path="split"), cap) == "partition"
    assert bench.use_pipeline(_args(schedule="groups"), cap) == "groups"
    assert bench.use_pipeline(_args(schedule="lockstep"), cap) == "lockstep"
    assert bench.use_pipeline(_args(schedule="serial"), cap) == "serial"
    assert bench.use_pipeline(_args(no_pipeline=True), cap) == "serial"
    assert bench.use_pipeline(_args(schedule="groups", path="fused"), cap) == "serial"
    # the 50K stream fits in L2 several times over: serial, L2 flushed per step
    assert bench.use_pipeline(_args(), single) == "serial"
    # one session (of enough layers to stream past L2): no groups to alternate
    assert bench.use_pipeline(_args(), cap.with_(sessions=1, layers=8)) == "lockstep"


def test_headline_defaults(monkeypatch):
    assert bench.SCORE_SMS == 120 and bench.GROUPS == 2
    monkeypatch.setattr("sys.argv", ["bench.py"])
    a = bench.parse()
    assert a.score_sms == 120 and a.groups == 2 and a.schedule is None and a.path is None
    assert a.gpus == 1 and a.config == 4 and a.warmup >= 3      # the capacity batch


def test_reference_arm_prints_the_contract_line():
    """`bench.py --impl reference` times the oracle on the host cores and
    prints one JSON line with the GPU arm's metric, unit and workload."""
    import json
    import os
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--steps", "1", "--warmup", "3"],
                       cwd=root, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    line = json.loads(r.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["metric"] == bench.METRIC
    assert line["unit"] == "layer-steps/s" and line["higher_is_better"] is True and line["value"] > 0
    assert line["n_gpus"] == 1 and line["steps"] == 1 and line["warmup"] >= 3
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] >= 1
    assert line["cpu_baseline"]["value"] == line["value"] and line["cpu_baseline"]["sample"]
    assert line["e2e"] == {"value": line["value"], "unit": line["unit"], "h2d_bytes_per_step": 0,
                           "d2h_bytes_per_step": 0}
    assert line["config"]["workload"].startswith("capacity batch")
