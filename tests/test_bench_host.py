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
