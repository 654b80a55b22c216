"""The partition schedule's stream ordering, checked on the CPU.

bench.py's partition schedule (WorkloadRun._record_partition) issues each
session group's step over several streams: the scoring partition's stream,
the group's stream on the other partition, and (end to end) ordinary copy
streams, ordered only by cross-stream waits. This runs that very code against
recording stand-ins for the streams, events, tensors and library calls, builds
the happens-before graph (each stream in order; a wait orders everything the
signalling stream had queued when the wait was issued before everything the
waiting stream queues after it), and checks that every pair of accesses to one
buffer that conflict (at least one write) is ordered on the device the way the
host issued it: no step reads inputs before they land or after the next ones
overwrite them, no attention overwrites an output before it is copied out.
"""
import contextlib
import itertools
import types

import pytest

import bench


class Stream:
    def __init__(self, sim, name):
        self.sim, self.name, self.ops = sim, name, []

    def wait_stream(self, other):
        self.sim.wait(self, other, len(other.ops))

    def wait_event(self, ev):
        if ev.at is not None:
            self.sim.wait(self, ev.at[0], ev.at[1])


class Event:
    def __init__(self, sim, **_):
        self.sim, self.at = sim, None

    def record(self, stream=None):
        st = stream if stream is not None else self.sim.current
        self.at = (st, len(st.ops))


class Tensor:
    """A named buffer; views and indexing keep the buffer they belong to."""

    def __init__(self, sim, name):
        self.sim, self.name = sim, name

    def __getitem__(self, k):
        if isinstance(k, slice):
            return Tensor(self.sim, f"{self.name}[{k.start}:{k.stop}]")
        return Tensor(self.sim, f"{self.name}[{k}]")

    def copy_(self, src, non_blocking=False):
        self.sim.op(self.sim.current, "copy", reads=[src.name], writes=[self.name])

    def add_(self, other):
        self.sim.op(self.sim.current, "add", reads=[other.name, self.name], writes=[self.name])


class Sim:
    def __init__(self):
        self.nodes = []          # (stream, index, kind, reads, writes)
        self.edges = []          # (from node, to node)
        self.pending_waits = {}  # stream -> [(signaller stream, position)]
        self.main = Stream(self, "main")
        self.current = self.main

    def op(self, stream, kind, reads=(), writes=()):
        node = len(self.nodes)
        self.nodes.append((stream, len(stream.ops), kind, tuple(reads), tuple(writes)))
        if stream.ops:
            self.edges.append((stream.ops[-1], node))
        for sig, pos in self.pending_waits.pop(stream, []):
            if pos > 0:
                self.edges.append((sig.ops[pos - 1], node))
        stream.ops.append(node)
        return node

    def wait(self, waiter, signaller, pos):
        # a wait is itself an (empty) operation of the waiting stream
        self.pending_waits.setdefault(waiter, []).append((signaller, pos))
        self.op(waiter, "wait")

    def reach(self):
        n = len(self.nodes)
        succ = [[] for _ in range(n)]
        for a, b in self.edges:
            succ[a].append(b)
        out = [set() for _ in range(n)]
        for v in reversed(range(n)):          # edges go from earlier to later nodes
            for w in succ[v]:
                out[v].add(w)
                out[v] |= out[w]
        return out

    def check(self):
        after = self.reach()
        for a, b in itertools.combinations(range(len(self.nodes)), 2):
            _, _, ka, ra, wa = self.nodes[a]
            _, _, kb, rb, wb = self.nodes[b]
            clash = (set(wa) & (set(rb) | set(wb))) | (set(ra) & set(wb))
            if clash:
                # issued a before b: the device must run a before b
                assert b in after[a], f"{ka} {self.nodes[a][0].name} and {kb} {self.nodes[b][0].name} race on {clash}"


def make_run(sim, fused, e2e, K=5, ngroups=2):
    abi = types.SimpleNamespace(ROUND_AUTO=-1)
    abi.dsa_stream_wait_stream = lambda waiter, sig: sim.wait(waiter, sig, len(sig.ops))

    @contextlib.contextmanager
    def on(stream):
        prev, sim.current = sim.current, stream
        try:
            yield
        finally:
            sim.current = prev

    cuda = types.SimpleNamespace(current_stream=lambda: sim.current, stream=on,
                                 Event=lambda **k: Event(sim, **k))
    torch = types.SimpleNamespace(cuda=cuda)
    run = object.__new__(bench.WorkloadRun)
    run.torch, run.abi, run.K, run.fused = torch, abi, K, fused
    run.granges = bench.session_groups(2 * ngroups, 2, ngroups)
    run.pstream = Stream(sim, "score")
    run.pext = run.pstream
    run.tstreams = [Stream(sim, f"rest{g}") for g in range(ngroups)]
    run.text = run.tstreams
    run.cin = [Stream(sim, f"in{g}") for g in range(ngroups)]
    run.cout = [Stream(sim, f"out{g}") for g in range(ngroups)]
    run.ev_in = [[Event(sim), Event(sim)] for _ in range(ngroups)]
    run.ctr = Tensor(sim, "ctr")
    run.gpaths = []
    names = ("q_idx", "w", "q_lat", "q_rope", "new_rows", "new_keys")
    for g in range(ngroups):
        t = f"g{g}."

        def score(qi, w, stream, t=t):
            sim.op(stream, "score", [qi.name, w.name], [t + "ws"])

        def select(stream, t=t):
            sim.op(stream, "select", [t + "ws"], [t + "ws", t + "topk"])

        def gather_attend(rnd, ql, qr, stream, t=t):
            sim.op(stream, "gather_attend", [t + "topk", t + "cache", ql.name, qr.name],
                   [t + "out", t + "counters", t + "cache", t + "cls"])

        def attend(ql, qr, stream, t=t):
            sim.op(stream, "attend", [t + "rows", t + "topk", ql.name, qr.name], [t + "out"])

        def append(nr, nk, stream, t=t):
            sim.op(stream, "append", [nr.name, nk.name, t + "cache"], [t + "cache"])

        p = types.SimpleNamespace(score=score, select=select, gather_attend=gather_attend, attend=attend,
                                  append=append, u=types.SimpleNamespace(units=None, U=1, dev_err=None),
                                  R=1, K=1, topk=Tensor(sim, t + "topk"), cls=Tensor(sim, t + "cls"),
                                  rows=Tensor(sim, t + "rows"), ws_gather=Tensor(sim, t + "ws_gather"),
                                  ws_gather_bytes=0, out=Tensor(sim, t + "out"),
                                  counters=Tensor(sim, t + "counters"))
        run.gpaths.append(p)

    def assign(units, U, R, K, rnd, topk, cls, counters, ws, ws_bytes, dev_err, stream):
        g = topk.name.split(".")[0] + "."
        sim.op(stream, "assign", [topk.name, g + "cache"], [cls.name, counters.name, ws.name, g + "cache"])

    def copy(units, U, R, K, topk, cls, rows, ws, ws_bytes, dev_err, stream):
        g = topk.name.split(".")[0] + "."
        sim.op(stream, "copy", [topk.name, cls.name, ws.name, g + "cache"], [rows.name, g + "cache"])

    abi.hot_gather_assign, abi.hot_gather_copy = assign, copy
    # without e2e the inputs are resident per step (never overwritten)
    run.step_args = lambda s: tuple(Tensor(sim, f"{n}[{s}]") for n in names)
    packs = None
    if e2e:
        packs = []
        for g in range(ngroups):
            hpack = Tensor(sim, f"g{g}.hpack")
            dpack = [Tensor(sim, f"g{g}.dpack{b}") for b in range(2)]
            dev_in = [{n: dpack[b] for n in names} for b in range(2)]
            out_host = Tensor(sim, f"g{g}.out_host")
            packs.append((hpack, dpack, dev_in, out_host, None))
    return run, packs


@pytest.mark.parametrize("fused", [True, False], ids=["fused", "split"])
@pytest.mark.parametrize("e2e", [False, True], ids=["device", "e2e"])
@pytest.mark.parametrize("ngroups", [2, 3])
def test_partition_schedule_orders_every_conflicting_access(fused, e2e, ngroups):
    sim = Sim()
    run, packs = make_run(sim, fused, e2e, ngroups=ngroups)
    run._record_partition(10, packs)
    sim.check()


def test_the_check_catches_a_missing_wait():
    """Drop the wait that keeps the next attention off an output still being
    copied out: the check must report the race."""
    sim = Sim()
    run, packs = make_run(sim, True, True)
    real = run.abi.dsa_stream_wait_stream

    def skip_output_wait(waiter, sig):
        if sig in run.cout and waiter in run.tstreams:
            return
        real(waiter, sig)

    run.abi.dsa_stream_wait_stream = skip_output_wait
    run._record_partition(10, packs)
    with pytest.raises(AssertionError, match="out"):
        sim.check()
