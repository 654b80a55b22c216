#!/usr/bin/env python3
"""Benchmark of the sparse-attention decode path on GB300.

One *step* is one decode step of every unit of the workload through the whole
path: DSA score + Top-K, hot gather, Q8G64 dequant + MLA attention, append with
batched write-back. The headline workload is the capacity batch (16 sessions x
2 layers, 1,048,576-position histories, Top-2048, 64 heads, 32,768 hot slots
per unit, mirror in pinned host memory): the largest single-GPU workload. The
value is layer-steps/s (units x steps / time).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--config C] [--sessions S]
                  [--mirror host|device] [--impl gb300|reference] [--reps R]

Timing: the cache is initialised and W >= 3 untimed warm-up steps run; then
R consecutive K-step segments of the same decode run, each from its own CUDA
graph, so every timed step selects rows that no earlier step has read; L2 is
flushed (a 512 MiB write) before every timed step, outside its CUDA-event
bracket, and the sum of the per-step event times is a segment's total. The
value is the median over the R segments. Clocks are sampled through NVML
every ~2 ms and only samples inside the timed segments are kept. Three more
segments give the per-call breakdown (events around each call, calls serial)
and three more ``e2e``: each step copies its inputs from pinned host memory
and the attention output back, inside the bracket, through the C ABI.

Beside the headline the same line carries the 50K single-stream workload
(``secondary``), and the offload gate (``gate``): the MTP=3 verify workload
with the mirror in pinned host memory and in HBM, in interleaved repetitions,
and the gap between them. The CPU baseline (the oracle, float64, one host
thread, on a bounded sample) runs after all GPU work.

``--impl reference`` times the oracle (the only reference there is: the pages
publish no code) on the host cores, on one unit-step per step. Under torchrun
(N > 1) every rank runs an independent replica of the workload (the path runs
on one GPU; there is no collective on the data path).
"""
from __future__ import annotations

import argparse
import ctypes
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "DSA+gather+MLA-attn layer-steps/s; tok/s; achieved GB/s vs HBM/PCIe roofline"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
DTYPE = "bf16 indexer operands, fp32 scores / Q8G64 rows / fp16 MMA operands, fp32 accumulate"


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=None)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--config", type=int, default=4)
    ap.add_argument("--sessions", type=int, default=None,
                    help="run the workload with fewer sessions (a reduced case for profiling)")
    ap.add_argument("--reps", type=int, default=5, help="timed repetitions of the K steps (median reported)")
    ap.add_argument("--mirror", choices=["host", "device"], default="host")
    ap.add_argument("--policy", choices=["ring", "clock"], default="ring",
                    help="hot-cache replacement of the headline workload")
    ap.add_argument("--impl", choices=["gb300", "reference"], default="gb300")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-graph", action="store_true", help="launch steps directly, no CUDA graph")
    ap.add_argument("--no-secondary", action="store_true", help="skip the 50K single-stream line")
    ap.add_argument("--no-gate", action="store_true", help="skip the offloaded-vs-resident gate")
    ap.add_argument("--reuse-every", type=int, default=1,
                    help="layer l reuses the selection of layer l - l %% N (1: every layer scores)")
    ap.add_argument("--path", choices=["fused", "split"], default=None,
                    help="fused: hot_gather_attn; split: hot_gather + mla_decode_attn with the append "
                         "overlapping the attention (default: fused in the partition schedule, else split)")
    ap.add_argument("--no-pipeline", action="store_true",
                    help="run every step serially, all units in lockstep (same as --schedule serial)")
    ap.add_argument("--score-sms", type=int, default=SCORE_SMS,
                    help="partition schedule: SMs of the partition the scoring runs on")
    ap.add_argument("--groups", type=int, default=GROUPS,
                    help="partition schedule: session groups whose scorings take turns on the scoring partition")
    ap.add_argument("--schedule", choices=["partition", "groups", "lockstep", "serial"], default=None,
                    help="partition: the sessions in two halves, each decoding step after step; the GPU "
                         "split into two SM partitions, every scoring on the first, the rest of each step "
                         "on the second, so one half's selection, gather and attention run beside the "
                         "other half's scoring (the default where the workload streams more than L2 and "
                         "has two or more sessions); groups: the same halves on ordinary streams, one "
                         "half's gather copy and attention overlapping the other half's scoring; "
                         "lockstep: all units, each step's copy and attention overlapping the next step's "
                         "scoring (a step's next query would have to be known before its attention "
                         "ends); serial: one step after the other")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-sample-steps", type=int, default=None)
    ap.add_argument("--oracle-child", type=str, default=None, help=argparse.SUPPRESS)
    return ap.parse_args()


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    except Exception:
        return dict(FALLBACK_PEAKS), "fallback"


def workload(args, cid=None):
    from synth import workloads as W
    wl = W.WORKLOADS[args.config if cid is None else cid]
    if cid is None and args.sessions:
        wl = wl.with_(sessions=args.sessions)
    if args.reuse_every > 1:
        wl = wl.with_(reuse_every=args.reuse_every)
    if cid is None and args.policy != "ring":
        wl = wl.with_(policy=args.policy)
    return wl


def default_steps(wl):
    return min(wl.steps, 64)


# ---------------------------------------------------------------- CPU oracle leg

# The oracle replays unit 0 of the workload: each unit-step is one decode step
# of one (session, layer) history, exactly as the GPU computes it.
CPU_UNITS = (0,)


def oracle_child(spec: str) -> None:
    """Run in a fresh interpreter: time the oracle on a bounded sample."""
    import numpy as np
    from oracle.decode import OracleUnit, decode_step
    from synth import workloads as W
    cfg = json.loads(spec)
    wl = W.WORKLOADS[cfg["config"]]
    if cfg.get("sessions"):
        wl = wl.with_(sessions=cfg["sessions"])
    nsteps, warm = cfg["steps"], cfg["warmup"]
    units = [u for u in CPU_UNITS if u < wl.U]
    wl2 = wl.with_(steps=max(wl.steps, nsteps + warm + 1))
    ous = {}
    t0 = time.time()
    for u in units:
        keys = W.keys_bits(wl2, u, np.arange(wl.L0))
        ous[u] = OracleUnit.create(wl.S, wl2.lmax, wl.L0, keys,
                                   (lambda pos, u=u: W.rows_bytes(wl2, u, pos)), wl.warm)
    setup = time.time() - t0
    nxt = {u: 0 for u in units}

    def one(i):
        u = units[i % len(units)]
        st = nxt[u]
        nxt[u] += 1
        x = W.step_inputs(wl2, u, st)
        decode_step(ous[u], st, wl.K, wl.scale(), x.q_idx, x.w, x.q_lat, x.q_rope, x.new_rows,
                    x.new_keys)
    for i in range(warm):
        one(i)
    t0 = time.perf_counter()
    for i in range(nsteps):
        one(warm + i)
    dt = time.perf_counter() - t0
    print(json.dumps({"seconds": dt, "unit_steps": nsteps, "setup_s": setup, "threads": 1,
                      "units": units}))


def run_oracle(config: int, sessions, steps: int, warmup: int) -> dict:
    env = dict(os.environ, OPENBLAS_NUM_THREADS="1", OMP_NUM_THREADS="1", MKL_NUM_THREADS="1")
    spec = json.dumps({"config": config, "sessions": sessions, "steps": steps, "warmup": warmup})
    r = subprocess.run([sys.executable, os.path.abspath(__file__), "--oracle-child", spec],
                       capture_output=True, text=True, env=env, cwd=ROOT)
    if r.returncode != 0:
        raise RuntimeError("oracle leg failed:\n" + r.stderr[-2000:])
    return json.loads(r.stdout.strip().splitlines()[-1])


def workload_config(wl, extra=None):
    d = {"workload": wl.name, "config_id": wl.cid, "sessions": wl.sessions, "layers": wl.layers,
         "units": wl.U, "history": wl.L0, "query_rows": wl.R, "appended_rows_per_step": wl.A,
         "topk": wl.K, "heads": wl.H, "hot_slots": wl.S, "ring_rows": 64, "row_bytes": 656}
    if extra:
        d.update(extra)
    return d


def sample_text(wl, n, r):
    return (f"{n} unit-steps of unit(s) {r['units']} of the {wl.name} workload (each replaying its own "
            f"decode steps from the start), float64 oracle, 1 host thread ({r['seconds']:.1f} s; "
            f"history set-up {r['setup_s']:.1f} s untimed)")


def reference_arm(args) -> dict:
    wl = workload(args)
    steps = args.steps or default_steps(wl)
    warm = max(3, args.warmup)
    r = run_oracle(args.config, args.sessions, steps, warm)
    value = r["unit_steps"] / r["seconds"]
    sample = sample_text(wl, steps, r)
    return {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "layer-steps/s",
        "n_gpus": args.gpus, "steps": steps, "warmup": warm,
        "ms_per_step": 1e3 * r["seconds"] / steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded counter-based generator)",
        "config": workload_config(wl, {"sample": sample}),
        "tok_per_s": value * wl.A / wl.layers,
        "cpu_baseline": {"value": value, "unit": "layer-steps/s", "cores": r["threads"],
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": "layer-steps/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


# ---------------------------------------------------------------- clocks

class ClockSampler:
    """SM clock, power and clock-event reasons every ~2 ms through NVML (read
    only), with host timestamps so that samples can be matched to the timed
    replays; nvidia-smi at 50 ms if NVML cannot be loaded."""

    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}

    def __init__(self, torch_index: int):
        self.samples = []          # (t, sm_mhz, reasons_mask)
        self.max_mhz = None
        self.source = None
        self._stop = threading.Event()
        self._thread = None
        self._proc = None
        self.windows = []
        try:
            import torch
            lib = ctypes.CDLL("libnvidia-ml.so.1")
            if lib.nvmlInit_v2() != 0:
                raise RuntimeError("nvmlInit")
            h = ctypes.c_void_p()
            uuid = "GPU-" + str(torch.cuda.get_device_properties(torch_index).uuid)
            if lib.nvmlDeviceGetHandleByUUID(uuid.encode(), ctypes.byref(h)) != 0:
                if lib.nvmlDeviceGetHandleByIndex_v2(torch_index, ctypes.byref(h)) != 0:
                    raise RuntimeError("nvml handle")
            self.lib, self.h = lib, h
            mx = ctypes.c_uint()
            if lib.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(mx)) == 0:
                self.max_mhz = float(mx.value)
            self._reasons = getattr(lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
                lib.nvmlDeviceGetCurrentClocksThrottleReasons
            self.source = "nvml"
        except Exception:
            self.lib = None
            self.torch_index = torch_index
            self.source = "nvidia-smi"

    def _poll_nvml(self):
        c, r = ctypes.c_uint(), ctypes.c_ulonglong()
        while not self._stop.is_set():
            ok = self.lib.nvmlDeviceGetClockInfo(self.h, 1, ctypes.byref(c)) == 0
            ok = ok and self._reasons(self.h, ctypes.byref(r)) == 0
            if ok:
                self.samples.append((time.perf_counter(), float(c.value), int(r.value)))
            time.sleep(0.002)

    def _poll_smi(self):
        q = ("clocks.sm,clocks.max.sm,clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
        self._proc = subprocess.Popen(["nvidia-smi", f"--id={self.torch_index}", f"--query-gpu={q}",
                                       "--format=csv,noheader,nounits", "-lms", "50"],
                                      stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        bits = [0x8, 0x40, 0x20, 0x4]
        for ln in self._proc.stdout:
            f = [x.strip() for x in ln.split(",")]
            try:
                mask = sum(b for b, v in zip(bits, f[2:6]) if v.lower() == "active")
                self.max_mhz = float(f[1])
                self.samples.append((time.perf_counter(), float(f[0]), mask))
            except (ValueError, IndexError):
                continue

    def start(self):
        target = self._poll_nvml if self.lib is not None else self._poll_smi
        self._thread = threading.Thread(target=target, daemon=True)
        try:
            self._thread.start()
        except Exception:
            self._thread = None
        time.sleep(0.05)

    def window(self, t0, t1):
        self.windows.append((t0, t1))

    def stop(self) -> dict:
        self._stop.set()
        if self._proc is not None:
            self._proc.terminate()
            try:
                self._proc.wait(timeout=5)
            except Exception:
                self._proc.kill()
        if self._thread is not None:
            self._thread.join(timeout=5)
        inside = [s for s in self.samples if any(a <= s[0] <= b for a, b in self.windows)]
        use = inside if inside else self.samples
        reasons = sorted({n for s in use for b, n in self.REASONS.items() if s[2] & b})
        return {"sm_mhz": statistics.median(s[1] for s in use) if use else None,
                "sm_max_mhz": self.max_mhz, "reasons": reasons, "samples": len(use),
                "samples_in_timed_region": len(inside), "source": self.source,
                "timed_region_s": round(sum(b - a for a, b in self.windows), 4)}


# ---------------------------------------------------------------- GPU arm

def session_groups(sessions: int, layers: int, n: int):
    """`n` contiguous groups of the sessions, as unit ranges [lo, hi) (units
    are session-major), sizes differing by at most one session."""
    n = max(1, min(n, sessions))
    b = [round(i * sessions / n) for i in range(n + 1)]
    return [(b0 * layers, b1 * layers) for b0, b1 in zip(b, b[1:])]


def traffic_for(kernel: str):
    """DRAM bytes per launch from the committed ncu summary, if the kernel's
    source has not changed since it was captured."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(p) as f:
            t = json.load(f)
        e = t[kernel]
        src = os.path.join(ROOT, e["source"])
        h = hashlib.sha256(open(src, "rb").read()).hexdigest()[:16]
        return e["bytes_per_launch"] if h == e["source_sha"] else None
    except Exception:
        return None


class WorkloadRun:
    """One workload on the device: unit set, decode path, inputs for W + n*K
    steps (generated on the device), and one CUDA graph per K-step segment.
    The timed segments are consecutive parts of one continuous decode, so
    every timed step selects rows no earlier step has read."""

    def __init__(self, wl, K, Wm, nseg, mirror, fused, use_graph, pipeline="serial", score_sms=None, ngroups=2):
        import torch
        from decode_attention_dsa_gb300 import abi
        from decode_attention_dsa_gb300.step import DecodePath
        from decode_attention_dsa_gb300.units import UnitSet
        from synth import gpu as sg
        self.torch, self.abi = torch, abi
        self.wl, self.K, self.Wm, self.fused, self.use_graph = wl, K, Wm, fused, use_graph
        self.mirror = mirror
        self.total = Wm + nseg * K
        wlr = wl.with_(steps=self.total)
        U = wl.U
        self.units = UnitSet(U, wl.S, wlr.lmax, mirror=mirror, policy=wl.policy)
        src = [wl.selection_source(u) for u in range(U)] if wl.reuse_every > 1 else None
        self.path = DecodePath(self.units, wl.R, wl.K, wl.H, wl.A, wl.scale(), selection_source=src)
        sg.history(wlr, self.units)
        self.inp = sg.step_inputs(wlr, 0, self.total)
        if self.path.sources:
            # only the source units' indexer queries are scored (set up before timing)
            self.inp["q_idx"] = self.inp["q_idx"][:, self.path.sources].contiguous()
            self.inp["w"] = self.inp["w"][:, self.path.sources].contiguous()
        self.flush = torch.empty(512 << 20, dtype=torch.uint8, device="cuda")
        self.side = torch.cuda.Stream()
        self.warm = abi.WARM_LAST_S if wl.warm == "last_s" else abi.WARM_EMPTY
        self.ctr = torch.zeros((U, 4), dtype=torch.int64, device="cuda")
        self.next_seg = 0
        self.pipeline = pipeline == "lockstep"
        self.groups = None
        self.part = None
        if pipeline in ("groups", "partition"):
            # contiguous groups of sessions (units are session-major); the
            # group schedule alternates two of them
            self.granges = session_groups(wl.sessions, wl.layers, ngroups if pipeline == "partition" else 2)
            self.gpaths = [DecodePath(self.units.subset(lo, hi), wl.R, wl.K, wl.H, wl.A, wl.scale())
                           for lo, hi in self.granges]
            self.gstreams = [torch.cuda.Stream() for _ in self.granges]
            self.g_assigned = [torch.cuda.Event() for _ in self.granges]
            self.groups = True
        if pipeline == "partition":
            # the scorings run on one SM partition, the rest of the steps on the other
            assert not use_graph, "a partition's streams are not captured into a CUDA graph"
            self.part, self.rest = abi.dsa_partition_split(score_sms or SCORE_SMS)
            self.part_sms, self.rest_sms = abi.dsa_partition_sms(self.part), abi.dsa_partition_sms(self.rest)
            self.pstream = abi.dsa_partition_stream(self.part)
            self.tstreams = [abi.dsa_partition_stream(self.rest) for _ in self.granges]
            self.text = [torch.cuda.ExternalStream(st) for st in self.tstreams]
            # the gathers read the host mirrors from the second partition
            abi.dsa_touch_mirror(self.units.units, U, wlr.lmax, self.tstreams[0])
            abi.dsa_stream_wait_stream(torch.cuda.current_stream(), self.tstreams[0])
            # (e2e) a group's input and output copies run on ordinary streams
            self.cin = [torch.cuda.Stream() for _ in self.granges]
            self.cout = [torch.cuda.Stream() for _ in self.granges]
            self.ev_in = [[torch.cuda.Event(), torch.cuda.Event()] for _ in self.granges]
            self.pext = torch.cuda.ExternalStream(self.pstream)
            if fused:
                for p in self.gpaths:
                    p.prepare_fused()
        if self.pipeline:
            self.path.enable_pipeline()
            # (e2e) input copies of the next step, issued on a copy stream
            self.ev_in = [torch.cuda.Event(), torch.cuda.Event()]
            self.ev_main_prev = torch.cuda.Event()
        torch.cuda.synchronize()

    def step_args(self, s):
        i = self.inp
        return (i["q_idx"][s], i["w"][s], i["q_lat"][s], i["q_rope"][s], i["new_rows"][s], i["new_keys"][s])

    def start(self):
        """Initialise the cache and run the W warm-up steps."""
        self.units.init([self.wl.L0] * self.wl.U, self.warm)
        for s in range(self.Wm):
            self.path.step(self.abi.ROUND_AUTO, *self.step_args(s))
        self.torch.cuda.synchronize()

    def _record_pipelined(self, s0, e2e=None):
        """K steps with each step's gather copy and attention overlapping the
        next step's scoring (no L2 flush between steps: every step streams
        far more than L2 holds); one event pair brackets the K steps."""
        torch, path, rnd = self.torch, self.path, self.abi.ROUND_AUTO
        path.begin_graph()
        ev = [torch.cuda.Event(enable_timing=True, external=self.use_graph) for _ in range(2)]
        ev[0].record()
        for i in range(self.K):
            s = s0 + i
            if e2e is None:
                path.step_pipelined(rnd, *self.step_args(s))
            else:
                # step s's inputs arrive in buffer i & 1 (one copy, issued on
                # the copy stream during the step before); the copy of step
                # s + 1 goes into the other buffer once step s - 1, its last
                # reader, is done on both streams
                hpack, dpack, dev_in, out_host, cs = e2e
                main = torch.cuda.current_stream()
                b = i & 1
                if i == 0:
                    cs.wait_stream(main)
                    with torch.cuda.stream(cs):
                        dpack[0].copy_(hpack[s], non_blocking=True)
                    self.ev_in[0].record(cs)
                if i + 1 < self.K:
                    if i >= 1:
                        cs.wait_event(self.ev_main_prev)
                        cs.wait_event(path.ev_done)
                    with torch.cuda.stream(cs):
                        dpack[b ^ 1].copy_(hpack[s + 1], non_blocking=True)
                    self.ev_in[b ^ 1].record(cs)
                main.wait_event(self.ev_in[b])
                names = ("q_idx", "w", "q_lat", "q_rope", "new_rows", "new_keys")
                path.step_pipelined(rnd, *(dev_in[b][n] for n in names), out_host=out_host[i])
                self.ev_main_prev.record(main)
            self.ctr.add_(path.counters)
        path.join()
        ev[1].record()
        return [ev]

    def _record_groups(self, s0, e2e=None):
        """K steps of each session group, step after step on the group's own
        stream (score + select, gather assignment, gather copy, attention,
        append; a step's scoring follows the group's previous attention). The
        groups' scorings alternate: a group scores once the other group's
        last gather assignment is done, so each group's host-link copy runs
        beside the other group's scoring. One event pair brackets them."""
        torch, abi, rnd = self.torch, self.abi, self.abi.ROUND_AUTO
        main = torch.cuda.current_stream()
        names = ("q_idx", "w", "q_lat", "q_rope", "new_rows", "new_keys")
        ev = [torch.cuda.Event(enable_timing=True, external=self.use_graph) for _ in range(2)]
        ev[0].record()
        for st in self.gstreams:
            st.wait_stream(main)
        for i in range(self.K):
            s = s0 + i
            for g, ((lo, hi), p, st) in enumerate(zip(self.granges, self.gpaths, self.gstreams)):
                u = p.u
                with torch.cuda.stream(st):
                    if e2e is None:
                        qi, w, ql, qr, nr, nk = tuple(x[lo:hi] for x in self.step_args(s))
                    else:
                        hpack, dpack, dev_in, out_host, _ = e2e[g]
                        dpack[0].copy_(hpack[s], non_blocking=True)
                        qi, w, ql, qr, nr, nk = (dev_in[0][n] for n in names)
                    if i > 0 or g > 0:
                        st.wait_event(self.g_assigned[1 - g])
                    p.score_topk(qi, w, st)
                    abi.hot_gather_assign(u.units, u.U, p.R, p.K, rnd, p.topk, p.cls, p.counters, p.ws_gather,
                                          p.ws_gather_bytes, u.dev_err, st)
                    self.g_assigned[g].record(st)
                    abi.hot_gather_copy(u.units, u.U, p.R, p.K, p.topk, p.cls, p.rows, p.ws_gather,
                                        p.ws_gather_bytes, u.dev_err, st)
                    p.attend(ql, qr, st)
                    p.append(nr, nk, st)
                    if e2e is not None:
                        out_host[i].copy_(p.out, non_blocking=True)
                    self.ctr[lo:hi].add_(p.counters)
        for st in self.gstreams:
            main.wait_stream(st)
        ev[1].record()
        return [ev]

    def _record_partition(self, s0, e2e=None):
        """K steps of each session group, step after step on the group's own
        stream of the second SM partition, with every scoring on the first
        partition's stream (the groups' scorings alternate there): a group's
        selection, gather and attention, and append run on their own SMs
        beside the other group's scoring. A group's scoring follows its
        previous step; its selection follows its scoring. With e2e, a group's
        inputs reach the device two steps ahead (two buffers, an ordinary
        copy stream) and its outputs leave on another ordinary stream, which
        the group's next attention waits for. One event pair brackets them."""
        torch, abi, rnd = self.torch, self.abi, self.abi.ROUND_AUTO
        main = torch.cuda.current_stream()
        names = ("q_idx", "w", "q_lat", "q_rope", "new_rows", "new_keys")
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
        ev[0].record()
        for ts in self.tstreams + [self.pstream]:
            abi.dsa_stream_wait_stream(ts, main)
        if e2e is not None:
            for g in range(len(self.granges)):
                hpack, dpack, _, _, _ = e2e[g]
                self.cin[g].wait_stream(main)
                self.cout[g].wait_stream(main)
                for s in (s0, s0 + 1):
                    with torch.cuda.stream(self.cin[g]):
                        dpack[s & 1].copy_(hpack[s], non_blocking=True)
                    self.ev_in[g][s & 1].record(self.cin[g])
        for i in range(self.K):
            s = s0 + i
            for g, ((lo, hi), p, ts) in enumerate(zip(self.granges, self.gpaths, self.tstreams)):
                u = p.u
                if e2e is None:
                    qi, w, ql, qr, nr, nk = tuple(x[lo:hi] for x in self.step_args(s))
                else:
                    hpack, dpack, dev_in, out_host, _ = e2e[g]
                    qi, w, ql, qr, nr, nk = (dev_in[s & 1][n] for n in names)
                    self.pext.wait_event(self.ev_in[g][s & 1])        # this step's inputs are in
                abi.dsa_stream_wait_stream(self.pstream, ts)
                p.score(qi, w, self.pstream)
                abi.dsa_stream_wait_stream(ts, self.pstream)
                p.select(ts)
                if e2e is not None:
                    abi.dsa_stream_wait_stream(ts, self.cout[g])     # the previous output is read out
                if self.fused:
                    p.gather_attend(rnd, ql, qr, ts)
                else:
                    abi.hot_gather_assign(u.units, u.U, p.R, p.K, rnd, p.topk, p.cls, p.counters, p.ws_gather,
                                          p.ws_gather_bytes, u.dev_err, ts)
                    abi.hot_gather_copy(u.units, u.U, p.R, p.K, p.topk, p.cls, p.rows, p.ws_gather,
                                        p.ws_gather_bytes, u.dev_err, ts)
                    p.attend(ql, qr, ts)
                p.append(nr, nk, ts)
                with torch.cuda.stream(self.text[g]):
                    self.ctr[lo:hi].add_(p.counters)
                if e2e is not None:
                    abi.dsa_stream_wait_stream(self.cout[g], ts)
                    with torch.cuda.stream(self.cout[g]):
                        out_host[i].copy_(p.out, non_blocking=True)
                    if i + 2 < self.K:
                        # step s + 2's inputs into the buffer this step has finished with
                        abi.dsa_stream_wait_stream(self.cin[g], ts)
                        with torch.cuda.stream(self.cin[g]):
                            dpack[s & 1].copy_(hpack[s + 2], non_blocking=True)
                        self.ev_in[g][s & 1].record(self.cin[g])
        for ts in self.tstreams:
            abi.dsa_stream_wait_stream(main, ts)
        if e2e is not None:
            for st in self.cin + self.cout:
                main.wait_stream(st)
        ev[1].record()
        return [ev]

    def _record(self, s0, per_call, e2e=None):
        torch, path, rnd = self.torch, self.path, self.abi.ROUND_AUTO
        if self.part is not None and not per_call:
            return self._record_partition(s0, e2e)
        if self.groups and not per_call:
            return self._record_groups(s0, e2e)
        if self.pipeline and not per_call:
            return self._record_pipelined(s0, e2e)
        nev = 5 if per_call else 2
        ev = [[torch.cuda.Event(enable_timing=True, external=self.use_graph) for _ in range(nev)]
              for _ in range(self.K)]
        for i in range(self.K):
            s = s0 + i
            qi, w, ql, qr, nr, nk = self.step_args(s)
            self.flush.fill_(i & 0xFF)
            e = ev[i]
            e[0].record()
            if e2e is not None:
                hpack, dpack, dev_in2, out_host, _ = e2e
                dpack[0].copy_(hpack[s], non_blocking=True)
                qi, w, ql, qr, nr, nk = (dev_in2[0][n] for n in ("q_idx", "w", "q_lat", "q_rope", "new_rows", "new_keys"))
            if per_call:
                path.score_topk(qi, w)
                e[1].record()
                path.gather(rnd)
                e[2].record()
                path.attend(ql, qr)
                e[3].record()
                path.append(nr, nk)
            elif self.fused:
                path.step(rnd, qi, w, ql, qr, nr, nk, fused=True)
            else:
                path.step(rnd, qi, w, ql, qr, nr, nk, side=self.side)
            if e2e is not None:
                e2e[3][i].copy_(path.out, non_blocking=True)
            e[-1].record()
            if not per_call:
                self.ctr.add_(path.counters)
        return ev

    def segment(self, per_call=False, e2e=None):
        """The next K-step segment of the decode, captured as a graph (or, with
        --no-graph, a closure that launches it). Segments must be run in the
        order they were made."""
        s0 = self.Wm + self.next_seg * self.K
        self.next_seg += 1
        assert s0 + self.K <= self.total
        torch = self.torch
        if not self.use_graph:
            return (None, lambda: self._record(s0, per_call, e2e))
        graph = torch.cuda.CUDAGraph()
        cap = torch.cuda.Stream()
        cap.wait_stream(torch.cuda.current_stream())
        with torch.cuda.graph(graph, stream=cap):
            ev = self._record(s0, per_call, e2e)
        torch.cuda.synchronize()
        return (graph, ev)

    def run_segment(self, seg, clocks=None):
        """Run a segment; returns its per-step events."""
        torch = self.torch
        graph, ev = seg
        self.ctr.zero_()
        t0 = time.perf_counter()
        if graph is not None:
            graph.replay()
        else:
            ev = ev()
        torch.cuda.synchronize()
        t1 = time.perf_counter()
        if clocks is not None:
            clocks.window(t0, t1)
        err = self.units.check()
        if err:
            raise RuntimeError(f"device error word {err:#x}")
        return ev

    def _pack(self, lo, hi, out_shape):
        """Packed per-step inputs of units [lo, hi): one pinned host buffer
        per step (the six tensors at 256-byte aligned offsets), two device
        buffers of that layout with typed views, pinned host outputs, a copy
        stream; and the bytes in and out per step."""
        torch = self.torch
        names = ["q_idx", "w", "q_lat", "q_rope", "new_rows", "new_keys"]
        nst = self.inp[names[0]].shape[0]
        src = {n: self.inp[n][:, lo:hi] for n in names}
        offs, nbytes, total = {}, {}, 0
        for n in names:
            nb = src[n][0].numel() * src[n][0].element_size()
            offs[n], nbytes[n] = total, nb
            total += (nb + 255) // 256 * 256
        hpack = torch.empty((nst, total), dtype=torch.uint8).pin_memory()
        for n in names:
            hpack[:, offs[n]:offs[n] + nbytes[n]].copy_(src[n].reshape(nst, -1).view(torch.uint8))
        dev = self.inp[names[0]].device
        dpack = [torch.empty(total, dtype=torch.uint8, device=dev) for _ in range(2)]
        dev_in = [{n: dpack[b][offs[n]:offs[n] + nbytes[n]].view(src[n].dtype).view(src[n][0].shape)
                   for n in names} for b in range(2)]
        out_host = torch.empty((self.K,) + tuple(out_shape), dtype=torch.float32).pin_memory()
        nout = 1
        for x in out_shape:
            nout *= x
        return (hpack, dpack, dev_in, out_host, torch.cuda.Stream()), sum(nbytes.values()), nout * 4

    def e2e_buffers(self):
        """The inputs a caller hands over per step and the outputs it reads
        back (per session group with the group schedule)."""
        if self.groups:
            packs = [self._pack(lo, hi, p.out.shape) for (lo, hi), p in zip(self.granges, self.gpaths)]
            return [x[0] for x in packs], sum(x[1] for x in packs), sum(x[2] for x in packs)
        return self._pack(0, self.wl.U, self.path.out.shape)

    def close(self):
        if self.part is not None:
            self.abi.dsa_partition_destroy(self.part)
            self.abi.dsa_partition_destroy(self.rest)
            self.part = self.rest = None
        self.units.close()
        del self.inp, self.flush
        self.torch.cuda.synchronize()
        self.torch.cuda.empty_cache()


def host_link_gbs(torch):
    """Pinned host -> device copy bandwidth (DMA), the host link's rate."""
    hb = torch.empty(256 << 20, dtype=torch.uint8).pin_memory()
    db = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")
    for _ in range(2):
        db.copy_(hb, non_blocking=True)
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    for _ in range(4):
        db.copy_(hb, non_blocking=True)
    b.record()
    torch.cuda.synchronize()
    gbs = 4 * hb.numel() / (a.elapsed_time(b) * 1e6)
    del hb, db
    return gbs


def measure_restore(run, n_units):
    """kv_restore_full on the first n units after the timed steps: their whole
    history as dense rows, almost all of it read from the mirror over the host
    link with zero-copy 16-byte loads (the append-prefill restore)."""
    import torch
    from decode_attention_dsa_gb300 import abi
    g = run.units
    st = g.state[:n_units].cpu().numpy()
    rows = int(st[:, abi.ST_LEN].max())
    dst = torch.empty((n_units, rows, abi.ROW_BYTES), dtype=torch.uint8, device="cuda")
    sub = g.units[:n_units * ctypes.sizeof(abi.DsaUnit)]
    ms = []
    for _ in range(3):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        abi.kv_restore_full(sub, n_units, dst, rows, g.dev_err)
        b.record()
        torch.cuda.synchronize()
        ms.append(a.elapsed_time(b))
    nbytes = float(st[:, abi.ST_LEN].sum()) * abi.ROW_BYTES
    host_b = float(st[:, abi.ST_RAM].sum()) * abi.ROW_BYTES
    t = min(ms)
    del dst
    return {"units": n_units, "rows": int(st[:, abi.ST_LEN].sum()), "bytes": nbytes, "ms": t,
            "GB/s": nbytes / (t * 1e6), "host_GB/s": host_b / (t * 1e6),
            "note": "kv_restore_full (append-prefill restore) of the first units' whole history, best of 3; "
                    "rows below RAM are zero-copy reads of the pinned mirror"}


BREAKDOWN_SEGS = 3
SCORE_SMS = 120           # partition schedule: SMs the scorings run on
GROUPS = 2                # partition schedule: session groups taking turns on them
E2E_SEGS = 3
L2_BYTES = 126 << 20


def use_pipeline(args, wl):
    """The step schedule: "partition" (two halves of the sessions, each
    decoding step after step, every scoring on one SM partition and the rest
    of the steps on the other), "groups" (the same halves on ordinary streams,
    overlapping each other) or "lockstep"
    (every unit; a step's gather copy and attention overlap the next step's
    scoring) where the path allows it (one appended row, no selection reuse,
    split path) and every step streams more than L2 holds, so that no L2 flush
    is needed between the steps; else "serial" (no overlap)."""
    if args.no_pipeline or args.schedule == "serial":
        return "serial"
    # the fused gather runs in the partition schedule (the default) or serially
    ok = (wl.A == 1 and wl.reuse_every == 1 and (args.path != "fused" or args.schedule in (None, "partition"))
          and wl.U * wl.L0 * 128 > 4 * L2_BYTES)
    if not ok:
        return "serial"
    if args.schedule == "lockstep" or wl.sessions < 2:
        return "lockstep"
    return "groups" if args.schedule == "groups" else "partition"


def measure(args, wl, K, Wm, mirror, reps, world, clocks=None, e2e=False, breakdown=True):
    """Time one workload: `reps` consecutive K-step segments of one decode
    (median reported), then the per-call breakdown (median over 3 segments
    with events around each call, calls serial), the cache counters and
    (optionally) e2e over 3 more segments. Returns a dict."""
    import torch
    sched = use_pipeline(args, wl)
    use_graph = not args.no_graph and sched != "partition"
    # the partition schedule gathers inside the attention unless told otherwise
    fused = args.path == "fused" or (args.path is None and sched == "partition")
    # the partition schedule's kernels load into their green contexts at
    # their first launches there: one untimed segment first
    warm_seg = 1 if sched == "partition" else 0
    nseg = warm_seg + reps + (BREAKDOWN_SEGS if breakdown else 0) + (E2E_SEGS if e2e else 0)
    run = WorkloadRun(wl, K, Wm, nseg, mirror, fused, use_graph, pipeline=sched, score_sms=args.score_sms,
                      ngroups=args.groups)
    path, U = run.path, wl.U
    warm = [run.segment() for _ in range(warm_seg)]
    heads = [run.segment() for _ in range(reps)]
    bds = [run.segment(per_call=True) for _ in range(BREAKDOWN_SEGS)] if breakdown else []
    e2e_bufs = None
    if e2e:
        e2e_bufs, h2d, d2h = run.e2e_buffers()
        e2es = [run.segment(e2e=e2e_bufs) for _ in range(E2E_SEGS)]
    run.start()
    for seg in warm:
        run.run_segment(seg)
    totals, ctrs = [], []
    for seg in heads:
        ev = run.run_segment(seg, clocks=clocks)
        totals.append(sum(e[0].elapsed_time(e[-1]) for e in ev))
        ctrs.append(run.ctr.cpu().numpy().sum(axis=0))      # HOT, RING, RAM entries, fills over K steps
    total_ms = statistics.median(totals)
    if world > 1:
        t = torch.tensor([total_ms], dtype=torch.float64, device="cuda")
        torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
        total_ms = float(t.item())
    import numpy as np
    lps = (sum(p.launches_per_step(fused) for p in run.gpaths) if run.groups else
           path.launches_per_step(fused and not run.pipeline))
    res = {"run": run, "totals_ms": totals, "total_ms": total_ms, "ctr": np.mean(ctrs, axis=0),
           "launches_per_step": lps}
    if breakdown:
        per = []
        for seg in bds:
            evb = run.run_segment(seg)
            per.append([statistics.mean(e[j].elapsed_time(e[j + 1]) for e in evb) for j in range(4)] +
                       [statistics.mean(e[0].elapsed_time(e[4]) for e in evb)])
        res["call_ms"] = [statistics.median(p[j] for p in per) for j in range(4)]
        res["breakdown_step_ms"] = statistics.median(p[4] for p in per)
    if e2e:
        ms = []
        for seg in e2es:
            ee = run.run_segment(seg)
            ms.append(sum(e[0].elapsed_time(e[-1]) for e in ee))
        e2e_ms = statistics.median(ms)
        if world > 1:
            t = torch.tensor([e2e_ms], dtype=torch.float64, device="cuda")
            torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
            e2e_ms = float(t.item())
        res["e2e"] = {"value": world * U * K / (e2e_ms / 1e3), "unit": "layer-steps/s",
                      "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h), "ms_per_step": e2e_ms / K}
    del heads, bds
    if e2e:
        del e2es
    return res


def roofline(wl, res, K, Wm, host_gbs, path, host_kind="DMA pinned->device copy"):
    """Per-call achieved rates, the dominant call's roofline fraction and the
    step roofline (the slower of HBM bytes, host-link bytes and attention
    FLOPs at their peaks)."""
    peaks, peak_kind = load_peaks()
    hbm_peak = float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
    tc_peak = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
    U, R, A = wl.U, wl.R, wl.A
    ctr = res["ctr"]
    mean_L = wl.L0 + (Wm + (K - 1) / 2.0) * A
    key_bytes = (path.Us if path.sources else U) * mean_L * 128.0   # per score_topk call
    ram_b = ctr[2] / K * 656.0                                      # host-link bytes per step
    hbm_rows_b = (ctr[0] + ctr[1]) / K * 656.0 + ctr[3] / K * 656.0
    attn_flops = U * R * wl.H * wl.K * (576 + 512) * 2.0
    out = {}
    if "call_ms" in res:
        cm = res["call_ms"]
        calls = [
            ("dsa_score_topk", "hbm", key_bytes, cm[0]),
            ("hot_gather", "hbm", hbm_rows_b + ram_b, cm[1]),
            ("mla_decode_attn", "tensor", attn_flops, cm[2]),
            ("kv_append_writeback", "hbm", U * A * (656 + 128.0), cm[3]),
        ]
        name, bound, work, ms = max(calls, key=lambda c: c[3])
        if bound == "hbm":
            achieved, peak, unit = work / (ms * 1e6), hbm_peak, "GB/s"
        else:
            achieved, peak, unit = work / (ms * 1e9), tc_peak, "TFLOP/s"
        out["roofline"] = {"kernel": name, "bound": bound, "achieved": achieved, "peak": peak, "unit": unit,
                           "frac": achieved / peak, "peak_source": peak_kind, "traffic": traffic_for(name),
                           "work_per_launch": work,
                           "note": "achieved = algorithmic bytes (or FLOPs) per call / mean call time "
                                   "(CUDA events around the call, serial replay)"}
        out["per_call"] = {n: ({"ms": m, "GB/s": wk / (m * 1e6)} if bd == "hbm" else
                               {"ms": m, "TFLOP/s": wk / (m * 1e9)}) for n, bd, wk, m in calls}
    ms_step = res["total_ms"] / K
    hbm_step_b = key_bytes + hbm_rows_b
    t_roof = max(hbm_step_b / (hbm_peak * 1e6), ram_b / (host_gbs * 1e6), attn_flops / (tc_peak * 1e9))
    out["step_roofline"] = {"t_roof_ms": t_roof, "frac": t_roof / ms_step, "hbm_bytes": hbm_step_b,
                            "host_bytes": ram_b, "attn_flops": attn_flops, "host_link_gbs": host_gbs,
                            "host_link_kind": host_kind, "peak_source": peak_kind}
    out["cache"] = {"hot": int(ctr[0]), "ring": int(ctr[1]), "ram": int(ctr[2]), "fills": int(ctr[3]),
                    "miss_frac": float(ctr[2] / max(1, ctr[:3].sum()))}
    return out


def run_gpu(args, rank: int, world: int):
    import torch
    wl = workload(args)
    K = args.steps or default_steps(wl)
    Wm = max(3, args.warmup)
    reps = max(1, args.reps)
    host_gbs = host_link_gbs(torch)
    clocks = ClockSampler(torch.cuda.current_device())
    if world > 1:
        torch.distributed.barrier()
    clocks.start()
    pipe = use_pipeline(args, wl)
    res = measure(args, wl, K, Wm, args.mirror, reps, world, clocks=clocks, e2e=not args.no_e2e)
    clk = clocks.stop()
    run = res.pop("run")
    restore = measure_restore(run, min(4, wl.U)) if args.mirror == "host" else None
    # the host link's rate as the kernels meet it: the better of the DMA copy
    # and the zero-copy sequential read of the restore
    link, link_kind = host_gbs, "DMA pinned->device copy"
    if restore and restore["host_GB/s"] > link:
        link, link_kind = restore["host_GB/s"], "zero-copy sequential read (kv_restore_full)"
    value = world * wl.U * K / (res["total_ms"] / 1e3)
    line = {
        "metric": METRIC, "value": value, "unit": "layer-steps/s", "n_gpus": world, "steps": K,
        "warmup": Wm, "ms_per_step": res["total_ms"] / K, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": DTYPE,
        "data": "synthetic (seeded counter-based generator, generated on the device)",
        "config": workload_config(wl, {
            "mirror": args.mirror, "replacement": wl.policy,
            "l2": ("not flushed: every step streams more than L2 holds (keys of all units)" if pipe != "serial" else
                   "flushed before every timed step (512 MiB write outside the bracket)"),
            "selection_reuse_every": wl.reuse_every,
            "path": "hot_gather_attn (fused)" if args.path == "fused" and pipe != "partition" else {
                "partition": (f"{len(getattr(run, 'granges', ()))} session groups (contiguous, sizes "
                              f"{[(hi - lo) // wl.layers for lo, hi in getattr(run, 'granges', ())]} sessions), "
                              "each decoding step after step; the GPU split into two SM partitions (green "
                              "contexts): every scoring runs "
                              f"on the first ({getattr(run, 'part_sms', 0)} SMs), the groups' scorings "
                              "taking turns there; a group's selection, "
                              + ("gather fused into the attention (hot_gather_attn)" if run.fused else
                                 "gather (hot_gather_assign + hot_gather_copy), attention")
                              + f" and append run on the second ({getattr(run, 'rest_sms', 0)} SMs), beside "
                              "the other groups' scorings"),
                "groups": ("two session groups (sessions [0, S/2) and [S/2, S)), each decoding step after "
                           "step on its own stream (score, select, gather, attention, append); one group's "
                           "gather copy and attention overlap the other group's scoring"),
                "lockstep": ("lockstep pipeline: each step's gather copy and attention (side stream) overlap "
                             "the next step's score and select"),
                "serial": "hot_gather + mla_decode_attn, append concurrent"}[pipe],
            "timing": f"median of {reps} consecutive {K}-step segments of one decode "
                      f"({'one CUDA graph each' if run.use_graph else 'launched directly'}) "
                      f"after {Wm} warm-up steps"
                      + (f" and one untimed {K}-step segment of the schedule" if pipe == "partition" else ""),
            "parallelism": "replicas" if world > 1 else "single GPU"}),
        "tok_per_s": value * wl.A / wl.layers,
        "segments_ms_per_step": [t / K for t in res["totals_ms"]],
    }
    line.update(roofline(wl, res, K, Wm, link, run.path, link_kind))
    line["host_link"] = {"dma_copy_gbs": host_gbs, "restore": restore}
    line["per_call_note"] = (f"median over {BREAKDOWN_SEGS} further {K}-step segments with events around each "
                             f"call, calls serial ({res['breakdown_step_ms']:.4f} ms/step there)")
    line["clocks"] = clk
    line["gpu_launches"] = res["launches_per_step"] * K
    line["cuda_graph"] = run.use_graph
    if "e2e" in res:
        line["e2e"] = res["e2e"]
    run.close()
    del run

    if rank == 0 and world == 1 and not args.no_secondary and args.config != 1:
        wl1 = workload(args, 1)
        r1 = measure(args, wl1, K, Wm, "host", reps, 1)
        run1 = r1.pop("run")
        v1 = wl1.U * K / (r1["total_ms"] / 1e3)
        sec = {"workload": wl1.name, "value": v1, "unit": "layer-steps/s", "ms_per_step": r1["total_ms"] / K,
               "tok_per_s": v1 * wl1.A / wl1.layers, "steps": K}
        rf = roofline(wl1, r1, K, Wm, link, run1.path, link_kind)
        sec.update({k: rf[k] for k in ("step_roofline", "per_call", "cache")})
        line["secondary"] = sec
        run1.close()
        del run1
    if rank == 0 and world == 1 and not args.no_gate:
        line["gate"] = offload_gate(args, K, Wm)
    return line


def offload_gate(args, K, Wm):
    """The MTP=3 verify workload with the mirror in pinned host memory
    (offloaded) and in HBM (resident), same kernels; the two decodes run
    their segments interleaved (host, device, host, ...); the gap is
    (offloaded - resident) / resident in step time (best segment of each)."""
    import torch
    wl2 = workload(args, 2)
    use_graph = not args.no_graph
    nrep = max(3, min(5, args.reps))
    runs = {m: WorkloadRun(wl2, K, Wm, nrep, m, args.path == "fused", use_graph) for m in ("host", "device")}
    segs = {m: [r.segment() for _ in range(nrep)] for m, r in runs.items()}
    for r in runs.values():
        r.start()
    ms = {"host": [], "device": []}
    for i in range(nrep):
        for m in ("host", "device"):
            ev = runs[m].run_segment(segs[m][i])
            ms[m].append(sum(e[0].elapsed_time(e[-1]) for e in ev) / K)
    del segs
    for m in runs:
        runs[m].close()
    del runs
    torch.cuda.empty_cache()
    best = {m: min(v) for m, v in ms.items()}
    gap = (best["host"] - best["device"]) / best["device"] * 100.0
    return {"workload": wl2.name, "steps": K, "offloaded_ms_per_step": best["host"],
            "resident_ms_per_step": best["device"], "gap_pct": gap, "within_5pct": gap <= 5.0,
            "segments_ms_per_step": ms,
            "note": "best of interleaved segments of two continuous decodes (host, device, host, ...)"}


def main():
    args = parse()
    if args.oracle_child:
        oracle_child(args.oracle_child)
        return 0
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        if rank != 0:
            return 0
        print(json.dumps(reference_arm(args)), flush=True)
        return 0
    import torch
    torch.cuda.set_device(local)
    if world > 1:
        torch.distributed.init_process_group("nccl")
    line = run_gpu(args, rank, world)
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        # after all GPU work: the oracle on a bounded sample of the same workload
        wl = workload(args)
        n = args.cpu_sample_steps or 12
        try:
            r = run_oracle(args.config, args.sessions, n, 1)
            v = r["unit_steps"] / r["seconds"]
            line["cpu_baseline"] = {"value": v, "unit": "layer-steps/s", "cores": r["threads"], "kind": "oracle",
                                    "sample": sample_text(wl, n, r)}
        except Exception as e:  # reported, not fatal
            line["cpu_baseline"] = {"value": None, "unit": "layer-steps/s", "cores": 1, "kind": "oracle",
                                    "sample": "failed: " + str(e)[-300:]}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
