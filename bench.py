#!/usr/bin/env python3
"""Benchmark of the sparse-attention decode path on GB300.

One *step* is one decode step of every unit of the workload through the whole
path: DSA score + Top-K, hot gather, Q8G64 dequant + MLA attention, append with
batched write-back. The default workload is the 50K single stream (50,023-token
history, 4 layers, 1 query row, Top-2048, 64 heads, 32,768 hot slots, mirror in
pinned host memory). The value is layer-steps/s (units x steps / time).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--config C]
                  [--mirror host|device] [--impl gb300|reference]

Timing: W >= 3 untimed warm-up steps, then K steps; L2 is flushed (a 512 MiB
write) before every timed step, outside its CUDA-event bracket; the sum of the
per-step event times is the timed total. The K timed steps (flushes and event
records included) are captured once into a CUDA graph and replayed once, so
host launch cost is off the device timeline; ``--no-graph`` launches directly. Inputs are generated on the device
before timing. ``e2e`` repeats the K steps from the same initial state through
the C ABI with host buffers: each step copies its inputs from pinned host
memory and the attention output back, inside the bracket.

``--impl reference`` times the CPU oracle (the only reference there is: the
pages publish no code) on the host cores, on one unit-step per step.
Under torchrun (N > 1) every rank runs an independent replica of the workload
(the path runs on one GPU; there is no collective on the data path).
"""
from __future__ import annotations

import argparse
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


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=None)
    ap.add_argument("--warmup", type=int, default=8)
    ap.add_argument("--config", type=int, default=1)
    ap.add_argument("--mirror", choices=["host", "device"], default="host")
    ap.add_argument("--impl", choices=["gb300", "reference"], default="gb300")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-graph", action="store_true", help="launch steps directly, no CUDA graph")
    ap.add_argument("--reuse-every", type=int, default=1,
                    help="layer l reuses the selection of layer l - l %% N (1: every layer scores)")
    ap.add_argument("--path", choices=["fused", "split"], default=None,
                    help="fused: hot_gather_attn; split: hot_gather + mla_decode_attn with the append "
                         "overlapping the attention (default: split, the faster one measured)")
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


# ---------------------------------------------------------------- CPU oracle leg

def oracle_child(spec: str) -> None:
    """Run in a fresh interpreter: time the oracle on a bounded sample."""
    os.environ.setdefault("OPENBLAS_NUM_THREADS", "1")
    os.environ.setdefault("OMP_NUM_THREADS", "1")
    os.environ.setdefault("MKL_NUM_THREADS", "1")
    import numpy as np
    from oracle.decode import OracleUnit, decode_step
    from synth import workloads as W
    cfg = json.loads(spec)
    wl = W.WORKLOADS[cfg["config"]]
    nsteps, warm = cfg["steps"], cfg["warmup"]
    units = list(range(wl.U))
    wl2 = wl.with_(steps=max(wl.steps, nsteps + warm + 1))
    ous = {}
    t0 = time.time()
    for u in units:
        keys = W.keys_bits(wl2, u, np.arange(wl.L0))
        ous[u] = OracleUnit.create(wl.S, wl2.lmax, wl.L0, keys,
                                   (lambda pos, u=u: W.rows_bytes(wl2, u, pos)), wl.warm)
    setup = time.time() - t0
    # one unit-step per bench step, units round robin; each unit keeps its own
    # step counter so every unit replays its own decode sequence
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
    print(json.dumps({"seconds": dt, "unit_steps": nsteps, "setup_s": setup, "threads": 1}))


def run_oracle(config: int, steps: int, warmup: int) -> dict:
    env = dict(os.environ, OPENBLAS_NUM_THREADS="1", OMP_NUM_THREADS="1", MKL_NUM_THREADS="1")
    spec = json.dumps({"config": config, "steps": steps, "warmup": warmup})
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


def reference_arm(args) -> dict:
    from synth import workloads as W
    wl = W.WORKLOADS[args.config]
    steps = args.steps or wl.steps
    warm = max(3, args.warmup)
    r = run_oracle(args.config, steps, warm)
    value = r["unit_steps"] / r["seconds"]
    sample = (f"{steps} unit-steps (units round robin, each replaying its own decode steps from "
              f"the start) of the {wl.name} workload, float64 oracle, 1 thread")
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
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []
        self.t = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
            time.sleep(0.3)
        except Exception:
            self.proc = None

    def _read(self):
        for ln in self.proc.stdout:
            self.lines.append(ln.strip())

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.2)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = float(f[2])
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------- GPU arm

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


def run_gpu(args, rank: int, world: int):
    import torch
    from decode_attention_dsa_gb300 import abi
    from decode_attention_dsa_gb300.step import DecodePath
    from decode_attention_dsa_gb300.units import UnitSet
    from synth import gpu as sg
    from synth import workloads as W

    wl = W.WORKLOADS[args.config]
    if args.reuse_every > 1:
        wl = wl.with_(reuse_every=args.reuse_every)
    K = args.steps or wl.steps
    Wm = max(3, args.warmup)
    total = Wm + K
    wlr = wl.with_(steps=total)
    U, R, A = wl.U, wl.R, wl.A
    dev = torch.device("cuda")
    units = UnitSet(U, wl.S, wlr.lmax, mirror=args.mirror)
    src = [wl.selection_source(u) for u in range(U)] if wl.reuse_every > 1 else None
    path = DecodePath(units, R, wl.K, wl.H, A, wl.scale(), selection_source=src)
    sg.history(wlr, units)
    inp = sg.step_inputs(wlr, 0, total)
    if path.sources:
        # only the source units' indexer queries are scored (set up before timing)
        inp["q_idx"] = inp["q_idx"][:, path.sources].contiguous()
        inp["w"] = inp["w"][:, path.sources].contiguous()
    torch.cuda.synchronize()
    flush = torch.empty(512 << 20, dtype=torch.uint8, device=dev)
    warm = abi.WARM_LAST_S if wl.warm == "last_s" else abi.WARM_EMPTY

    def step_args(s):
        return (inp["q_idx"][s], inp["w"][s], inp["q_lat"][s], inp["q_rope"][s],
                inp["new_rows"][s], inp["new_keys"][s])

    # ---- device-resident run
    units.init([wl.L0] * U, warm)
    for s in range(Wm):
        path.step(abi.ROUND_AUTO, *step_args(s))
    torch.cuda.synchronize()
    use_graph = not args.no_graph
    rnd = abi.ROUND_AUTO

    side = torch.cuda.Stream()
    fused = args.path == "fused"

    def record_steps(nsteps, per_call, ctr_acc=None):
        """Enqueue nsteps timed steps; returns the events. per_call adds
        events between the four calls and runs them one after another (a
        separate breakdown run); otherwise the append runs on a side stream
        concurrently with the attention, as the API allows."""
        nev = 5 if per_call else 2
        ev = [[torch.cuda.Event(enable_timing=True, external=use_graph) for _ in range(nev)]
              for _ in range(nsteps)]
        for i in range(nsteps):
            s = Wm + i
            qi, w, ql, qr, nr, nk = step_args(s)
            flush.fill_(i & 0xFF)
            e = ev[i]
            e[0].record()
            if per_call:
                path.score_topk(qi, w)
                e[1].record()
                path.gather(rnd)
                e[2].record()
                path.attend(ql, qr)
                e[3].record()
                path.append(nr, nk)
            elif fused:
                path.step(rnd, qi, w, ql, qr, nr, nk, fused=True)
            else:
                path.step(rnd, qi, w, ql, qr, nr, nk, side=side)
            e[-1].record()
            if ctr_acc is not None:
                ctr_acc.add_(path.counters)
        return ev

    def run_steps(nsteps, per_call, ctr_acc=None):
        if use_graph:
            graph = torch.cuda.CUDAGraph()
            cap = torch.cuda.Stream()
            cap.wait_stream(torch.cuda.current_stream())
            with torch.cuda.graph(graph, stream=cap):
                ev = record_steps(nsteps, per_call, ctr_acc)
            torch.cuda.synchronize()
            return ev, graph
        return None, None

    def warm_start():
        units.init([wl.L0] * U, warm)
        for s in range(Wm):
            path.step(rnd, *step_args(s))
        torch.cuda.synchronize()

    # ---- headline run: events only at step boundaries
    ctr_acc = torch.zeros((U, 4), dtype=torch.int64, device=dev)
    ev, graph = run_steps(K, False, ctr_acc)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    clocks = ClockSampler(torch.cuda.current_device())
    clocks.start()
    wall0 = time.perf_counter()
    if graph is not None:
        graph.replay()
    else:
        ev = record_steps(K, False, ctr_acc)
    torch.cuda.synchronize()
    wall = time.perf_counter() - wall0
    clk = clocks.stop()
    err = units.check()
    if err:
        raise RuntimeError(f"device error word {err:#x}")
    step_ms = [e[0].elapsed_time(e[-1]) for e in ev]
    total_ms = sum(step_ms)
    if world > 1:
        t = torch.tensor([total_ms], dtype=torch.float64, device=dev)
        torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
        total_ms = float(t.item())
    del graph

    # ---- breakdown run (same start state): events around each call
    KB = min(K, 256)
    warm_start()
    evb, gb = run_steps(KB, True)
    if gb is not None:
        gb.replay()
    else:
        evb = record_steps(KB, True)
    torch.cuda.synchronize()
    call_ms = [statistics.mean(e[j].elapsed_time(e[j + 1]) for e in evb) for j in range(4)]
    breakdown_step_ms = statistics.mean(e[0].elapsed_time(e[4]) for e in evb)
    del gb
    ctr = ctr_acc.cpu().numpy().sum(axis=0)    # HOT, RING, RAM entries, fills over K steps

    # ---- end to end through the C ABI with host buffers (same K steps, same start state)
    e2e = None
    if not args.no_e2e:
        names = ["q_idx", "w", "q_lat", "q_rope", "new_rows", "new_keys"]
        host = {n: torch.empty_like(inp[n][Wm:], device="cpu").pin_memory() for n in names}
        for n in names:
            host[n].copy_(inp[n][Wm:])
        dev_in = {n: torch.empty_like(inp[n][0]) for n in names}
        out_host = torch.empty((K,) + tuple(path.out.shape), dtype=torch.float32).pin_memory()
        h2d = sum(host[n][0].numel() * host[n][0].element_size() for n in names)
        d2h = path.out.numel() * 4
        units.init([wl.L0] * U, warm)
        for s in range(Wm):
            path.step(abi.ROUND_AUTO, *step_args(s))
        torch.cuda.synchronize()
        ee = [(torch.cuda.Event(enable_timing=True, external=use_graph),
               torch.cuda.Event(enable_timing=True, external=use_graph)) for _ in range(K)]

        def e2e_steps():
            for i in range(K):
                flush.fill_(i & 0xFF)
                ee[i][0].record()
                for n in names:
                    dev_in[n].copy_(host[n][i], non_blocking=True)
                path.step(abi.ROUND_AUTO, dev_in["q_idx"], dev_in["w"], dev_in["q_lat"],
                          dev_in["q_rope"], dev_in["new_rows"], dev_in["new_keys"], side=side, fused=fused)
                out_host[i].copy_(path.out, non_blocking=True)
                ee[i][1].record()
        if use_graph:
            g2 = torch.cuda.CUDAGraph()
            cap = torch.cuda.Stream()
            cap.wait_stream(torch.cuda.current_stream())
            with torch.cuda.graph(g2, stream=cap):
                e2e_steps()
            torch.cuda.synchronize()
            g2.replay()
        else:
            e2e_steps()
        torch.cuda.synchronize()
        e2e_ms = sum(a.elapsed_time(b) for a, b in ee)
        if world > 1:
            t = torch.tensor([e2e_ms], dtype=torch.float64, device=dev)
            torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
            e2e_ms = float(t.item())
        e2e = {"value": world * U * K / (e2e_ms / 1e3), "unit": "layer-steps/s",
               "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
               "ms_per_step": e2e_ms / K}

    # ---- host-link copy bandwidth (DMA, pinned -> device), for the roofline's host term
    hb = torch.empty(256 << 20, dtype=torch.uint8).pin_memory()
    db = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    for _ in range(2):
        db.copy_(hb, non_blocking=True)
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    for _ in range(4):
        db.copy_(hb, non_blocking=True)
    b.record()
    torch.cuda.synchronize()
    host_gbs = 4 * hb.numel() / (a.elapsed_time(b) * 1e6)
    del hb, db

    peaks, peak_kind = load_peaks()
    hbm_peak = float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
    tc_peak = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
    mean_L = wl.L0 + (Wm + (K - 1) / 2.0) * A
    key_bytes = (path.Us if path.sources else U) * mean_L * 128.0   # per score_topk launch
    ent = ctr[:3].sum() / K
    ram_b = ctr[2] / K * 656.0                              # host-link bytes per step
    hbm_rows_b = (ctr[0] + ctr[1]) / K * 656.0 + ctr[3] / K * 656.0
    attn_flops = U * R * wl.H * wl.K * (576 + 512) * 2.0
    calls = [
        ("dsa_score_topk", "hbm", key_bytes, call_ms[0]),
        ("hot_gather", "hbm", hbm_rows_b + ram_b, call_ms[1]),
        ("mla_decode_attn", "tensor", attn_flops, call_ms[2]),
        ("kv_append_writeback", "hbm", U * A * (656 + 128.0), call_ms[3]),
    ]
    dom = max(calls, key=lambda c: c[3])
    name, bound, work, ms = dom
    if bound == "hbm":
        achieved, peak, unit = work / (ms * 1e6), hbm_peak, "GB/s"
    else:
        achieved, peak, unit = work / (ms * 1e9), tc_peak, "TFLOP/s"
    per_call = {}
    for n, bd, wk, m in calls:
        if bd == "hbm":
            per_call[n] = {"ms": m, "GB/s": wk / (m * 1e6)}
        else:
            per_call[n] = {"ms": m, "TFLOP/s": wk / (m * 1e9)}
    ms_step = total_ms / K
    hbm_step_b = key_bytes + hbm_rows_b
    t_roof_ms = max(hbm_step_b / (hbm_peak * 1e6), ram_b / (host_gbs * 1e6),
                    attn_flops / (tc_peak * 1e9))
    value = world * U * K / (total_ms / 1e3)
    line = {
        "metric": METRIC, "value": value, "unit": "layer-steps/s", "n_gpus": world, "steps": K,
        "warmup": Wm, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "fp32 score / u8 rows / fp32 attention",
        "data": "synthetic (seeded counter-based generator, generated on the device)",
        "config": workload_config(wl, {"mirror": args.mirror, "l2": "flushed before every timed step",
                                       "selection_reuse_every": wl.reuse_every,
                                       "path": "hot_gather_attn (fused)" if fused else
                                               "hot_gather + mla_decode_attn, append concurrent",
                                       "parallelism": "replicas" if world > 1 else "single GPU"}),
        "tok_per_s": value * A / wl.layers,
        "roofline": {"kernel": name, "bound": bound, "achieved": achieved, "peak": peak,
                     "unit": unit, "frac": achieved / peak, "peak_source": peak_kind,
                     "traffic": traffic_for(name)},
        "step_roofline": {"t_roof_ms": t_roof_ms, "frac": t_roof_ms / ms_step,
                          "hbm_bytes": hbm_step_b, "host_bytes": ram_b, "attn_flops": attn_flops,
                          "host_link_gbs": host_gbs, "host_link_kind": "DMA pinned->device copy",
                          "peak_source": peak_kind},
        "per_call": per_call,
        "per_call_note": (f"mean over a separate replay of {KB} steps from the same start with "
                          f"events around each call ({breakdown_step_ms:.4f} ms/step there)"),
        "cache": {"hot": int(ctr[0]), "ring": int(ctr[1]), "ram": int(ctr[2]), "fills": int(ctr[3]),
                  "miss_frac": float(ctr[2] / max(1, ctr[:3].sum()))},
        "clocks": clk,
        "gpu_launches": path.launches_per_step() * K,
        "cuda_graph": use_graph,
        "wall_s": wall,
    }
    if e2e:
        line["e2e"] = e2e
    units.close()
    return line


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
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        # the CPU leg runs in a child process started before any CUDA work
        from synth import workloads as W
        wl = W.WORKLOADS[args.config]
        n = args.cpu_sample_steps or min(64, wl.steps) * 1
        cpu_res = {}

        def go():
            try:
                cpu_res.update(run_oracle(args.config, n, 2))
            except Exception as e:  # reported, not fatal
                cpu_res["error"] = str(e)[-300:]
        th = threading.Thread(target=go)
        th.start()
    import torch
    torch.cuda.set_device(local)
    if world > 1:
        torch.distributed.init_process_group("nccl")
    line = run_gpu(args, rank, world)
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        th.join()
        if "seconds" in cpu_res:
            v = cpu_res["unit_steps"] / cpu_res["seconds"]
            cpu = {"value": v, "unit": "layer-steps/s", "cores": cpu_res["threads"], "kind": "oracle",
                   "sample": f"{cpu_res['unit_steps']} unit-steps of the same workload, units round "
                             f"robin, float64 oracle, 1 thread ({cpu_res['seconds']:.1f} s)"}
        else:
            cpu = {"value": None, "unit": "layer-steps/s", "cores": 1, "kind": "oracle",
                   "sample": "failed: " + cpu_res.get("error", "?")}
        line["cpu_baseline"] = cpu
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
