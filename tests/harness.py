"""Shared set-up for the GPU parity tests: builds the same workload on the
CUDA path (through the C ABI) and in the oracle, from the numpy generator."""
from __future__ import annotations

import numpy as np

from oracle.decode import OracleUnit, decode_step
from oracle.hotcache import PAD
from synth import workloads as W


def gpu_modules():
    import torch
    from decode_attention_dsa_gb300 import abi
    from decode_attention_dsa_gb300.step import DecodePath
    from decode_attention_dsa_gb300.units import UnitSet
    return torch, abi, UnitSet, DecodePath


class Pair:
    """A workload run side by side on the GPU and in the oracle."""

    def __init__(self, wl: W.Workload, units=None, mirror="host", oracle_units=None, gpu_gen=False):
        torch, abi, UnitSet, DecodePath = gpu_modules()
        self.torch, self.abi = torch, abi
        self.wl = wl
        self.uidx = list(range(wl.U)) if units is None else list(units)
        self.oidx = self.uidx if oracle_units is None else list(oracle_units)
        U = len(self.uidx)
        self.g = UnitSet(U, wl.S, wl.lmax, mirror=mirror, policy=wl.policy)
        self.o = {}
        hist = np.arange(wl.L0)
        if gpu_gen:
            # history drawn on the device (same bytes as the numpy generator);
            # the oracle regenerates its units with numpy, mirror rows on demand
            from synth import gpu as sg
            assert self.uidx == list(range(wl.U))
            sg.history(wl, self.g)
            for u in self.oidx:
                keys = W.keys_bits(wl, u, hist)
                self.o[u] = OracleUnit.create(wl.S, wl.lmax, wl.L0, keys,
                                              (lambda pos, u=u: W.rows_bytes(wl, u, pos)), wl.warm,
                                              policy=wl.policy)
        for i, u in enumerate(self.uidx):
            if gpu_gen:
                break
            keys = W.keys_bits(wl, u, hist)
            rows = W.rows_bytes(wl, u, hist)
            self.g.set_keys(i, 0, keys)
            self.g.set_mirror_rows(i, 0, rows)
            if u in self.oidx:
                self.o[u] = OracleUnit.create(wl.S, wl.lmax, wl.L0, keys, rows, wl.warm, policy=wl.policy)
        self.g.init([wl.L0] * U, abi.WARM_LAST_S if wl.warm == "last_s" else abi.WARM_EMPTY)
        src = [wl.selection_source(u) for u in self.uidx] if wl.reuse_every > 1 else None
        self.p = DecodePath(self.g, wl.R, wl.K, wl.H, wl.A, wl.scale(), selection_source=src)
        torch.cuda.synchronize()

    def inputs(self, step):
        torch = self.torch
        per = [W.step_inputs(self.wl, u, step) for u in self.uidx]
        dev = self.g.device

        def t16(a):
            return torch.from_numpy(np.ascontiguousarray(np.stack(a)).view(np.int16)).to(dev)
        sel = (lambda a: [a[i] for i, u in enumerate(self.uidx) if self.wl.selection_source(u) == u]) \
            if self.wl.reuse_every > 1 else (lambda a: a)
        return per, dict(
            q_idx=t16(sel([x.q_idx for x in per])),
            w=torch.from_numpy(np.stack(sel([x.w for x in per]))).to(dev),
            q_lat=t16([x.q_lat for x in per]),
            q_rope=t16([x.q_rope for x in per]),
            new_rows=torch.from_numpy(np.stack([x.new_rows for x in per])).to(dev),
            new_keys=t16([x.new_keys for x in per]),
        )

    def step(self, step, rnd=None, attention=True, oracle_rnd=None, side=None):
        """Run one step on both sides; return (gpu dict, oracle dict per unit).
        With a ``side`` stream the append runs there, concurrently with the
        attention."""
        rnd = step if rnd is None else rnd
        ornd = rnd if oracle_rnd is None else oracle_rnd
        per, t = self.inputs(step)
        self.last_inputs = per
        p = self.p
        if side == "fused":
            p.step(rnd, t["q_idx"], t["w"], t["q_lat"], t["q_rope"], t["new_rows"], t["new_keys"], fused=True)
        elif side is not None:
            assert attention
            p.step(rnd, t["q_idx"], t["w"], t["q_lat"], t["q_rope"], t["new_rows"], t["new_keys"], side=side)
        else:
            p.score_topk(t["q_idx"], t["w"])
            p.gather(rnd)
            if attention:
                p.attend(t["q_lat"], t["q_rope"])
            p.append(t["new_rows"], t["new_keys"])
        self.torch.cuda.synchronize()
        g = dict(topk=p.topk.cpu().numpy(), cls=p.cls.cpu().numpy(), counters=p.counters.cpu().numpy())
        if attention:
            g["out"] = p.out.cpu().numpy()
            g["lse"] = p.lse.cpu().numpy()
        g["rows"] = p.rows.cpu().numpy()
        ores = {}
        for i, u in enumerate(self.uidx):
            if u not in self.o:
                continue
            x = per[i]
            given = None
            if self.wl.reuse_every > 1 and self.wl.selection_source(u) != u:
                given = ores[self.wl.selection_source(u)]["topk"]   # sources come first in unit order
            ores[u] = decode_step(self.o[u], ornd, self.wl.K, self.wl.scale(), x.q_idx, x.w, x.q_lat,
                                  x.q_rope, x.new_rows, x.new_keys, attention=attention, topk=given)
        return g, ores

    def state(self, i):
        g = self.g
        return dict(slot_pos=g.slot_pos[i].cpu().numpy(), fill_round=g.fill_round[i].cpu().numpy(),
                    pos_slot=g.pos_slot[i].cpu().numpy(), st=g.state[i].cpu().numpy(),
                    ring=g.ring[i].cpu().numpy(), ref=g.ref[i].cpu().numpy())


def lse_bound(pair, per_q, r, i):
    """Per-head bound on |lse_gpu - lse_oracle|: the tensor-core operands are
    rounded once to fp16 (relative error <= 2^-11 each), so every logit moves by
    at most scale * 2^-11 * sum_d |q_d| * |k_d| * 2 (one rounding on each side
    of the product, q is exact for these bf16 inputs but is counted anyway);
    log-sum-exp moves by at most the largest logit change. 1e-5 covers fp32
    accumulation and the exp/log evaluations."""
    from oracle.q8g64 import dequant_latent, rope_values
    from oracle.indexer import bf16_to_f64
    wl = pair.wl
    rows = per_q["rows"][r][per_q["cls"][r] != PAD]
    k = np.concatenate([np.abs(dequant_latent(rows)), np.abs(rope_values(rows))], axis=1)
    x = pair.last_inputs[i]
    q = np.concatenate([np.abs(bf16_to_f64(x.q_lat[r])), np.abs(bf16_to_f64(x.q_rope[r]))], axis=1)
    return wl.scale() * 2.0 ** -11 * 2 * (q @ k.T).max(axis=1) + 1e-5


def lse_fp16_operands(pair, per_q, r, i):
    """log-sum-exp of one query row with the tensor cores' operands: the
    query (bf16) and the dequantised key values (int8 * fp16 scale, RoPE bf16)
    each rounded once to fp16 (round to nearest even, as the kernel's
    conversions do), everything else in float64. Against this the kernel's
    lse differs only by fp32 accumulation and exp/log evaluation (well under
    2e-4 for these magnitudes), a check ~100x tighter than lse_bound's, which
    has to cover the fp16 roundings themselves."""
    from oracle.q8g64 import dequant_latent, rope_values
    from oracle.indexer import bf16_to_f64
    wl = pair.wl
    rows = per_q["rows"][r][per_q["cls"][r] != PAD]
    f16 = lambda a: np.asarray(a, np.float64).astype(np.float16).astype(np.float64)
    k = np.concatenate([f16(dequant_latent(rows)), f16(rope_values(rows))], axis=1)
    x = pair.last_inputs[i]
    q = np.concatenate([f16(bf16_to_f64(x.q_lat[r])), f16(bf16_to_f64(x.q_rope[r]))], axis=1)
    lg = wl.scale() * (q @ k.T)
    m = lg.max(axis=1)
    return m + np.log(np.exp(lg - m[:, None]).sum(axis=1))


def check_step(pair: Pair, g, ores, attention=True, rows=True, full_state=True, atol_rel=1e-3):
    """Element-by-element comparison of one step; returns the worst attention error ratio."""
    worst = 0.0
    wl = pair.wl
    for i, u in enumerate(pair.uidx):
        if u not in ores:
            continue
        o = ores[u]
        oc = pair.o[u].cache
        assert np.array_equal(g["topk"][i], o["topk"]), f"unit {u}: Top-K differs"
        assert np.array_equal(g["cls"][i], o["cls"]), f"unit {u}: classification differs"
        assert np.array_equal(g["counters"][i], o["counters"]), f"unit {u}: counters differ"
        if rows:
            assert np.array_equal(g["rows"][i], o["rows"]), f"unit {u}: gathered rows differ"
        if full_state and getattr(pair, "check_slots", False):
            gs = pair.g.slots[i].cpu().numpy()
            occ = oc.slot_pos >= 0
            assert np.array_equal(gs[occ], oc.slots[occ]), f"unit {u}: slot bytes differ"
        s = pair.state(i)
        assert np.array_equal(s["slot_pos"], oc.slot_pos), f"unit {u}: slot map differs"
        assert np.array_equal(s["fill_round"], oc.fill_round), f"unit {u}: fill rounds differ"
        assert s["st"][0] == oc.length and s["st"][1] == oc.rows_in_ram, f"unit {u}: len/ram"
        assert s["st"][2] == oc.hand, f"unit {u}: hand differs"
        if wl.policy == "clock":
            assert np.array_equal(s["ref"], oc.ref), f"unit {u}: reference bits differ"
        if full_state:
            assert np.array_equal(s["pos_slot"], oc.pos_slot[:wl.lmax]), f"unit {u}: pos_slot"
            assert np.array_equal(s["ring"], oc.ring), f"unit {u}: ring differs"
        if attention:
            for r in range(wl.R):
                ref = o["out"][r]
                err = np.abs(g["out"][i, r].astype(np.float64) - ref).max()
                scale = np.abs(ref).max()
                ratio = err / (atol_rel * scale) if scale > 0 else err
                worst = max(worst, ratio)
                assert err <= atol_rel * scale or (scale == 0 and err == 0), \
                    f"unit {u} row {r}: attention err {err:.3e} > {atol_rel}*{scale:.3e}"
                valid = o["cls"][r] != PAD
                if valid.any():
                    tol = lse_bound(pair, per_q=ores[u], r=r, i=i)
                    d = np.abs(g["lse"][i, r].astype(np.float64) - o["lse"][r])
                    assert (d <= tol).all(), f"unit {u} row {r}: lse err {d.max():.3e}"
                    d16 = np.abs(g["lse"][i, r].astype(np.float64) - lse_fp16_operands(pair, ores[u], r, i))
                    assert (d16 <= 2e-4).all(), f"unit {u} row {r}: lse vs fp16-operand lse {d16.max():.3e}"
                else:
                    assert np.isneginf(g["lse"][i, r]).all()
    return worst
