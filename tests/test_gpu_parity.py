"""GPU parity: the CUDA path through the C ABI against the oracle, element by
element. Index sets, classification, counters, slot map, ring and gathered
bytes must be bit-exact; attention within max|gpu - oracle| <= 1e-3 * max|oracle|
per (step, unit, query row), the bound the decode path is specified to."""
import numpy as np
import pytest

from oracle.decode import decode_step
from synth import workloads as W
from tests.harness import Pair, check_step

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _need_gpu():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def run(wl, steps=None, rnds=None, mirror="host", check_every=1, attention_every=1,
        full_state=True, units=None, oracle_units=None, oracle_rnds=None, gpu_gen=False,
        side_stream=False):
    pair = Pair(wl, units=units, mirror=mirror, oracle_units=oracle_units, gpu_gen=gpu_gen)
    side = pair.torch.cuda.Stream() if side_stream is True else side_stream or None
    pair.check_slots = True
    steps = range(wl.steps) if steps is None else steps
    worst = 0.0
    for k, st in enumerate(steps):
        rnd = None if rnds is None else rnds[k]
        ornd = None if oracle_rnds is None else oracle_rnds[k]
        att = (k % attention_every) == 0 or k == len(steps) - 1
        g, o = pair.step(st, rnd=rnd, attention=att or side is not None, oracle_rnd=ornd, side=side)
        if (k % check_every) == 0 or k == len(steps) - 1:
            worst = max(worst, check_step(pair, g, o, attention=att or side is not None,
                                          full_state=full_state, rows=side != "fused"))
        assert pair.g.check() == 0, f"device error word {pair.g.check():#x}"
    return pair, worst


def test_config0_tiny_smoke_all_steps():
    pair, worst = run(W.WORKLOADS[0])
    assert worst < 1.0


SMALL = [
    # R=4 verify rows with duplicates, evictions every step, 4 appends per step
    dict(L0=1500, S=64, R=4, A=4, K=128, H=64, warm="last_s", mode="mtp", steps=20),
    # one query row, heavy eviction from an empty cache
    dict(L0=700, S=16, R=1, A=1, K=64, H=16, warm="empty", steps=24),
    # history shorter than K: -1 padding, then it grows past K
    dict(L0=100, S=32, R=2, A=3, K=128, H=32, warm="empty", steps=16),
    # ragged score tiles and cluster ranges, 48 heads, ragged attention clusters
    dict(L0=3 * 512 + 37, S=256, R=1, A=1, K=200, H=48, warm="last_s", steps=6),
    dict(L0=9000, S=300, R=3, A=2, K=1000, H=64, warm="last_s", mode="mtp", steps=4),
    # K = 1 and tiny history
    dict(L0=5, S=4, R=1, A=1, K=1, H=16, warm="empty", steps=70),
    # cluster sizes that are not powers of two before padding: 3 -> 4, 5 -> 8,
    # 12 -> 16 CTAs (the padding CTAs hold no rows)
    dict(L0=2500, S=512, R=1, A=1, K=300, H=16, warm="last_s", steps=4),
    dict(L0=3000, S=700, R=2, A=2, K=640, H=32, warm="empty", steps=3),
    dict(L0=5000, S=2048, R=1, A=1, K=1500, H=64, warm="last_s", steps=3),
]


@pytest.mark.parametrize("cfg", SMALL, ids=[f"L{c['L0']}_S{c['S']}_R{c['R']}_K{c['K']}" for c in SMALL])
def test_small_variants(cfg):
    base = W.WORKLOADS[0]
    wl = base.with_(name="variant", **cfg)
    run(wl)


def test_empty_history_then_growth():
    wl = W.WORKLOADS[0].with_(name="empty", L0=0, S=8, K=16, H=16, steps=80)
    run(wl)


def test_repeated_round_visibility():
    """Calls that repeat a round number: slots filled earlier in the same round
    are RAM (not HOT) and are not evicted in that round."""
    wl = W.WORKLOADS[0].with_(name="rep", L0=800, S=32, K=48, H=16, steps=10, warm="empty")
    rnds = [0, 0, 0, 1, 1, 2, 2, 2, 3, 3]
    run(wl, rnds=rnds)


def test_round_auto_matches_explicit_rounds():
    """hot_gather with DSA_ROUND_AUTO uses the call count as the round."""
    wl = W.WORKLOADS[0].with_(name="auto", L0=900, S=48, K=64, H=16, steps=12, warm="empty")
    run(wl, rnds=[-1] * 12, oracle_rnds=list(range(12)))


def test_append_concurrent_with_attention():
    """The append on a side stream, concurrent with the attention, across
    several 64-row write-backs: results identical to the serial order."""
    wl = W.WORKLOADS[0].with_(name="side", L0=700, S=48, K=64, H=16, steps=140, A=1, warm="last_s")
    run(wl, side_stream=True)


FUSED = [
    W.WORKLOADS[0],
    W.WORKLOADS[0].with_(name="fused-mtp", L0=1500, S=64, R=4, A=4, K=128, H=64, warm="last_s", mode="mtp",
                         steps=20),
    W.WORKLOADS[0].with_(name="fused-ragged", L0=3 * 512 + 37, S=256, K=200, H=48, warm="last_s", steps=6),
    W.WORKLOADS[0].with_(name="fused-evict", L0=700, S=16, K=64, H=16, warm="empty", steps=70),
    W.WORKLOADS[0].with_(name="fused-pad3", L0=2500, S=512, K=300, H=16, warm="last_s", steps=4),
]


def test_two_session_groups_on_two_streams():
    """Two groups of sessions, each with its own DecodePath over its units
    (UnitSet.subset) and its own stream, the groups' scorings alternating
    through events as in the bench's group schedule: within a step one group's
    gather copy, attention and append run beside the other group's scoring.
    After every step every unit matches the oracle (selection, classes,
    counters, gathered rows, cache state, attention)."""
    import torch
    from decode_attention_dsa_gb300.step import DecodePath
    from oracle.decode import decode_step
    wl = W.WORKLOADS[0].with_(name="groups", sessions=2, layers=2, L0=3000, S=256, K=256, H=16, steps=6,
                              warm="last_s")
    pair = Pair(wl)
    pair.check_slots = True
    abi = pair.abi
    ranges = [(0, 2), (2, 4)]
    paths = [DecodePath(pair.g.subset(lo, hi), wl.R, wl.K, wl.H, wl.A, wl.scale()) for lo, hi in ranges]
    streams = [torch.cuda.Stream() for _ in ranges]
    assigned = [torch.cuda.Event() for _ in ranges]
    for st in streams:
        st.wait_stream(torch.cuda.current_stream())
    for step in range(wl.steps):
        per, t = pair.inputs(step)
        for st in streams:
            st.wait_stream(torch.cuda.current_stream())     # the step's inputs
        for g, ((lo, hi), p, st) in enumerate(zip(ranges, paths, streams)):
            u = p.u
            with torch.cuda.stream(st):
                if step > 0 or g > 0:
                    st.wait_event(assigned[1 - g])
                p.score_topk(t["q_idx"][lo:hi], t["w"][lo:hi], st)
                abi.hot_gather_assign(u.units, u.U, p.R, p.K, step, p.topk, p.cls, p.counters, p.ws_gather,
                                      p.ws_gather_bytes, u.dev_err, st)
                assigned[g].record(st)
                abi.hot_gather_copy(u.units, u.U, p.R, p.K, p.topk, p.cls, p.rows, p.ws_gather,
                                    p.ws_gather_bytes, u.dev_err, st)
                p.attend(t["q_lat"][lo:hi], t["q_rope"][lo:hi], st)
                p.append(t["new_rows"][lo:hi], t["new_keys"][lo:hi], st)
        torch.cuda.synchronize()
        cat = lambda name: np.concatenate([getattr(p, name).cpu().numpy() for p in paths])
        g = dict(topk=cat("topk"), cls=cat("cls"), counters=cat("counters"), out=cat("out"), lse=cat("lse"),
                 rows=cat("rows"))
        pair.last_inputs = per
        ores = {}
        for i, u in enumerate(pair.uidx):
            x = per[i]
            ores[u] = decode_step(pair.o[u], step, wl.K, wl.scale(), x.q_idx, x.w, x.q_lat, x.q_rope,
                                  x.new_rows, x.new_keys, attention=True)
        check_step(pair, g, ores)
        assert pair.g.check() == 0


@pytest.mark.parametrize("fused", [False, True], ids=["split", "fused"])
def test_scoring_on_sm_partition_beside_the_other_group(fused):
    """The partition schedule: two session groups; the GPU split into two SM
    partitions; every scoring (dsa_score) on the first partition's stream, the
    groups' scorings alternating there; each group's selection, gather
    (split, or fused into the attention), attention and append on its own
    stream of the second partition; the order kept by dsa_stream_wait_stream.
    After every step every unit matches the oracle."""
    import torch
    from decode_attention_dsa_gb300.step import DecodePath
    from oracle.decode import decode_step
    wl = W.WORKLOADS[0].with_(name="partition", sessions=2, layers=2, L0=3000, S=256, K=256, H=16, steps=6,
                              warm="last_s")
    pair = Pair(wl)
    pair.check_slots = True
    abi = pair.abi
    first, second = abi.dsa_partition_split(64)
    ranges = [(0, 2), (2, 4)]
    paths = [DecodePath(pair.g.subset(lo, hi), wl.R, wl.K, wl.H, wl.A, wl.scale()) for lo, hi in ranges]
    try:
        assert abi.dsa_partition_sms(first) >= 64 and abi.dsa_partition_sms(second) >= 8
        pstream = abi.dsa_partition_stream(first)
        streams = [abi.dsa_partition_stream(second) for _ in ranges]
        if fused:
            for p in paths:
                p.prepare_fused()
            torch.cuda.synchronize()
        for step in range(wl.steps):
            per, t = pair.inputs(step)
            cur = torch.cuda.current_stream()
            for st in streams:
                abi.dsa_stream_wait_stream(st, cur)     # the step's inputs
            for g, ((lo, hi), p, st) in enumerate(zip(ranges, paths, streams)):
                u = p.u
                abi.dsa_stream_wait_stream(pstream, st)
                p.score(t["q_idx"][lo:hi], t["w"][lo:hi], pstream)
                abi.dsa_stream_wait_stream(st, pstream)
                p.select(st)
                if fused:
                    p.gather_attend(step, t["q_lat"][lo:hi], t["q_rope"][lo:hi], st)
                else:
                    abi.hot_gather_assign(u.units, u.U, p.R, p.K, step, p.topk, p.cls, p.counters,
                                          p.ws_gather, p.ws_gather_bytes, u.dev_err, st)
                    abi.hot_gather_copy(u.units, u.U, p.R, p.K, p.topk, p.cls, p.rows, p.ws_gather,
                                        p.ws_gather_bytes, u.dev_err, st)
                    p.attend(t["q_lat"][lo:hi], t["q_rope"][lo:hi], st)
                p.append(t["new_rows"][lo:hi], t["new_keys"][lo:hi], st)
            for st in streams:
                abi.dsa_stream_wait_stream(cur, st)
            torch.cuda.synchronize()
            cat = lambda name: np.concatenate([getattr(p, name).cpu().numpy() for p in paths])
            g = dict(topk=cat("topk"), cls=cat("cls"), counters=cat("counters"), out=cat("out"),
                     lse=cat("lse"), rows=cat("rows"))
            pair.last_inputs = per
            ores = {}
            for i, u in enumerate(pair.uidx):
                x = per[i]
                ores[u] = decode_step(pair.o[u], step, wl.K, wl.scale(), x.q_idx, x.w, x.q_lat, x.q_rope,
                                      x.new_rows, x.new_keys, attention=True)
            check_step(pair, g, ores, rows=not fused)
            assert pair.g.check() == 0
    finally:
        abi.dsa_partition_destroy(first)
        abi.dsa_partition_destroy(second)


@pytest.mark.parametrize("wl", FUSED, ids=[w.name[:12] for w in FUSED])
def test_fused_gather_attention(wl):
    """hot_gather_attn: same classification, state, slot bytes and attention
    as hot_gather + mla_decode_attn (compared with the oracle)."""
    run(wl, side_stream="fused")


@pytest.mark.slow
def test_fused_config1_full_size_first_steps():
    run(W.WORKLOADS[1], steps=range(66), side_stream="fused", attention_every=1)


def test_resident_mirror_same_results():
    wl = W.WORKLOADS[0].with_(name="resident", steps=4)
    run(wl, mirror="device")


def test_flush_makes_ram_complete():
    wl = W.WORKLOADS[0].with_(name="flush", L0=300, S=16, K=32, H=16, steps=30, A=3)
    pair, _ = run(wl)
    p = pair
    p.abi.kv_flush(p.g.units, p.g.U, p.g.dev_err)
    p.torch.cuda.synchronize()
    oc = p.o[0].cache
    oc.flush()
    st = p.g.state[0].cpu().numpy()
    assert st[0] == st[1] == oc.length == oc.rows_in_ram
    got = p.g.get_mirror_rows(0, 0, oc.length)
    want = oc.mirror.rows(np.arange(oc.length))
    assert np.array_equal(got, want)


def test_selection_reuse_across_layers():
    """Layers 1 and 3 reuse the selections of layers 0 and 2 (same session);
    every layer keeps its own cache."""
    wl = W.WORKLOADS[0].with_(name="reuse", sessions=2, layers=4, L0=2000, S=128, K=128, H=16, steps=8,
                              warm="last_s", reuse_every=2)
    run(wl)


@pytest.mark.slow
def test_selection_reuse_config1_first_steps():
    run(W.WORKLOADS[1].with_(reuse_every=2), steps=range(8), attention_every=4)


def test_export_restore_round_trip():
    """Flush, export to the host, rebuild a fresh unit set from the snapshot and
    continue: every later step matches the oracle, which flushed at the same
    point (the export/restore barrier: RAM rows equal logical rows first)."""
    from decode_attention_dsa_gb300.step import DecodePath
    from decode_attention_dsa_gb300.units import UnitSet
    wl = W.WORKLOADS[0].with_(name="restore", L0=900, S=64, K=96, H=16, steps=50, A=1, warm="last_s")
    pair = Pair(wl)
    pair.check_slots = True
    for st in range(25):
        g, o = pair.step(st)
        check_step(pair, g, o)
    pair.abi.kv_flush(pair.g.units, pair.g.U, pair.g.dev_err)
    pair.o[0].cache.flush()
    snap = pair.g.export_state()
    st0 = snap["snapshot"][:64].view(np.int64)
    assert st0[0] == st0[1] == pair.o[0].cache.length, "flush must bring RAM rows to the logical rows"
    fresh = UnitSet(pair.g.U, wl.S, wl.lmax, mirror="host")
    fresh.import_state(snap)
    pair.g.close()
    pair.g = fresh
    pair.p = DecodePath(fresh, wl.R, wl.K, wl.H, wl.A, wl.scale())
    for st in range(25, 50):
        g, o = pair.step(st)
        check_step(pair, g, o)
    assert fresh.check() == 0


CLOCK = [
    # every warm slot referenced, few misses: long first turns of the hand
    dict(L0=1500, S=512, R=1, A=1, K=256, H=16, warm="last_s", steps=12),
    # MTP rows with duplicates and evictions from an empty cache
    dict(L0=1500, S=64, R=4, A=4, K=128, H=64, warm="last_s", mode="mtp", steps=16),
    dict(L0=700, S=16, R=1, A=1, K=64, H=16, warm="empty", steps=40),
    # more misses than eligible slots (the second turn runs out)
    dict(L0=900, S=8, R=2, A=1, K=48, H=16, warm="last_s", steps=10),
]


@pytest.mark.parametrize("cfg", CLOCK, ids=[f"clock_L{c['L0']}_S{c['S']}_R{c['R']}" for c in CLOCK])
def test_clock_policy_matches_oracle(cfg):
    """Clock replacement with reference bits: classification, victims, bits,
    hand and slot bytes identical to the oracle's walk of the hand."""
    wl = W.WORKLOADS[0].with_(name="clock", policy="clock", **cfg)
    run(wl)


def test_clock_policy_fused_path():
    wl = W.WORKLOADS[0].with_(name="clock-fused", policy="clock", L0=1500, S=64, R=4, A=4, K=128, H=64,
                              warm="last_s", mode="mtp", steps=10)
    run(wl, side_stream="fused")


@pytest.mark.slow
def test_config3_clock_policy_first_steps():
    """The cache-stress workload (full window, every slot referenced, 1% of
    the Top-2048 outside the hot set) under the clock policy."""
    wl = W.WORKLOADS[3].with_(policy="clock")
    run(wl, steps=range(6), attention_every=3)


def test_decreasing_round_is_refused_on_the_device():
    """A gather whose round is below the unit's previous round would break the
    visibility rule: the unit is left unchanged and DSA_DEVERR_ROUND is set."""
    wl = W.WORKLOADS[0].with_(name="round", L0=600, S=32, K=48, H=16, steps=4, warm="empty")
    pair, _ = run(wl, rnds=[0, 1, 2, 3])
    torch, abi, g, p = pair.torch, pair.abi, pair.g, pair.p
    before = {k: getattr(g, k).clone() for k in ("slot_pos", "pos_slot", "fill_round", "state", "slots")}
    p.gather(2)
    torch.cuda.synchronize()
    assert g.check() == abi.DEVERR_ROUND
    assert (p.cls == abi.CLS_PAD).all() and (p.counters == 0).all() and (p.rows == 0).all()
    for k, v in before.items():
        assert torch.equal(getattr(g, k), v), f"{k} changed"
    g.dev_err.zero_()
    p.gather(3)                      # the same round again is allowed
    torch.cuda.synchronize()
    assert g.check() == 0


def test_bounded_wait_gives_up_with_an_error_status():
    """The bounded wait every kernel uses: a phase that nothing completes makes
    it give up after its limit and report DSA_DEVERR_TIMEOUT; the context stays
    usable (a completed phase right after reports nothing)."""
    import torch
    from decode_attention_dsa_gb300 import abi
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    abi.dsa_wait_selftest(1 << 16, False, err)
    torch.cuda.synchronize()
    assert int(err.item()) == abi.DEVERR_TIMEOUT
    assert abi.dsa_check(int(err.item())) == abi.DSA_ERR_DEVICE_CHECK
    err.zero_()
    abi.dsa_wait_selftest(1 << 16, True, err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0


@pytest.mark.parametrize("policy", ["ring", "clock"])
def test_snapshot_restore_is_bit_exact(policy):
    """dsa_export after kv_flush, dsa_restore into a fresh unit set whose
    mirror holds the same rows: every array of the cache state comes back
    bit for bit, and slot bytes are re-read from the mirror."""
    from decode_attention_dsa_gb300.units import UnitSet
    wl = W.WORKLOADS[0].with_(name="snap", sessions=2, layers=2, L0=1200, S=96, K=64, H=16, steps=70, A=1,
                              warm="last_s", policy=policy)
    pair, _ = run(wl, steps=range(37), check_every=12, attention_every=12)
    g, abi, torch = pair.g, pair.abi, pair.torch
    before = {f: getattr(g, f).clone() for f in ("slot_pos", "fill_round", "ref", "ring", "state", "keys")}
    abi.kv_flush(g.units, g.U, g.dev_err)
    snap = g.export_state()
    assert g.check() == 0
    fresh = UnitSet(g.U, wl.S, wl.lmax, mirror="host", policy=policy)
    fresh.import_state(snap)
    assert fresh.check() == 0
    st = g.state.cpu().numpy()
    for f in ("slot_pos", "fill_round", "ref", "ring"):
        assert torch.equal(getattr(fresh, f), getattr(g, f)), f
    assert torch.equal(fresh.state, g.state)
    assert torch.equal(g.slot_pos, before["slot_pos"]) and torch.equal(g.ring, before["ring"])
    for u in range(g.U):
        L = int(st[u, 0])
        assert st[u, 1] == L
        assert torch.equal(fresh.keys[u, :L], g.keys[u, :L])
        assert torch.equal(fresh.pos_slot[u], g.pos_slot[u])
        occ = g.slot_pos[u] >= 0
        assert torch.equal(fresh.slots[u][occ], g.slots[u][occ])
    assert (fresh.pin_epoch == -1).all()
    fresh.close()


def test_export_of_an_unflushed_unit_is_refused():
    wl = W.WORKLOADS[0].with_(name="noflush", L0=300, S=16, K=32, H=16, steps=5, A=1)
    pair, _ = run(wl)
    g, abi, torch = pair.g, pair.abi, pair.torch
    stride = g.snapshot_stride()
    snap = torch.zeros(stride, dtype=torch.uint8, device="cuda")
    abi.dsa_export(g.units, g.U, snap, stride, g.S, g.lmax, g.dev_err)
    torch.cuda.synchronize()
    assert g.check() == abi.DEVERR_STATE
    assert int(snap.sum().item()) == 0


def test_full_history_restore_for_append_prefill():
    """kv_restore_full: the dense history [0, LEN) of every unit, rows below
    RAM from the mirror and the rest from the ring, equals the oracle's rows."""
    wl = W.WORKLOADS[0].with_(name="prefill", sessions=3, layers=1, L0=2000, S=64, K=64, H=16, steps=50, A=3)
    pair, _ = run(wl, steps=range(50), check_every=25, attention_every=25)
    g, abi, torch = pair.g, pair.abi, pair.torch
    dst = torch.full((g.U, wl.lmax, 656), 0xAB, dtype=torch.uint8, device="cuda")
    abi.kv_restore_full(g.units, g.U, dst, wl.lmax, g.dev_err)
    torch.cuda.synchronize()
    got = dst.cpu().numpy()
    for u in range(g.U):
        oc = pair.o[u].cache
        L = oc.length
        assert oc.rows_in_ram < L, "the case must leave rows in the ring"
        want = np.concatenate([oc.mirror.rows(np.arange(oc.rows_in_ram)),
                               np.stack([oc.ring[p % 64] for p in range(oc.rows_in_ram, L)])])
        assert np.array_equal(got[u, :L], want), f"unit {u}"
        assert (got[u, L:] == 0xAB).all()


def test_append_beyond_capacity_sets_device_flag():
    wl = W.WORKLOADS[0].with_(name="cap", L0=10, S=4, K=4, H=16, steps=1, A=1)
    pair = Pair(wl)
    torch, abi = pair.torch, pair.abi
    rows = torch.zeros((1, 1, 656), dtype=torch.uint8, device="cuda")
    keys = torch.zeros((1, 1, 64), dtype=torch.int16, device="cuda")
    abi.kv_append_writeback(pair.g.units, 1, 1, rows, keys, pair.g.dev_err)   # fills lmax
    torch.cuda.synchronize()
    assert pair.g.check() == 0
    abi.kv_append_writeback(pair.g.units, 1, 1, rows, keys, pair.g.dev_err)   # one too many
    torch.cuda.synchronize()
    assert pair.g.check() & abi.DEVERR_CAPACITY
    assert pair.g.state[0, 0].item() == wl.lmax


@pytest.mark.slow
def test_config1_full_size_first_steps():
    """50K single stream, 4 layers, full sizes and the bench's launch shapes;
    66 steps cross the first 64-row write-back."""
    wl = W.WORKLOADS[1]
    _, worst = run(wl, steps=range(66), attention_every=11)
    assert worst < 1.0


@pytest.mark.slow
def test_config2_mtp_verify_first_steps():
    """34 steps of 4 appended rows cross two 64-row write-backs (steps 15 and
    31) with steps after each."""
    wl = W.WORKLOADS[2]
    _, worst = run(wl, steps=range(34), attention_every=8)
    assert worst < 1.0


@pytest.mark.slow
def test_config3_cache_stress_first_steps():
    wl = W.WORKLOADS[3]
    pair, worst = run(wl, steps=range(6), attention_every=3)
    c = pair.p.counters.cpu().numpy()[0]
    assert c[2] / wl.K < 0.05          # phase 1: about 1% of the Top-K misses


@pytest.mark.slow
def test_config3_cache_stress_high_miss_phase():
    """The second phase of the cache-stress workload (about 30% of the
    Top-2048 outside the hot set: eviction scans and miss bandwidth), started
    at step 0 from the full warm cache, compared for 10 steps."""
    wl = W.WORKLOADS[3].with_(phases=((0, 88), (1024, 36)))
    pair, worst = run(wl, steps=range(10), attention_every=3)
    c = pair.p.counters.cpu().numpy()[0]
    assert 0.15 < c[2] / wl.K < 0.5
    assert worst < 1.0


@pytest.mark.slow
def test_config4_capacity_batch_other_units_more_steps():
    """Units 5 (session 2, layer 1) and 22 (session 11, layer 0) of the
    capacity batch, 9 steps, in the full 32-unit launch."""
    import torch
    free, _ = torch.cuda.mem_get_info()
    if free < 12 * 2**30:
        pytest.skip("not enough device memory")
    wl = W.WORKLOADS[4].with_(steps=9)
    run(wl, steps=range(9), oracle_units=[5, 22], gpu_gen=True, attention_every=4)


@pytest.mark.slow
def test_config4_capacity_batch_sampled_units():
    """16 sessions x 2 layers x 1,048,576-position histories in one launch per
    call (32 units, 20.5 GiB pinned host mirror); units 0 and 31 are compared
    with the oracle element by element on the first steps."""
    import torch
    free, _ = torch.cuda.mem_get_info()
    if free < 12 * 2**30:
        pytest.skip("not enough device memory")
    wl = W.WORKLOADS[4].with_(steps=3)
    run(wl, steps=range(3), oracle_units=[0, 31], gpu_gen=True, attention_every=2)


def _run_pipelined(wl, nsteps, units=None, oracle_units=None, gpu_gen=False):
    """Enqueue nsteps pipelined steps back to back (no synchronisation in
    between, so each step's copy and attention overlap the next step's score),
    keeping each step's outputs on the stream that orders them, then compare
    every step with the oracle."""
    pair = Pair(wl, units=units, oracle_units=oracle_units, gpu_gen=gpu_gen)
    torch, p = pair.torch, pair.p
    p.enable_pipeline()
    U, R, K = pair.g.U, wl.R, wl.K
    keep = {k: [] for k in ("topk", "cls", "ctr", "out", "rows")}
    inputs = []
    for st in range(nsteps):
        per, t = pair.inputs(st)
        inputs.append((per, t))
        p.step_pipelined(st, t["q_idx"], t["w"], t["q_lat"], t["q_rope"], t["new_rows"], t["new_keys"])
        keep["cls"].append(p.cls.clone())              # main stream: before the next assign
        keep["ctr"].append(p.counters.clone())
        with torch.cuda.stream(p.side):                # side stream: after this step's attention
            keep["out"].append(p.out.clone())
            keep["topk"].append(p.cur_topk.clone())
            keep["rows"].append(p.rows.clone())
    p.join()
    torch.cuda.synchronize()
    assert pair.g.check() == 0, f"device error word {pair.g.check():#x}"
    worst = 0.0
    for st in range(nsteps):
        per, _ = inputs[st]
        pair.last_inputs = per
        g = {k: v[st].cpu().numpy() for k, v in keep.items()}
        g["counters"] = g.pop("ctr")
        g["lse"] = None
        for i, u in enumerate(pair.uidx):
            if u not in pair.o:
                continue
            x = per[i]
            o = decode_step(pair.o[u], st, wl.K, wl.scale(), x.q_idx, x.w, x.q_lat, x.q_rope, x.new_rows, x.new_keys)
            assert np.array_equal(g["topk"][i], o["topk"]), f"step {st} unit {u}: Top-K"
            assert np.array_equal(g["cls"][i], o["cls"]), f"step {st} unit {u}: classification"
            assert np.array_equal(g["counters"][i], o["counters"]), f"step {st} unit {u}: counters"
            assert np.array_equal(g["rows"][i], o["rows"]), f"step {st} unit {u}: gathered rows"
            for r in range(R):
                ref = o["out"][r]
                err = np.abs(g["out"][i, r].astype(np.float64) - ref).max()
                assert err <= 1e-3 * np.abs(ref).max(), f"step {st} unit {u} row {r}: attention"
                worst = max(worst, err / (1e-3 * np.abs(ref).max()))
    # the final cache state
    for i, u in enumerate(pair.uidx):
        if u not in pair.o:
            continue
        oc, s = pair.o[u].cache, pair.state(i)
        assert np.array_equal(s["slot_pos"], oc.slot_pos) and s["st"][2] == oc.hand
        assert s["st"][0] == oc.length and s["st"][1] == oc.rows_in_ram
    return worst


def test_pipelined_steps_match_oracle():
    """Steps whose gather copy and attention run on a side stream while the
    next step scores: results identical to the serial path's (the oracle)."""
    wl = W.WORKLOADS[0].with_(name="pipe", sessions=2, layers=1, L0=3000, S=128, K=256, H=64, steps=70, A=1,
                              warm="last_s")
    from decode_attention_dsa_gb300 import abi  # noqa: F401
    assert _run_pipelined(wl, 70) < 1.0


def test_pipelined_steps_mtp_rows():
    wl = W.WORKLOADS[0].with_(name="pipe-mtp", L0=1500, S=64, R=4, A=1, K=128, H=16, warm="last_s", mode="mtp",
                              steps=24)
    _run_pipelined(wl, 24)


@pytest.mark.slow
def test_config4_capacity_batch_pipelined_steps():
    """The bench's launch shape of the capacity batch (pipelined steps),
    units 0 and 31 against the oracle for 6 steps."""
    import torch
    free, _ = torch.cuda.mem_get_info()
    if free < 12 * 2**30:
        pytest.skip("not enough device memory")
    wl = W.WORKLOADS[4].with_(steps=6)
    _run_pipelined(wl, 6, oracle_units=[0, 31], gpu_gen=True)
