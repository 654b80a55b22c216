"""Pins for oracle.hotcache: a hand trace, a second naive simulator on many
random tiny cases, per-round invariants and closed-form special cases."""
import numpy as np
import pytest

from oracle.hotcache import HOT, PAD, RAM, RING, UnitCache
from oracle.naive_cache import NaiveCache

CLS = {"H": HOT, "G": RING, "M": RAM, "P": PAD}


def _mirror(L0):
    rows = np.zeros((L0, 656), dtype=np.uint8)
    rows[:, :8] = np.arange(L0, dtype="<i8").view(np.uint8).reshape(L0, 8)
    return rows


def _row_pos(row):
    return int(row[:8].view("<i8")[0])


def test_hand_trace(golden):
    lines = golden("hotcache_trace.txt")
    cfg = dict(kv.split("=") for kv in lines[0].split()[1:])
    S, L0 = int(cfg["S"]), int(cfg["L0"])
    uc = UnitCache(S, L0 + 16, L0, _mirror(L0), cfg["warm"])
    for ln in lines[1:]:
        if ln.startswith("append"):
            n = int(ln.split()[1])
            rows = np.zeros((n, 656), np.uint8)
            uc.append(rows)
            continue
        lhs, rhs = ln[len("call "):].split("=>")
        rnd, tk = lhs.split(";")
        topk = np.array([[int(x) for x in r.split(",")] for r in tk.strip().split("|")])
        c_want, sp, fr, hand, ctr = [x.strip() for x in rhs.split(";")]
        cls, rows, counters = uc.gather(int(rnd), topk)
        want = [[CLS[x] for x in r.split(",")] for r in c_want.split("|")]
        assert cls.tolist() == want, ln
        assert uc.slot_pos.tolist() == [int(x) for x in sp.split(",")], ln
        assert uc.fill_round.tolist() == [int(x) for x in fr.split(",")], ln
        assert uc.hand == int(hand), ln
        assert counters.tolist() == [int(x) for x in ctr.split(",")], ln
        uc.check_invariants()


def _random_topk(rng, R, K, L, dup_frac):
    base = np.sort(rng.choice(L, size=min(K, L), replace=False))
    rows = []
    for r in range(R):
        if r == 0:
            sel = base
        else:
            keep = base[rng.random(base.size) < dup_frac]
            extra = rng.choice(L, size=min(K, L), replace=False)
            sel = np.unique(np.concatenate([keep, extra]))[:min(K, L)]
            sel = np.sort(rng.choice(sel, size=min(K, L, sel.size), replace=False))
        t = np.full(K, -1)
        t[:sel.size] = sel
        rows.append(t)
    return np.stack(rows)


@pytest.mark.parametrize("seed", range(40))
def test_against_naive_simulator(seed):
    rng = np.random.default_rng(1000 + seed)
    S = int(rng.choice([4, 8, 16, 64]))
    L0 = int(rng.integers(8, 512))
    R = int(rng.choice([1, 4]))
    K = int(rng.integers(1, min(48, L0) + 1))
    warm = str(rng.choice(["empty", "last_s"]))
    rounds = int(rng.integers(5, 25))
    lmax = L0 + rounds * 4 + 8
    uc = UnitCache(S, lmax, L0, _mirror(L0), warm)
    nc = NaiveCache(S, L0, warm)
    rnd = 0
    for t in range(rounds):
        L = uc.length
        topk = _random_topk(rng, R, K, L, dup_frac=0.75)
        if rng.random() < 0.2 and t > 0:
            rnd_call = rnd          # a repeated round number
        else:
            rnd += 1
            rnd_call = rnd
        pinned_before = uc.slot_pos.copy()
        cls, rows, counters = uc.gather(rnd_call, topk)
        ncls, nfilled = nc.gather(rnd_call, topk.tolist())
        assert cls.tolist() == ncls
        assert counters[3] == nfilled
        assert uc.slot_pos.tolist() == [(-1 if o is None else o) for o in nc.owner]
        assert uc.fill_round.tolist() == nc.filled
        assert uc.hand == nc.hand
        uc.check_invariants()
        # pinned (HOT) slots did not change
        for i in range(R):
            for j in range(K):
                if cls[i, j] == HOT:
                    s = uc.pos_slot[topk[i, j]]
                    assert pinned_before[s] == topk[i, j]
        # no position is HOT in the round its slot was filled
        for i in range(R):
            for j in range(K):
                if cls[i, j] == HOT:
                    assert uc.fill_round[uc.pos_slot[topk[i, j]]] < rnd_call
        # duplicates of a RAM position are RAM in every row; RING never RAM
        for p in set(topk[cls == RAM].tolist()):
            assert (cls[topk == p] == RAM).all()
            assert p < uc.rows_in_ram or p >= L
        assert (topk[cls == RING] >= uc.rows_in_ram).all()
        # bytes: every emitted row is the row of its position; slots hold their rows
        for i in range(R):
            for j in range(K):
                if cls[i, j] != PAD:
                    assert _row_pos(rows[i, j]) == topk[i, j] or cls[i, j] == RING
        for s in range(S):
            if uc.slot_pos[s] >= 0:
                assert _row_pos(uc.slots[s]) == uc.slot_pos[s]
        assert counters[:3].sum() + (cls == PAD).sum() == R * K
        # append like decode does
        a = int(rng.integers(0, 5))
        if uc.length + a <= lmax:
            new = np.zeros((a, 656), np.uint8)
            for k in range(a):
                new[k, :8] = np.array([uc.length + k], "<i8").view(np.uint8)
            uc.append(new)
            nc.append(a)
            assert uc.rows_in_ram == nc.rows_in_ram


def test_closed_form_no_eviction_when_cache_covers_history():
    """S >= L, EMPTY start, R = 1, increasing rounds: the misses of a round are
    exactly the selected positions never selected before."""
    rng = np.random.default_rng(7)
    L0 = 300
    uc = UnitCache(512, L0, L0, _mirror(L0), "empty")
    seen = set()
    for r in range(30):
        sel = np.sort(rng.choice(L0, size=40, replace=False))
        cls, _, counters = uc.gather(r, sel[None])
        want = [RAM if int(p) not in seen else HOT for p in sel]
        assert cls[0].tolist() == want
        seen.update(int(p) for p in sel)
        assert counters[3] == want.count(RAM)
        assert uc.hand == len(seen) % 512


def test_no_misses_leaves_map_unchanged():
    L0 = 100
    uc = UnitCache(64, L0, L0, _mirror(L0), "last_s")
    before = (uc.slot_pos.copy(), uc.fill_round.copy(), uc.hand)
    cls, _, counters = uc.gather(3, np.arange(36, 100)[None])
    assert (cls == HOT).all() and counters[3] == 0
    assert (uc.slot_pos == before[0]).all() and (uc.fill_round == before[1]).all()
    assert uc.hand == before[2]


def test_all_misses_without_pins_take_consecutive_slots():
    L0 = 1000
    uc = UnitCache(64, L0, L0, _mirror(L0), "last_s")
    uc.hand = 10
    sel = np.arange(0, 40)               # none of these is hot (hot: 936..999)
    uc.gather(0, sel[None])
    assert uc.slot_pos[10:50].tolist() == list(range(40))
    assert uc.hand == 50


def test_excess_misses_are_not_inserted():
    L0 = 200
    uc = UnitCache(8, L0, L0, _mirror(L0), "last_s")   # slots hold 192..199
    sel = np.concatenate([np.arange(192, 198), np.arange(0, 10)])  # 6 hot, 10 misses
    cls, _, counters = uc.gather(0, np.sort(sel)[None])
    assert counters.tolist() == [6, 0, 10, 2]
    assert sorted(uc.slot_pos.tolist()) == [0, 1, 192, 193, 194, 195, 196, 197]


def test_write_back_batches_and_flush():
    L0 = 10
    uc = UnitCache(4, 10 + 200, L0, _mirror(L0), "empty")
    for k in range(130):
        row = np.zeros((1, 656), np.uint8)
        row[0, :8] = np.array([L0 + k], "<i8").view(np.uint8)
        uc.append(row)
    assert uc.writebacks == 2 and uc.rows_in_ram == L0 + 128 and uc.length == L0 + 130
    assert _row_pos(uc.mirror.rows([L0 + 127])[0]) == L0 + 127
    uc.flush()
    assert uc.rows_in_ram == uc.length
    assert _row_pos(uc.mirror.rows([L0 + 129])[0]) == L0 + 129
    cls, rows, _ = uc.gather(0, np.array([[L0 + 129]]))
    assert cls[0, 0] == RAM and _row_pos(rows[0, 0]) == L0 + 129
