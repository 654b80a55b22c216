"""Pins for the clock-with-reference-bits policy of oracle.hotcache (C8): a
hand trace, an independent closed form of the hand's walk on many random
states, the special case that reduces to ring replacement, and the stress
shape of the pages (full window, every bit set, few misses)."""
import numpy as np
import pytest

from oracle.hotcache import HOT, PAD, RAM, RING, UnitCache

CLS = {"H": HOT, "G": RING, "M": RAM, "P": PAD}


def _ints(s):
    return [int(x) for x in s.split(",")]


def test_clock_hand_trace(golden):
    lines = golden("clock_trace.txt")
    cfg = dict(kv.split("=") for kv in lines[0].split()[1:])
    S, L0 = int(cfg["S"]), int(cfg["L0"])
    uc = UnitCache(S, L0 + 8, L0, np.zeros((L0, 656), np.uint8), cfg["warm"], policy="clock")
    for ln in lines[1:]:
        lhs, rhs = ln[len("call "):].split("=>")
        rnd, tk = lhs.split(";")
        cls, _, ctr = uc.gather(int(rnd), np.array([_ints(tk.strip())]))
        c, sp, ref, fr, hand, sweep, cnt = [x.strip() for x in rhs.split(";")]
        assert cls[0].tolist() == [CLS[x] for x in c.split(",")], ln
        assert uc.slot_pos.tolist() == _ints(sp), ln
        assert uc.ref.tolist() == _ints(ref), ln
        assert uc.fill_round.tolist() == _ints(fr), ln
        assert uc.hand == int(hand) and uc.last_sweep == int(sweep), ln
        assert ctr.tolist() == _ints(cnt), ln
        uc.check_invariants()


def _closed_form(ref, fill_round, pinned, hand, r, m):
    """Victims, bits after the walk (before the fills) and sweep length,
    stated without walking: the eligible slots with a clear bit in cyclic
    order from the hand come first, then those with a set bit (cleared on the
    first turn); bits are cleared up to the last victim of the first turn,
    or all of them if a second turn was needed."""
    S = len(ref)
    order = [(hand + t) % S for t in range(S)]
    elig = [s for s in order if s not in pinned and fill_round[s] < r]
    a = [s for s in elig if ref[s] == 0]
    b = [s for s in elig if ref[s] == 1]
    ref2 = np.array(ref)
    if m == 0:
        return [], ref2, 0
    if m <= len(a):
        v = a[:m]
        stop = order.index(v[-1])
        for s in b:
            if order.index(s) < stop:
                ref2[s] = 0
        return v, ref2, stop + 1
    for s in b:
        ref2[s] = 0
    v = a + b[:m - len(a)]
    sweep = S + order.index(v[-1]) + 1 if m - len(a) <= len(b) and len(v) == m else 2 * S
    if len(v) < m:
        sweep = 2 * S
    return v, ref2, sweep


@pytest.mark.parametrize("seed", range(300))
def test_walk_equals_closed_form(seed):
    rng = np.random.default_rng(seed)
    S = int(rng.choice([1, 2, 3, 5, 8, 17, 64]))
    uc = UnitCache(S, 4, 0, np.zeros((0, 656), np.uint8), "empty", policy="clock")
    uc.ref[:] = rng.integers(0, 2, S)
    r = 5
    uc.fill_round[:] = np.where(rng.random(S) < 0.15, r, rng.integers(-1, r, S))
    pinned = set(np.nonzero(rng.random(S) < 0.2)[0].tolist())
    uc.hand = int(rng.integers(0, S))
    m = int(rng.integers(0, S + 3))
    ref0, fr0, hand0 = uc.ref.copy(), uc.fill_round.copy(), uc.hand
    v = uc._clock_victims(pinned, r, m)
    want_v, want_ref, want_sweep = _closed_form(ref0, fr0, pinned, hand0, r, m)
    assert v == want_v
    assert uc.ref.tolist() == want_ref.tolist()
    assert uc.last_sweep == want_sweep


def _rows(L):
    rows = np.zeros((L, 656), np.uint8)
    rows[:, :8] = np.arange(L, dtype="<i8").view(np.uint8).reshape(L, 8)
    return rows


def test_clear_bits_give_the_ring_choice():
    """With every bit clear the hand takes the first eligible slots in
    cyclic order, exactly as ring replacement does (one call)."""
    rng = np.random.default_rng(7)
    for _ in range(50):
        S, L0 = int(rng.integers(2, 40)), int(rng.integers(40, 200))
        ring = UnitCache(S, L0 + 4, L0, _rows(L0), "last_s", policy="ring")
        clock = UnitCache(S, L0 + 4, L0, _rows(L0), "last_s", policy="clock")
        clock.ref[:] = 0
        h = int(rng.integers(0, S))
        ring.hand = clock.hand = h
        K = int(rng.integers(1, 30))
        topk = np.sort(rng.choice(L0, size=min(K, L0), replace=False))[None]
        a = ring.gather(0, topk)
        b = clock.gather(0, topk)
        assert np.array_equal(a[0], b[0]) and np.array_equal(a[2], b[2])
        assert np.array_equal(ring.slot_pos, clock.slot_pos) and ring.hand == clock.hand


def test_stress_full_window_every_bit_set():
    """The pages' stress shape: the window is full, every bit is set and a
    few positions miss. The hand clears the whole cache on its first turn
    and takes its victims on the second: S + m visits."""
    S, L0, m = 1024, 5000, 10
    uc = UnitCache(S, L0 + 4, L0, _rows(L0), "last_s", policy="clock")
    assert uc.ref.all()
    hits = np.arange(L0 - S + m, L0)                 # slots m..S-1 hit (pinned, bits stay set)
    misses = np.arange(m) * 7                        # positions outside the window
    topk = np.sort(np.concatenate([hits, misses]))[None]
    cls, _, ctr = uc.gather(0, topk)
    assert ctr.tolist() == [S - m, 0, m, m]
    victims = np.arange(m)                           # the only unpinned slots
    assert uc.last_sweep == S + m
    assert uc.slot_pos[victims].tolist() == misses.tolist()
    assert uc.ref.all()                              # hits keep their bits, fills set theirs
    # the same shape under ring replacement needs no sweep beyond the victims
    ring = UnitCache(S, L0 + 4, L0, _rows(L0), "last_s", policy="ring")
    ring.gather(0, topk)
    assert ring.slot_pos[victims].tolist() == misses.tolist()
