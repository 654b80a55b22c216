"""The score kernel's barrier protocol, simulated on the CPU.

The warp-specialised score kernel runs three roles per CTA that meet only at
mbarriers: the producer copies tile j into stage j % NST (waiting for the
stage's previous use to be read), the MMA warp multiplies it into accumulator
j % 2 (waiting for the keys and for the accumulator to be read), and the
epilogue reads the accumulator. Each wait is a parity wait on a barrier
phase. This restates the waits the kernel issues, with the same parities,
drives the roles in random interleavings with copies and products that
complete after random delays, and checks that no wait ever passes before the
event it stands for has happened (no phase aliasing), that the roles never
deadlock, and that a unit change rewrites the query operand only once every
product that read it is done.
"""
import random

import pytest


class Barrier:
    """An mbarrier: `count` arrivals complete a phase; try_wait.parity(P)
    passes when the phase of parity P has completed (the current phase has
    the other parity)."""

    def __init__(self, count):
        self.count, self.pending, self.done = count, count, 0

    def arrive(self):
        self.pending -= 1
        assert self.pending >= 0
        if self.pending == 0:
            self.done += 1
            self.pending = self.count

    def passes(self, parity):
        return (self.done & 1) != parity


def simulate(nst, units, seed, wrong_epilogue_parity=False):
    """units: tiles per unit of one CTA's range, in order. With
    `wrong_epilogue_parity` the epilogue waits on parity j & 1 instead of
    (j >> 1) & 1 (a plausible slip the checks must catch)."""
    rng = random.Random(seed)
    tiles = [u for u, n in enumerate(units) for _ in range(n)]
    n = len(tiles)
    full = [Barrier(1) for _ in range(nst)]
    empty = [Barrier(1) for _ in range(nst)]
    acc_full = [Barrier(1) for _ in range(2)]
    acc_empty = [Barrier(4) for _ in range(2)]     # one arrival per epilogue warp
    landed, mma_done, reads = [False] * n, [False] * n, [0] * n
    pending = []                                   # (time, action) of async completions
    clock = [0]
    last_mma = [0]

    def later(action, in_order=False):
        t = clock[0] + rng.randint(1, 6)
        if in_order:
            # one thread's tensor-core products complete in issue order, and a
            # commit arrives once every product issued before it is done
            t = max(t, last_mma[0])
            last_mma[0] = t
        pending.append((t, len(pending), action))

    def producer():
        s, use_par = 0, 0
        for j in range(n):
            if j >= nst:
                while not empty[s].passes(use_par ^ 1):
                    yield
                # the stage's previous tile has been multiplied
                assert mma_done[j - nst]
            def land(j=j, s=s):
                landed[j] = True
                full[s].arrive()
            later(land)
            yield
            s += 1
            if s == nst:
                s, use_par = 0, use_par ^ 1

    def mma():
        s, use_par, unit = 0, 0, -1
        for j in range(n):
            if tiles[j] != unit:
                if j > 0:
                    while not acc_full[(j - 1) & 1].passes(((j - 1) >> 1) & 1):
                        yield
                    # every product issued so far is done: the other operand
                    # buffer may be rewritten
                    assert all(mma_done[:j])
                unit = tiles[j]
            while not full[s].passes(use_par):
                yield
            assert landed[j]
            acc = j & 1
            if j >= 2:
                while not acc_empty[acc].passes(((j >> 1) - 1) & 1):
                    yield
                assert reads[j - 2] == 4     # all four warps read the accumulator's previous tile
            def complete(j=j, s=s, acc=acc):
                mma_done[j] = True
                empty[s].arrive()
                acc_full[acc].arrive()
            later(complete, in_order=True)
            yield
            s += 1
            if s == nst:
                s, use_par = 0, use_par ^ 1

    def epilogue(w):
        for j in range(n):
            acc = j & 1
            parity = (j & 1) if wrong_epilogue_parity else ((j >> 1) & 1)
            while not acc_full[acc].passes(parity):
                yield
            assert mma_done[j]
            yield                            # this warp reads the accumulator
            reads[j] += 1
            acc_empty[acc].arrive()
            yield

    roles = [producer(), mma()] + [epilogue(w) for w in range(4)]
    alive = list(roles)
    steps = 0
    while alive or pending:
        steps += 1
        assert steps < 20000, "deadlock"
        clock[0] += 1
        due = [p for p in pending if p[0] <= clock[0]]
        for p in due:
            pending.remove(p)
        rng.shuffle(due)
        # same-time products keep their issue order (a commit never overtakes an earlier one)
        mmas = sorted((p for p in due if p[2].__name__ == "complete"), key=lambda p: p[1])
        others = [p for p in due if p[2].__name__ != "complete"]
        for _, _, action in others + mmas:
            action()
        order = list(alive)
        rng.shuffle(order)
        for r in order:
            if rng.random() < 0.7:
                try:
                    next(r)
                except StopIteration:
                    alive.remove(r)
    assert all(landed) and all(mma_done) and all(r == 4 for r in reads)


@pytest.mark.parametrize("nst", [2, 3, 4, 6])
@pytest.mark.parametrize("units", [[1], [2], [3], [7], [40], [1, 1, 1], [5, 1, 9, 2], [13, 13]])
def test_roles_never_pass_a_wait_early_nor_deadlock(nst, units):
    for seed in range(20):
        simulate(nst, units, seed)


def test_the_epilogue_warps_may_drift_apart():
    """The epilogue warps wait independently; a slow warp holds the
    accumulator (the MMA two tiles on waits for all four), never a wrong one."""
    for seed in range(50):
        simulate(2, [64], 1000 + seed)


def test_a_wrong_parity_is_caught():
    """The simulation is a check, not a formality: the epilogue waiting on the
    wrong phase parity either passes a wait early or deadlocks."""
    caught = 0
    for seed in range(20):
        try:
            simulate(2, [16], 2000 + seed, wrong_epilogue_parity=True)
        except AssertionError:
            caught += 1
    assert caught == 20
