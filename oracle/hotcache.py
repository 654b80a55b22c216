"""GPU-managed hot cache, recent ring and batched write-back (oracle).

One ``UnitCache`` is the cache state of one (session, layer) unit. Sources:

* [P3] section "起点" (starting point): the hot cache is not a sliding window;
  old positions stay in RAM and stay selectable, a miss reads them from RAM.
* [P3] section "第三次决策：让 GPU 直接管理热缓存" (third decision: the GPU
  manages the hot cache): the selection stays on the GPU, the GPU looks up hot
  slots, a hit reads VRAM, a miss reads the registered RAM mirror, and the
  result is the compact selected set attention uses; new KV goes to a GPU
  recent ring and is written back to the RAM history in batches.
* [P3] section "第二次决策" (second decision): write-back in 64-row batches.
* [P3] section "GPU 管缓存也会犯错：跨 block 可见性与置换长扫描" (GPU-managed
  caching errs too: cross-block visibility and long replacement sweeps):
  slots filled in a round are hit sources only from the next round, duplicate
  misses in the same round read RAM, slots in use this round are pinned, rows
  not yet written back are protected by the recent ring, and replacement is a
  ring that skips the pinned slots.
* [P3] section "容量优化必须通过会话生命周期" (capacity work must survive the
  session lifecycle): before export, flush the log and make the RAM row count
  reach the logical row count.

Rules as implemented (round ``r`` = the ``round`` argument of a gather call):

C1 classify, with the state as it is when the call starts: a position
   ``p >= rows_in_ram`` is RING (read ring row ``p % 64``); else if
   ``pos_slot[p] = s >= 0`` and ``fill_round[s] < r`` it is HOT (read slot
   ``s``); else it is RAM (read ``mirror[p]``). -1 entries are PAD.
C2 every slot classified HOT by any query row of the call is pinned.
C3 the insertion list M is the ascending list of distinct RAM positions that
   hold no slot; every occurrence of a RAM position, duplicates included,
   reads RAM in this round.
C4 a fill made in round r sets ``fill_round = r``, so it is never HOT before
   round r + 1.
C5 eligible slots E are the slots that are neither pinned nor filled in round
   r, in cyclic order starting at ``hand``. The i-th position of M takes the
   i-th slot of E: the old position of that slot loses its mapping, the slot
   gets the new position, ``fill_round = r`` and the mirror row's bytes.
   Afterwards ``hand`` = (last slot assigned + 1) mod S. Positions of M beyond
   ``len(E)`` are not inserted (they are still served from RAM).
C6 warm start: EMPTY (all slots free) or LAST_S (slot i holds position
   ``L0 - n + i`` for ``n = min(S, L0)``, ``fill_round = -1``), hand 0.
C7 append: the row at position ``p = len`` goes to ring row ``p % 64`` and its
   indexer key to ``keys[p]``; ``len += 1``; when ``len - rows_in_ram == 64``
   the 64 ring rows of positions ``[rows_in_ram, rows_in_ram + 64)`` are copied
   to the mirror and ``rows_in_ram += 64``. Appended rows are not inserted into
   the hot cache. ``flush`` copies the partial batch and sets
   ``rows_in_ram = len``.

The ascending assignment order of C5, the hand update and the insertion filter
of C3 are readings of "ring replacement skipping pinned slots".

C8 clock with reference bits (the policy the pages replaced by the ring; a
   unit built with ``policy="clock"``). Section "GPU 管缓存也会犯错" describes
   it only by its cost: with a full window, every reference bit set and 1%
   misses, the few missing blocks had to sweep far. Readings: each slot has a
   reference bit; a HOT hit sets it; warm slots start with it set, empty ones
   clear. To find victims for M (same list as C3), the hand walks the slots
   cyclically from ``hand``: a slot pinned in this call, filled in this round
   or already taken in this walk is passed over; a slot whose bit is set gets
   it cleared and is passed over; a slot whose bit is clear is the next
   victim. The walk stops when every position of M has a victim or after two
   turns (after one turn every eligible bit is clear). A fill sets the bit
   (the row was just referenced). ``hand`` = last victim + 1; ``last_sweep``
   is the number of slots the hand visited.
"""
from __future__ import annotations

import numpy as np

from .q8g64 import ROW_BYTES

HOT, RING, RAM, PAD = 0, 1, 2, 3
RING_ROWS = 64


class MirrorStore:
    """Host RAM mirror of one unit: initial history plus written-back rows.

    ``initial`` is either a uint8 array ``[L0, 656]`` or a function
    ``positions -> uint8 [n, 656]`` for the history present at start.
    """

    def __init__(self, initial, L0: int):
        self._initial = initial
        self.L0 = L0
        self._written: dict[int, np.ndarray] = {}

    def rows(self, positions) -> np.ndarray:
        positions = np.asarray(positions, dtype=np.int64).reshape(-1)
        out = np.empty((positions.size, ROW_BYTES), dtype=np.uint8)
        base = [i for i, p in enumerate(positions) if int(p) not in self._written]
        for i, p in enumerate(positions):
            if int(p) in self._written:
                out[i] = self._written[int(p)]
        if base:
            bp = positions[base]
            if np.any(bp >= self.L0) or np.any(bp < 0):
                raise IndexError("mirror read of a position never written to RAM")
            out[base] = (self._initial[bp] if isinstance(self._initial, np.ndarray)
                         else self._initial(bp))
        return out

    def write(self, p: int, row: np.ndarray) -> None:
        self._written[int(p)] = np.array(row, dtype=np.uint8, copy=True)


class UnitCache:
    def __init__(self, S: int, lmax: int, L0: int, mirror_initial, warm: str, policy: str = "ring"):
        if policy not in ("ring", "clock"):
            raise ValueError(policy)
        self.policy = policy
        self.S = S
        self.lmax = lmax
        self.slot_pos = np.full(S, -1, dtype=np.int64)
        self.pos_slot = np.full(lmax, -1, dtype=np.int64)
        self.fill_round = np.full(S, -1, dtype=np.int64)
        self.hand = 0
        self.slots = np.zeros((S, ROW_BYTES), dtype=np.uint8)
        self.ring = np.zeros((RING_ROWS, ROW_BYTES), dtype=np.uint8)
        self.mirror = MirrorStore(mirror_initial, L0)
        self.rows_in_ram = L0
        self.length = L0
        self.writebacks = 0
        self.ref = np.zeros(S, dtype=np.uint8)      # C8 reference bits
        self.last_sweep = 0
        if warm == "last_s":
            n = min(S, L0)
            pos = np.arange(L0 - n, L0, dtype=np.int64)
            self.slot_pos[:n] = pos
            self.pos_slot[pos] = np.arange(n)
            self.slots[:n] = self.mirror.rows(pos)
            self.ref[:n] = 1
        elif warm != "empty":
            raise ValueError(warm)

    # -- C1
    def classify(self, p: int, r: int) -> int:
        if p < 0:
            return PAD
        if p >= self.rows_in_ram:
            return RING
        s = self.pos_slot[p]
        if s >= 0 and self.fill_round[s] < r:
            return HOT
        return RAM

    def gather(self, r: int, topk: np.ndarray):
        """One gather call for round ``r`` over ``topk [R, K]``.

        Returns ``(cls [R, K] uint8, rows [R, K, 656] uint8, counters [4])``
        where counters are (HOT, RING, RAM, slots filled).
        """
        topk = np.asarray(topk)
        R, K = topk.shape
        cls = np.full((R, K), PAD, dtype=np.uint8)
        rows = np.zeros((R, K, ROW_BYTES), dtype=np.uint8)
        pinned = set()
        for i in range(R):
            for j in range(K):
                p = int(topk[i, j])
                c = self.classify(p, r)
                cls[i, j] = c
                if c == HOT:
                    pinned.add(int(self.pos_slot[p]))
                    self.ref[self.pos_slot[p]] = 1
        # rows as read at call start (pinned HOT slots and the ring do not change below)
        for i in range(R):
            for j in range(K):
                p = int(topk[i, j])
                c = cls[i, j]
                if c == HOT:
                    rows[i, j] = self.slots[self.pos_slot[p]]
                elif c == RING:
                    rows[i, j] = self.ring[p % RING_ROWS]
                elif c == RAM:
                    rows[i, j] = self.mirror.rows([p])[0]
        # C3
        M = sorted({int(topk[i, j]) for i in range(R) for j in range(K)
                    if cls[i, j] == RAM and self.pos_slot[int(topk[i, j])] < 0})
        if self.policy == "ring":
            # C5
            E = []
            for t in range(self.S):
                if len(E) == len(M):
                    break
                s = (self.hand + t) % self.S
                if s not in pinned and self.fill_round[s] < r:
                    E.append(s)
        else:
            E = self._clock_victims(pinned, r, len(M))
        n = min(len(M), len(E))
        for i in range(n):
            s, p = E[i], M[i]
            q = self.slot_pos[s]
            if q >= 0:
                self.pos_slot[q] = -1
            self.slot_pos[s] = p
            self.pos_slot[p] = s
            self.fill_round[s] = r
            self.slots[s] = self.mirror.rows([p])[0]
            self.ref[s] = 1
        if n > 0:
            self.hand = (E[n - 1] + 1) % self.S
        counters = np.array([(cls == HOT).sum(), (cls == RING).sum(), (cls == RAM).sum(), n],
                            dtype=np.int64)
        return cls, rows, counters

    # -- C8
    def _clock_victims(self, pinned, r: int, m: int) -> list:
        """The clock hand's walk for m victims (see C8); one slot per visit."""
        E, taken = [], set()
        s, visits = self.hand, 0
        while len(E) < m and visits < 2 * self.S:
            visits += 1
            if s not in pinned and s not in taken and self.fill_round[s] < r:
                if self.ref[s]:
                    self.ref[s] = 0
                else:
                    E.append(s)
                    taken.add(s)
            s = (s + 1) % self.S
        self.last_sweep = visits
        return E

    # -- C7
    def append(self, new_rows: np.ndarray, keys=None, new_keys=None) -> None:
        for a in range(new_rows.shape[0]):
            p = self.length
            if p >= self.lmax:
                raise IndexError("append beyond capacity")
            self.ring[p % RING_ROWS] = new_rows[a]
            if keys is not None:
                keys[p] = new_keys[a]
            self.length += 1
            if self.length - self.rows_in_ram == RING_ROWS:
                self._write_back(self.length)

    def _write_back(self, upto: int) -> None:
        for q in range(self.rows_in_ram, upto):
            self.mirror.write(q, self.ring[q % RING_ROWS])
        self.rows_in_ram = upto
        self.writebacks += 1

    def flush(self) -> None:
        if self.length > self.rows_in_ram:
            self._write_back(self.length)

    # -- invariants used by the tests
    def check_invariants(self) -> None:
        occ = self.slot_pos >= 0
        assert np.all(self.pos_slot[self.slot_pos[occ]] == np.nonzero(occ)[0])
        mapped = np.nonzero(self.pos_slot >= 0)[0]
        assert np.all(self.slot_pos[self.pos_slot[mapped]] == mapped)
        assert len(np.unique(self.slot_pos[occ])) == occ.sum()
        assert 0 <= self.hand < self.S
        assert 0 <= self.length - self.rows_in_ram < RING_ROWS
