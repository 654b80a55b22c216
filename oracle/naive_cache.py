"""A second, deliberately naive hot-cache simulator (oracle pin only).

Same rules as ``oracle.hotcache`` (see its docstring) written differently, so a
bookkeeping mistake in one is unlikely to be repeated in the other: there is no
position->slot index (every lookup is a linear scan over the slots), misses are
collected as a plain list and sorted, and the replacement hand walks slot by
slot for each miss, skipping pinned slots and slots filled in the current round,
and never examines more than S slots in one call. Only positions are tracked
(no bytes).
"""
from __future__ import annotations

HOT, RING, RAM, PAD = 0, 1, 2, 3


class NaiveCache:
    def __init__(self, S: int, L0: int, warm: str):
        self.S = S
        self.owner = [None] * S       # position held by each slot
        self.filled = [-1] * S        # round of the last fill
        self.hand = 0
        self.rows_in_ram = L0
        self.length = L0
        if warm == "last_s":
            n = min(S, L0)
            for i in range(n):
                self.owner[i] = L0 - n + i

    def _find(self, p):
        for s in range(self.S):
            if self.owner[s] == p:
                return s
        return None

    def gather(self, r, topk):
        R = len(topk)
        K = len(topk[0])
        cls = [[PAD] * K for _ in range(R)]
        pinned = [False] * self.S
        for i in range(R):
            for j in range(K):
                p = int(topk[i][j])
                if p < 0:
                    continue
                if p >= self.rows_in_ram:
                    cls[i][j] = RING
                    continue
                s = self._find(p)
                if s is not None and self.filled[s] < r:
                    cls[i][j] = HOT
                    pinned[s] = True
                else:
                    cls[i][j] = RAM
        misses = []
        for i in range(R):
            for j in range(K):
                p = int(topk[i][j])
                if cls[i][j] == RAM and self._find(p) is None and p not in misses:
                    misses.append(p)
        misses.sort()
        start = self.hand
        examined = 0
        last = None
        filled = 0
        for p in misses:
            got = None
            while examined < self.S:
                s = (start + examined) % self.S
                examined += 1
                if not pinned[s] and self.filled[s] < r:
                    got = s
                    break
            if got is None:
                break
            self.owner[got] = p
            self.filled[got] = r
            last = got
            filled += 1
        if last is not None:
            self.hand = (last + 1) % self.S
        return cls, filled

    def append(self, n):
        for _ in range(n):
            self.length += 1
            if self.length - self.rows_in_ram == 64:
                self.rows_in_ram = self.length

    def flush(self):
        self.rows_in_ram = self.length
