"""One decode step of one unit, composed from the oracle's steps.

Order within a step (the pages' per-layer path, [P3] "第三次决策" diagram):
score all history positions and keep the Top-K ([P3] "起点"), hot gather
(``hotcache``), dequantise and attend (``attention``), then append the step's
new rows to the recent ring with batched write-back (``hotcache`` C7).

Pinned by ``tests/test_oracle_decode.py``: a row appended in step t is not a
candidate before step t + 1, the gather sees the state of the step start (not
the step's own append or write-back), attention reads the gathered rows, and
the selection-reuse branch does not score.
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np

from .attention import mla_decode_attention
from .hotcache import PAD, UnitCache
from .indexer import score_topk


@dataclass
class OracleUnit:
    cache: UnitCache
    keys: np.ndarray          # bf16 bits [lmax, 64]; rows >= length are unused

    @classmethod
    def create(cls, S, lmax, L0, keys_initial, mirror_initial, warm, policy="ring"):
        keys = np.zeros((lmax, keys_initial.shape[1]), dtype=np.uint16)
        keys[:L0] = keys_initial[:L0]
        return cls(UnitCache(S, lmax, L0, mirror_initial, warm, policy=policy), keys)


def decode_step(unit: OracleUnit, rnd: int, K: int, scale: float, q_idx, w,
                q_lat, q_rope, new_rows, new_keys, attention: bool = True, topk=None):
    """Run one step; returns a dict with scores, topk, cls, rows, counters, out, lse.

    ``topk`` given: the unit reuses that selection (made by an earlier layer of
    the same session, [P3] section "起点": some later layers reuse the
    selection while every layer keeps its own KV) and does not score.
    """
    L = unit.cache.length
    if topk is None:
        scores, topk = score_topk(unit.keys[:L], q_idx, w, K)
    else:
        scores = None
    cls, rows, counters = unit.cache.gather(rnd, topk)
    res = dict(L=L, scores=scores, topk=topk, cls=cls, rows=rows, counters=counters)
    if attention:
        outs, lses = [], []
        for r in range(topk.shape[0]):
            o, s = mla_decode_attention(q_lat[r], q_rope[r], rows[r], cls[r] != PAD, scale)
            outs.append(o)
            lses.append(s)
        res["out"] = np.stack(outs)
        res["lse"] = np.stack(lses)
    unit.cache.append(new_rows, unit.keys, new_keys)
    return res
