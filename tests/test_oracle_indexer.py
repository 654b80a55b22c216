"""Pins for oracle.indexer: a hand-computed example, Python-integer brute force,
and the Top-K invariants."""
import itertools

import numpy as np
import pytest

from oracle import indexer
from synth.rng import f32_to_bf16_bits


def _bits(a):
    return f32_to_bf16_bits(np.asarray(a, dtype=np.float32))


def test_worked_example(golden):
    lines = golden("topk_worked_example.txt")
    d = {}
    tk = {}
    for ln in lines:
        k, *rest = ln.split()
        if k == "topk":
            tk[int(rest[0])] = [int(x) for x in rest[1].split(",")]
        else:
            d[k] = rest
    keys = np.array([[int(x) for x in v.split(",")] for v in d["keys"]], dtype=np.float32)
    q = np.array([[int(x) for x in v.split(",")] for v in d["q"]], dtype=np.float32)[None]
    w = np.array([[float(x) for x in d["w"]]], dtype=np.float32)
    s = indexer.dsa_scores(_bits(keys), _bits(q), w)
    assert s[0].tolist() == [float(x) for x in d["scores"]]
    for K, want in tk.items():
        assert indexer.topk_positions(s[0], K).tolist() == want


def _brute(keys, q, w, K):
    """Python integers, nested loops, a full sort of (-score, position) tuples."""
    L = len(keys)
    res = []
    for r in range(len(q)):
        sc = []
        for s in range(L):
            tot = 0
            for h in range(len(q[r])):
                dot = sum(int(a) * int(b) for a, b in zip(q[r][h], keys[s]))
                tot += int(w[r][h]) * max(0, dot)
            sc.append((-tot, s))
        sc.sort()
        sel = sorted(p for _, p in sc[:K])
        res.append(sel + [-1] * (K - len(sel)))
    return res


@pytest.mark.parametrize("seed", range(12))
def test_brute_force_small(seed):
    rng = np.random.default_rng(seed)
    L = int(rng.integers(1, 200))
    d = int(rng.integers(1, 9))
    HI = int(rng.integers(1, 5))
    R = int(rng.integers(1, 4))
    K = int(rng.integers(1, 64))
    lim = int(rng.integers(1, 5))          # small value range forces ties
    keys = rng.integers(-lim, lim + 1, size=(L, d))
    q = rng.integers(-lim, lim + 1, size=(R, HI, d))
    w = rng.integers(1, 5, size=(R, HI))
    s, sel = indexer.score_topk(_bits(keys), _bits(q), w.astype(np.float32), K)
    assert sel.tolist() == _brute(keys.tolist(), q.tolist(), w.tolist(), K)


def test_invariants_random():
    rng = np.random.default_rng(1)
    for _ in range(20):
        L = int(rng.integers(50, 3000))
        K = int(rng.integers(1, 300))
        keys = rng.integers(-4, 5, size=(L, 64))
        q = rng.integers(-4, 5, size=(1, 8, 64))
        w = rng.integers(1, 5, size=(1, 8)).astype(np.float32)
        s, sel = indexer.score_topk(_bits(keys), _bits(q), w, K)
        sel = sel[0]
        n = min(K, L)
        assert (sel[n:] == -1).all()
        chosen = sel[:n]
        assert (np.diff(chosen) > 0).all()
        mask = np.zeros(L, bool)
        mask[chosen] = True
        if n < L:
            lo = s[0][mask].min()
            assert lo >= s[0][~mask].max()
            # at the boundary score every excluded position is above every included one
            inc = np.nonzero(mask & (s[0] == lo))[0]
            exc = np.nonzero(~mask & (s[0] == lo))[0]
            if len(exc):
                assert inc.max() < exc.min()


def test_all_equal_scores_take_lowest_positions():
    keys = np.zeros((100, 64))
    q = np.ones((1, 8, 64))
    s, sel = indexer.score_topk(_bits(keys), _bits(q), np.ones((1, 8), np.float32), 10)
    assert sel[0].tolist() == list(range(10))


def test_empty_history():
    s, sel = indexer.score_topk(np.zeros((0, 64), np.uint16), _bits(np.ones((1, 8, 64))),
                                np.ones((1, 8), np.float32), 4)
    assert sel.tolist() == [[-1, -1, -1, -1]]
