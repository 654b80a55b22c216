"""Pins for oracle.decode.decode_step, the composition of one decode step.

The pieces are pinned on their own (indexer, hot cache, attention); these
tests pin the ORDER in which a step uses them, on tiny hand-built units whose
expected results follow from the rules by hand:

* the Top-K candidates are the positions [0, L) with L the history length at
  the start of the step: a row appended by step t is never selected in step t,
  even with the largest score, and is selectable from step t + 1 ([P3] section
  "起点": the indexer selects from the history);
* the gather classifies with the cache state of the step start, before the
  step's own append (a write-back triggered by that append must not turn a
  RING position of this step into RAM);
* attention reads the rows the gather returned (a ring row selected with K = 1
  comes back exactly as its dequantised latent);
* the selection-reuse branch (``topk=`` given) does not score, and classifies
  and updates the cache exactly as a gather on that selection does.
"""
import numpy as np

from oracle.decode import OracleUnit, decode_step
from oracle.hotcache import HOT, PAD, RAM, RING, UnitCache
from oracle.q8g64 import dequant_latent
from synth.rng import f32_to_bf16_bits

SC = 1.0 / 24.0


def _key(v):
    """An indexer key whose first dimension is v, the rest 0 (bf16 bits)."""
    k = np.zeros(64, np.float32)
    k[0] = v
    return f32_to_bf16_bits(k)


def _row(tag):
    """A 656-byte row: latent[0] = tag (int8), every group scale 1.0 (fp16)."""
    r = np.zeros(656, np.uint8)
    r[0] = np.int8(tag).view(np.uint8)
    r[512:528] = np.full(8, 1.0, dtype="<f2").view(np.uint8)
    return r


def _unit(L0, S, lmax, warm="empty", key_of=lambda p: p % 4):
    keys = np.stack([_key(key_of(p)) for p in range(L0)])
    rows = np.stack([_row(p % 100) for p in range(L0)])
    return OracleUnit.create(S, lmax, L0, keys, rows, warm)


def _q():
    """One query row, indexer head 0 reads key dimension 0; w = (1, 0, ...)."""
    q = np.zeros((1, 8, 64), np.float32)
    q[0, 0, 0] = 1.0
    w = np.zeros((1, 8), np.float32)
    w[0, 0] = 1.0
    return f32_to_bf16_bits(q), w


def _attn_q(H=2):
    return np.zeros((1, H, 512), np.uint16), np.zeros((1, H, 64), np.uint16)


def test_row_appended_in_a_step_is_selected_only_from_the_next_step():
    L0 = 10
    u = _unit(L0, S=4, lmax=L0 + 4)
    q, w = _q()
    ql, qr = _attn_q()
    big = np.stack([_key(4.0)])            # larger than every history score (at most 3)
    r0 = decode_step(u, 0, 1, SC, q, w, ql, qr, np.stack([_row(77)]), big)
    assert r0["L"] == L0
    assert r0["scores"].shape == (1, L0)   # scored over [0, L) only
    # the best history score 3 is taken by positions 3 and 7: the lower wins
    assert r0["topk"].tolist() == [[3]]
    r1 = decode_step(u, 1, 1, SC, q, w, ql, qr, np.stack([_row(78)]), np.stack([_key(0.0)]))
    assert r1["L"] == L0 + 1
    assert r1["topk"].tolist() == [[L0]]   # the row appended by step 0 wins now
    assert r1["cls"].tolist() == [[RING]]  # not yet written back: served by the ring
    # K = 1: attention returns that ring row's dequantised latent exactly
    assert np.array_equal(r1["rows"][0, 0], _row(77))
    assert np.array_equal(r1["out"][0], np.repeat(dequant_latent(_row(77)[None]), 2, axis=0))
    assert u.cache.length == L0 + 2


def test_gather_uses_the_state_before_the_steps_own_append():
    L0 = 8
    u = _unit(L0, S=4, lmax=L0 + 80, key_of=lambda p: 0)
    q, w = _q()
    ql, qr = _attn_q()
    # step 0 appends 63 rows (positions 8..70, still in the ring); the key of
    # position 13 is the only positive one
    keys63 = np.stack([_key(5.0 if L0 + a == 13 else 0.0) for a in range(63)])
    rows63 = np.stack([_row(a) for a in range(63)])
    r0 = decode_step(u, 0, 1, SC, q, w, ql, qr, rows63, keys63)
    assert u.cache.length == L0 + 63 and u.cache.rows_in_ram == L0
    # all history scores are 0: position 0 wins the tie, misses and takes slot 0
    assert r0["topk"].tolist() == [[0]] and r0["cls"].tolist() == [[RAM]]
    assert u.cache.slot_pos.tolist() == [0, -1, -1, -1]
    # step 1 selects 13, then appends the 64th pending row, which triggers the
    # write-back of positions 8..71: the selection must still be RING
    r = decode_step(u, 1, 1, SC, q, w, ql, qr, np.stack([_row(99)]), np.stack([_key(0.0)]))
    assert r["topk"].tolist() == [[13]]
    assert r["cls"].tolist() == [[RING]]
    assert r["counters"].tolist() == [0, 1, 0, 0]
    assert np.array_equal(r["rows"][0, 0], _row(13 - L0))
    assert u.cache.rows_in_ram == L0 + 64 and u.cache.writebacks == 1
    assert u.cache.slot_pos.tolist() == [0, -1, -1, -1]  # a RING read fills no slot
    # one step later the same position is RAM (now in the mirror, no slot yet)
    r2 = decode_step(u, 2, 1, SC, q, w, ql, qr, np.stack([_row(98)]), np.stack([_key(0.0)]))
    assert r2["topk"].tolist() == [[13]]
    assert r2["cls"].tolist() == [[RAM]]
    assert u.cache.slot_pos.tolist() == [0, 13, -1, -1]


def test_reuse_branch_does_not_score_and_matches_a_plain_gather():
    L0, S, K = 40, 8, 6
    topk = np.array([[1, 5, 9, 33, 36, 39], [5, 9, 20, 33, -1, -1]])
    ql, qr = np.zeros((2, 2, 512), np.uint16), np.zeros((2, 2, 64), np.uint16)
    u = _unit(L0, S, L0 + 8, warm="last_s")
    ref = UnitCache(S, L0 + 8, L0, np.stack([_row(p % 100) for p in range(L0)]), "last_s")
    for rnd in range(3):
        new = np.stack([_row(50 + rnd)])
        # q_idx and w are None: the branch must not touch the indexer
        r = decode_step(u, rnd, K, SC, None, None, ql, qr, new, np.stack([_key(0.0)]), topk=topk)
        cls, rows, ctr = ref.gather(rnd, topk)
        ref.append(new)
        assert r["scores"] is None
        assert np.array_equal(r["topk"], topk)
        assert np.array_equal(r["cls"], cls) and np.array_equal(r["rows"], rows)
        assert np.array_equal(r["counters"], ctr)
        assert np.array_equal(u.cache.slot_pos, ref.slot_pos)
        assert np.array_equal(u.cache.fill_round, ref.fill_round) and u.cache.hand == ref.hand
    # round 0: warm slots hold 32..39, so 33, 36, 39 are HOT, the rest RAM; PAD stays PAD
    first = UnitCache(S, L0 + 8, L0, np.stack([_row(p % 100) for p in range(L0)]), "last_s")
    c0, _, _ = first.gather(0, topk)
    assert c0.tolist() == [[RAM, RAM, RAM, HOT, HOT, HOT], [RAM, RAM, RAM, HOT, PAD, PAD]]
