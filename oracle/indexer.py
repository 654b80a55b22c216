"""DSA indexer scores and Top-K selection (oracle).

[P3] section "起点" (starting point): the DSA indexer picks the Top-2048
positions from the history and MLA attention consumes the selected KV; section
"第一次决策" (first decision): the selection stays on the GPU as the exact DSA
path with a BF16 query, because a quantised query changed the cutoff set.
[ALG] table of attention schemes: DSA uses a learned indexer and each query
selects only its Top-K tokens.

Readings where the pages are silent:

* Score (the DSA "lightning indexer" form, a ReLU-gated sum over indexer heads):
  ``I[r][s] = sum_h w[r][h] * max(0, sum_d q[r][h][d] * k[s][d])``; keys are
  shared by the heads, queries and weights belong to each query row.
* Candidates are positions ``[0, L)`` with ``L`` the history length at the
  start of the step (rows appended in the step are not candidates).
* The K largest scores win; equal scores are broken by the lower position.
  The selected positions are returned in ascending order, padded with -1 when
  ``L < K``.
"""
from __future__ import annotations

import numpy as np


def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    b = np.ascontiguousarray(bits, dtype=np.uint16).astype(np.uint32)
    return (b << np.uint32(16)).view(np.float32).astype(np.float64)


def dsa_scores(keys_bits: np.ndarray, q_bits: np.ndarray, w: np.ndarray) -> np.ndarray:
    """Indexer scores ``[R, L]`` in float64.

    keys_bits: bf16 bits ``[L, d]``; q_bits: bf16 bits ``[R, H_I, d]``;
    w: float32 ``[R, H_I]``.
    """
    k = bf16_to_f64(keys_bits)
    q = bf16_to_f64(q_bits)
    R, HI, d = q.shape
    L = k.shape[0]
    dots = (q.reshape(R * HI, d) @ k.T).reshape(R, HI, L)
    return np.einsum("rh,rhl->rl", np.asarray(w, dtype=np.float64), np.maximum(dots, 0.0))


def topk_positions(scores_row: np.ndarray, K: int) -> np.ndarray:
    """The K best positions of one row, ascending, -1 padded (int32 ``[K]``).

    Full sort by (score descending, position ascending), keep the first
    ``min(K, L)``, then sort the kept positions.
    """
    L = scores_row.shape[0]
    pos = np.arange(L, dtype=np.int64)
    order = np.lexsort((pos, -scores_row))
    n = min(K, L)
    out = np.full(K, -1, dtype=np.int32)
    out[:n] = np.sort(order[:n])
    return out


def score_topk(keys_bits, q_bits, w, K: int) -> tuple[np.ndarray, np.ndarray]:
    """Scores ``[R, L]`` and selections ``[R, K]`` for one unit."""
    s = dsa_scores(keys_bits, q_bits, w)
    return s, np.stack([topk_positions(s[r], K) for r in range(s.shape[0])])
