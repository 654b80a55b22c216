"""Counter-based SplitMix64 draws and value mappings (host side, numpy).

Draw ``i`` of the stream with key ``k`` is ``mix64(k + (i + 1) * GAMMA)``
(mod 2**64), where ``mix64`` is the SplitMix64 output finaliser. Each 64-bit
draw is split into four 16-bit *fields*, least significant first, so field
``f`` is bits ``16*(f % 4) .. 16*(f % 4) + 15`` of draw ``f // 4``.

Value mappings (all integer-exact, so that the numpy and CUDA generators agree
bit for bit):

* uniform integer in ``[lo, hi]``: ``lo + (field * (hi - lo + 1)) >> 16``.
* approximately standard normal: Irwin-Hall sum of 12 fields,
  ``z = (sum(field_i) + 6 - 6 * 65536) / 65536``; each uniform is
  ``(field + 1/2) / 65536`` so the sum has mean 6 and variance 1. ``z`` is an
  exact float32 (|numerator| < 2**20), rounded to bf16 by round-to-nearest-even.
"""
from __future__ import annotations

import numpy as np

MASK64 = (1 << 64) - 1
GAMMA = 0x9E3779B97F4A7C15
MIX_C1 = 0xBF58476D1CE4E5B9
MIX_C2 = 0x94D049BB133111EB
NORMAL_FIELDS = 12


def _mix64_int(z: int) -> int:
    z &= MASK64
    z = ((z ^ (z >> 30)) * MIX_C1) & MASK64
    z = ((z ^ (z >> 27)) * MIX_C2) & MASK64
    return z ^ (z >> 31)


def _mix64(z: np.ndarray) -> np.ndarray:
    z = z ^ (z >> np.uint64(30))
    z = z * np.uint64(MIX_C1)
    z = z ^ (z >> np.uint64(27))
    z = z * np.uint64(MIX_C2)
    return z ^ (z >> np.uint64(31))


def stream_key(*ids: int) -> int:
    """Fold a tuple of small non-negative integers into one 64-bit stream key."""
    k = 0x243F6A8885A308D3  # arbitrary fixed start value
    for i in ids:
        k = _mix64_int((k ^ (int(i) & MASK64)) + GAMMA)
    return k


def draws64(key: int, start: int, count: int) -> np.ndarray:
    """Draws ``start .. start+count-1`` of stream ``key`` as uint64."""
    with np.errstate(over="ignore"):
        idx = np.arange(count, dtype=np.uint64) + np.uint64(start + 1)
        z = idx * np.uint64(GAMMA) + np.uint64(key)
        return _mix64(z)


def fields16(key: int, start_field: int, count: int) -> np.ndarray:
    """16-bit fields ``start_field .. start_field+count-1`` (uint32 array)."""
    if count <= 0:
        return np.zeros(0, dtype=np.uint32)
    d0 = start_field // 4
    d1 = (start_field + count + 3) // 4
    d = draws64(key, d0, d1 - d0)
    f = np.empty((d1 - d0) * 4, dtype=np.uint32)
    for s in range(4):
        f[s::4] = ((d >> np.uint64(16 * s)) & np.uint64(0xFFFF)).astype(np.uint32)
    off = start_field - 4 * d0
    return f[off:off + count]


def fields16_items(key: int, items: np.ndarray, per_item: int) -> np.ndarray:
    """Fields of arbitrary items: item ``i`` owns fields ``[i*per_item, (i+1)*per_item)``.

    Returns uint32 ``[len(items), per_item]``.
    """
    items = np.asarray(items, dtype=np.int64).reshape(-1)
    n = items.size
    if n == 0:
        return np.zeros((0, per_item), dtype=np.uint32)
    if per_item % 4 == 0:
        nd = per_item // 4
        didx = (items[:, None] * nd + np.arange(nd, dtype=np.int64)[None, :]).astype(np.uint64)
        with np.errstate(over="ignore"):
            d = _mix64((didx + np.uint64(1)) * np.uint64(GAMMA) + np.uint64(key))
        f = np.empty((n, nd, 4), dtype=np.uint32)
        for s in range(4):
            f[:, :, s] = ((d >> np.uint64(16 * s)) & np.uint64(0xFFFF)).astype(np.uint32)
        return f.reshape(n, per_item)
    fidx = items[:, None] * per_item + np.arange(per_item, dtype=np.int64)[None, :]
    didx = (fidx // 4).astype(np.uint64)
    sub = (fidx % 4).astype(np.uint64)
    with np.errstate(over="ignore"):
        d = _mix64((didx + np.uint64(1)) * np.uint64(GAMMA) + np.uint64(key))
    return ((d >> (sub * np.uint64(16))) & np.uint64(0xFFFF)).astype(np.uint32)


def uniform_int_fields(f: np.ndarray, lo: int, hi: int) -> np.ndarray:
    """Map 16-bit fields to integers in ``[lo, hi]`` (int64)."""
    n = hi - lo + 1
    return lo + ((f.astype(np.int64) * n) >> 16)


def normal_fields_f32(f: np.ndarray) -> np.ndarray:
    """Map fields ``[..., 12*m]`` to ``m`` Irwin-Hall normals per row (exact float32)."""
    m = f.shape[-1] // NORMAL_FIELDS
    g = f.reshape(f.shape[:-1] + (m, NORMAL_FIELDS)).astype(np.int64)
    num = g.sum(axis=-1) + 6 - 6 * 65536
    return (num.astype(np.float64) / 65536.0).astype(np.float32)


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 to bf16 (round to nearest, ties to even); returns uint16 bits."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    r = ((u >> np.uint64(16)) & np.uint64(1)) + np.uint64(0x7FFF)
    return ((u + r) >> np.uint64(16)).astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)
