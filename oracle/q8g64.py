"""Q8G64 MLA row layout and dequantisation (oracle).

[P3] section "起点：把容量和当前计算的工作集分开" (Starting point: separate
capacity from the working set): one Q8G64 MLA row holds 512 B latent, 16 B
scale and 128 B RoPE data, 656 B in all; the capacity table on that page
(31.281 MiB for 50,000 rows, 1.28125 MiB for 2,048 rows, 20.5 MiB for a
32,768-row hot cache) follows from 656 B/row.

[ALG] section "3. KV Cache：历史信息的可复用表示" (KV cache): the MLA cache
stores the normalised low-rank latent and the RoPE part; the quantised layout
keeps the latent as INT8 per group and the RoPE part in 16-bit floats.

[QNT] section "三、基本思路：不是全局舍入，而是利用权重局部性" (basic idea:
use locality instead of one global scale): symmetric quantisation
``q = round(w / scale)``, ``w_hat = scale * q``, with one scale per group of
32/64/128/256 values; "G64" is one scale per 64 consecutive latent values.

Readings (the pages give sizes and listing order only): bytes [0, 512) are the
int8 latent, [512, 528) eight little-endian fp16 scales (group g covers latent
dims 64g..64g+63), [528, 656) 64 little-endian bf16 RoPE values.
"""
from __future__ import annotations

import numpy as np

ROW_BYTES = 656
LAT_DIM = 512
GROUP = 64
N_GROUPS = LAT_DIM // GROUP
ROPE_DIM = 64
OFF_SCALES = LAT_DIM
OFF_ROPE = LAT_DIM + 2 * N_GROUPS


def latent_int8(rows: np.ndarray) -> np.ndarray:
    rows = np.ascontiguousarray(rows, dtype=np.uint8)
    return rows[..., :LAT_DIM].view(np.int8)


def group_scales(rows: np.ndarray) -> np.ndarray:
    """The eight fp16 group scales of each row, as float64 ``[..., 8]``."""
    rows = np.ascontiguousarray(rows, dtype=np.uint8)
    b = np.ascontiguousarray(rows[..., OFF_SCALES:OFF_ROPE])
    return b.view("<f2").astype(np.float64)


def rope_values(rows: np.ndarray) -> np.ndarray:
    """The 64 bf16 RoPE values of each row, as float64 ``[..., 64]``."""
    rows = np.ascontiguousarray(rows, dtype=np.uint8)
    b = np.ascontiguousarray(rows[..., OFF_ROPE:]).view("<u2").astype(np.uint32)
    return (b << np.uint32(16)).view(np.float32).astype(np.float64)


def dequant_latent(rows: np.ndarray) -> np.ndarray:
    """``c[d] = q[d] * scale[d // 64]`` for each row, float64 ``[..., 512]``.

    Symmetric dequantisation, no offset ([QNT] ``w_hat = scale * q``). The
    product of an int8 and an fp16 is exact in float64.
    """
    q = latent_int8(rows).astype(np.float64)
    s = np.repeat(group_scales(rows), GROUP, axis=-1)
    return q * s


def quantize_row(latent_bf16, rope_bf16) -> np.ndarray:
    """Q8G64-quantise one new KV row (the owner quantises once).

    [QNT] section "三、基本思路": symmetric quantisation ``q = round(w / scale)``,
    one scale per group of 64. Readings (the pages give the formula only): the
    group scale is ``fp16_rn(amax / 127)`` with ``amax = max |w|`` over the group
    (division in float32); ``q = clamp(rint(w / scale), -127, 127)`` with the
    division in float32 and round-half-to-even; a group with ``amax = 0`` (or a
    scale that rounds to 0) gets scale 0 and all codes 0; the RoPE part is
    stored as given. Every rounding is an IEEE float32/float16 operation, the
    same ones the kernel performs, so both sides take identical integer
    decisions.

    latent_bf16: uint16 bf16 bits [512]; rope_bf16: uint16 bf16 bits [64].
    Returns the 656-byte row.
    """
    lat = (np.asarray(latent_bf16, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)
    row = np.zeros(ROW_BYTES, dtype=np.uint8)
    q = np.zeros(LAT_DIM, dtype=np.int8)
    scales = np.zeros(N_GROUPS, dtype="<f2")
    for g in range(N_GROUPS):
        x = lat[g * GROUP:(g + 1) * GROUP]
        amax = np.float32(np.max(np.abs(x)))
        s16 = np.float16(np.float32(amax) / np.float32(127.0))
        s = np.float32(s16)
        scales[g] = s16
        if s == 0 or not np.isfinite(s):
            scales[g] = np.float16(0.0)
            continue
        r = np.rint(x / s).astype(np.float32)
        q[g * GROUP:(g + 1) * GROUP] = np.clip(r, -127, 127).astype(np.int8)
    row[:LAT_DIM] = q.view(np.uint8)
    row[OFF_SCALES:OFF_ROPE] = scales.view(np.uint8)
    row[OFF_ROPE:] = np.asarray(rope_bf16, dtype="<u2").view(np.uint8)
    return row
