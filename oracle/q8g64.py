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
