"""Absorbed-MLA decode attention over the selected rows (oracle, float64).

[ALG] section "2. Attention：决定此刻应读取哪些信息" (attention decides what
to read now): ``Attention(Q, K, V) = softmax(Q K^T / sqrt(d_k) + mask) V``.
[ALG] section "3. KV Cache": MLA stores the normalised low-rank latent and the
RoPE part and rebuilds what it needs when reading.
[P3] section "第三次决策" (third decision): attention runs over the compact
selected KV set produced by the hot gather.

Readings: the absorbed form, where the query is already projected into the
latent space, so one selected row j gives the key ``[c_j, rho_j]`` (dequantised
latent and RoPE part, 576 values) and the value ``c_j`` (512 values):

    logit[h][j] = scale * (q_lat[h] . c_j + q_rope[h] . rho_j)
    out[h]      = sum_j softmax_j(logit[h]) * c_j

with ``scale = 1 / sqrt(576)``. Padding entries (position -1) are excluded.
The log-sum-exp ``lse[h] = log(sum_j exp(logit[h][j]))`` is returned as well.
"""
from __future__ import annotations

import numpy as np

from .indexer import bf16_to_f64
from .q8g64 import dequant_latent, rope_values


def mla_decode_attention(q_lat_bits: np.ndarray, q_rope_bits: np.ndarray,
                         rows: np.ndarray, valid: np.ndarray, scale: float):
    """One query row: ``q_lat [H, 512]``, ``q_rope [H, 64]`` bf16 bits,
    ``rows [K, 656]`` uint8, ``valid [K]`` bool. Returns ``(out [H, 512], lse [H])``
    in float64; with no valid row, out is 0 and lse is -inf.
    """
    ql = bf16_to_f64(q_lat_bits)
    qr = bf16_to_f64(q_rope_bits)
    sel = np.asarray(rows)[np.asarray(valid, dtype=bool)]
    H = ql.shape[0]
    if sel.shape[0] == 0:
        return np.zeros((H, ql.shape[1])), np.full(H, -np.inf)
    c = dequant_latent(sel)
    rho = rope_values(sel)
    logits = scale * (ql @ c.T + qr @ rho.T)
    m = logits.max(axis=1, keepdims=True)
    e = np.exp(logits - m)
    l = e.sum(axis=1, keepdims=True)
    out = (e / l) @ c
    return out, (m + np.log(l))[:, 0]
