"""The five synthetic decode workloads and per-unit input generation (numpy).

A *unit* is one (session, layer) pair, ``u = session * layers + layer``. Every
tensor is a pure function of (workload id, tensor id, unit, item), so a test can
regenerate exactly the rows or step inputs it needs.

Value distributions (same for every workload unless stated):

* indexer keys and queries: integers uniform in [-4, 4], stored as bf16;
  head weights ``w``: integers uniform in [1, 4], float32.
* MLA rows (656 B): 512 int8 latents uniform in [-127, 127]; 8 fp16 group
  scales ``k * 2**-16`` with ``k`` uniform in [328, 1311] (so in
  [0.005, 0.02] on an exact fp16 grid); 64 bf16 RoPE values ~ N(0, 1)
  (Irwin-Hall approximation, see ``synth.rng``).
* attention queries ``q_lat [H][512]`` and ``q_rope [H][64]``: bf16 ~ N(0, 1).
* the row and key appended at position ``p`` during decode are the same
  functions of ``p`` as the history rows, so "the history" and "what decode
  appended" are one sequence.

Workload-specific query structure:

* ``mtp`` (four verify rows): every row of a step is a common integer base plus
  a per-row perturbation ``N(0, sd**2)`` rounded to a multiple of 1/16 and the
  result clipped to [-8, 8]; ``w`` is shared by the rows of a step. Scores stay
  exact in float32 (values on a 1/16 grid, |score| < 2**17).
* ``tagged`` (cache stress): key dimension 63 is a tag, +4 for the positions
  that start in the hot cache (the last ``S`` history positions) and -4 for
  all others; query dimension 63 of every head is a per-phase bias ``b`` (a
  multiple of 1/16). ``b`` was chosen so that at the first step of the phase
  about 1% (phase 1) and about 30% (phase 2) of the Top-2048 fall outside the
  initially hot positions; the miss fraction actually seen is measured.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

from .rng import (
    bf16_bits_to_f32, f32_to_bf16_bits, fields16_items, normal_fields_f32,
    stream_key, uniform_int_fields, NORMAL_FIELDS,
)

ROW_BYTES = 656
LAT_DIM = 512
N_GROUPS = 8
ROPE_DIM = 64
IDX_HEADS = 8
IDX_DIM = 64
RING = 64

# tensor ids of the streams
T_KEY, T_LAT, T_SCALE, T_ROPE = 1, 2, 3, 4
T_QI, T_W, T_QLAT, T_QROPE, T_QI_BASE, T_QI_PERT = 5, 6, 7, 8, 9, 10

SCALE_K_LO, SCALE_K_HI = 328, 1311          # scale = k * 2**-16


@dataclass(frozen=True)
class Workload:
    cid: int
    name: str
    sessions: int
    layers: int
    L0: int            # history length at the first decode step
    R: int             # query rows per step (MTP verify: 4)
    A: int             # rows appended per unit per step
    steps: int
    K: int             # Top-K
    H: int             # attention heads
    S: int             # hot-cache slots per unit
    warm: str          # 'empty' or 'last_s'
    mode: str = "iid"  # 'iid' | 'mtp' | 'tagged'
    mtp_sd16: int = 8  # perturbation sd in 1/16 units (8 -> sd 0.5, variance 0.25)
    phases: tuple = field(default=())  # tagged: ((steps, bias in 1/16 units), ...)
    reuse_every: int = 1   # layer l reuses the selection of layer l - l % reuse_every (1: none)
    seed: int = 0
    policy: str = "ring"   # hot-cache replacement: 'ring' or 'clock' (reference bits)

    @property
    def U(self) -> int:
        return self.sessions * self.layers

    def selection_source(self, u: int) -> int:
        """Unit whose selection unit u uses (itself unless it reuses one)."""
        layer = u % self.layers
        return u - layer % self.reuse_every

    @property
    def lmax(self) -> int:
        return self.L0 + self.steps * self.A

    def bias_at(self, step: int) -> float:
        """Query tag bias of a step (tagged workload), in value units."""
        return self._bias16_at(step) / 16.0

    def _bias16_at(self, step: int) -> int:
        t = step
        for n, b in self.phases:
            if t < n:
                return b
            t -= n
        return self.phases[-1][1]

    def scale(self) -> float:
        return 1.0 / np.sqrt(float(LAT_DIM + ROPE_DIM))

    def with_(self, **kw) -> "Workload":
        d = dict(self.__dict__)
        d.update(kw)
        return Workload(**d)


WORKLOADS = {
    0: Workload(0, "tiny smoke: 4,096-position history, 1 layer, Top-256, 16 heads, "
                "1,024 slots (empty start)",
                sessions=1, layers=1, L0=4096, R=1, A=1, steps=8, K=256, H=16,
                S=1024, warm="empty"),
    1: Workload(1, "50K single stream: 50,023-token history, 4 layers, 1 query row, "
                "Top-2048, 64 heads, 32,768 slots",
                sessions=1, layers=4, L0=50023, R=1, A=1, steps=1024, K=2048, H=64,
                S=32768, warm="last_s"),
    2: Workload(2, "MTP=3 verify: 50,023-token history, 4 layers, 4 query rows, "
                "Top-2048, 64 heads, 32,768 slots",
                sessions=1, layers=4, L0=50023, R=4, A=4, steps=256, K=2048, H=64,
                S=32768, warm="last_s", mode="mtp"),
    3: Workload(3, "cache stress: 131,072-position history, 1 layer, full 32,768-slot "
                "cache, 512 low-miss then 512 high-miss steps",
                sessions=1, layers=1, L0=131072, R=1, A=1, steps=1024, K=2048, H=64,
                S=32768, warm="last_s", mode="tagged", phases=((512, 88), (512, 36))),
    4: Workload(4, "capacity batch: 16 sessions x 2 layers, 1,048,576-position history "
                "each, Top-2048, 64 heads, 32,768 slots per unit",
                sessions=16, layers=2, L0=1048576, R=1, A=1, steps=64, K=2048, H=64,
                S=32768, warm="last_s"),
}


def _key(wl: Workload, tensor: int, u: int) -> int:
    return stream_key(wl.cid, tensor, u, wl.seed)


# ---------------------------------------------------------------- history rows

def keys_bits(wl: Workload, u: int, positions) -> np.ndarray:
    """Indexer keys at ``positions``: bf16 bits ``[n, 64]``."""
    pos = np.asarray(positions, dtype=np.int64)
    v = uniform_int_fields(fields16_items(_key(wl, T_KEY, u), pos, IDX_DIM), -4, 4)
    if wl.mode == "tagged":
        hot0 = max(0, wl.L0 - wl.S)
        v[:, IDX_DIM - 1] = np.where((pos >= hot0) & (pos < wl.L0), 4, -4)
    return f32_to_bf16_bits(v.astype(np.float32))


def rows_bytes(wl: Workload, u: int, positions) -> np.ndarray:
    """Q8G64 MLA rows at ``positions``: uint8 ``[n, 656]``.

    Bytes [0,512) int8 latent, [512,528) eight little-endian fp16 group scales,
    [528,656) 64 little-endian bf16 RoPE values.
    """
    pos = np.asarray(positions, dtype=np.int64)
    n = pos.size
    out = np.empty((n, ROW_BYTES), dtype=np.uint8)
    lat = uniform_int_fields(fields16_items(_key(wl, T_LAT, u), pos, LAT_DIM), -127, 127)
    out[:, :LAT_DIM] = lat.astype(np.int8).view(np.uint8)
    k = uniform_int_fields(fields16_items(_key(wl, T_SCALE, u), pos, N_GROUPS),
                           SCALE_K_LO, SCALE_K_HI)
    sc = (k.astype(np.float64) * 2.0 ** -16).astype("<f2")
    out[:, LAT_DIM:LAT_DIM + 16] = sc.view(np.uint8).reshape(n, 16)
    rope = normal_fields_f32(fields16_items(_key(wl, T_ROPE, u), pos, ROPE_DIM * NORMAL_FIELDS))
    out[:, LAT_DIM + 16:] = f32_to_bf16_bits(rope).astype("<u2").view(np.uint8).reshape(n, 128)
    return out


# ---------------------------------------------------------------- step inputs

@dataclass
class UnitInputs:
    """One unit's inputs for one decode step (host arrays)."""
    q_idx: np.ndarray    # uint16 bf16 bits [R][8][64]
    w: np.ndarray        # float32 [R][8]
    q_lat: np.ndarray    # uint16 bf16 bits [R][H][512]
    q_rope: np.ndarray   # uint16 bf16 bits [R][H][64]
    new_rows: np.ndarray  # uint8 [A][656]
    new_keys: np.ndarray  # uint16 bf16 bits [A][64]
    positions: np.ndarray  # int64 [A], positions the new rows take


def step_q_idx(wl: Workload, u: int, step: int) -> tuple[np.ndarray, np.ndarray]:
    R = wl.R
    if wl.mode == "mtp":
        base = uniform_int_fields(fields16_items(_key(wl, T_QI_BASE, u), [step],
                                                 IDX_HEADS * IDX_DIM), -4, 4)[0]
        f = fields16_items(_key(wl, T_QI_PERT, u), step * R + np.arange(R),
                           IDX_HEADS * IDX_DIM * NORMAL_FIELDS)
        g = f.reshape(R, IDX_HEADS * IDX_DIM, NORMAL_FIELDS).astype(np.int64)
        num = g.sum(axis=-1) + 6 - 6 * 65536            # z * 65536
        # perturbation in 1/16 units: round(z * sd16), rounding half up
        m = np.floor_divide(num * wl.mtp_sd16 + 32768, 65536)
        q16 = np.clip(base[None, :] * 16 + m, -128, 128)
        q = (q16.astype(np.float32) / 16.0).reshape(R, IDX_HEADS, IDX_DIM)
        w = uniform_int_fields(fields16_items(_key(wl, T_W, u), [step], IDX_HEADS), 1, 4)
        w = np.repeat(w.astype(np.float32), R, axis=0).reshape(R, IDX_HEADS)
    else:
        v = uniform_int_fields(fields16_items(_key(wl, T_QI, u), step * R + np.arange(R),
                                              IDX_HEADS * IDX_DIM), -4, 4)
        q = v.astype(np.float32).reshape(R, IDX_HEADS, IDX_DIM)
        if wl.mode == "tagged":
            q[:, :, IDX_DIM - 1] = wl.bias_at(step)
        w = uniform_int_fields(fields16_items(_key(wl, T_W, u), step * R + np.arange(R),
                                              IDX_HEADS), 1, 4).astype(np.float32)
        w = w.reshape(R, IDX_HEADS)
    return f32_to_bf16_bits(q), w.astype(np.float32)


def step_q_attn(wl: Workload, u: int, step: int) -> tuple[np.ndarray, np.ndarray]:
    R, H = wl.R, wl.H
    items = step * R + np.arange(R)
    ql = normal_fields_f32(fields16_items(_key(wl, T_QLAT, u), items, H * LAT_DIM * NORMAL_FIELDS))
    qr = normal_fields_f32(fields16_items(_key(wl, T_QROPE, u), items, H * ROPE_DIM * NORMAL_FIELDS))
    return (f32_to_bf16_bits(ql).reshape(R, H, LAT_DIM),
            f32_to_bf16_bits(qr).reshape(R, H, ROPE_DIM))


def append_positions(wl: Workload, step: int) -> np.ndarray:
    return wl.L0 + step * wl.A + np.arange(wl.A, dtype=np.int64)


def step_inputs(wl: Workload, u: int, step: int) -> UnitInputs:
    q_idx, w = step_q_idx(wl, u, step)
    q_lat, q_rope = step_q_attn(wl, u, step)
    pos = append_positions(wl, step)
    return UnitInputs(q_idx, w, q_lat, q_rope, rows_bytes(wl, u, pos), keys_bits(wl, u, pos), pos)


def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    return bf16_bits_to_f32(bits).astype(np.float64)
