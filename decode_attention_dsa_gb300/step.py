"""One decode step over a UnitSet: the four C-ABI calls in order, with
persistent workspaces and outputs (marshalling only)."""
from __future__ import annotations

import ctypes

import torch

from . import abi
from .units import UnitSet


class DecodePath:
    """Workspaces and outputs for steps of ``R`` query rows, Top-``K``, ``H``
    heads and ``A`` appended rows per unit per step."""

    def __init__(self, units: UnitSet, R: int, K: int, H: int, A: int, scale: float,
                 max_len: int | None = None, selection_source=None):
        """``selection_source[u]``: the unit whose selection unit u reuses (a
        later layer reusing an earlier layer's selection); None: every unit is
        scored. With reuse, score_topk takes the query rows of the source
        units only, in ascending unit order."""
        self.u = units
        U = units.U
        self.R, self.K, self.H, self.A, self.scale = R, K, H, A, float(scale)
        self.max_len = units.lmax if max_len is None else max_len
        dev = units.device
        self.sources = None
        if selection_source is not None and any(int(x) != u for u, x in enumerate(selection_source)):
            self.sources = sorted(set(int(x) for x in selection_source))
            self.Us = len(self.sources)
            raw = units.units.view(-1, ctypes.sizeof(abi.DsaUnit))
            self.src_units = raw[self.sources].contiguous().view(-1)
            self.src_of = torch.tensor([self.sources.index(int(x)) for x in selection_source],
                                       dtype=torch.int32, device=dev)
            self.src_topk = torch.empty((self.Us, R, K), dtype=torch.int32, device=dev)
        n_scored = self.Us if self.sources else U
        self.ws_topk_bytes = abi.dsa_score_topk_workspace(n_scored, R, self.max_len)
        self.ws_topk = torch.zeros(self.ws_topk_bytes, dtype=torch.uint8, device=dev)
        self.ws_gather_bytes = abi.hot_gather_workspace(U, R, K)
        self.ws_gather = torch.zeros(self.ws_gather_bytes, dtype=torch.uint8, device=dev)
        self.ws_attn_bytes = abi.mla_decode_attn_workspace(U, R, H, K)
        self.ws_attn = (torch.zeros(self.ws_attn_bytes, dtype=torch.uint8, device=dev)
                        if self.ws_attn_bytes else None)
        self.topk = torch.empty((U, R, K), dtype=torch.int32, device=dev)
        self.cls = torch.empty((U, R, K), dtype=torch.uint8, device=dev)
        self.rows = torch.empty((U, R, K, abi.ROW_BYTES), dtype=torch.uint8, device=dev)
        self.counters = torch.zeros((U, 4), dtype=torch.int32, device=dev)
        self.out = torch.empty((U, R, H, abi.LAT_DIM), dtype=torch.float32, device=dev)
        self.lse = torch.empty((U, R, H), dtype=torch.float32, device=dev)

    def score_topk(self, q_idx, w, stream=None):
        u = self.u
        if self.sources:
            abi.dsa_score_topk(self.src_units, self.Us, self.R, self.K, q_idx, w, self.src_topk, self.max_len,
                               self.ws_topk, self.ws_topk_bytes, u.dev_err, stream)
            abi.dsa_reuse_selection(self.topk, self.src_topk, u.U, self.Us, self.R, self.K, self.src_of,
                                    u.dev_err, stream)
            return
        abi.dsa_score_topk(u.units, u.U, self.R, self.K, q_idx, w, self.topk, self.max_len,
                           self.ws_topk, self.ws_topk_bytes, u.dev_err, stream)

    def gather(self, rnd: int, stream=None):
        u = self.u
        abi.hot_gather(u.units, u.U, self.R, self.K, rnd, self.topk, self.cls, self.rows,
                       self.counters, self.ws_gather, self.ws_gather_bytes, u.dev_err, stream)

    def attend(self, q_lat, q_rope, stream=None):
        u = self.u
        abi.mla_decode_attn(u.U, self.R, self.H, self.K, q_lat, q_rope, self.rows, self.topk,
                            self.scale, self.out, self.lse, self.ws_attn, self.ws_attn_bytes,
                            u.dev_err, stream)

    def gather_attend(self, rnd: int, q_lat, q_rope, stream=None):
        """hot_gather + attention in one call (rows read from their sources)."""
        u = self.u
        if not hasattr(self, "ws_fused"):
            self.ws_fused_bytes = abi.hot_gather_attn_workspace(u.U, self.R, self.H, self.K)
            self.ws_fused = torch.zeros(self.ws_fused_bytes, dtype=torch.uint8, device=u.device)
        abi.hot_gather_attn(u.units, u.U, self.R, self.K, self.H, rnd, self.topk, q_lat, q_rope, self.scale,
                            self.cls, self.counters, self.out, self.lse, self.ws_fused, self.ws_fused_bytes,
                            u.dev_err, stream)

    def append(self, new_rows, new_keys, stream=None):
        u = self.u
        abi.kv_append_writeback(u.units, u.U, self.A, new_rows, new_keys, u.dev_err, stream)

    def step(self, rnd, q_idx, w, q_lat, q_rope, new_rows, new_keys, stream=None, side=None,
             fused=False):
        """One decode step. ``fused`` uses hot_gather_attn (no compact rows; the
        append follows it). Otherwise, with a ``side`` stream, the append runs
        there, concurrently with the attention (allowed once the gather is
        done)."""
        if fused:
            self.score_topk(q_idx, w, stream)
            self.gather_attend(rnd, q_lat, q_rope, stream)
            self.append(new_rows, new_keys, stream)
            return
        self.score_topk(q_idx, w, stream)
        self.gather(rnd, stream)
        if side is None:
            self.attend(q_lat, q_rope, stream)
            self.append(new_rows, new_keys, stream)
            return
        main = stream if stream is not None else torch.cuda.current_stream()
        side.wait_stream(main)
        self.append(new_rows, new_keys, side)
        self.attend(q_lat, q_rope, main)
        main.wait_stream(side)

    def launches_per_step(self) -> int:
        """Kernel launches one step enqueues (score, select, [reuse copy],
        classify+assign, copy, attention, append)."""
        return 7 if self.sources else 6
