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

    def score(self, q_idx, w, stream=None):
        """The scoring half of score_topk (dsa_score); select() completes it."""
        u = self.u
        units, U = (self.src_units, self.Us) if self.sources else (u.units, u.U)
        abi.dsa_score(units, U, self.R, self.K, q_idx, w, self.max_len, self.ws_topk, self.ws_topk_bytes,
                      u.dev_err, stream)

    def select(self, stream=None):
        """The selection half of score_topk (dsa_topk_select), ordered after
        score() by the caller."""
        u = self.u
        if self.sources:
            abi.dsa_topk_select(self.src_units, self.Us, self.R, self.K, self.src_topk, self.max_len,
                                self.ws_topk, self.ws_topk_bytes, u.dev_err, stream)
            abi.dsa_reuse_selection(self.topk, self.src_topk, u.U, self.Us, self.R, self.K, self.src_of,
                                    u.dev_err, stream)
            return
        abi.dsa_topk_select(u.units, u.U, self.R, self.K, self.topk, self.max_len, self.ws_topk,
                            self.ws_topk_bytes, u.dev_err, stream)

    def gather(self, rnd: int, stream=None):
        u = self.u
        abi.hot_gather(u.units, u.U, self.R, self.K, rnd, self.topk, self.cls, self.rows,
                       self.counters, self.ws_gather, self.ws_gather_bytes, u.dev_err, stream)

    def attend(self, q_lat, q_rope, stream=None):
        u = self.u
        abi.mla_decode_attn(u.U, self.R, self.H, self.K, q_lat, q_rope, self.rows, self.topk,
                            self.scale, self.out, self.lse, self.ws_attn, self.ws_attn_bytes,
                            u.dev_err, stream)

    def prepare_fused(self):
        """The workspace of gather_attend (zero-filled on the current stream;
        allocate it before the first call when that call runs on another
        stream)."""
        if not hasattr(self, "ws_fused"):
            u = self.u
            self.ws_fused_bytes = abi.hot_gather_attn_workspace(u.U, self.R, self.H, self.K)
            self.ws_fused = torch.zeros(self.ws_fused_bytes, dtype=torch.uint8, device=u.device)

    def gather_attend(self, rnd: int, q_lat, q_rope, stream=None):
        """hot_gather + attention in one call (rows read from their sources)."""
        u = self.u
        self.prepare_fused()
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

    # ------------------------------------------------------ pipelined steps
    def enable_pipeline(self):
        """Buffers and streams for step_pipelined: a second selection buffer,
        a side stream and the events that order the two halves of the gather."""
        if self.A != 1 or self.sources:
            raise ValueError("pipelined steps need one appended row per step and no selection reuse")
        dev = self.u.device
        self.topk_pipe = [self.topk, torch.empty_like(self.topk)]
        self.pipe_i = 0
        self.side = torch.cuda.Stream(dev)
        self.ev_assigned = torch.cuda.Event()
        self.ev_copied = torch.cuda.Event()
        self.ev_used = [torch.cuda.Event(), torch.cuda.Event()]   # attention done with topk_pipe[i]
        self.ev_done = torch.cuda.Event()
        self.copy_pending = False
        self.used_pending = [False, False]

    def step_pipelined(self, rnd, q_idx, w, q_lat, q_rope, new_rows, new_keys, stream=None, out_host=None,
                       stage_inputs=None):
        """One decode step whose gather copy and attention run on a side stream,
        overlapping the next step's scoring and selection (main stream). The
        order the C ABI requires is kept with events: the next step's
        hot_gather_assign waits for this step's hot_gather_copy (it may evict
        slots the copy reads); the append (one row) follows the assign on the
        main stream. Selections alternate between two buffers; ``cur_topk`` is
        this step's. ``out`` is this step's output once ``join()`` has made the
        main stream wait for the side stream (or, with ``out_host``, it is
        copied there on the side stream). ``stage_inputs(b)``, if given, is
        called on the main stream once the step before last has finished with
        input set b (b = step parity) and returns the six input tensors it has
        staged there (e.g. copies from host memory)."""
        u = self.u
        main = stream if stream is not None else torch.cuda.current_stream()
        b = self.pipe_i
        topk = self.topk_pipe[b]
        self.pipe_i ^= 1
        if self.used_pending[b]:
            main.wait_event(self.ev_used[b])     # the attention two steps back read this buffer
        if stage_inputs is not None:
            q_idx, w, q_lat, q_rope, new_rows, new_keys = stage_inputs(b)
        abi.dsa_score_topk(u.units, u.U, self.R, self.K, q_idx, w, topk, self.max_len,
                           self.ws_topk, self.ws_topk_bytes, u.dev_err, main)
        if self.copy_pending:
            main.wait_event(self.ev_copied)
        abi.hot_gather_assign(u.units, u.U, self.R, self.K, rnd, topk, self.cls, self.counters, self.ws_gather,
                              self.ws_gather_bytes, u.dev_err, main)
        self.ev_assigned.record(main)
        abi.kv_append_writeback(u.units, u.U, self.A, new_rows, new_keys, u.dev_err, main)
        self.side.wait_event(self.ev_assigned)
        abi.hot_gather_copy(u.units, u.U, self.R, self.K, topk, self.cls, self.rows, self.ws_gather,
                            self.ws_gather_bytes, u.dev_err, self.side)
        self.ev_copied.record(self.side)
        abi.mla_decode_attn(u.U, self.R, self.H, self.K, q_lat, q_rope, self.rows, topk, self.scale, self.out,
                            self.lse, self.ws_attn, self.ws_attn_bytes, u.dev_err, self.side)
        self.ev_used[b].record(self.side)
        self.used_pending[b] = True
        if out_host is not None:
            with torch.cuda.stream(self.side):
                out_host.copy_(self.out, non_blocking=True)
        self.ev_done.record(self.side)
        self.copy_pending = True
        self.cur_topk = topk

    def begin_graph(self):
        """The steps before this point have completed (e.g. an earlier CUDA
        graph replay on the same stream); steps captured from here on do not
        wait on their events (a graph capture cannot)."""
        self.copy_pending = False
        self.used_pending = [False, False]

    def join(self, stream=None):
        """Make `stream` (default: the current stream) wait for the side stream."""
        (stream if stream is not None else torch.cuda.current_stream()).wait_event(self.ev_done)

    def launches_per_step(self, fused: bool = False) -> int:
        """Kernel launches one step enqueues (score, select, [reuse copy],
        classify+assign, copy (not with the fused gather), attention parts,
        attention merge, append)."""
        return (8 if self.sources else 7) - (1 if fused else 0)
