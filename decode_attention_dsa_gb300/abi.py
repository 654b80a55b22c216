"""ctypes binding of ``libdsa_decode.so``: the C ABI of ``include/dsa_decode.h``
under the same names. Argument marshalling only: every step runs in the CUDA
kernels of the library. Pointers may be given as torch tensors (their
``data_ptr()``), plain integers, or None (NULL). Streams may be a
``torch.cuda.Stream``, an integer handle, or None (the current torch stream).

A non-zero status raises ``DsaError``. Loading fails loudly if the library is
missing: there is no fallback path.
"""
from __future__ import annotations

import ctypes
import os

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "libdsa_decode.so")

DSA_OK = 0
DSA_ERR_ARG, DSA_ERR_SHAPE, DSA_ERR_WS, DSA_ERR_CUDA, DSA_ERR_DEVICE_CHECK = -1, -2, -3, -4, -6
DSA_ERR_SCRATCH_LIMIT = -7
DEVERR_BOUNDS, DEVERR_CAPACITY, DEVERR_QRANGE, DEVERR_TIMEOUT, DEVERR_ROUND = 0x1, 0x2, 0x4, 0x8, 0x10
DEVERR_STATE = 0x20
ROW_BYTES, LAT_DIM, ROPE_DIM, IDX_HEADS, IDX_DIM, RING_ROWS = 656, 512, 64, 8, 64, 64
MAX_K, MAX_ROWS, MAX_ATTN_K, ROUND_AUTO = 4096, 8, 2048, -1
CLS_HOT, CLS_RING, CLS_RAM, CLS_PAD = 0, 1, 2, 3
WARM_EMPTY, WARM_LAST_S = 0, 1
POLICY_RING, POLICY_CLOCK = 0, 1
ST_LEN, ST_RAM, ST_HAND, ST_EPOCH, ST_WRITEBACKS, ST_ROUND, ST_WORDS = 0, 1, 2, 3, 4, 5, 8


class DsaError(RuntimeError):
    def __init__(self, fn: str, status: int):
        super().__init__(f"{fn} failed: {status} ({status_string(status)})")
        self.status = status


class DsaUnit(ctypes.Structure):
    """Mirror of ``struct dsa_unit``."""
    _fields_ = [
        ("keys", ctypes.c_void_p), ("slots", ctypes.c_void_p), ("slot_pos", ctypes.c_void_p),
        ("pos_slot", ctypes.c_void_p), ("fill_round", ctypes.c_void_p),
        ("pin_epoch", ctypes.c_void_p), ("ring", ctypes.c_void_p), ("mirror", ctypes.c_void_p),
        ("state", ctypes.c_void_p), ("slots_n", ctypes.c_int32), ("policy", ctypes.c_int32),
        ("lmax", ctypes.c_int64), ("ref", ctypes.c_void_p),
    ]


assert ctypes.sizeof(DsaUnit) == 96

_VP, _I32, _I64, _SZ, _F = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t, ctypes.c_float

# name -> (restype, argtypes), in the order of the header
SIGNATURES = {
    "dsa_abi_version": (ctypes.c_int, []),
    "dsa_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    "dsa_check": (ctypes.c_int, [_I32]),
    "dsa_wait_selftest": (ctypes.c_int, [_I64, _I32, _VP, _VP]),
    "dsa_host_alloc": (ctypes.c_int, [ctypes.POINTER(_VP), ctypes.POINTER(_VP), _SZ]),
    "dsa_host_free": (ctypes.c_int, [_VP]),
    "hc_init": (ctypes.c_int, [_VP, _I32, _I32, _VP, _I32, _I64, _VP, _VP]),
    "dsa_touch_mirror": (ctypes.c_int, [_VP, _I32, _I64, _VP]),
    "dsa_score_topk_workspace": (_SZ, [_I32, _I32, _I64]),
    "dsa_score_topk": (ctypes.c_int, [_VP, _I32, _I32, _I32, _VP, _VP, _VP, _I64, _VP, _SZ, _VP, _VP]),
    "dsa_score": (ctypes.c_int, [_VP, _I32, _I32, _I32, _VP, _VP, _I64, _VP, _SZ, _VP, _VP]),
    "dsa_topk_select": (ctypes.c_int, [_VP, _I32, _I32, _I32, _VP, _I64, _VP, _SZ, _VP, _VP]),
    "dsa_partition_split": (ctypes.c_int, [_I32, ctypes.POINTER(_VP), ctypes.POINTER(_VP)]),
    "dsa_partition_sms": (ctypes.c_int, [_VP]),
    "dsa_partition_stream": (ctypes.c_int, [_VP, ctypes.POINTER(_VP)]),
    "dsa_stream_wait_stream": (ctypes.c_int, [_VP, _VP]),
    "dsa_partition_destroy": (ctypes.c_int, [_VP]),
    "dsa_score_topk_noalloc": (ctypes.c_int, [_VP, _I32, _I32, _I32, _VP, _VP, _VP, _I64, _VP, _VP]),
    "dsa_reuse_selection": (ctypes.c_int, [_VP, _VP, _I32, _I32, _I32, _I32, _VP, _VP, _VP]),
    "hot_gather_workspace": (_SZ, [_I32, _I32, _I32]),
    "hot_gather": (ctypes.c_int, [_VP, _I32, _I32, _I32, _I32, _VP, _VP, _VP, _VP, _VP, _SZ, _VP, _VP]),
    "hot_gather_assign": (ctypes.c_int, [_VP, _I32, _I32, _I32, _I32, _VP, _VP, _VP, _VP, _SZ, _VP, _VP]),
    "hot_gather_copy": (ctypes.c_int, [_VP, _I32, _I32, _I32, _VP, _VP, _VP, _VP, _SZ, _VP, _VP]),
    "mla_decode_attn_workspace": (_SZ, [_I32, _I32, _I32, _I32]),
    "mla_decode_attn": (ctypes.c_int, [_I32, _I32, _I32, _I32, _VP, _VP, _VP, _VP, _F, _VP, _VP, _VP,
                                       _SZ, _VP, _VP]),
    "hot_gather_attn_workspace": (_SZ, [_I32, _I32, _I32, _I32]),
    "hot_gather_attn": (ctypes.c_int, [_VP, _I32, _I32, _I32, _I32, _I32, _VP, _VP, _VP, _F, _VP, _VP, _VP,
                                       _VP, _VP, _SZ, _VP, _VP]),
    "kv_append_writeback": (ctypes.c_int, [_VP, _I32, _I32, _VP, _VP, _VP, _VP]),
    "kv_append_quantize": (ctypes.c_int, [_VP, _I32, _I32, _VP, _VP, _VP, _VP, _VP]),
    "kv_flush": (ctypes.c_int, [_VP, _I32, _VP, _VP]),
    "dsa_snapshot_bytes": (_SZ, [_I32, _I64]),
    "dsa_export": (ctypes.c_int, [_VP, _I32, _VP, _SZ, _I32, _I64, _VP, _VP]),
    "dsa_restore": (ctypes.c_int, [_VP, _I32, _VP, _SZ, _I32, _I64, _VP, _VP]),
    "kv_restore_full": (ctypes.c_int, [_VP, _I32, _VP, _I64, _VP, _VP]),
}

_lib = None


def load(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load the library (once). Raises if it is missing or incomplete."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is missing: build it with __graft_entry__.build() "
                           "or python -m decode_attention_dsa_gb300.build")
    lib = ctypes.CDLL(path)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)          # AttributeError if a symbol is missing
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


def _p(x):
    if x is None:
        return None
    if hasattr(x, "data_ptr"):
        return x.data_ptr()
    return int(x)


def _s(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if hasattr(stream, "cuda_stream"):
        return stream.cuda_stream
    return int(stream)


def _ok(fn, st):
    if st != DSA_OK:
        raise DsaError(fn, st)
    return st


def dsa_abi_version() -> int:
    return load().dsa_abi_version()


def status_string(status: int) -> str:
    return load().dsa_status_string(status).decode()


dsa_status_string = status_string


def dsa_check(dev_err_value: int) -> int:
    return load().dsa_check(int(dev_err_value))


def dsa_wait_selftest(limit_cycles, complete, dev_err, stream=None):
    return _ok("dsa_wait_selftest", load().dsa_wait_selftest(int(limit_cycles), int(bool(complete)),
                                                             _p(dev_err), _s(stream)))


def dsa_host_alloc(nbytes: int) -> tuple[int, int]:
    """Pinned, mapped host memory: returns (host address, device alias)."""
    h, d = _VP(), _VP()
    _ok("dsa_host_alloc", load().dsa_host_alloc(ctypes.byref(h), ctypes.byref(d), nbytes))
    return h.value, d.value


def dsa_host_free(host_ptr: int) -> None:
    _ok("dsa_host_free", load().dsa_host_free(host_ptr))


def hc_init(units, U, warm, l0, max_slots, max_lmax, dev_err, stream=None):
    return _ok("hc_init", load().hc_init(_p(units), U, warm, _p(l0), max_slots, max_lmax,
                                         _p(dev_err), _s(stream)))


def dsa_touch_mirror(units, U, max_lmax, stream=None):
    return _ok("dsa_touch_mirror", load().dsa_touch_mirror(_p(units), U, max_lmax, _s(stream)))


def dsa_score_topk_workspace(U, R, max_len) -> int:
    return load().dsa_score_topk_workspace(U, R, max_len)


def dsa_score_topk(units, U, R, K, q, w, topk_idx, max_len, ws, ws_bytes, dev_err, stream=None):
    return _ok("dsa_score_topk", load().dsa_score_topk(
        _p(units), U, R, K, _p(q), _p(w), _p(topk_idx), max_len, _p(ws), ws_bytes, _p(dev_err),
        _s(stream)))


def dsa_score(units, U, R, K, q, w, max_len, ws, ws_bytes, dev_err, stream=None):
    return _ok("dsa_score", load().dsa_score(
        _p(units), U, R, K, _p(q), _p(w), max_len, _p(ws), ws_bytes, _p(dev_err), _s(stream)))


def dsa_topk_select(units, U, R, K, topk_idx, max_len, ws, ws_bytes, dev_err, stream=None):
    return _ok("dsa_topk_select", load().dsa_topk_select(
        _p(units), U, R, K, _p(topk_idx), max_len, _p(ws), ws_bytes, _p(dev_err), _s(stream)))


def dsa_partition_split(min_sms: int, first: bool = True, second: bool = True):
    """Split the current device's SMs: returns (first, second) partition
    handles (None where not asked for)."""
    p1, p2 = _VP(), _VP()
    _ok("dsa_partition_split", load().dsa_partition_split(
        int(min_sms), ctypes.byref(p1) if first else None, ctypes.byref(p2) if second else None))
    return (p1.value if first else None), (p2.value if second else None)


def dsa_partition_sms(part) -> int:
    return load().dsa_partition_sms(part)


def dsa_partition_stream(part) -> int:
    """A new stream of the partition (a raw cudaStream_t handle)."""
    s = _VP()
    _ok("dsa_partition_stream", load().dsa_partition_stream(part, ctypes.byref(s)))
    return s.value


def dsa_stream_wait_stream(waiter, signaller):
    return _ok("dsa_stream_wait_stream", load().dsa_stream_wait_stream(_s(waiter), _s(signaller)))


def dsa_partition_destroy(part):
    return _ok("dsa_partition_destroy", load().dsa_partition_destroy(part))


def dsa_score_topk_noalloc(units, U, R, K, q, w, topk_idx, max_len, dev_err, stream=None):
    """dsa_score_topk with the library's fixed built-in scratch (no workspace)."""
    return _ok("dsa_score_topk_noalloc", load().dsa_score_topk_noalloc(
        _p(units), U, R, K, _p(q), _p(w), _p(topk_idx), max_len, _p(dev_err), _s(stream)))


def dsa_reuse_selection(topk_idx, src_topk, U, Us, R, K, src_of, dev_err, stream=None):
    return _ok("dsa_reuse_selection", load().dsa_reuse_selection(
        _p(topk_idx), _p(src_topk), U, Us, R, K, _p(src_of), _p(dev_err), _s(stream)))


def hot_gather_workspace(U, R, K) -> int:
    return load().hot_gather_workspace(U, R, K)


def hot_gather(units, U, R, K, round_, topk_idx, cls, rows, counters, ws, ws_bytes, dev_err,
               stream=None):
    return _ok("hot_gather", load().hot_gather(
        _p(units), U, R, K, round_, _p(topk_idx), _p(cls), _p(rows), _p(counters), _p(ws), ws_bytes,
        _p(dev_err), _s(stream)))


def hot_gather_assign(units, U, R, K, round_, topk_idx, cls, counters, ws, ws_bytes, dev_err, stream=None):
    return _ok("hot_gather_assign", load().hot_gather_assign(
        _p(units), U, R, K, round_, _p(topk_idx), _p(cls), _p(counters), _p(ws), ws_bytes, _p(dev_err),
        _s(stream)))


def hot_gather_copy(units, U, R, K, topk_idx, cls, rows, ws, ws_bytes, dev_err, stream=None):
    return _ok("hot_gather_copy", load().hot_gather_copy(
        _p(units), U, R, K, _p(topk_idx), _p(cls), _p(rows), _p(ws), ws_bytes, _p(dev_err), _s(stream)))


def mla_decode_attn_workspace(U, R, H, K) -> int:
    return load().mla_decode_attn_workspace(U, R, H, K)


def mla_decode_attn(U, R, H, K, q_lat, q_rope, rows, topk_idx, scale, out, lse, ws, ws_bytes,
                    dev_err, stream=None):
    return _ok("mla_decode_attn", load().mla_decode_attn(
        U, R, H, K, _p(q_lat), _p(q_rope), _p(rows), _p(topk_idx), float(scale), _p(out), _p(lse),
        _p(ws), ws_bytes, _p(dev_err), _s(stream)))


def hot_gather_attn_workspace(U, R, H, K) -> int:
    return load().hot_gather_attn_workspace(U, R, H, K)


def hot_gather_attn(units, U, R, K, H, round_, topk_idx, q_lat, q_rope, scale, cls, counters, out, lse,
                    ws, ws_bytes, dev_err, stream=None):
    return _ok("hot_gather_attn", load().hot_gather_attn(
        _p(units), U, R, K, H, round_, _p(topk_idx), _p(q_lat), _p(q_rope), float(scale), _p(cls),
        _p(counters), _p(out), _p(lse), _p(ws), ws_bytes, _p(dev_err), _s(stream)))


def kv_append_writeback(units, U, A, new_rows, new_keys, dev_err, stream=None):
    return _ok("kv_append_writeback", load().kv_append_writeback(
        _p(units), U, A, _p(new_rows), _p(new_keys), _p(dev_err), _s(stream)))


def kv_append_quantize(units, U, A, new_latent, new_rope, new_keys, dev_err, stream=None):
    return _ok("kv_append_quantize", load().kv_append_quantize(
        _p(units), U, A, _p(new_latent), _p(new_rope), _p(new_keys), _p(dev_err), _s(stream)))


def kv_flush(units, U, dev_err, stream=None):
    return _ok("kv_flush", load().kv_flush(_p(units), U, _p(dev_err), _s(stream)))


def dsa_snapshot_bytes(S, lmax) -> int:
    return load().dsa_snapshot_bytes(S, lmax)


def dsa_export(units, U, snap, snap_stride, max_slots, max_lmax, dev_err, stream=None):
    return _ok("dsa_export", load().dsa_export(_p(units), U, _p(snap), snap_stride, max_slots, max_lmax,
                                               _p(dev_err), _s(stream)))


def dsa_restore(units, U, snap, snap_stride, max_slots, max_lmax, dev_err, stream=None):
    return _ok("dsa_restore", load().dsa_restore(_p(units), U, _p(snap), snap_stride, max_slots, max_lmax,
                                                 _p(dev_err), _s(stream)))


def kv_restore_full(units, U, dst, dst_rows, dev_err, stream=None):
    return _ok("kv_restore_full", load().kv_restore_full(_p(units), U, _p(dst), dst_rows, _p(dev_err),
                                                         _s(stream)))
