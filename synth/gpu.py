"""GPU generator: the same draws as ``synth.workloads``, written on the device.

Loads ``synth/libdsa_synth.so`` (built by ``build()``), which holds only the
counter-based generator kernels. Used to produce large workloads quickly
(history rows straight into the pinned mirror, all step inputs into HBM); the
numpy generator remains the definition and a GPU test checks byte equality.
"""
from __future__ import annotations

import ctypes
import os
import shutil
import subprocess

import numpy as np

from . import workloads as W

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "csrc", "synth_gen.cu")
LIB = os.path.join(HERE, "libdsa_synth.so")

_lib = None
_VP, _I32, _I64, _U64 = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_uint64


def build(force: bool = False) -> str:
    if not force and os.path.exists(LIB) and os.path.getmtime(LIB) >= os.path.getmtime(SRC):
        return LIB
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    cmd = [nvcc, "-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-std=c++17",
           "-Xcompiler", "-fPIC", "-shared", "-o", LIB + ".tmp", SRC]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(r.stdout + r.stderr)
    os.replace(LIB + ".tmp", LIB)
    return LIB


def load():
    global _lib
    if _lib is None:
        if not os.path.exists(LIB):
            raise RuntimeError(f"{LIB} is missing: run synth.gpu.build()")
        lib = ctypes.CDLL(LIB)
        lib.synth_keys.argtypes = [_U64, _VP, _I64, _I64, _I32, _I64, _I64, _VP]
        lib.synth_rows.argtypes = [_U64, _U64, _U64, _VP, _I64, _I64, _VP]
        lib.synth_normal_bf16.argtypes = [_U64, _VP, _I64, _I64, _I32, _VP]
        lib.synth_uniform_bf16.argtypes = [_U64, _VP, _I64, _I64, _I32, _I32, _I32, _I32, _I32, _VP]
        lib.synth_uniform_f32.argtypes = [_U64, _VP, _I64, _I64, _I32, _I32, _I32, _I32, _VP]
        lib.synth_mtp_qidx.argtypes = [_U64, _U64, _VP, _I64, _I32, _I32, _VP]
        for f in ("synth_keys", "synth_rows", "synth_normal_bf16", "synth_uniform_bf16",
                  "synth_uniform_f32", "synth_mtp_qidx"):
            getattr(lib, f).restype = ctypes.c_int
        _lib = lib
    return _lib


def _chk(rc):
    if rc != 0:
        raise RuntimeError(f"synth kernel launch failed ({rc})")


def _stream(stream):
    import torch
    return (stream or torch.cuda.current_stream()).cuda_stream


def keys(wl: W.Workload, u: int, out_ptr: int, pos0: int, n: int, stream=None):
    lib = load()
    hot_lo = max(0, wl.L0 - wl.S)
    _chk(lib.synth_keys(W._key(wl, W.T_KEY, u), out_ptr, pos0, n, int(wl.mode == "tagged"),
                        hot_lo, wl.L0, _stream(stream)))


def rows(wl: W.Workload, u: int, out_ptr: int, pos0: int, n: int, stream=None):
    """Rows of positions [pos0, pos0+n) to ``out_ptr`` (device or mapped host alias)."""
    lib = load()
    _chk(lib.synth_rows(W._key(wl, W.T_LAT, u), W._key(wl, W.T_SCALE, u), W._key(wl, W.T_ROPE, u),
                        out_ptr, pos0, n, _stream(stream)))


def step_inputs(wl: W.Workload, step0: int, nsteps: int, stream=None) -> dict:
    """All units' inputs for steps [step0, step0+nsteps) as device tensors with a
    leading step dimension (same layout as ``synth.workloads.step_inputs``)."""
    import torch
    lib = load()
    U, R, H, A = wl.U, wl.R, wl.H, wl.A
    dev = torch.device("cuda")
    q_idx = torch.empty((nsteps, U, R, 8, 64), dtype=torch.int16, device=dev)
    w = torch.empty((nsteps, U, R, 8), dtype=torch.float32, device=dev)
    q_lat = torch.empty((nsteps, U, R, H, 512), dtype=torch.int16, device=dev)
    q_rope = torch.empty((nsteps, U, R, H, 64), dtype=torch.int16, device=dev)
    new_rows = torch.empty((nsteps, U, A, 656), dtype=torch.uint8, device=dev)
    new_keys = torch.empty((nsteps, U, A, 64), dtype=torch.int16, device=dev)
    s = _stream(stream)
    for u in range(U):
        for k in range(nsteps):
            st = step0 + k
            if wl.mode == "mtp":
                _chk(lib.synth_mtp_qidx(W._key(wl, W.T_QI_BASE, u), W._key(wl, W.T_QI_PERT, u),
                                        q_idx[k, u].data_ptr(), st, R, wl.mtp_sd16, s))
                _chk(lib.synth_uniform_f32(W._key(wl, W.T_W, u), w[k, u].data_ptr(), st * R, R, 8,
                                           1, 4, R, s))
            else:
                tag = wl._bias16_at(st) if wl.mode == "tagged" else 0
                _chk(lib.synth_uniform_bf16(W._key(wl, W.T_QI, u), q_idx[k, u].data_ptr(), st * R, R,
                                            512, -4, 4, 64 if wl.mode == "tagged" else 0, tag, s))
                _chk(lib.synth_uniform_f32(W._key(wl, W.T_W, u), w[k, u].data_ptr(), st * R, R, 8,
                                           1, 4, 1, s))
            pos = wl.L0 + st * A
            rows(wl, u, new_rows[k, u].data_ptr(), pos, A, stream)
            keys(wl, u, new_keys[k, u].data_ptr(), pos, A, stream)
        # attention queries of all steps of this unit in one launch each
        # (items step*R + r are consecutive, so [step0*R, (step0+nsteps)*R))
        ql = torch.empty((nsteps, R, H, 512), dtype=torch.int16, device=dev)
        qr = torch.empty((nsteps, R, H, 64), dtype=torch.int16, device=dev)
        _chk(lib.synth_normal_bf16(W._key(wl, W.T_QLAT, u), ql.data_ptr(), step0 * R, nsteps * R,
                                   H * 512, s))
        _chk(lib.synth_normal_bf16(W._key(wl, W.T_QROPE, u), qr.data_ptr(), step0 * R, nsteps * R,
                                   H * 64, s))
        q_lat[:, u].copy_(ql)
        q_rope[:, u].copy_(qr)
    return dict(q_idx=q_idx, w=w, q_lat=q_lat, q_rope=q_rope, new_rows=new_rows, new_keys=new_keys)


def history(wl: W.Workload, units_set, stream=None, chunk: int = 1 << 20):
    """History keys and mirror rows [0, L0) of every unit of a UnitSet."""
    for u in range(wl.U):
        keys(wl, u, units_set.keys[u].data_ptr(), 0, wl.L0, stream)
        base = units_set._mirror_dev + u * units_set.lmax * 656
        for p0 in range(0, wl.L0, chunk):
            n = min(chunk, wl.L0 - p0)
            rows(wl, u, base + p0 * 656, p0, n, stream)
