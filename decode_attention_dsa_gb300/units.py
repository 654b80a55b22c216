"""Device buffers of a set of units and the device array of ``dsa_unit``.

Host plumbing only (allocation, pointer marshalling, host views of the pinned
mirror). Every array is carved so that the per-unit pieces keep the 16-byte
alignment the kernels require.
"""
from __future__ import annotations

import ctypes

import numpy as np
import torch

from . import abi


class UnitSet:
    """U units with S hot slots and capacity ``lmax`` positions each.

    ``mirror='host'`` puts the RAM mirror in pinned, mapped host memory
    (offloaded, the pages' design); ``mirror='device'`` puts it in HBM (the
    fully resident run of the same kernels).
    """

    def __init__(self, U: int, S: int, lmax: int, mirror: str = "host", device="cuda", policy: str = "ring"):
        abi.load()
        self.U, self.S, self.lmax, self.mirror_kind = U, S, lmax, mirror
        self.policy = {"ring": abi.POLICY_RING, "clock": abi.POLICY_CLOCK}[policy]
        dev = torch.device(device)
        self.device = dev
        self.keys = torch.zeros((U, lmax, abi.IDX_DIM), dtype=torch.int16, device=dev)
        self.slots = torch.zeros((U, S, abi.ROW_BYTES), dtype=torch.uint8, device=dev)
        self.slot_pos = torch.full((U, S), -1, dtype=torch.int32, device=dev)
        self.pos_slot = torch.full((U, lmax), -1, dtype=torch.int32, device=dev)
        self.fill_round = torch.full((U, S), -1, dtype=torch.int32, device=dev)
        self.pin_epoch = torch.full((U, S), -1, dtype=torch.int32, device=dev)
        self.ring = torch.zeros((U, abi.RING_ROWS, abi.ROW_BYTES), dtype=torch.uint8, device=dev)
        self.state = torch.zeros((U, abi.ST_WORDS), dtype=torch.int64, device=dev)
        self.ref = torch.zeros((U, S), dtype=torch.uint8, device=dev)
        nbytes = U * lmax * abi.ROW_BYTES
        self._host_ptr = None
        if mirror == "host":
            h, d = abi.dsa_host_alloc(max(nbytes, 16))
            self._host_ptr = h
            self._mirror_dev = d
            buf = (ctypes.c_uint8 * max(nbytes, 16)).from_address(h)
            self.mirror_host = np.ctypeslib.as_array(buf)[:nbytes].reshape(U, lmax, abi.ROW_BYTES)
            self.mirror_dev_tensor = None
        elif mirror == "device":
            self.mirror_dev_tensor = torch.zeros((U, lmax, abi.ROW_BYTES), dtype=torch.uint8, device=dev)
            self._mirror_dev = self.mirror_dev_tensor.data_ptr()
            self.mirror_host = None
        else:
            raise ValueError(mirror)
        arr = (abi.DsaUnit * U)()
        for u in range(U):
            arr[u] = abi.DsaUnit(
                self.keys[u].data_ptr(), self.slots[u].data_ptr(), self.slot_pos[u].data_ptr(),
                self.pos_slot[u].data_ptr(), self.fill_round[u].data_ptr(),
                self.pin_epoch[u].data_ptr(), self.ring[u].data_ptr(),
                self._mirror_dev + u * lmax * abi.ROW_BYTES, self.state[u].data_ptr(), S, self.policy, lmax,
                self.ref[u].data_ptr())
        raw = np.frombuffer(bytes(arr), dtype=np.uint8).copy()
        self.units = torch.from_numpy(raw).to(dev)
        self.dev_err = torch.zeros(1, dtype=torch.int32, device=dev)

    # -------------------------------------------------------------- mirror
    def mirror_unit(self, u: int):
        """Host-visible view (numpy, host mirror) or tensor (device mirror) of unit u."""
        return self.mirror_host[u] if self.mirror_host is not None else self.mirror_dev_tensor[u]

    def set_mirror_rows(self, u: int, start: int, rows: np.ndarray) -> None:
        n = rows.shape[0]
        if self.mirror_host is not None:
            self.mirror_host[u, start:start + n] = rows
        else:
            self.mirror_dev_tensor[u, start:start + n] = torch.from_numpy(rows).to(self.device)

    def get_mirror_rows(self, u: int, start: int, n: int) -> np.ndarray:
        if self.mirror_host is not None:
            return np.array(self.mirror_host[u, start:start + n])
        return self.mirror_dev_tensor[u, start:start + n].cpu().numpy()

    def set_keys(self, u: int, start: int, keys_bits: np.ndarray) -> None:
        t = torch.from_numpy(np.ascontiguousarray(keys_bits, dtype=np.uint16).view(np.int16))
        self.keys[u, start:start + keys_bits.shape[0]] = t.to(self.device)

    def init(self, l0, warm: int, stream=None) -> None:
        l0t = torch.as_tensor(np.asarray(l0, dtype=np.int64).reshape(self.U), device=self.device)
        self._l0 = l0t
        abi.hc_init(self.units, self.U, warm, l0t, self.S, self.lmax, self.dev_err, stream)

    # ----------------------------------------------------------- snapshots
    def snapshot_stride(self) -> int:
        return abi.dsa_snapshot_bytes(self.S, self.lmax)

    def export_state(self, stream=None) -> dict:
        """Host snapshot of every unit: dsa_export into pinned, mapped host
        memory (slot map, bits, ring, keys, state words) plus a copy of the
        mirror. Call kv_flush first on the same stream; a unit that was not
        flushed is not exported (DSA_DEVERR_STATE)."""
        stride = self.snapshot_stride()
        h, d = abi.dsa_host_alloc(self.U * stride)
        try:
            abi.dsa_export(self.units, self.U, d, stride, self.S, self.lmax, self.dev_err, stream)
            torch.cuda.synchronize(self.device)
            buf = (ctypes.c_uint8 * (self.U * stride)).from_address(h)
            snap = np.array(np.ctypeslib.as_array(buf))
        finally:
            abi.dsa_host_free(h)
        mirror = (np.array(self.mirror_host) if self.mirror_host is not None
                  else self.mirror_dev_tensor.cpu().numpy())
        return {"snapshot": snap, "stride": stride, "mirror": mirror}

    def import_state(self, d: dict, stream=None) -> None:
        """Restore a snapshot from export_state into a unit set of the same
        shape: the mirror rows are put back, then dsa_restore rebuilds the
        cache state (and re-reads every slot's bytes from the mirror)."""
        if self.mirror_host is not None:
            self.mirror_host[...] = d["mirror"]
        else:
            self.mirror_dev_tensor.copy_(torch.from_numpy(d["mirror"]).to(self.device))
        snap = torch.from_numpy(d["snapshot"]).to(self.device)
        abi.dsa_restore(self.units, self.U, snap, d["stride"], self.S, self.lmax, self.dev_err, stream)
        torch.cuda.synchronize(self.device)

    def check(self) -> int:
        return int(self.dev_err.item())

    def subset(self, lo: int, hi: int) -> "UnitRange":
        """Units [lo, hi) as a unit set of their own, for a DecodePath that
        runs them apart from the others (for example two groups of sessions
        decoding on two streams). Same device buffers and error word."""
        return UnitRange(self, lo, hi)


    def close(self) -> None:
        if self._host_ptr is not None:
            torch.cuda.synchronize(self.device)
            self.mirror_host = None
            abi.dsa_host_free(self._host_ptr)
            self._host_ptr = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


class UnitRange:
    """Units [lo, hi) of a UnitSet: a device copy of their ``dsa_unit``
    descriptors (pointing at the parent's buffers), the parent's error word.
    Calls on different ranges touch disjoint units and may run concurrently;
    calls on one range follow the C ABI's ordering rules."""

    def __init__(self, parent: UnitSet, lo: int, hi: int):
        if not (0 <= lo < hi <= parent.U):
            raise ValueError(f"unit range [{lo}, {hi}) outside [0, {parent.U})")
        self.parent, self.lo, self.hi = parent, lo, hi
        self.U, self.S, self.lmax, self.device = hi - lo, parent.S, parent.lmax, parent.device
        self.dev_err = parent.dev_err
        raw = parent.units.view(-1, ctypes.sizeof(abi.DsaUnit))
        self.units = raw[lo:hi].contiguous().view(-1)

    def check(self) -> int:
        return self.parent.check()
