"""The C-ABI library (no GPU needed): it loads, exports every function that
include/dsa_decode.h declares, and its host-side checks reject bad arguments
before any CUDA call."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "dsa_decode.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?[a-z_0-9]+\s*\**\s+\**([a-z_0-9]+)\s*\(", text, flags=re.M)
    return [n for n in names if n not in ("if", "while")]


@pytest.fixture(scope="module")
def lib():
    from decode_attention_dsa_gb300 import abi, build
    build.build()
    return abi


def test_header_declares_the_boundary():
    names = set(declared_functions())
    for n in ("dsa_score_topk", "hot_gather", "mla_decode_attn", "kv_append_writeback", "kv_flush",
              "hc_init", "dsa_host_alloc", "dsa_host_free", "dsa_check"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    so = ctypes.CDLL(lib.LIB_PATH)
    for n in declared_functions():
        assert hasattr(so, n), n
    assert set(declared_functions()) <= set(lib.SIGNATURES)


def test_housekeeping(lib):
    assert lib.dsa_abi_version() == 2
    assert lib.dsa_check(0) == 0
    assert lib.dsa_check(0x4) == lib.DSA_ERR_DEVICE_CHECK
    assert "workspace" in lib.status_string(lib.DSA_ERR_WS)


def test_workspace_sizes(lib):
    assert lib.dsa_score_topk_workspace(0, 1, 10) == 0
    a = lib.dsa_score_topk_workspace(4, 1, 51047)
    b = lib.dsa_score_topk_workspace(4, 1, 100000)
    assert 0 < a < b and a % 256 == 0
    assert lib.hot_gather_workspace(1, 4, 2048) > lib.hot_gather_workspace(1, 1, 2048) > 0
    assert lib.mla_decode_attn_workspace(1, 1, 64, 2048) > 0


def _raw(lib, fn, *args):
    return getattr(lib.load(), fn)(*args)


def test_host_side_validation(lib):
    L = lib.load()
    fake = 0x1000   # never dereferenced: every call below fails validation first
    assert L.dsa_score_topk(None, 1, 1, 8, fake, fake, fake, 10, fake, 1 << 20, None, None) == lib.DSA_ERR_ARG
    assert L.dsa_score_topk(fake, 1, 1, 5000, fake, fake, fake, 10, fake, 1 << 20, None, None) == lib.DSA_ERR_SHAPE
    assert L.dsa_score_topk(fake, 1, 9, 8, fake, fake, fake, 10, fake, 1 << 20, None, None) == lib.DSA_ERR_ARG
    assert L.dsa_score_topk(fake, 1, 1, 8, fake, fake, fake, 10, fake, 16, None, None) == lib.DSA_ERR_WS
    assert L.hot_gather(fake, 1, 1, 8, 0, None, fake, fake, fake, fake, 1 << 20, None, None) == lib.DSA_ERR_ARG
    assert L.hot_gather(fake, 1, 1, 0, 0, fake, fake, fake, fake, fake, 1 << 20, None, None) == lib.DSA_ERR_SHAPE
    assert L.hot_gather(fake, 1, 1, 8, 0, fake, fake, fake, fake, None, 0, None, None) == lib.DSA_ERR_WS
    assert L.mla_decode_attn(1, 1, 24, 8, fake, fake, fake, fake, 0.04, fake, None, fake, 1 << 30, None, None) == lib.DSA_ERR_SHAPE
    assert L.mla_decode_attn(1, 1, 64, 8, fake, fake, fake, fake, -1.0, fake, None, fake, 1 << 30, None, None) == lib.DSA_ERR_ARG
    assert L.mla_decode_attn(1, 1, 64, 4096, fake, fake, fake, fake, 0.04, fake, None, None, 0, None, None) == lib.DSA_ERR_SHAPE
    assert L.mla_decode_attn(1, 1, 64, 64, fake, fake, fake, fake, 0.04, fake, None, None, 0, None, None) == lib.DSA_ERR_WS
    assert L.mla_decode_attn(1, 1, 128, 64, fake, fake, fake, fake, 0.04, fake, None, None, 0, None, None) == lib.DSA_ERR_SHAPE
    assert L.kv_append_writeback(fake, 1, 0, fake, fake, None, None) == lib.DSA_ERR_ARG
    assert L.kv_append_writeback(fake, 1, 65, fake, fake, None, None) == lib.DSA_ERR_ARG
    assert L.kv_flush(None, 1, None, None) == lib.DSA_ERR_ARG
    assert L.hc_init(fake, 1, 7, fake, 4, 10, None, None) == lib.DSA_ERR_ARG
    assert L.dsa_wait_selftest(100, 0, None, None) == lib.DSA_ERR_ARG
    sb = lib.dsa_snapshot_bytes(64, 1000)
    assert sb % 16 == 0 and sb > 1000 * 128 and lib.dsa_snapshot_bytes(0, 10) == 0
    assert L.dsa_export(fake, 1, fake, sb - 16, 64, 1000, None, None) == lib.DSA_ERR_ARG     # stride too small
    assert L.dsa_export(fake, 1, fake + 8, sb, 64, 1000, None, None) == lib.DSA_ERR_ARG      # misaligned
    assert L.dsa_restore(None, 1, fake, sb, 64, 1000, None, None) == lib.DSA_ERR_ARG
    assert L.kv_restore_full(fake, 1, fake + 4, 100, None, None) == lib.DSA_ERR_ARG
    assert L.kv_restore_full(fake, 1, fake, 0, None, None) == lib.DSA_ERR_ARG
    assert L.dsa_wait_selftest(-1, 0, fake, None) == lib.DSA_ERR_ARG
    # attention: K beyond 2048 or H off the 16-grid are refused before any launch
    for K in (0, 2049, 4096):
        assert L.mla_decode_attn(1, 1, 64, K, fake, fake, fake, fake, 0.04, fake, None, fake, 1 << 30,
                                 None, None) == lib.DSA_ERR_SHAPE
        assert L.hot_gather_attn(fake, 1, 1, K, 64, 0, fake, fake, fake, 0.04, fake, fake, fake, None,
                                 fake, 1 << 30, None, None) == lib.DSA_ERR_SHAPE
    # the two halves of dsa_score_topk check the same arguments
    assert L.dsa_score(fake, 1, 1, 8, None, fake, 10, fake, 1 << 20, None, None) == lib.DSA_ERR_ARG
    assert L.dsa_score(fake, 1, 1, 5000, fake, fake, 10, fake, 1 << 20, None, None) == lib.DSA_ERR_SHAPE
    assert L.dsa_score(fake, 1, 1, 8, fake, fake, 10, fake, 16, None, None) == lib.DSA_ERR_WS
    assert L.dsa_score(fake, 1, 1, 8, fake + 8, fake, 10, fake, 1 << 24, None, None) == lib.DSA_ERR_ARG
    assert L.dsa_topk_select(fake, 1, 1, 8, None, 10, fake, 1 << 20, None, None) == lib.DSA_ERR_ARG
    assert L.dsa_topk_select(fake, 1, 9, 8, fake, 10, fake, 1 << 20, None, None) == lib.DSA_ERR_ARG
    assert L.dsa_topk_select(fake, 1, 1, 8, fake, 10, fake + 4, 1 << 24, None, None) == lib.DSA_ERR_ARG
    assert L.dsa_touch_mirror(None, 1, 10, None) == lib.DSA_ERR_ARG
    assert L.dsa_touch_mirror(fake, 0, 10, None) == lib.DSA_ERR_ARG
    # SM partitions: argument checks come before any driver call
    p1, p2 = ctypes.c_void_p(), ctypes.c_void_p()
    assert L.dsa_partition_split(0, ctypes.byref(p1), ctypes.byref(p2)) == lib.DSA_ERR_ARG
    assert L.dsa_partition_split(8, None, None) == lib.DSA_ERR_ARG
    assert L.dsa_partition_stream(None, ctypes.byref(p1)) == lib.DSA_ERR_ARG
    assert L.dsa_partition_destroy(None) == lib.DSA_ERR_ARG
    assert L.dsa_partition_sms(None) == 0
    h, d = ctypes.c_void_p(), ctypes.c_void_p()
    assert L.dsa_host_alloc(None, ctypes.byref(d), 16) == lib.DSA_ERR_ARG
    assert L.dsa_host_alloc(ctypes.byref(h), ctypes.byref(d), 0) == lib.DSA_ERR_ARG
    assert L.dsa_host_free(None) == lib.DSA_ERR_ARG
