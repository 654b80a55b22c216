"""The allocation-free variant of the score + Top-K entry point.

Some callers cannot allocate device memory (a host framework that owns every
allocation, a loop that must not stall on the allocator), so the library also
offers dsa_score_topk_noalloc, whose scratch is a fixed array built into the
library. These tests call it through the C ABI twice in a row and check that
both calls select exactly what the workspace-based dsa_score_topk selects and
what the oracle selects (indices are integers, so the comparison is exact);
that a call at exactly the size limit of the built-in array works; and that a
problem larger than the array is refused. The file is named to be collected
last.
"""
import numpy as np
import pytest

from oracle.indexer import score_topk
from synth import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _need_gpu():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def _setup(wl):
    import torch
    from decode_attention_dsa_gb300 import abi
    from decode_attention_dsa_gb300.step import DecodePath
    from decode_attention_dsa_gb300.units import UnitSet
    U = wl.U
    g = UnitSet(U, wl.S, wl.lmax, mirror="device")
    keys = [W.keys_bits(wl, u, np.arange(wl.L0)) for u in range(U)]
    for u in range(U):
        g.set_keys(u, 0, keys[u])
    g.init([wl.L0] * U, abi.WARM_EMPTY)
    path = DecodePath(g, wl.R, wl.K, wl.H, wl.A, wl.scale())
    return torch, abi, g, path, keys


def _queries(torch, wl, step):
    U = wl.U
    q = np.stack([W.step_q_idx(wl, u, step)[0] for u in range(U)])
    w = np.stack([W.step_q_idx(wl, u, step)[1] for u in range(U)])
    return q, w, torch.from_numpy(q.view(np.int16)).cuda(), torch.from_numpy(w).cuda()


def test_noalloc_matches_workspace_entry_point_and_oracle_on_two_calls():
    wl = W.WORKLOADS[2].with_(name="noalloc", layers=3, L0=20000, K=512, S=1024, steps=4)
    torch, abi, g, path, keys = _setup(wl)
    U, R = wl.U, wl.R
    got = torch.empty_like(path.topk)
    for step in range(2):
        q, w, qt, wt = _queries(torch, wl, step)
        path.score_topk(qt, wt)
        got.fill_(-7)
        abi.dsa_score_topk_noalloc(g.units, U, R, wl.K, qt, wt, got, path.max_len, g.dev_err)
        torch.cuda.synchronize()
        assert torch.equal(got, path.topk), f"call {step}: selections differ from dsa_score_topk"
        if step == 0:
            for u in range(U):
                _, want = score_topk(keys[u], q[u], w[u], wl.K)
                assert np.array_equal(got[u].cpu().numpy(), want), f"unit {u}: differs from the oracle"
    assert g.check() == 0
    with pytest.raises(abi.DsaError) as e:
        abi.dsa_score_topk_noalloc(g.units, U, R, wl.K, qt, wt, got, 70000, g.dev_err)
    assert e.value.status == abi.DSA_ERR_SCRATCH_LIMIT
    g.close()


def test_noalloc_at_the_size_limit():
    """U x R = 16 (unit, row) pairs and max_len = 65,536 use the whole array."""
    wl = W.WORKLOADS[2].with_(name="noalloc-limit", sessions=1, layers=4, L0=65536 - 4, K=2048, S=64, steps=1)
    torch, abi, g, path, keys = _setup(wl)
    assert wl.U * wl.R == 16
    got = torch.empty_like(path.topk)
    for step in range(2):
        q, w, qt, wt = _queries(torch, wl, step)
        got.fill_(-7)
        abi.dsa_score_topk_noalloc(g.units, wl.U, wl.R, wl.K, qt, wt, got, 65536, g.dev_err)
        torch.cuda.synchronize()
        u = 3 if step else 0
        _, want = score_topk(keys[u], q[u], w[u], wl.K)
        assert np.array_equal(got[u].cpu().numpy(), want), f"call {step}: unit {u} differs from the oracle"
    assert g.check() == 0
    g.close()
