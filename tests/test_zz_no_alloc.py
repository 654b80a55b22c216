"""The allocation-free variant of the score + Top-K entry point.

Some callers cannot allocate device memory (a host framework that owns every
allocation, a loop that must not stall on the allocator), so the library also
offers dsa_score_topk_noalloc, whose scratch is a fixed array built into the
library. This test calls it through the C ABI twice in a row and checks that
both calls select exactly what the workspace-based dsa_score_topk selects
(indices are integers, so the comparison is exact), and that a problem larger
than the fixed scratch is refused. The file is named to be collected last.
"""
import numpy as np
import pytest

from synth import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _need_gpu():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def test_noalloc_matches_workspace_entry_point_on_two_calls():
    import torch
    from decode_attention_dsa_gb300 import abi
    from decode_attention_dsa_gb300.step import DecodePath
    from decode_attention_dsa_gb300.units import UnitSet

    wl = W.WORKLOADS[2].with_(name="noalloc", layers=3, L0=20000, K=512, S=1024, steps=4)
    U, R = wl.U, wl.R
    g = UnitSet(U, wl.S, wl.lmax, mirror="device")
    for u in range(U):
        g.set_keys(u, 0, W.keys_bits(wl, u, np.arange(wl.L0)))
    g.init([wl.L0] * U, abi.WARM_EMPTY)
    path = DecodePath(g, R, wl.K, wl.H, wl.A, wl.scale())
    got = torch.empty_like(path.topk)
    for step in range(2):
        q = np.stack([W.step_q_idx(wl, u, step)[0] for u in range(U)])
        w = np.stack([W.step_q_idx(wl, u, step)[1] for u in range(U)])
        qt = torch.from_numpy(q.view(np.int16)).cuda()
        wt = torch.from_numpy(w).cuda()
        path.score_topk(qt, wt)
        got.fill_(-7)
        abi.dsa_score_topk_noalloc(g.units, U, R, wl.K, qt, wt, got, path.max_len, g.dev_err)
        torch.cuda.synchronize()
        assert torch.equal(got, path.topk), f"call {step}: selections differ"
    assert g.check() == 0
    with pytest.raises(abi.DsaError) as e:
        abi.dsa_score_topk_noalloc(g.units, U, R, wl.K, qt, wt, got, 70000, g.dev_err)
    assert e.value.status == abi.DSA_ERR_SCRATCH_LIMIT
    g.close()
