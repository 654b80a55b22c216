"""The GPU input generator writes exactly the bytes of the numpy generator
(the definition), so large workloads can be generated on the device."""
import numpy as np
import pytest

from synth import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _need_gpu():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


@pytest.mark.parametrize("cid", [0, 2, 3, 4])
def test_gpu_generator_matches_numpy(cid):
    import torch
    from synth import gpu as sg
    sg.build()
    wl = W.WORKLOADS[cid].with_(steps=3)
    u = wl.U - 1
    pos = np.array([0, 1, 17, wl.L0 - wl.S, wl.L0 - 1, wl.L0 + 2])
    for p0 in (int(pos[0]), int(pos[2]), int(pos[4])):
        k = torch.empty((5, 64), dtype=torch.int16, device="cuda")
        sg.keys(wl, u, k.data_ptr(), p0, 5)
        r = torch.empty((5, 656), dtype=torch.uint8, device="cuda")
        sg.rows(wl, u, r.data_ptr(), p0, 5)
        torch.cuda.synchronize()
        assert np.array_equal(k.cpu().numpy().view(np.uint16), W.keys_bits(wl, u, np.arange(p0, p0 + 5)))
        assert np.array_equal(r.cpu().numpy(), W.rows_bytes(wl, u, np.arange(p0, p0 + 5)))
    inp = sg.step_inputs(wl, 1, 2)
    torch.cuda.synchronize()
    for k in range(2):
        x = W.step_inputs(wl, u, 1 + k)
        assert np.array_equal(inp["q_idx"][k, u].cpu().numpy().view(np.uint16), x.q_idx)
        assert np.array_equal(inp["w"][k, u].cpu().numpy(), x.w)
        assert np.array_equal(inp["q_lat"][k, u].cpu().numpy().view(np.uint16), x.q_lat)
        assert np.array_equal(inp["q_rope"][k, u].cpu().numpy().view(np.uint16), x.q_rope)
        assert np.array_equal(inp["new_rows"][k, u].cpu().numpy(), x.new_rows)
        assert np.array_equal(inp["new_keys"][k, u].cpu().numpy().view(np.uint16), x.new_keys)
