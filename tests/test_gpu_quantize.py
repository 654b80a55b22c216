"""Quantise-on-append on the GPU against the oracle quantiser, byte for byte
(codes are integer decisions taken in the same IEEE fp32/fp16 steps)."""
import numpy as np
import pytest

from oracle.q8g64 import quantize_row
from synth.rng import f32_to_bf16_bits

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _need_gpu():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def test_append_quantize_matches_oracle():
    import torch
    from decode_attention_dsa_gb300 import abi
    from decode_attention_dsa_gb300.units import UnitSet
    rng = np.random.default_rng(7)
    U, L0, A, calls = 2, 10, 5, 14
    g = UnitSet(U, 8, L0 + A * calls + 4, mirror="host")
    g.init([L0] * U, abi.WARM_EMPTY)
    want = {u: [] for u in range(U)}
    for c in range(calls):
        lat = rng.standard_normal((U, A, 512)).astype(np.float32)
        lat *= rng.choice([1e-6, 1e-3, 1.0, 40.0, 3e4], size=(U, A, 8)).repeat(64, axis=2)
        lat[:, :, 64:128] *= (c % 3 == 0)                          # zero groups
        lat[:, :, 5] = -0.0
        latb = f32_to_bf16_bits(lat)
        rope = rng.integers(0, 65535, size=(U, A, 64)).astype(np.uint16)
        keys = rng.integers(0, 65535, size=(U, A, 64)).astype(np.uint16)
        for u in range(U):
            for a in range(A):
                want[u].append(quantize_row(latb[u, a], rope[u, a]))
        dev = lambda x: torch.from_numpy(x.view(np.int16)).cuda()
        abi.kv_append_quantize(g.units, U, A, dev(latb), dev(rope), dev(keys), g.dev_err)
        torch.cuda.synchronize()
        for u in range(U):
            got_keys = g.keys[u, L0 + c * A:L0 + (c + 1) * A].cpu().numpy().view(np.uint16)
            assert np.array_equal(got_keys, keys[u])
    abi.kv_flush(g.units, U, g.dev_err)
    torch.cuda.synchronize()
    assert g.check() == 0
    for u in range(U):
        got = g.get_mirror_rows(u, L0, A * calls)
        exp = np.stack(want[u])
        bad = np.nonzero((got != exp).any(axis=1))[0]
        assert bad.size == 0, f"unit {u}: rows {bad[:5]} differ"
    g.close()
