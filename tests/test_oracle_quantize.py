"""Pins for oracle.q8g64.quantize_row: a hand-derived example, the error bound
of symmetric rounding, idempotence, and dequantisation consistency."""
import numpy as np

from oracle import q8g64
from synth.rng import f32_to_bf16_bits


def _bits(a):
    return f32_to_bf16_bits(np.asarray(a, dtype=np.float32))


def test_worked_example(golden):
    lat = np.zeros(512, np.float32)
    exp_s, exp_q = {}, {}
    for ln in golden("q8g64_quantize_example.txt"):
        k, a, b = ln.split()
        if k == "value":
            lat[int(a)] = float(b)
        elif k == "expect_scale":
            exp_s[int(a)] = int(b, 16)
        elif k == "expect_q":
            exp_q[int(a)] = int(b)
    row = q8g64.quantize_row(_bits(lat), np.zeros(64, np.uint16))
    sc = row[512:528].copy().view("<u2")
    q = row[:512].view(np.int8)
    for g, v in exp_s.items():
        assert sc[g] == v, g
    for d, v in exp_q.items():
        assert q[d] == v, d


def test_error_bound_and_idempotence():
    rng = np.random.default_rng(0)
    for _ in range(200):
        lat = (rng.standard_normal(512) * rng.choice([1e-3, 1.0, 30.0])).astype(np.float32)
        lat[rng.integers(0, 512, 20)] = 0
        bits = _bits(lat)
        x = (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
        rope = rng.integers(0, 65535, 64).astype(np.uint16)
        row = q8g64.quantize_row(bits, rope)
        c = q8g64.dequant_latent(row[None])[0]
        s = q8g64.group_scales(row[None])[0]
        for g in range(8):
            xs = x[64 * g:64 * g + 64]
            cs = c[64 * g:64 * g + 64]
            amax = np.abs(xs).max()
            # symmetric rounding: half a step, plus the fp16 rounding of the scale
            assert np.abs(xs - cs).max() <= s[g] / 2 + amax * 2.0 ** -10 + 1e-30
            assert np.abs(row[:512].view(np.int8)[64 * g:64 * g + 64]).max() == (127 if s[g] > 0 else 0)
        assert np.array_equal(row[528:].view("<u2"), rope)
        # quantising the dequantised row (exact in bf16? only if c is bf16) is idempotent
        cb = f32_to_bf16_bits(c.astype(np.float32))
        if np.array_equal((cb.astype(np.uint32) << 16).view(np.float32).astype(np.float64), c):
            assert np.array_equal(q8g64.quantize_row(cb, rope), row)


def test_zero_group_and_signs():
    lat = np.zeros(512, np.float32)
    lat[64:128] = -np.arange(64) / 8.0
    row = q8g64.quantize_row(_bits(lat), np.zeros(64, np.uint16))
    assert (row[:64] == 0).all() and row[512:514].view("<u2")[0] == 0
    q = row[64:128].view(np.int8)
    assert q[0] == 0 and (q[1:] < 0).all() and q[63] == -127
