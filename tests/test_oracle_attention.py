"""Pins for oracle.attention: closed forms, invariances and an independent
high-precision (decimal) evaluation on tiny inputs."""
from decimal import Decimal, getcontext
from fractions import Fraction

import numpy as np

from oracle import attention, q8g64
from synth.rng import f32_to_bf16_bits, bf16_bits_to_f32


def _rows(rng, K, scale_bits=None):
    rows = np.zeros((K, 656), np.uint8)
    rows[:, :512] = rng.integers(-127, 128, size=(K, 512)).astype(np.int8).view(np.uint8)
    sc = (rng.integers(328, 1312, size=(K, 8)) * 2.0 ** -16).astype("<f2")
    rows[:, 512:528] = sc.view(np.uint8).reshape(K, 16)
    rope = f32_to_bf16_bits(rng.standard_normal((K, 64)).astype(np.float32))
    rows[:, 528:] = rope.astype("<u2").view(np.uint8).reshape(K, 128)
    return rows


def _q(rng, H):
    return (f32_to_bf16_bits(rng.standard_normal((H, 512)).astype(np.float32)),
            f32_to_bf16_bits(rng.standard_normal((H, 64)).astype(np.float32)))


SC = 1.0 / 24.0


def test_single_row_returns_that_row():
    rng = np.random.default_rng(0)
    rows = _rows(rng, 1)
    ql, qr = _q(rng, 4)
    out, lse = attention.mla_decode_attention(ql, qr, rows, np.ones(1, bool), SC)
    assert (out == q8g64.dequant_latent(rows)[0][None]).all()


def test_zero_query_gives_mean():
    rng = np.random.default_rng(1)
    rows = _rows(rng, 37)
    z = np.zeros((3, 512), np.uint16), np.zeros((3, 64), np.uint16)
    out, lse = attention.mla_decode_attention(z[0], z[1], rows, np.ones(37, bool), SC)
    want = q8g64.dequant_latent(rows).mean(axis=0)
    assert np.allclose(out, want[None], rtol=0, atol=1e-14)
    assert np.allclose(lse, np.log(37.0))


def test_dominant_logit_selects_row():
    rng = np.random.default_rng(2)
    rows = _rows(rng, 20)
    c = q8g64.dequant_latent(rows)
    ql = f32_to_bf16_bits((c[7] * 40.0).astype(np.float32))[None]  # aligned with row 7
    qr = np.zeros((1, 64), np.uint16)
    out, _ = attention.mla_decode_attention(ql, qr, rows, np.ones(20, bool), SC)
    assert np.abs(out[0] - c[7]).max() < 1e-6 * np.abs(c[7]).max()


def test_common_rope_is_a_shift_and_permutation_invariance():
    rng = np.random.default_rng(3)
    rows = _rows(rng, 50)
    rows[:, 528:] = rows[0, 528:]          # same RoPE part on every row
    ql, qr = _q(rng, 5)
    a, la = attention.mla_decode_attention(ql, qr, rows, np.ones(50, bool), SC)
    b, lb = attention.mla_decode_attention(ql, np.zeros_like(qr), rows, np.ones(50, bool), SC)
    assert np.allclose(a, b, rtol=0, atol=1e-13)
    perm = rng.permutation(50)
    c, lc = attention.mla_decode_attention(ql, qr, rows[perm], np.ones(50, bool), SC)
    assert np.allclose(a, c, rtol=0, atol=1e-13) and np.allclose(la, lc)


def test_padding_is_excluded():
    rng = np.random.default_rng(4)
    rows = _rows(rng, 30)
    ql, qr = _q(rng, 2)
    valid = np.ones(30, bool)
    valid[[3, 17, 29]] = False
    a, _ = attention.mla_decode_attention(ql, qr, rows, valid, SC)
    b, _ = attention.mla_decode_attention(ql, qr, rows[valid], np.ones(27, bool), SC)
    assert (a == b).all()
    e, le = attention.mla_decode_attention(ql, qr, rows, np.zeros(30, bool), SC)
    assert (e == 0).all() and np.isneginf(le).all()


def test_against_decimal_high_precision():
    """Exact rational logits, then exp/sums in 50-digit decimal arithmetic."""
    getcontext().prec = 50
    rng = np.random.default_rng(5)
    K, H = 4, 2
    rows = _rows(rng, K)
    ql, qr = _q(rng, H)
    out, lse = attention.mla_decode_attention(ql, qr, rows, np.ones(K, bool), SC)
    lat = rows[:, :512].view(np.int8).astype(int)
    sc = rows[:, 512:528].copy().view("<f2").astype(float)
    rope = bf16_bits_to_f32(rows[:, 528:].copy().view("<u2")).astype(float)
    qlf = bf16_bits_to_f32(ql).astype(float)
    qrf = bf16_bits_to_f32(qr).astype(float)
    cs = [[Fraction(int(lat[j, d])) * Fraction(sc[j, d // 64]) for d in range(512)] for j in range(K)]
    for h in range(H):
        logits = []
        for j in range(K):
            t = sum(Fraction(qlf[h, d]) * cs[j][d] for d in range(512))
            t += sum(Fraction(qrf[h, d]) * Fraction(rope[j, d]) for d in range(64))
            logits.append(t / 24)
        ex = [Decimal(l.numerator) / Decimal(l.denominator) for l in logits]
        ex = [x.exp() for x in ex]
        tot = sum(ex)
        for d in (0, 1, 100, 511):
            v = sum(e * Decimal(cs[j][d].numerator) / Decimal(cs[j][d].denominator)
                    for j, e in enumerate(ex)) / tot
            assert abs(float(v) - out[h, d]) <= 1e-13 * max(1.0, abs(float(v)))
        assert abs(float(tot.ln()) - lse[h]) < 1e-12
