"""Pins for oracle.q8g64: the printed capacity table and a hand-derived row."""
from fractions import Fraction

import numpy as np

from oracle import q8g64


def test_capacity_table_reproduces_from_row_size(golden):
    lines = golden("capacity_table.txt")
    assert lines[0] == "row_bytes 656"
    assert q8g64.ROW_BYTES == 656
    # the row is the sum of its parts
    assert q8g64.LAT_DIM * 1 + q8g64.N_GROUPS * 2 + q8g64.ROPE_DIM * 2 == 656
    for ln in lines[1:]:
        rows, layers, copies, sessions, unit, value = ln.split()
        b = int(rows) * int(layers) * int(copies) * int(sessions) * q8g64.ROW_BYTES
        div = {"MiB": 2 ** 20, "GiB": 2 ** 30}[unit]
        printed = float(value)
        decimals = len(value.split(".")[1]) if "." in value else 0
        assert round(b / div, decimals) == printed, ln


def _build_row(lines):
    row = np.zeros(656, dtype=np.uint8)
    lat = np.zeros(512, dtype=np.int8)
    scales = np.full(8, 0x3C00, dtype="<u2")
    rope = np.zeros(64, dtype="<u2")
    exp_c, exp_r = {}, {}
    for ln in lines:
        k, a, b = ln.split()
        if k == "latent":
            lat[int(a)] = int(b)
        elif k == "scale":
            scales[int(a)] = int(b, 16)
        elif k == "rope":
            rope[int(a)] = int(b, 16)
        elif k == "expect_c":
            exp_c[int(a)] = Fraction(b)
        elif k == "expect_rope":
            exp_r[int(a)] = Fraction(b)
    row[:512] = lat.view(np.uint8)
    row[512:528] = scales.view(np.uint8)
    row[528:] = rope.view(np.uint8)
    return row, exp_c, exp_r


def test_worked_example(golden):
    row, exp_c, exp_r = _build_row(golden("q8g64_worked_example.txt"))
    c = q8g64.dequant_latent(row[None])[0]
    rho = q8g64.rope_values(row[None])[0]
    for d, v in exp_c.items():
        assert Fraction(c[d]) == v, d
    for d, v in exp_r.items():
        assert Fraction(rho[d]) == v, d


def test_group_boundaries_and_exactness():
    rng = np.random.default_rng(5)
    rows = rng.integers(0, 256, size=(7, 656), dtype=np.uint8)
    sc = rng.integers(0x1000, 0x5000, size=(7, 8)).astype("<u2")  # finite fp16 scales
    rows[:, 512:528] = sc.view(np.uint8).reshape(7, 16)
    c = q8g64.dequant_latent(rows)
    lat = rows[:, :512].view(np.int8).astype(np.int64)
    for i in range(7):
        for d in (0, 63, 64, 127, 128, 511):
            s = Fraction(float(np.array([sc[i, d // 64]], dtype="<u2").view("<f2")[0]))
            assert Fraction(c[i, d]) == lat[i, d] * s
