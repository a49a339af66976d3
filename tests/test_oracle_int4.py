"""Pins for the oracle's INT4 group quantiser (CPU only): hand-worked groups, a brute-force
nearest-integer search with ties to even, the reconstruction bound and the group maximum."""
import os
from fractions import Fraction

import numpy as np
import pytest

from oracle import int4

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "int4_groups.txt")


def _golden():
    rows = []
    for line in open(GOLDEN):
        if not line.strip() or line.startswith("#"):
            continue
        name, vals, sc, codes = [f.strip() for f in line.split("|")]
        v = np.zeros(64, np.float32)
        for item in vals.split():
            i, x = item.split(":")
            v[int(i)] = np.float32(float(x))
        c = np.full(64, 8, np.uint8)
        for item in codes.split():
            i, x = item.split(":")
            c[int(i)] = int(x, 16)
        rows.append((name, v, int(sc, 16), c))
    return rows


@pytest.mark.parametrize("row", _golden(), ids=lambda r: r[0])
def test_hand_worked_groups(row):
    _, v, scale_bits, codes = row
    c, s = int4.quantize_groups(v[None, :])
    assert int(np.float32(s[0, 0]).view(np.uint32)) == scale_bits
    assert np.array_equal(c[0], codes)


def _nearest_even(t):
    """Nearest integer to the float t by exact rational comparison, ties to the even one,
    clamped to [-7, 7]."""
    ft = Fraction(float(t))
    lo = ft.numerator // ft.denominator
    d = ft - lo
    if d > Fraction(1, 2) or (d == Fraction(1, 2) and lo % 2):
        lo += 1
    return max(-7, min(7, lo))


def test_codes_against_bruteforce_nearest():
    rng = np.random.default_rng(7)
    v = (rng.standard_normal((40, 256)) * np.exp2(rng.uniform(-10, 10, (40, 1)))).astype(np.float32)
    v[3, :64] = 0
    v[5, 64:128] = np.float32(2.5) * np.sign(rng.standard_normal(64)).astype(np.float32)   # many ties
    c, s = int4.quantize_groups(v)
    for r in range(v.shape[0]):
        for g in range(4):
            sg = s[r, g]
            if sg == 0:
                assert np.all(c[r, 64 * g:64 * g + 64] == 8)
                continue
            rcp = np.float32(np.float32(1.0) / sg)
            for k in range(64 * g, 64 * g + 64):
                t = np.float32(v[r, k] * rcp)
                assert int(c[r, k]) - 8 == _nearest_even(t), (r, k)


def test_scale_and_reconstruction_bound():
    rng = np.random.default_rng(8)
    v = (rng.standard_normal((64, 512)) * np.exp2(rng.uniform(-6, 6, (64, 1)))).astype(np.float32)
    c, s = int4.quantize_groups(v)
    blk = v.reshape(64, 8, 64).astype(np.float64)
    amax = np.max(np.abs(blk), axis=2)
    # s = fl32(amax / 7), one rounding
    assert np.all(s == (amax.astype(np.float32) / np.float32(7)).astype(np.float32))
    deq = int4.dequantize_groups(c, s).reshape(64, 8, 64)
    assert np.all(np.abs(deq - blk) <= 0.5 * s[:, :, None] * (1 + 1e-6))
    # the group's largest magnitude lands on q = +-7
    q = c.reshape(64, 8, 64).astype(np.int64) - 8
    idx = np.argmax(np.abs(blk), axis=2)
    top = np.take_along_axis(q, idx[:, :, None], axis=2)[:, :, 0]
    assert np.all(np.abs(top) == 7)
    assert np.all(np.abs(q) <= 7)
