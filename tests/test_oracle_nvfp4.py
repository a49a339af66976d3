"""Pins for the oracle's NVFP4 encodings (CPU only).

Each check ties oracle.nvfp4 to something other than itself: hand-worked blocks,
a brute-force nearest-grid search, torch's own float8_e4m3fn conversion, and
invariants of the block quantiser.
"""
import os

import numpy as np
import pytest
import torch

from oracle import nvfp4

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "nvfp4_blocks.txt")


def _grid_nearest_e2m1(v):
    """Brute force: nearest of the 8 magnitudes, ties to the even code, sign from the IEEE bit."""
    out = []
    for x in np.asarray(v, np.float32):
        a = abs(float(x))
        d = [abs(a - m) for m in nvfp4.E2M1_MAGNITUDES]
        best = min(d)
        cands = [i for i, di in enumerate(d) if di == best]
        code = cands[0] if len(cands) == 1 else [c for c in cands if c % 2 == 0][0]
        if a > 6.0:
            code = 7
        out.append(code | (8 if np.signbit(x) else 0))
    return np.array(out, np.uint8)


def test_e2m1_grid_roundtrip():
    codes = np.arange(16, dtype=np.uint8)
    vals = nvfp4.e2m1_decode(codes)
    assert list(vals[:8]) == [0, 0.5, 1, 1.5, 2, 3, 4, 6]
    assert list(vals[8:]) == [-0.0, -0.5, -1, -1.5, -2, -3, -4, -6]
    assert np.array_equal(nvfp4.e2m1_encode(vals.astype(np.float32)), codes)


def test_e2m1_ties_go_to_even_code():
    mids = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0], np.float32)
    want = np.array([0, 2, 2, 4, 4, 6, 6], np.uint8)
    assert np.array_equal(nvfp4.e2m1_encode(mids), want)
    assert np.array_equal(nvfp4.e2m1_encode(-mids), want | 8)


def test_e2m1_midpoints_plus_minus_ulp_and_bruteforce():
    mids = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, 6.0], np.float32)
    up = np.nextafter(mids, np.float32(np.inf))
    dn = np.nextafter(mids, np.float32(0))
    rng = np.random.default_rng(1)
    rand = (rng.standard_normal(20000) * 3).astype(np.float32)
    v = np.concatenate([mids, up, dn, -mids, -up, -dn, rand, np.float32([0.0, -0.0, 7.0, 1e30, -1e-30])])
    assert np.array_equal(nvfp4.e2m1_encode(v), _grid_nearest_e2m1(v))


def test_e2m1_negative_zero_keeps_sign():
    assert nvfp4.e2m1_encode(np.float32([-0.0]))[0] == 8
    assert nvfp4.e2m1_encode(np.float32([-0.1]))[0] == 8
    assert nvfp4.e2m1_encode(np.float32([0.1]))[0] == 0


def test_e4m3_matches_torch_in_range():
    rng = np.random.default_rng(2)
    v = np.concatenate([
        np.exp2(rng.uniform(-12, np.log2(448), 200000)),
        np.arange(0, 256, dtype=np.float64) * 2.0 ** -9,       # subnormal grid and midpoints
        (np.arange(0, 512) + 0.5) * 2.0 ** -10,
        [448.0, 447.9, 2.0 ** -6, 2.0 ** -9, 2.0 ** -10, 0.0],
    ]).astype(np.float32)
    v = v[v <= 448]
    ours = nvfp4.e4m3_encode_nonneg(v)
    theirs = torch.from_numpy(v).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(ours, theirs)


def test_e4m3_saturates_and_decodes():
    assert nvfp4.e4m3_encode_nonneg(np.float32([1000.0, 464.0, 449.0]))[0] == 0x7E
    assert nvfp4.e4m3_decode(np.uint8([0x7E]))[0] == 448.0
    assert nvfp4.e4m3_decode(np.uint8([0x01]))[0] == 2.0 ** -9
    assert nvfp4.e4m3_decode(np.uint8([0x08]))[0] == 2.0 ** -6
    allc = np.arange(0x7F, dtype=np.uint8)            # every finite non-negative code
    assert np.array_equal(nvfp4.e4m3_encode_nonneg(nvfp4.e4m3_decode(allc).astype(np.float32)), allc)


def _golden():
    rows = []
    for line in open(GOLDEN):
        if not line.strip() or line.startswith("#"):
            continue
        name, sg, vals, sc, codes = [f.strip() for f in line.split("|")]
        rows.append((name, np.float32(sg), np.float32([float(x) for x in vals.split()]),
                     int(sc, 16), np.uint8([int(c, 16) for c in codes.split()])))
    return rows


@pytest.mark.parametrize("row", _golden(), ids=lambda r: r[0])
def test_hand_worked_blocks(row):
    _, sg, vals, scale, codes = row
    c, s = nvfp4.quantize_blocks(vals[None, :], sg)
    assert s[0, 0] == scale
    assert np.array_equal(c[0], codes)


def test_block_invariants():
    rng = np.random.default_rng(3)
    v = (rng.standard_normal((256, 512)) * np.exp2(rng.uniform(-8, 8, (256, 1)))).astype(np.float32)
    v[0, :16] = 0
    sg = nvfp4.global_scale(np.max(np.abs(v)))
    codes, scales = nvfp4.quantize_blocks(v, sg)
    d = nvfp4.e4m3_decode(scales) * np.float64(sg)
    blk = v.reshape(256, 32, 16).astype(np.float64)
    deq = nvfp4.dequantize_blocks(codes, scales).reshape(256, 32, 16) * np.float64(sg)
    # reconstruction error <= half the local grid step (step <= 2 d), except saturation
    q = np.abs(blk) / np.where(d > 0, d, 1)[:, :, None]
    step = np.where(q < 2, 0.5, np.where(q < 4, 1.0, 2.0))
    sat = q > 6.0
    err = np.abs(deq - blk)
    bound = 0.5 * step * d[:, :, None] * (1 + 1e-6) + 1e-300
    assert np.all((err <= bound) | sat)
    # with a normal (non-subnormal) block scale, the block maximum maps to code 6.0
    mag = (codes.reshape(256, 32, 16) & 7).max(axis=2)
    normal = (scales >> 3) > 0
    assert np.all(mag[normal] == 7)
    assert scales[0, 0] == 0 and np.all(codes[0, :16] == 0)


# ------------------------------------------------------------------ global scale
def _f32_nearest(q):
    """The float32 nearest to a positive rational q, ties to even, in exact integer
    arithmetic (normal range): independent of numpy's float32 division."""
    from fractions import Fraction
    e = q.numerator.bit_length() - q.denominator.bit_length()
    if Fraction(2) ** e > q:
        e -= 1
    if Fraction(2) ** (e + 1) <= q:
        e += 1
    s = q / Fraction(2) ** (e - 23)                 # in [2^23, 2^24)
    n, rem = divmod(s.numerator, s.denominator)
    if 2 * rem > s.denominator or (2 * rem == s.denominator and n % 2):
        n += 1
    return n * 2.0 ** (e - 23)


def _bits(x):
    return int(np.float32(x).view(np.uint32))


def test_global_scale_hand_values():
    """s_g = fl32(amax / 2688) with 2688 = 6 * 448 (the largest E2M1 magnitude times the
    largest E4M3 scale), one rounding; 1.0 for an all-zero tensor."""
    assert nvfp4.global_scale(2688.0) == np.float32(1.0)
    assert nvfp4.global_scale(0.0) == np.float32(1.0)
    # fl32(1 / 2688) written out: 0x39C30C31
    assert _bits(nvfp4.global_scale(1.0)) == 0x39C30C31
    assert _bits(nvfp4.global_scale(5376.0)) == _bits(2.0)


def test_global_scale_is_one_rounding():
    """amax = 64.0592041015625 (0x42801E50): one correctly rounded quotient gives 0x3CC33A62,
    while dividing by 6 and then by 448 (two roundings) gives 0x3CC33A61.  The expected bits
    come from exact rational arithmetic."""
    from fractions import Fraction
    a = np.uint32(0x42801E50).view(np.float32)
    assert _bits(nvfp4.global_scale(a)) == 0x3CC33A62
    two = np.float32(np.float32(a / np.float32(6)) / np.float32(448))
    assert _bits(two) == 0x3CC33A61                  # the slip this pin catches
    rng = np.random.default_rng(11)
    for v in rng.uniform(1e-3, 1e4, 2000).astype(np.float32):
        assert _bits(nvfp4.global_scale(v)) == _bits(_f32_nearest(Fraction(float(v)) / 2688))
