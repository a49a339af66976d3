"""NVFP4 encodings for the oracle (test infrastructure only).

The Nunchaku/SVDQuant pages say the Blackwell build quantises both operands to
NVFP4 ("How Nunchaku four bit quantization actually works", aiflownews article;
same page, "Risks, limitations" and "Takeaways" sections) but never spell the
format out.  The reading used here is the standard one:

  * element codes are E2M1 (1 sign, 2 exponent, 1 mantissa bit), magnitudes
    {0, 0.5, 1, 1.5, 2, 3, 4, 6} for codes 0..7, sign in bit 3;
  * one unsigned E4M3 scale (bias 7, max 448, subnormal step 2^-9) per 16
    consecutive elements along the reduction dimension;
  * one float32 global scale per tensor.

Rounding (not fixed by the pages, taken from the layer spec): round to nearest,
ties to even code, saturating at the largest finite value.  A value whose IEEE
sign bit is set keeps sign bit 3 of its code even when its magnitude rounds to
zero (so -0.0 and -0.1 encode to 0x8).

Block quantiser Qz(v, s_g), each step a float32 IEEE operation:
    s_raw = amax(|v_blk|) / fl32(6 * s_g)
    s8    = E4M3(s_raw)
    if s8 == 0: all 16 codes are +0
    else:  d = fl32(E4M3value(s8) * s_g);  rcp = fl32(1 / d)
           code_i = E2M1(fl32(v_i * rcp))

Pins (tests/test_oracle_nvfp4.py): exhaustive tie midpoints and +-1 ulp, a
brute-force nearest-grid search, torch.float8_e4m3fn on in-range values, two
hand-worked blocks in tests/golden/, and the block invariants (reconstruction
error within half a grid step; the block maximum lands on code 6.0).  The global
scale is pinned to hand values (0x39C30C31 for amax = 1) and to the correctly
rounded quotient computed in exact rational arithmetic, including an amax where
two successive roundings (by 6, then by 448) would differ in the last bit.
"""
from __future__ import annotations

import numpy as np

E2M1_MAGNITUDES = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])
E4M3_MAX = 448.0
BLOCK = 16


def e2m1_encode(v) -> np.ndarray:
    """float32 values -> E2M1 codes (uint8 in 0..15), RNE, saturating."""
    v = np.asarray(v, dtype=np.float32)
    a = np.abs(v).astype(np.float64)
    # grid spacing of the binade a falls in: [0,2) -> 0.5, [2,4) -> 1, [4,inf) -> 2
    step = np.where(a < 2.0, 0.5, np.where(a < 4.0, 1.0, 2.0))
    m = np.minimum(np.rint(a / step) * step, 6.0)   # rint rounds half to even
    # magnitude -> code: 0,.5,1,1.5,2 -> 0..4 ; 3 -> 5 ; 4 -> 6 ; 6 -> 7
    mag = np.where(m <= 2.0, m * 2.0, np.where(m == 3.0, 5.0, np.where(m == 4.0, 6.0, 7.0)))
    sign = np.signbit(v).astype(np.uint8)
    return (mag.astype(np.uint8) | (sign << 3)).astype(np.uint8)


def e2m1_decode(c) -> np.ndarray:
    c = np.asarray(c, dtype=np.uint8)
    mag = E2M1_MAGNITUDES[c & 7]
    return np.where(c & 8, -mag, mag)


def e4m3_decode(b) -> np.ndarray:
    """E4M3 bit patterns -> float64 (0x7F/0xFF are NaN)."""
    b = np.asarray(b, dtype=np.uint8).astype(np.int64)
    s = np.where(b & 0x80, -1.0, 1.0)
    e = (b >> 3) & 0xF
    m = b & 7
    val = np.where(e == 0, m * 2.0 ** -9, (1.0 + m / 8.0) * np.exp2(e - 7.0))
    val = np.where((e == 15) & (m == 7), np.nan, val)
    return s * val


def e4m3_encode_nonneg(s) -> np.ndarray:
    """Non-negative float32 -> unsigned E4M3 bits, RNE, saturating to 448."""
    a = np.asarray(s, dtype=np.float32).astype(np.float64)
    if np.any(a < 0) or np.any(np.isnan(a)):
        raise ValueError("scales are non-negative and finite")
    a = np.minimum(a, E4M3_MAX)
    _, ex = np.frexp(a)                       # a = f * 2^ex, f in [0.5, 1)
    e = np.maximum(ex - 1, -6)                # binade exponent, clamped at min normal
    q = np.exp2(e - 3.0)                      # 3 mantissa bits
    r = np.rint(a / q) * q                    # exact scaling, half to even
    r = np.minimum(r, E4M3_MAX)
    out = np.zeros(a.shape, dtype=np.uint8)
    nz = r > 0
    sub = nz & (r < 2.0 ** -6)
    out[sub] = np.rint(r[sub] / 2.0 ** -9).astype(np.uint8)
    nrm = nz & ~sub
    _, ex2 = np.frexp(r[nrm])
    e2 = ex2 - 1
    mant = np.rint((r[nrm] / np.exp2(e2) - 1.0) * 8.0).astype(np.int64)
    out[nrm] = (((e2 + 7) << 3) | mant).astype(np.uint8)
    return out


def quantize_blocks(v, s_g):
    """Qz: rows of float32 values (K % 16 == 0) -> (codes uint8 rows x K, scales uint8 rows x K/16)."""
    v = np.asarray(v, dtype=np.float32)
    rows, K = v.shape
    if K % BLOCK:
        raise ValueError("K must be a multiple of 16")
    s_g = np.float32(s_g)
    blk = v.reshape(rows, K // BLOCK, BLOCK)
    amax = np.max(np.abs(blk), axis=2)                      # exact
    six_sg = np.float32(6.0) * s_g                           # fp32 product
    s_raw = (amax / six_sg).astype(np.float32)               # fp32 division
    s8 = e4m3_encode_nonneg(s_raw)
    d = (e4m3_decode(s8).astype(np.float32) * s_g).astype(np.float32)
    zero = s8 == 0
    d_safe = np.where(zero, np.float32(1.0), d).astype(np.float32)
    rcp = (np.float32(1.0) / d_safe).astype(np.float32)      # fp32 reciprocal
    q = (blk * rcp[:, :, None]).astype(np.float32)           # fp32 product
    codes = e2m1_encode(q)
    codes[zero] = 0
    return codes.reshape(rows, K), s8


def dequantize_blocks(codes, scales) -> np.ndarray:
    """codes (rows x K), scales (rows x K/16) -> float64 values without the global scale (exact)."""
    codes = np.asarray(codes)
    rows, K = codes.shape
    val = e2m1_decode(codes).reshape(rows, K // BLOCK, BLOCK)
    return (val * e4m3_decode(scales)[:, :, None]).reshape(rows, K)


def global_scale(amax) -> np.float32:
    """s_g = fl32(amax / (6 * 448)); 1.0 for an all-zero tensor."""
    amax = np.float32(amax)
    if amax == 0:
        return np.float32(1.0)
    return np.float32(amax / np.float32(6.0 * E4M3_MAX))
