"""INT4 encoding of SVDQuant's INT4 variant, for the oracle (test infrastructure only).

The pages say SVDQuant supports both INT4 and FP4, and that Nunchaku ships fused kernels for
both, using the INT4 paths on hardware older than Blackwell ("What SVDQuant actually does" and
"How Nunchaku four bit quantization actually works", aiflownews article).  They give no group
size or scale format for INT4.  The reading used here, the plainest symmetric group quantiser:

  * element codes are signed integers q in [-7, 7] (the grid is kept symmetric: -8 is unused);
  * one float32 scale per 64 consecutive elements along the reduction dimension K (per row and
    group), s = fl32(amax / 7);
  * q = clamp(rint(fl32(v * fl32(1 / s))), -7, 7), ties to even; a group whose amax is 0 has
    s = 0 and q = 0;
  * a code is stored as the offset-binary nibble c = q + 8 (element k of a row in byte k/2, low
    nibble for even k), so c = 8 means zero.

Every step is one float32 IEEE operation, so a kernel doing the same operations in the same
order produces the same codes and scales.

Pins (tests/test_oracle_int4.py): hand-worked groups in tests/golden/int4_groups.txt, every
code against a brute-force nearest-integer search with ties to even, the reconstruction bound
|q s - v| <= s / 2, and the group's largest magnitude landing on q = +-7.
"""
from __future__ import annotations

import numpy as np

GROUP = 64
QMAX = 7


def quantize_groups(v):
    """rows of float32 values (K % 64 == 0) -> (codes uint8 rows x K, nibbles q + 8;
    scales float32 rows x K/64)."""
    v = np.asarray(v, dtype=np.float32)
    rows, K = v.shape
    if K % GROUP:
        raise ValueError("K must be a multiple of 64")
    blk = v.reshape(rows, K // GROUP, GROUP)
    amax = np.max(np.abs(blk), axis=2)                              # exact
    s = (amax / np.float32(QMAX)).astype(np.float32)                # fp32 division
    zero = s == 0
    s_safe = np.where(zero, np.float32(1.0), s).astype(np.float32)
    rcp = (np.float32(1.0) / s_safe).astype(np.float32)             # fp32 reciprocal
    t = (blk * rcp[:, :, None]).astype(np.float32)                  # fp32 product
    q = np.clip(np.rint(t), -QMAX, QMAX)                            # rint: half to even
    q[zero] = 0
    codes = (q + 8).astype(np.uint8)
    return codes.reshape(rows, K), s


def dequantize_groups(codes, scales) -> np.ndarray:
    """codes (rows x K nibbles), scales (rows x K/64) -> float64 values q * s (exact)."""
    codes = np.asarray(codes)
    rows, K = codes.shape
    q = codes.astype(np.float64).reshape(rows, K // GROUP, GROUP) - 8.0
    return (q * np.asarray(scales, np.float64)[:, :, None]).reshape(rows, K)
