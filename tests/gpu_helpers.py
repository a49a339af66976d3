"""Shared helpers of the GPU tests: device buffers, layout decoding, comparisons.

Layout decoding follows the device layouts documented in include/svdq.h; it is
written here from that description, not taken from the library.
"""
from __future__ import annotations

import numpy as np
import torch

from oracle import svdquant as sq

# spec tolerances for Y (float32 accumulation, bfloat16 output)
Y_REL_FRO = 5e-3
Y_MAX_ABS_FRAC = 2e-2


def dev_u16(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).cuda()


def host_u16(t: torch.Tensor) -> np.ndarray:
    return t.cpu().numpy().view(np.uint16)


def unpack_codes(packed: np.ndarray) -> np.ndarray:
    """rows x K/2 bytes -> rows x K nibbles (even k in the low nibble)."""
    out = np.empty((packed.shape[0], packed.shape[1] * 2), np.uint8)
    out[:, 0::2] = packed & 0xF
    out[:, 1::2] = packed >> 4
    return out


def untile_scales(buf: np.ndarray, M: int, K: int) -> np.ndarray:
    """Tiled activation scales (include/svdq.h) -> M x K/16 row-major."""
    KG = 4 * ((K + 255) // 256)
    m = np.arange(M)[:, None]
    j = np.arange(K // 16)[None, :]
    off = ((m // 128) * KG + j // 4) * 512 + (m % 32) * 16 + ((m % 128) // 32) * 4 + (j % 4)
    return buf[off]


def tile_scales(sc: np.ndarray, M: int, K: int) -> np.ndarray:
    """Inverse of untile_scales (padding rows and groups hold 0)."""
    KG = 4 * ((K + 255) // 256)
    buf = np.zeros(((M + 127) // 128) * KG * 512, np.uint8)
    m = np.arange(M)[:, None]
    j = np.arange(K // 16)[None, :]
    off = ((m // 128) * KG + j // 4) * 512 + (m % 32) * 16 + ((m % 128) // 32) * 4 + (j % 4)
    buf[off] = sc
    return buf


def oracle_packed(exp: dict) -> dict:
    """The library's exported packed layer in the oracle's form (codes as nibbles)."""
    p = dict(exp)
    p["R_codes"] = unpack_codes(exp["R_codes"])
    return p


def y_errors(Y: np.ndarray, ref: np.ndarray):
    rel = float(np.linalg.norm(Y - ref) / np.linalg.norm(ref))
    mx = float(np.max(np.abs(Y - ref)) / np.max(np.abs(ref)))
    return rel, mx


def assert_y_close(Y: np.ndarray, ref: np.ndarray, what=""):
    rel, mx = y_errors(Y, ref)
    assert rel <= Y_REL_FRO and mx <= Y_MAX_ABS_FRAC, f"{what}: rel_fro={rel:.3e} max_abs/max={mx:.3e}"
    return rel, mx


# Per-tile check: each 256 x 256 output tile (the GEMM's pair tile) on its own, so that an error
# confined to some TMEM lanes, one epilogue warp's rows or one tile cannot hide in the global
# norm.  A tile's error is the same mix of bf16 output rounding and 4-bit product noise as the
# whole output's (about 3e-3 relative), so twice the global bound leaves a wide margin.
Y_TILE_REL_FRO = 1e-2


def assert_tiles_close(Y: np.ndarray, ref: np.ndarray, what="", tile=256):
    M, N = ref.shape
    worst = (0.0, None)
    for m0 in range(0, M, tile):
        for n0 in range(0, N, tile):
            r = ref[m0:m0 + tile, n0:n0 + tile]
            nr = np.linalg.norm(r)
            if nr == 0:
                assert np.all(Y[m0:m0 + tile, n0:n0 + tile] == 0), f"{what}: tile ({m0}, {n0})"
                continue
            e = float(np.linalg.norm(Y[m0:m0 + tile, n0:n0 + tile] - r) / nr)
            if e > worst[0]:
                worst = (e, (m0, n0))
    assert worst[0] <= Y_TILE_REL_FRO, f"{what}: tile {worst[1]} rel_fro={worst[0]:.3e}"
    return worst


def bf16_bits_to_f64(b: np.ndarray) -> np.ndarray:
    return sq.bf16_to_f64(b)
