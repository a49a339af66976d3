"""AWQ-style W4A16 linear layer, restated on the CPU (test infrastructure only).

Per the pages, Nunchaku treats the adaptive-normalisation and modulation layers differently
from the transformer blocks, because 4-bit activations hurt them more: it keeps their
activations in 16 bits and quantises only their weights to four bits, AWQ style (aiflownews article on Nunchaku,
"How Nunchaku four bit quantization actually works").  They give no group size, scale
format or search rule; the readings below are the plainest ones (each also listed in the
design notes):

  * weights: asymmetric unsigned 4-bit codes per group of G = 64 consecutive input channels
    of an output row, float32 scale s and integer zero point z in [0, 15]:
        s = fl32(max(w_max - w_min, 1e-5) / 15),  z = clamp(rint(-w_min / s), 0, 15),
        q = clamp(rint(w / s) + z, 0, 15),          w ~ (q - z) * s
    (float32 arithmetic, rint = round half to even; the quotients w / s are correctly
    rounded float32 divisions);
  * activation-aware scaling: per input channel c, a = mean_m |Xcal_mc| (float64),
    s_c = a_c^alpha normalised by sqrt(max s * min s), stored as float32, with alpha picked
    from {0, 0.05, ..., 0.95} as the one that minimises the calibration output error
    || Xcal W^T - (Xcal diag(1/s)) deq(Q(W diag(s)))^T ||_F^2; channels with a_c = 0 get
    s_c = 1;
  * forward: x' = fl32(x * fl32(1 / s)), Y = x' deq(Q)^T + b, in float64.

Pins (tests/test_oracle_awq.py): weights already on a group's grid are reproduced
exactly; the per-group extremes map to codes 0 and 15 (up to the zero point's rounding);
the reconstruction error is at most half a step per element; alpha = 0 is plain
round-to-nearest quantisation of W; the forward against Python loops on a tiny case; on
activations with outlier channels the searched alpha does no worse than alpha = 0 on the
calibration error.
"""
from __future__ import annotations

import numpy as np

from oracle import svdquant as sq

GROUP = 64
ALPHAS = [i / 20 for i in range(20)]


def quantize_groups(w32: np.ndarray, group: int = GROUP):
    """Rows of float32 weights -> (codes uint8 in [0, 15], scales float32, zeros uint8)."""
    w = np.asarray(w32, dtype=np.float32)
    N, K = w.shape
    assert K % group == 0
    g = w.reshape(N, K // group, group)
    mn = g.min(axis=2)
    mx = g.max(axis=2)
    rng = np.maximum(mx - mn, np.float32(1e-5)).astype(np.float32)
    s = (rng / np.float32(15.0)).astype(np.float32)
    z = np.clip(np.rint((-mn / s).astype(np.float32)), 0, 15).astype(np.uint8)
    q = np.rint((g / s[:, :, None]).astype(np.float32)) + z[:, :, None].astype(np.float32)
    q = np.clip(q, 0, 15).astype(np.uint8)
    return q.reshape(N, K), s, z


def dequantize_groups(q: np.ndarray, s: np.ndarray, z: np.ndarray, group: int = GROUP) -> np.ndarray:
    """Codes, scales and zero points -> float64 weights (q - z) * s."""
    N, K = q.shape
    d = (q.reshape(N, K // group, group).astype(np.float64) - z[:, :, None].astype(np.float64)) * s[:, :, None].astype(np.float64)
    return d.reshape(N, K)


def channel_magnitudes(Xcal_bits) -> np.ndarray:
    return np.mean(np.abs(sq.bf16_to_f64(Xcal_bits)), axis=0)


def awq_scales(a: np.ndarray, alpha: float) -> np.ndarray:
    """s_c = a_c^alpha / sqrt(max s * min s) over channels with a_c > 0; 1 elsewhere; float32."""
    s = np.ones_like(a)
    pos = a > 0
    if np.any(pos):
        v = a[pos] ** alpha
        v = v / np.sqrt(v.max() * v.min())
        s[pos] = v
    return s.astype(np.float32)


def scaled_weight(W_bits, s32) -> np.ndarray:
    """fl32(w * s_c)."""
    return (sq.bf16_to_f32(W_bits) * s32[None, :]).astype(np.float32)


def scaled_act(X_bits, s32) -> np.ndarray:
    """x' = fl32(x * fl32(1 / s_c))."""
    inv = (np.float32(1.0) / s32).astype(np.float32)
    return (sq.bf16_to_f32(X_bits) * inv[None, :]).astype(np.float32)


def search_alpha(W_bits, Xcal_bits, group: int = GROUP):
    """The grid search over alpha; returns (alpha, s32, error per alpha)."""
    a = channel_magnitudes(Xcal_bits)
    ref = sq.bf16_to_f64(Xcal_bits) @ sq.bf16_to_f64(W_bits).T
    errs = []
    best = None
    for alpha in ALPHAS:
        s = awq_scales(a, alpha)
        q, sc, z = quantize_groups(scaled_weight(W_bits, s), group)
        Y = scaled_act(Xcal_bits, s).astype(np.float64) @ dequantize_groups(q, sc, z, group).T
        e = float(np.sum((Y - ref) ** 2))
        errs.append(e)
        if best is None or e < best[0]:
            best = (e, alpha, s)
    return best[1], best[2], errs


def pack(W_bits, bias_bits, Xcal_bits=None, s32=None, group: int = GROUP):
    """Offline step: scales (searched, given, or all ones), then the group quantiser."""
    K = np.asarray(W_bits).shape[1]
    alpha = None
    if s32 is None:
        if Xcal_bits is None:
            s32 = np.ones(K, np.float32)
        else:
            alpha, s32, _ = search_alpha(W_bits, Xcal_bits, group)
    q, sc, z = quantize_groups(scaled_weight(W_bits, s32), group)
    return {"s": np.asarray(s32, np.float32), "alpha": alpha, "codes": q, "scales": sc, "zeros": z,
            "bias": np.asarray(bias_bits), "group": group}


def forward(X_bits, p, rows=None) -> np.ndarray:
    """Y = x' deq(Q)^T + b in float64."""
    Xb = np.asarray(X_bits)
    if rows is not None:
        Xb = Xb[rows]
    xs = scaled_act(Xb, p["s"]).astype(np.float64)
    return xs @ dequantize_groups(p["codes"], p["scales"], p["zeros"], p["group"]).T + sq.bf16_to_f64(p["bias"])[None, :]
