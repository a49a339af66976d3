"""Pins for oracle/awq.py (the AWQ-style W4A16 layer), independent of its own code paths."""
import numpy as np
import pytest

from oracle import awq
from oracle import svdquant as sq


def test_weights_on_the_grid_are_reproduced_exactly():
    rng = np.random.default_rng(0)
    N, K = 5, 256
    s = np.float32(2.0) ** rng.integers(-8, -2, size=(N, K // 64)).astype(np.float32)
    z = rng.integers(1, 15, size=(N, K // 64))
    q = rng.integers(0, 16, size=(N, K))
    q[:, ::64] = 0                        # each group spans the whole code range
    q[:, 1::64] = 15
    w = ((q.reshape(N, K // 64, 64) - z[:, :, None]) * s[:, :, None]).reshape(N, K).astype(np.float32)
    q2, s2, z2 = awq.quantize_groups(w)
    assert np.array_equal(s2, s) and np.array_equal(z2, z) and np.array_equal(q2, q)
    assert np.array_equal(awq.dequantize_groups(q2, s2, z2), w.astype(np.float64))


def test_codes_span_the_range_and_error_is_half_a_step():
    rng = np.random.default_rng(1)
    w = rng.standard_normal((7, 512)).astype(np.float32)     # every group holds both signs
    q, s, z = awq.quantize_groups(w)
    g = q.reshape(7, 8, 64)
    assert np.all(g.min(axis=2) <= 1) and np.all(g.max(axis=2) >= 14)
    err = np.abs(awq.dequantize_groups(q, s, z) - w).reshape(7, 8, 64)
    assert np.all(err <= 0.5 * s[:, :, None].astype(np.float64) * (1 + 1e-6))


def test_one_signed_group_is_clipped_at_the_top_code():
    """A group with no negative value gets zero point 0, so values above 15 s saturate (the
    asymmetric quantiser's known limitation, kept as the plainest reading)."""
    w = np.linspace(1.0, 2.0, 64, dtype=np.float32)[None, :]
    q, s, z = awq.quantize_groups(w)
    assert z[0, 0] == 0 and q.max() == 15
    assert np.isclose(float(s[0, 0]), 1.0 / 15, rtol=1e-6)


def test_scales_normalisation_and_alpha_zero():
    a = np.array([0.1, 2.0, 0.0, 5.0, 0.7])
    s = awq.awq_scales(a, 0.5)
    pos = a > 0
    assert s[2] == 1.0
    assert np.isclose(np.sqrt(s[pos].max() * s[pos].min()), 1.0, rtol=1e-6)
    assert np.allclose(s[pos] / s[pos][0], (a[pos] / a[pos][0]) ** 0.5, rtol=1e-6)
    assert np.all(awq.awq_scales(a, 0.0) == 1.0)


def test_forward_against_python_loops():
    rng = np.random.default_rng(2)
    M, K, N = 2, 128, 3
    X = sq.f64_to_bf16(rng.standard_normal((M, K)))
    W = sq.f64_to_bf16(rng.standard_normal((N, K)) * 0.1)
    b = sq.f64_to_bf16(rng.standard_normal(N) * 0.1)
    s = np.float32(1.0) + rng.random(K).astype(np.float32)
    p = awq.pack(W, b, s32=s)
    ref = np.zeros((M, N))
    for m in range(M):
        for n in range(N):
            acc = 0.0
            for k in range(K):
                xs = np.float32(sq.bf16_to_f32(X[m, k]) * np.float32(np.float32(1.0) / s[k]))
                grp = k // 64
                d = (float(p["codes"][n, k]) - float(p["zeros"][n, grp])) * float(p["scales"][n, grp])
                acc += float(xs) * d
            ref[m, n] = acc + float(sq.bf16_to_f64(b[n]))
    assert np.allclose(awq.forward(X, p), ref, rtol=1e-12, atol=1e-12)


def test_search_helps_on_outlier_channels():
    """Activation-aware scaling protects the weights of large-activation channels: the
    searched alpha gives a smaller calibration error than alpha = 0 (plain round-to-nearest)."""
    rng = np.random.default_rng(3)
    M, K, N = 64, 256, 96
    X = rng.standard_normal((M, K))
    X[:, rng.choice(K, 6, replace=False)] *= 40.0
    Xb = sq.f64_to_bf16(X)
    W = sq.f64_to_bf16(rng.standard_normal((N, K)) / np.sqrt(K))
    alpha, s, errs = awq.search_alpha(W, Xb)
    assert errs[awq.ALPHAS.index(alpha)] == min(errs)
    assert min(errs) < 0.9 * errs[0]
