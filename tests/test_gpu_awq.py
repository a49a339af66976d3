"""AWQ-style W4A16 layer on the GPU (svdq_awq_forward) against the oracle.

Y is compared with the oracle's forward (float64) evaluated on the library's own packed
layer (svdq_awq_export): relative Frobenius error <= 5e-3 and max-abs error
<= 2e-2 * max|Y_ref| (bf16 output, float32 accumulation).
"""
import numpy as np
import pytest
import torch

from oracle import awq
from oracle import svdquant as sq
from tests import gpu_helpers as gh
from w4a4_rank_corrected_e2m1_b300 import svdq, synthetic

pytestmark = pytest.mark.gpu


def _oracle_packed(o):
    return {"s": o["s"], "codes": np.stack([o["codes"] & 15, o["codes"] >> 4], -1).reshape(o["codes"].shape[0], -1),
            "scales": o["scales"], "zeros": o["zeros"], "bias": o["bias"], "group": 64}


def _run(layer, X, M):
    Xd = gh.dev_u16(X)
    Y = torch.full((max(M, 1), layer.N), float("nan"), dtype=torch.bfloat16, device="cuda")
    layer.forward(Xd, Y, M)
    torch.cuda.synchronize()
    layer.check_error()
    return sq.bf16_to_f64(gh.host_u16(Y.view(torch.int16)))[:M]


def _case(M, K, N, seed, n_cal=32):
    w = synthetic.scaled(synthetic.MOD, name=f"awq_{M}_{K}_{N}", M=M, K=K, N=N, seed=seed)
    d = synthetic.make(w)
    Xcal = synthetic.make_x(w, n_cal, seed=seed + 100)
    return w, d, Xcal


@pytest.mark.parametrize("M,K,N", [(1, 256, 40), (3, 512, 1000), (8, 1024, 520), (9, 1024, 264), (21, 512, 96)])
def test_awq_forward_matches_oracle(M, K, N):
    w, d, Xcal = _case(M, K, N, seed=M + K)
    layer = svdq.AwqLayer(d["W"], bias=d["bias"], Xcal=Xcal)
    o = layer.export()
    Y = _run(layer, d["X"], M)
    ref = awq.forward(d["X"], _oracle_packed(o))
    gh.assert_y_close(Y, ref, f"awq M={M} K={K} N={N}")
    layer.close()


@pytest.mark.parametrize("w", synthetic.AWQ_WORKLOADS, ids=lambda w: w.name)
def test_awq_modulation_shapes(w):
    """FLUX modulation shapes (K = 3072, N = 6 x 3072) in the bench's launch configuration."""
    d = synthetic.make(w)
    Xcal = synthetic.make_x(w, 64, seed=7)
    layer = svdq.AwqLayer(d["W"], bias=d["bias"], Xcal=Xcal)
    o = layer.export()
    Y = _run(layer, d["X"], w.M)
    gh.assert_y_close(Y, awq.forward(d["X"], _oracle_packed(o)), w.name)
    layer.close()


def test_awq_wide_k_and_repeatability():
    """K = 12288 (fewer rows of x' fit in shared memory per pass); two calls identical."""
    w, d, Xcal = _case(5, 12288, 384, seed=11)
    layer = svdq.AwqLayer(d["W"], bias=d["bias"], Xcal=Xcal)
    o = layer.export()
    Y1 = _run(layer, d["X"], 5)
    Y2 = _run(layer, d["X"], 5)
    assert np.array_equal(Y1, Y2)
    gh.assert_y_close(Y1, awq.forward(d["X"], _oracle_packed(o)), "awq K=12288")
    layer.close()


def test_awq_errors_and_m_zero():
    w, d, Xcal = _case(2, 256, 64, seed=1)
    layer = svdq.AwqLayer(d["W"], bias=d["bias"])
    X = torch.zeros((4, 256), dtype=torch.int16, device="cuda")
    Y = torch.zeros((4, 64), dtype=torch.int16, device="cuda")
    layer.forward(X, Y, 0)                                       # no-op
    with pytest.raises(svdq.SvdqError) as e:
        layer.forward(X.view(-1)[1:], Y, 1)                      # misaligned
    assert e.value.status == svdq.ERR_INVALID_ARG
    with pytest.raises(svdq.SvdqError) as e:
        layer.forward(X, X, 1)                                   # aliasing
    assert e.value.status == svdq.ERR_INVALID_ARG
    layer.close()


@pytest.mark.parametrize("amp", [400.0, 560.0, 3000.0, 60000.0])
def test_awq_large_activations_do_not_overflow(amp):
    """Rows of x' far beyond the range where four fp16 products x' (q - z) would overflow
    (|x'| * 15 * 4 > 65504 from |x'| ~ 1092): the kernel scales such a row by a power of two
    for its fp16 part.  One row stays small (scale 1), the others peak at `amp`; Y is finite
    and matches the oracle within the layer's tolerance."""
    w, d, _ = _case(4, 1024, 520, seed=23)
    layer = svdq.AwqLayer(d["W"], bias=d["bias"])          # s = 1: x' = x
    rng = np.random.default_rng(5)
    X = rng.standard_normal((4, 1024))
    X[1:] *= amp / np.max(np.abs(X[1:]), axis=1, keepdims=True)
    Xb = synthetic.f64_to_bf16_bits(X)
    o = layer.export()
    Y = _run(layer, Xb, 4)
    assert np.all(np.isfinite(Y))
    ref = awq.forward(Xb, _oracle_packed(o))
    for m in range(4):
        gh.assert_y_close(Y[m:m + 1], ref[m:m + 1], f"awq row {m} amp={amp}")
    layer.close()
