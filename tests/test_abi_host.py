"""The C-ABI library on the CPU: symbols, argument checks, and the host pack against the oracle.

No kernel runs here.  svdq_pack_host is the library's offline step (smoothing,
randomized SVD, residual NVFP4 quantisation) in C++; the oracle does the same
steps in numpy with LAPACK.  Where both take the same factors (the L1/L2
override) every byte must agree; the library's own SVD is held to Eckart-Young.
"""
import ctypes

import numpy as np
import pytest

from oracle import nvfp4
from oracle import svdquant as sq
from w4a4_rank_corrected_e2m1_b300 import svdq, synthetic


def test_every_declared_symbol_is_exported():
    names = svdq.header_functions()
    assert len(names) >= 15
    for n in names:
        assert hasattr(svdq.LIB, n), n
        assert ctypes.cast(getattr(svdq.LIB, n), ctypes.c_void_p).value


def test_binding_declares_every_header_function():
    """The ctypes layer sets argument and result types for every C-ABI function, so no call
    falls back to ctypes' int defaults (which would truncate pointers and 64-bit sizes)."""
    missing = [n for n in svdq.header_functions() if n not in svdq._SIGS]
    assert not missing, missing


def test_batch_host_forward_rejects_null_handle():
    # argument checks run before any device work, so they are testable without a GPU
    assert svdq.LIB.svdq_linear_forward_host_batch(None, None, None, 1, 1, None) == svdq.ERR_INVALID_ARG
    assert svdq.LIB.svdq_linear_forward_host(None, None, None, 1, None) == svdq.ERR_INVALID_ARG


def test_status_strings():
    for s in range(8):
        assert svdq.LIB.svdq_status_string(s)
    assert svdq.LIB.svdq_status_string(99) == b"unknown status"


def test_scale_buffer_size():
    assert svdq.scales_bytes(0, 256) == 0
    assert svdq.scales_bytes(1, 256) == 512 * 4
    assert svdq.scales_bytes(129, 3072) == 2 * 4 * 12 * 512
    assert svdq.scales_bytes(64, 320) == 1 * 8 * 512          # K padded to whole 256-column stages


def test_null_and_bad_arguments():
    assert svdq.LIB.svdq_pack_host(None, None) == svdq.ERR_INVALID_ARG
    assert svdq.LIB.svdq_pack_weights(None, None) == svdq.ERR_INVALID_ARG
    assert svdq.LIB.svdq_destroy(None) == svdq.OK
    assert svdq.LIB.svdq_linear_forward(None, None, None, 4, None) == svdq.ERR_INVALID_ARG
    assert svdq.LIB.svdq_set_wait_limit(None, 0, 0) == svdq.ERR_INVALID_ARG
    assert svdq.LIB.svdq_linear_forward_noalloc(None, None, None, 4, None) == svdq.ERR_INVALID_ARG
    W = np.zeros((32, 48), np.uint16)
    with pytest.raises(svdq.SvdqError) as e:
        svdq.pack_host(W, rank=40)                      # rank > min(N, K)
    assert e.value.status == svdq.ERR_UNSUPPORTED_SHAPE
    with pytest.raises(svdq.SvdqError) as e:
        svdq.pack_host(np.zeros((32, 40), np.uint16), rank=0)   # K % 16
    assert e.value.status == svdq.ERR_UNSUPPORTED_SHAPE
    with pytest.raises(svdq.SvdqError) as e:
        svdq.pack_host(W, rank=4, lam=np.full(48, -1.0, np.float32))
    assert e.value.status == svdq.ERR_INVALID_ARG


@pytest.mark.parametrize("case", ["tiny", "qkv_small", "down_small"])
def test_host_pack_bit_exact_with_oracle_factors(case):
    w = {c.name: c for c in synthetic.parity_cases()}[case]
    d = synthetic.make(w)
    ref = sq.pack(d["W"], d["bias"], w.rank, Xcal_bits=d["X"])
    got = svdq.pack_host(d["W"], w.rank, bias=d["bias"], Xcal=d["X"], L1=ref["L1"], L2=ref["L2"])
    assert np.array_equal(got["lam"], ref["lam"])
    assert np.array_equal(got["inv_lambda"], ref["inv_lambda"])
    assert got["s_gW"] == ref["s_gW"] and got["s_gX"] == ref["s_gX"]
    assert got["alpha"] == sq.alpha(ref)
    packed = (ref["R_codes"][:, 0::2] | (ref["R_codes"][:, 1::2] << 4)).astype(np.uint8)
    assert np.array_equal(got["R_codes"], packed)
    assert np.array_equal(got["R_scales"], ref["R_scales"])
    assert np.array_equal(got["bias"], ref["bias"])


def test_host_pack_without_smoothing_is_plain_w4a4():
    d = synthetic.make(synthetic.TINY)
    got = svdq.pack_host(d["W"], 0, smooth=False)
    wf = sq.bf16_to_f32(d["W"])
    cw, sw = nvfp4.quantize_blocks(wf, nvfp4.global_scale(np.max(np.abs(wf))))
    assert np.array_equal(got["R_codes"], (cw[:, 0::2] | (cw[:, 1::2] << 4)).astype(np.uint8))
    assert np.array_equal(got["R_scales"], sw)
    assert np.all(got["inv_lambda"] == 1.0)


def test_host_quantizer_on_hand_worked_and_edge_rows():
    """Rows with ties, -0, saturation and zero blocks through the library's quantiser (lambda = 1,
    rank 0, so R = W exactly) against the oracle quantiser."""
    rng = np.random.default_rng(11)
    K = 64
    rows = [
        [3, -3, 1, 0.25, 0.125, 0.375, -0.625, 2.5, 1.75, -0.875, 0, -0.0, 2, 1.25, 0.625, -2.875] * 4,
        [0.0] * 64,
        list(np.float32(rng.standard_normal(64) * 1e-3)),
        [448.0 * 6] + [1e-3] * 63,
    ]
    rows += [list(np.float32(rng.standard_normal(K) * 10 ** rng.uniform(-3, 3))) for _ in range(12)]
    W = synthetic.f64_to_bf16_bits(np.array(rows, np.float64))
    got = svdq.pack_host(W, 0, smooth=False)
    wf = sq.bf16_to_f32(W)
    cw, sw = nvfp4.quantize_blocks(wf, nvfp4.global_scale(np.max(np.abs(wf))))
    assert np.array_equal(got["R_codes"], (cw[:, 0::2] | (cw[:, 1::2] << 4)).astype(np.uint8))
    assert np.array_equal(got["R_scales"], sw)


# ------------------------------------------------------------------ INT4 variant host pack
def _pack_nibbles(c):
    return (c[:, 0::2] | (c[:, 1::2] << 4)).astype(np.uint8)


@pytest.mark.parametrize("case", ["tiny", "qkv_small", "down_small"])
def test_int4_host_pack_bit_exact_with_oracle_factors(case):
    w = {c.name: c for c in synthetic.parity_cases()}[case]
    d = synthetic.make(w)
    ref = sq.pack_int4(d["W"], d["bias"], w.rank, Xcal_bits=d["X"])
    got = svdq.int4_pack_host(d["W"], w.rank, bias=d["bias"], Xcal=d["X"], L1=ref["L1"], L2=ref["L2"])
    assert np.array_equal(got["lam"], ref["lam"]) and np.array_equal(got["inv_lambda"], ref["inv_lambda"])
    assert np.array_equal(got["R_codes"], _pack_nibbles(ref["R_codes"]))
    assert np.array_equal(got["R_scales"].view(np.uint32), ref["R_scales"].view(np.uint32))
    assert np.array_equal(got["bias"], ref["bias"])


def test_int4_host_quantizer_on_edge_rows():
    """Zero groups, ties, negative zeros and wide magnitude ranges through the library's INT4
    quantiser (lambda = 1, rank 0: R = W exactly) against the oracle's."""
    from oracle import int4
    rng = np.random.default_rng(12)
    rows = [[0.0] * 128, ([7, -7, 2.5, -2.5, 3.5, -3.5, 0.5, -0.5, -0.0, 1.5] + [0.0] * 54) * 2]
    rows += [list(rng.standard_normal(128) * 10 ** rng.uniform(-4, 4)) for _ in range(30)]
    W = synthetic.f64_to_bf16_bits(np.array(rows, np.float64))
    got = svdq.int4_pack_host(W, 0, smooth=False)
    cw, sw = int4.quantize_groups(sq.bf16_to_f32(W))
    assert np.array_equal(got["R_codes"], _pack_nibbles(cw))
    assert np.array_equal(got["R_scales"].view(np.uint32), sw.view(np.uint32))


def test_int4_shape_errors():
    W = np.zeros((32, 96), np.uint16)                 # K % 64 != 0
    with pytest.raises(svdq.SvdqError) as e:
        svdq.int4_pack_host(W, 0)
    assert e.value.status == svdq.ERR_UNSUPPORTED_SHAPE
    assert svdq.LIB.svdq_int4_forward(None, None, None, 4, None) == svdq.ERR_INVALID_ARG
    assert svdq.LIB.svdq_int4_destroy(None) == svdq.OK
    assert svdq.int4_scale_ld(1) == 128 and svdq.int4_scale_ld(129) == 256


@pytest.mark.parametrize("shape", [(256, 256, 16), (512, 768, 32), (384, 1024, 64)])
def test_randomized_svd_near_eckart_young(shape):
    N, K, r = shape
    w = synthetic.scaled(synthetic.QKV, M=64, K=K, N=N, rank=r, n_outlier=max(1, K // 100))
    d = synthetic.make(w)
    got = svdq.pack_host(d["W"], r, Xcal=d["X"])
    Wh = sq.smooth_weight(d["W"], got["lam"])
    L1 = sq.bf16_to_f64(got["L1"])
    L2 = sq.bf16_to_f64(got["L2"])
    res = np.sum((Wh.T - L1 @ L2) ** 2)
    s = np.linalg.svd(Wh, compute_uv=False)
    opt = np.sum(s[r:] ** 2)
    # bf16 rounding of the factors adds ~2^-9 relative error to the captured part
    assert res <= 1.01 * opt + 2 ** -16 * np.sum(s[:r] ** 2), (res, opt)
    # residual codes follow from the library's own factors, through the oracle quantiser
    R = sq.residual(Wh, got["L1"], got["L2"])
    cw, sw = nvfp4.quantize_blocks(R, nvfp4.global_scale(np.max(np.abs(R))))
    assert np.array_equal(got["R_codes"], (cw[:, 0::2] | (cw[:, 1::2] << 4)).astype(np.uint8))
    assert np.array_equal(got["R_scales"], sw)


# ------------------------------------------------------------------ AWQ-style W4A16 host pack
def _awq_case(seed, N=48, K=256, M=24):
    rng = np.random.default_rng(seed)
    W = sq.f64_to_bf16(rng.standard_normal((N, K)) * 0.05)
    W[:, 5] = sq.f64_to_bf16(np.linspace(0.5, 1.5, N))          # an all-positive column
    X = rng.standard_normal((M, K))
    X[:, rng.choice(K, 4, replace=False)] *= 35.0
    return W, sq.f64_to_bf16(X), sq.f64_to_bf16(rng.standard_normal(N) * 0.1)


def _nibbles(codes):
    return np.stack([codes & 15, codes >> 4], axis=-1).reshape(codes.shape[0], -1)


def test_awq_host_quantiser_bit_exact_with_oracle_given_scales():
    from oracle import awq
    W, X, b = _awq_case(0)
    s = (1.0 + np.random.default_rng(9).random(W.shape[1])).astype(np.float32)
    o = svdq.awq_pack_host(W, bias=b, s=s)
    p = awq.pack(W, b, s32=s)
    assert np.array_equal(_nibbles(o["codes"]), p["codes"])
    assert np.array_equal(o["scales"], p["scales"]) and np.array_equal(o["zeros"], p["zeros"])
    assert np.array_equal(o["inv_s"], (np.float32(1.0) / s).astype(np.float32))
    assert np.array_equal(o["bias"], b)


def test_awq_host_search_matches_oracle():
    from oracle import awq
    W, X, b = _awq_case(1)
    o = svdq.awq_pack_host(W, bias=b, Xcal=X)
    p = awq.pack(W, b, Xcal_bits=X)
    assert abs(o["alpha"] - p["alpha"]) < 1e-6
    assert np.array_equal(o["s"], p["s"])
    assert np.array_equal(_nibbles(o["codes"]), p["codes"])


def test_awq_host_without_calibration_is_plain_rounding():
    from oracle import awq
    W, X, b = _awq_case(2)
    o = svdq.awq_pack_host(W)
    assert np.all(o["s"] == 1.0) and o["alpha"] == -1.0
    q, sc, z = awq.quantize_groups(sq.bf16_to_f32(W))
    assert np.array_equal(_nibbles(o["codes"]), q) and np.array_equal(o["scales"], sc)


def test_awq_host_rejects_bad_shapes():
    rng = np.random.default_rng(3)
    W = sq.f64_to_bf16(rng.standard_normal((8, 96)))
    with pytest.raises(svdq.SvdqError) as e:
        svdq.awq_pack_host(W)                                    # K % 64 != 0
    assert e.value.status == svdq.ERR_UNSUPPORTED_SHAPE
