"""GPU parity of the SVDQuant layer's INT4 variant against the CPU oracle (oracle.int4,
oracle.svdquant.pack_int4 / forward_int4), through the C ABI.

  * kernel int4_k1 (svdq_int4_quantize_act): INT4 codes and float32 group scales bit-exact with
    the oracle's quantiser given the library's inv_lambda; T = X^ L1 within bf16 accuracy;
  * the forward (svdq_int4_forward): Y against the oracle's INT4 forward evaluated on the
    library's own packed layer (svdq_int4_export), within relative Frobenius error 5e-3 and
    max-abs error 2e-2 * max|Y_ref|, like the NVFP4 layer; also each 128 x 128 tile on its own;
  * ragged M / N / K, rank 0 and 128, M = 0, the FLUX MLP-up shape on every element.
"""
import numpy as np
import pytest
import torch

from oracle import svdquant as sq
from tests import gpu_helpers as gh
from w4a4_rank_corrected_e2m1_b300 import svdq, synthetic

pytestmark = pytest.mark.gpu


def _oracle_packed(exp):
    p = dict(exp)
    p["R_codes"] = gh.unpack_codes(exp["R_codes"])
    return p


def _layer(w):
    d = synthetic.make(w)
    layer = svdq.Int4Layer(d["W"], w.rank, bias=d["bias"], Xcal=d["X"], M_max=w.M)
    return d, layer, _oracle_packed(layer.export())


def _forward(layer, X, M):
    Y = torch.full((max(M, 1), layer.N), float("nan"), dtype=torch.bfloat16, device="cuda")
    layer.forward(gh.dev_u16(X), Y, M)
    torch.cuda.synchronize()
    layer.check_error()
    return sq.bf16_to_f64(gh.host_u16(Y.view(torch.int16)))[:M]


CASES = [
    synthetic.TINY,
    synthetic.scaled(synthetic.QKV, name="qkv_small", M=300, K=512, N=768, rank=32, n_outlier=5),
    synthetic.scaled(synthetic.MLP_DOWN, name="down_ragged", M=77, K=1088, N=272, rank=16),
    synthetic.scaled(synthetic.QKV, name="rank128", M=200, K=640, N=384, rank=128, n_outlier=6),
    synthetic.scaled(synthetic.QKV, name="rank0", M=129, K=256, N=160, rank=0, n_outlier=3),
]


@pytest.mark.parametrize("w", CASES, ids=lambda w: w.name)
def test_int4_k1_codes_scales_bitexact_and_T(w):
    d, layer, p = _layer(w)
    M, K = w.M, w.K
    ld = svdq.int4_scale_ld(M)
    codes = torch.zeros((M, K // 2), dtype=torch.uint8, device="cuda")
    scales = torch.full((K // 64, ld), float("nan"), dtype=torch.float32, device="cuda")
    T = torch.zeros((M, max(layer.r_pad, 8)), dtype=torch.int16, device="cuda") if w.rank else None
    layer.quantize_act(gh.dev_u16(d["X"]), M, codes, scales, T)
    torch.cuda.synchronize()
    layer.check_error()
    rc, rs, xh = sq.quantize_act_int4(d["X"], p["inv_lambda"])
    got_c = gh.unpack_codes(codes.cpu().numpy())
    got_s = scales.cpu().numpy()[:, :M].T
    assert np.array_equal(got_s.view(np.uint32), rs.view(np.uint32)), f"scale mismatches {np.sum(got_s != rs)}"
    assert np.array_equal(got_c, rc), f"code mismatches {np.sum(got_c != rc)}"
    if w.rank:
        t = sq.bf16_to_f64(gh.host_u16(T))[:, : w.rank]
        tref = sq.lowrank_down(xh, p["L1"])
        assert np.linalg.norm(t - tref) <= 1e-2 * np.linalg.norm(tref)
        assert np.all(sq.bf16_to_f64(gh.host_u16(T))[:, w.rank: layer.r_pad] == 0)
    layer.close()


@pytest.mark.parametrize("w", CASES, ids=lambda w: w.name)
def test_int4_forward_matches_oracle(w):
    d, layer, p = _layer(w)
    Y = _forward(layer, d["X"], w.M)
    ref = sq.forward_int4(d["X"], p)
    gh.assert_y_close(Y, ref, w.name)
    gh.assert_tiles_close(Y, ref, w.name, tile=128)
    layer.close()


def test_int4_edge_cases_and_repeatability():
    w = CASES[1]
    d, layer, p = _layer(w)
    Y1 = _forward(layer, d["X"], w.M)
    Y2 = _forward(layer, d["X"], w.M)
    assert np.array_equal(Y1, Y2)
    for M in (1, 31, 129):
        Y = _forward(layer, d["X"][:M], M)
        gh.assert_y_close(Y, sq.forward_int4(d["X"][:M], p), f"M={M}")
    layer.forward(gh.dev_u16(d["X"]), torch.zeros((1, w.N), dtype=torch.int16, device="cuda"), 0)   # no-op
    with pytest.raises(svdq.SvdqError) as e:
        _forward(layer, np.concatenate([d["X"], d["X"]]), 2 * w.M)                # above the workspace
    assert e.value.status == svdq.ERR_WORKSPACE
    layer.close()


def test_int4_full_size_mlp_up():
    """FLUX MLP-up shape (4608 x 3072 -> 12288, rank 32), every element."""
    w = synthetic.MLP_UP
    d, layer, p = _layer(w)
    Y = _forward(layer, d["X"], w.M)
    ref = sq.forward_int4(d["X"], p)
    gh.assert_y_close(Y, ref, "int4 mlp_up")
    gh.assert_tiles_close(Y, ref, "int4 mlp_up")
    layer.close()
