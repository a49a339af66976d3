"""LoRA adapter on the low-rank branch (svdq_attach_lora) against the oracle.

The adapter's factors are concatenated onto L1 and L2, so kernel 1's down-projection and
kernel 2's up-projection run with rank + r_lora.  Y is compared with the oracle's forward on
the library's own packed operands plus the oracle's LoRA term scale * (X A) B, within the
same bound as the plain layer.
"""
import numpy as np
import pytest
import torch

from oracle import svdquant as sq
from tests import gpu_helpers as gh
from w4a4_rank_corrected_e2m1_b300 import svdq, synthetic

pytestmark = pytest.mark.gpu


def _lora(K, N, r_lora, seed, amp=0.05):
    rng = np.random.default_rng(seed)
    A = synthetic.f64_to_bf16_bits(rng.standard_normal((K, r_lora)) / np.sqrt(K))
    B = synthetic.f64_to_bf16_bits(rng.standard_normal((r_lora, N)) * amp)
    return A, B


def _forward(layer, X, M):
    Xd = gh.dev_u16(X)
    Y = torch.empty((M, layer.N), dtype=torch.bfloat16, device="cuda")
    layer.forward(Xd, Y, M)
    torch.cuda.synchronize()
    layer.check_error()
    return sq.bf16_to_f64(gh.host_u16(Y.view(torch.int16)))


@pytest.mark.parametrize("r_lora,scale", [(16, 0.5), (32, 1.0), (64, 2.0)])
def test_lora_forward_matches_oracle(r_lora, scale):
    w = synthetic.parity_cases()[1]                  # 300 x 512 x 768, rank 32
    d = synthetic.make(w)
    layer = svdq.Layer(d["W"], w.rank, bias=d["bias"], Xcal=d["X"], M_max=w.M)
    exp = layer.export()
    A, B = _lora(w.K, w.N, r_lora, seed=5 + r_lora, amp=0.2)
    layer.attach_lora(A, B, scale)
    info = layer.info
    assert info.rank == w.rank and info.lora_rank == r_lora and info.r_pad == 64 * -(-(w.rank + r_lora) // 64)
    Y = _forward(layer, d["X"], w.M)
    ref = sq.forward(d["X"], gh.oracle_packed(exp)) + sq.lora_delta(d["X"], A, B, scale)
    gh.assert_y_close(Y, ref, f"lora r={r_lora}")
    # the adapter really contributes: without it the output is measurably different
    base = sq.forward(d["X"], gh.oracle_packed(exp))
    assert gh.y_errors(base, ref)[0] > 10 * gh.y_errors(Y, ref)[0]
    layer.close()


def test_lora_detach_restores_the_plain_layer():
    w = synthetic.parity_cases()[1]
    d = synthetic.make(w)
    layer = svdq.Layer(d["W"], w.rank, bias=d["bias"], Xcal=d["X"], M_max=w.M)
    Y0 = _forward(layer, d["X"], w.M)
    A, B = _lora(w.K, w.N, 16, seed=3)
    layer.attach_lora(A, B, 1.0)
    layer.attach_lora(None, None)
    assert layer.info.lora_rank == 0
    Y1 = _forward(layer, d["X"], w.M)
    assert np.array_equal(Y0, Y1)
    layer.close()


def test_lora_quantised_activations_unchanged():
    """The adapter touches neither the activation quantiser nor the residual."""
    w = synthetic.parity_cases()[1]
    d = synthetic.make(w)
    layer = svdq.Layer(d["W"], w.rank, bias=d["bias"], Xcal=d["X"], M_max=w.M)
    exp = layer.export()
    A, B = _lora(w.K, w.N, 32, seed=4)
    layer.attach_lora(A, B, 1.0)
    K = w.K
    codes = torch.empty((w.M, K // 2), dtype=torch.uint8, device="cuda")
    scales = torch.full((svdq.scales_bytes(w.M, K),), 0xFF, dtype=torch.uint8, device="cuda")
    T = torch.empty((w.M, layer.info.r_pad), dtype=torch.int16, device="cuda")
    layer.quantize_act(gh.dev_u16(d["X"]), w.M, codes, scales, T)
    torch.cuda.synchronize()
    layer.check_error()
    rc, rs, _ = sq.quantize_act(d["X"], exp["inv_lambda"], exp["s_gX"])
    assert np.array_equal(gh.unpack_codes(codes.cpu().numpy()), rc)
    assert np.array_equal(gh.untile_scales(scales.cpu().numpy(), w.M, K), rs)
    # T's LoRA columns are (X bf16(A)) / alpha
    t = sq.bf16_to_f64(gh.host_u16(T))
    ref = (sq.bf16_to_f64(d["X"]) @ sq.bf16_to_f64(A)) / float(exp["alpha"])
    got = t[:, w.rank:w.rank + 32]
    assert np.max(np.abs(got - ref)) <= 1e-2 * np.max(np.abs(ref))
    layer.close()


def test_lora_errors():
    w = synthetic.parity_cases()[1]
    d = synthetic.make(w)
    layer = svdq.Layer(d["W"], w.rank, bias=d["bias"], Xcal=d["X"])
    A, B = _lora(w.K, w.N, 24, seed=1)
    with pytest.raises(svdq.SvdqError) as e:
        layer.attach_lora(A, B)                          # not a multiple of 16
    assert e.value.status == svdq.ERR_UNSUPPORTED_SHAPE
    A, B = _lora(w.K, w.N, 112, seed=1)
    with pytest.raises(svdq.SvdqError) as e:
        layer.attach_lora(A, B)                          # 32 + 112 > 128
    assert e.value.status == svdq.ERR_UNSUPPORTED_SHAPE
    # a lent workspace sized for the plain rank is too small for rank + LoRA
    nbytes = layer.workspace_size(w.M)
    buf = torch.empty(nbytes + 256, dtype=torch.uint8, device="cuda")
    off = (-buf.data_ptr()) % 256
    layer.set_workspace(buf[off:off + nbytes], w.M)
    A, B = _lora(w.K, w.N, 64, seed=1)
    with pytest.raises(svdq.SvdqError) as e:
        layer.attach_lora(A, B)
    assert e.value.status == svdq.ERR_WORKSPACE
    assert layer.info.lora_rank == 0
    layer.set_workspace(None, 0)
    layer.close()


def test_lora_full_size_mlp_up():
    """FLUX MLP-up shape, rank 32 + LoRA 32, in the bench's launch configuration; every element."""
    w = synthetic.MLP_UP
    d = synthetic.make(w)
    layer = svdq.Layer(d["W"], w.rank, bias=d["bias"], Xcal=d["X"], M_max=w.M)
    exp = layer.export()
    A, B = _lora(w.K, w.N, 32, seed=9, amp=0.1)
    layer.attach_lora(A, B, 1.0)
    Y = _forward(layer, d["X"], w.M)
    ref = sq.forward(d["X"], gh.oracle_packed(exp)) + sq.lora_delta(d["X"], A, B, 1.0)
    gh.assert_y_close(Y, ref, "mlp_up + lora 32")
    gh.assert_tiles_close(Y, ref, "mlp_up + lora 32")
    layer.close()
