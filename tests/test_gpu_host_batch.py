"""Pipelined host-buffer calls (svdq_linear_forward_host_batch): every step's Y equals the same
layer's device-buffer forward on that step's X, bit for bit, while uploads, kernels and
downloads of neighbouring steps overlap."""
from __future__ import annotations

import numpy as np
import pytest
import torch

from oracle import svdquant as sq
from tests import gpu_helpers as gh
from w4a4_rank_corrected_e2m1_b300 import svdq, synthetic

pytestmark = pytest.mark.gpu


def _device_forward(layer, X, M):
    Y = torch.empty((M, layer.N), dtype=torch.bfloat16, device="cuda")
    layer.forward(gh.dev_u16(X), Y, M)
    torch.cuda.synchronize()
    layer.check_error()
    return gh.host_u16(Y.view(torch.int16))


def _pinned(a):
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).pin_memory()


@pytest.mark.parametrize("w,B", [(synthetic.parity_cases()[1], 5),
                                 (synthetic.scaled(synthetic.QKV, name="qkv_ragged", M=257, K=512, N=272, rank=16), 4),
                                 (synthetic.MLP_UP, 3)],
                         ids=["qkv_small_B5", "ragged_B4", "mlp_up_B3"])
def test_batch_matches_device_forward(w, B):
    d = synthetic.make(w)
    layer = svdq.Layer(d["W"], w.rank, bias=d["bias"], Xcal=d["X"], M_max=w.M)
    Xs = [synthetic.make_x(w, w.M, seed=100 + b) for b in range(B)]
    expect = [_device_forward(layer, X, w.M) for X in Xs]
    layer.reserve(w.M, host_staging=2)
    Xh = [_pinned(X) for X in Xs]
    Yh = [torch.full((w.M, layer.N), -1, dtype=torch.int16).pin_memory() for _ in range(B)]
    layer.forward_host_batch(Xh, Yh, w.M)
    layer.check_error()
    for b in range(B):
        assert np.array_equal(Yh[b].numpy().view(np.uint16), expect[b]), f"step {b}"
    # a second batch on the same handle reuses the streams, events and slots
    Yh2 = [torch.full((w.M, layer.N), -1, dtype=torch.int16).pin_memory() for _ in range(B)]
    layer.forward_host_batch(Xh[::-1], Yh2, w.M)
    for b in range(B):
        assert np.array_equal(Yh2[b].numpy().view(np.uint16), expect[B - 1 - b]), f"second batch step {b}"
    layer.close()


def test_batch_against_oracle_small():
    w = synthetic.parity_cases()[1]
    d = synthetic.make(w)
    layer = svdq.Layer(d["W"], w.rank, bias=d["bias"], Xcal=d["X"], M_max=w.M)
    layer.reserve(w.M, host_staging=2)
    Xh = [_pinned(d["X"])]
    Yh = [torch.empty((w.M, layer.N), dtype=torch.int16).pin_memory()]
    layer.forward_host_batch(Xh, Yh, w.M)
    Y = sq.bf16_to_f64(Yh[0].numpy().view(np.uint16))
    gh.assert_y_close(Y, sq.forward(d["X"], gh.oracle_packed(layer.export())), "host batch")
    layer.close()


def test_batch_errors_and_empty():
    w = synthetic.parity_cases()[0]
    d = synthetic.make(w)
    layer = svdq.Layer(d["W"], w.rank, bias=d["bias"], Xcal=d["X"], M_max=w.M)
    Xh = [_pinned(d["X"])]
    Yh = [torch.empty((w.M, layer.N), dtype=torch.int16).pin_memory()]
    # one staging slot is not enough
    layer.reserve(w.M, host_staging=1)
    with pytest.raises(svdq.SvdqError) as e:
        layer.forward_host_batch(Xh, Yh, w.M)
    assert e.value.status == svdq.ERR_WORKSPACE
    layer.reserve(w.M, host_staging=2)
    # M too large for the workspace
    with pytest.raises(svdq.SvdqError) as e:
        layer.forward_host_batch(Xh, Yh, w.M + 1)
    assert e.value.status == svdq.ERR_WORKSPACE
    # empty batch and M = 0 do nothing
    layer.forward_host_batch([], [], w.M)
    layer.forward_host_batch(Xh, Yh, 0)
    # a null host pointer in the list
    with pytest.raises(svdq.SvdqError) as e:
        layer.forward_host_batch([None], Yh, w.M)
    assert e.value.status == svdq.ERR_INVALID_ARG
    layer.check_error()
    layer.close()
