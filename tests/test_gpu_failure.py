"""Failure detection on the GPU, without faulting it.

Every wait inside the kernels is bounded; when one runs out the kernel records a timeout in the
handle's device error word, waits out the work it started (copies in flight, MMAs issued) and
returns, and svdq_check_error reports SVDQ_ERR_TIMEOUT.  The tests make a wait run out on purpose
with the library's stall hook: the MMA warp of kernel 1 or kernel 2 waits on a barrier that
nothing completes, under a 1 ms limit.  Afterwards the same handle, back at the default limit,
must compute the layer correctly: the context is still usable.  A workspace request far beyond
device memory must report SVDQ_ERR_OOM and leave the handle's workspace as it was.
"""
import numpy as np
import pytest
import torch

from oracle import svdquant as sq
from tests import gpu_helpers as gh
from w4a4_rank_corrected_e2m1_b300 import svdq, synthetic

pytestmark = pytest.mark.gpu

QKV_SMALL = synthetic.parity_cases()[1]        # kernel 1 whole-K path
DOWN_SPLIT = synthetic.parity_cases()[4]       # kernel 1 split-K path (K = 6464)


def _forward(layer, X, M):
    Y = torch.full((M, layer.N), float("nan"), dtype=torch.bfloat16, device="cuda")
    layer.forward(gh.dev_u16(X), Y, M)
    return Y


@pytest.mark.parametrize("w", [QKV_SMALL, DOWN_SPLIT], ids=lambda w: w.name)
@pytest.mark.parametrize("kernel", [1, 2])
def test_stalled_wait_reports_timeout_and_the_handle_recovers(w, kernel):
    d = synthetic.make(w)
    layer = svdq.Layer(d["W"], w.rank, bias=d["bias"], Xcal=d["X"], M_max=w.M)
    ref = sq.forward(d["X"], gh.oracle_packed(layer.export()))
    layer.set_wait_limit(1_000_000, kernel)                    # 1 ms, this kernel's MMA warp stalls
    _forward(layer, d["X"], w.M)
    with pytest.raises(svdq.SvdqError) as e:
        layer.check_error()
    assert e.value.status == svdq.ERR_TIMEOUT
    layer.check_error()                                        # the error word was cleared
    layer.set_wait_limit(0, 0)                                 # default limit, no stall
    Y = _forward(layer, d["X"], w.M)
    torch.cuda.synchronize()
    layer.check_error()
    gh.assert_y_close(sq.bf16_to_f64(gh.host_u16(Y.view(torch.int16))), ref, f"{w.name} after a stall")
    layer.close()


def test_wait_limit_arguments():
    w = synthetic.TINY
    d = synthetic.make(w)
    layer = svdq.Layer(d["W"], w.rank, bias=d["bias"], Xcal=d["X"], M_max=w.M)
    with pytest.raises(svdq.SvdqError) as e:
        layer.set_wait_limit(0, 3)
    assert e.value.status == svdq.ERR_INVALID_ARG
    layer.close()


def test_workspace_beyond_device_memory_reports_oom():
    w = QKV_SMALL
    d = synthetic.make(w)
    layer = svdq.Layer(d["W"], w.rank, bias=d["bias"], Xcal=d["X"], M_max=w.M)
    ref = sq.forward(d["X"], gh.oracle_packed(layer.export()))
    with pytest.raises(svdq.SvdqError) as e:
        layer.reserve(1 << 40)                                 # ~1.7 PB of scratch
    assert e.value.status == svdq.ERR_OOM
    assert layer.info.M_max == w.M                             # the old workspace stays
    Y = _forward(layer, d["X"], w.M)
    torch.cuda.synchronize()
    layer.check_error()
    gh.assert_y_close(sq.bf16_to_f64(gh.host_u16(Y.view(torch.int16))), ref, "after a failed reserve")
    layer.close()
