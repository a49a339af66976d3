"""svdq_linear_forward_noalloc: the forward for callers that cannot allocate device memory.

Callers running inside a framework's memory pool, inside CUDA graph capture or in a
latency-critical loop cannot let a library call cudaMalloc.  This entry point takes its scratch
from a statically sized device array held by the library, so it allocates nothing.  Here it is
called through the C ABI and compared with svdq_linear_forward (the entry point that uses the
handle's workspace) on the same inputs, twice in a row, so that leftover scratch contents from
the first call cannot change the second.  This file is collected last on purpose: if it fails, a
run that stops at the first failure has already run every other test.
"""
import ctypes

import numpy as np
import pytest
import torch

from oracle import svdquant as sq
from tests import gpu_helpers as gh
from w4a4_rank_corrected_e2m1_b300 import svdq, synthetic

pytestmark = pytest.mark.gpu

_fn = svdq.LIB.svdq_linear_forward_noalloc
_fn.restype = ctypes.c_int32
_fn.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p]


def _forward_noalloc(layer, X, Y, M):
    st = _fn(layer.h, X.data_ptr(), Y.data_ptr(), M, torch.cuda.current_stream().cuda_stream)
    return st


@pytest.mark.parametrize("w", [synthetic.parity_cases()[1], synthetic.TINY], ids=lambda w: w.name)
def test_noalloc_matches_workspace_forward_twice(w):
    d = synthetic.make(w)
    layer = svdq.Layer(d["W"], w.rank, bias=d["bias"], Xcal=d["X"], M_max=w.M)
    X = gh.dev_u16(d["X"])
    Y_ref = torch.empty((w.M, layer.N), dtype=torch.bfloat16, device="cuda")
    layer.forward(X, Y_ref, w.M)
    torch.cuda.synchronize()
    ref = sq.bf16_to_f64(gh.host_u16(Y_ref.view(torch.int16)))
    for call in range(2):
        Y = torch.full((w.M, layer.N), float("nan"), dtype=torch.bfloat16, device="cuda")
        assert _forward_noalloc(layer, X, Y, w.M) == svdq.OK, svdq.LIB.svdq_last_error()
        torch.cuda.synchronize()
        layer.check_error()
        got = sq.bf16_to_f64(gh.host_u16(Y.view(torch.int16)))
        gh.assert_y_close(got, ref, f"{w.name} call {call}")
    layer.close()


def test_noalloc_rejects_sizes_beyond_the_static_scratch():
    rng = np.random.default_rng(3)
    K, N = 3072, 256
    W = synthetic.f64_to_bf16_bits(rng.standard_normal((N, K)) / 50)
    layer = svdq.Layer(W, 32, s_gX=1.0)
    X = torch.zeros((8, K), dtype=torch.int16, device="cuda")
    Y = torch.zeros((8, N), dtype=torch.int16, device="cuda")
    M_big = 32768                                   # needs well over 32 MiB of scratch
    assert layer.workspace_size(M_big) > (32 << 20)
    assert _forward_noalloc(layer, X, Y, M_big) == svdq.ERR_WORKSPACE
    assert b"static scratch" in svdq.LIB.svdq_last_error()
    layer.close()
