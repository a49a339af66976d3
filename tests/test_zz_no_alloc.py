"""svdq_linear_forward_noalloc: the forward for callers that cannot allocate device memory.

Callers running under a framework's memory pool or budget, or in a latency-critical loop that
cannot take cudaMalloc's implicit synchronisation, cannot let a library allocate.  This entry
point takes its scratch from a statically sized device array held by the library, so it
allocates nothing.  Here it is called through the C ABI and compared bit for bit with
svdq_linear_forward (the entry point that uses the handle's workspace): both run the same
kernels on the same inputs, and kernel 1's split-K partial sums are added in a fixed order, so
the outputs must be identical.  The cases cover both kernel-1 paths (whole-K and split-K, whose
arrival words live in the shared array), called alternately through different handles and with
calls of another layer and size in between, so every call starts from another call's leftover
contents and epochs.  Each reference output is also checked against the CPU oracle.  This file
is collected last on purpose: if it fails, a run that stops at the first failure has already
run every other test.
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

_STATIC_BYTES = 32 << 20


def _forward_noalloc(layer, X, Y, M):
    return _fn(layer.h, X.data_ptr(), Y.data_ptr(), M, torch.cuda.current_stream().cuda_stream)


def _setup(w):
    d = synthetic.make(w)
    layer = svdq.Layer(d["W"], w.rank, bias=d["bias"], Xcal=d["X"], M_max=w.M)
    X = gh.dev_u16(d["X"])
    Y_ref = torch.empty((w.M, layer.N), dtype=torch.bfloat16, device="cuda")
    layer.forward(X, Y_ref, w.M)
    torch.cuda.synchronize()
    layer.check_error()
    return d, layer, X, Y_ref


def test_noalloc_bitexact_with_workspace_forward_across_handles():
    cases = [synthetic.parity_cases()[1], synthetic.TINY, synthetic.parity_cases()[4]]
    assert cases[2].name == "down_split"                 # K = 6464 at M = 300: split-K kernel 1
    # another layer and size whose call fills the front of the array with its own codes,
    # scales and T (about 15 MB), over every offset the cases above use
    filler = synthetic.scaled(synthetic.QKV, name="filler", M=8192, K=3072, N=256, rank=32, n_outlier=31)
    runs = {w.name: _setup(w) for w in cases + [filler]}
    for w in cases:                                      # the reference path against the oracle
        d, layer, _, Y_ref = runs[w.name]
        ref = sq.forward(d["X"], gh.oracle_packed(layer.export()))
        gh.assert_y_close(sq.bf16_to_f64(gh.host_u16(Y_ref.view(torch.int16))), ref, w.name)
    order = ["filler", "qkv_small", "tiny", "down_split", "qkv_small", "down_split", "tiny",
             "filler", "down_split", "down_split", "qkv_small"]
    for i, name in enumerate(order):
        d, layer, X, Y_ref = runs[name]
        M = X.shape[0]
        Y = torch.full((M, layer.N), float("nan"), dtype=torch.bfloat16, device="cuda")
        assert _forward_noalloc(layer, X, Y, M) == svdq.OK, svdq.LIB.svdq_last_error()
        torch.cuda.synchronize()
        layer.check_error()
        if name != "filler":
            same = torch.equal(Y.view(torch.int16), Y_ref.view(torch.int16))
            assert same, f"call {i} ({name}): {int((Y.view(torch.int16) != Y_ref.view(torch.int16)).sum())} differ"
    for _, layer, _, _ in runs.values():
        layer.close()


def test_noalloc_rejects_sizes_beyond_the_static_scratch_and_overlaps():
    rng = np.random.default_rng(3)
    K, N = 3072, 256
    W = synthetic.f64_to_bf16_bits(rng.standard_normal((N, K)) / 50)
    layer = svdq.Layer(W, 32, s_gX=1.0)
    X = torch.zeros((8, K), dtype=torch.int16, device="cuda")
    Y = torch.zeros((8, N), dtype=torch.int16, device="cuda")
    M_big = 32768                                   # needs well over 32 MiB of scratch
    assert layer.workspace_size(M_big) > _STATIC_BYTES
    assert _forward_noalloc(layer, X, Y, M_big) == svdq.ERR_WORKSPACE
    assert b"static scratch" in svdq.LIB.svdq_last_error()
    # Y starting inside X's rows
    buf = torch.zeros((8, K + N), dtype=torch.int16, device="cuda")
    st = _fn(layer.h, buf.data_ptr(), buf.data_ptr() + 1024, 8, torch.cuda.current_stream().cuda_stream)
    assert st == svdq.ERR_INVALID_ARG
    assert b"overlap" in svdq.LIB.svdq_last_error()
    layer.close()
