"""GPU parity: the CUDA path through the C ABI against the CPU oracle.

  * kernel 1 (svdq_quantize_act): FP4 codes and E4M3 block scales bit-exact with
    the oracle quantiser given the library's inv_lambda and s_gX; T = X^ L1
    within bf16 accuracy;
  * the full forward (svdq_linear_forward): Y against the oracle's forward
    evaluated on the library's own packed operands (svdq_export), within
    relative Frobenius error 5e-3 and max-abs error 2e-2 * max|Y_ref|;
  * kernel 2 alone on operands the oracle quantised;
  * ragged M, M = 0, two calls in a row, host-buffer entry point, error codes.
Full FLUX-shaped sizes run in the launch configuration the benchmark times;
there Y is compared on every element (and each 256 x 256 output tile on its own)
and kernel 1 on every row.
"""
import numpy as np
import pytest
import torch

from oracle import nvfp4
from oracle import svdquant as sq
from tests import gpu_helpers as gh
from w4a4_rank_corrected_e2m1_b300 import svdq, synthetic

pytestmark = pytest.mark.gpu

_CACHE = {}


def case(w: synthetic.Workload, **pack_kw):
    key = (w, tuple(sorted(pack_kw.items())))
    if key not in _CACHE:
        d = synthetic.make(w)
        layer = svdq.Layer(d["W"], w.rank, bias=d["bias"], Xcal=d["X"], M_max=w.M, **pack_kw)
        exp = layer.export()
        _CACHE[key] = (d, layer, exp)
    return _CACHE[key]


def run_k1(layer, X, M):
    K = layer.K
    codes = torch.empty((max(M, 1), K // 2), dtype=torch.uint8, device="cuda")
    # 0xFF is an E4M3 NaN: any byte kernel 1 leaves unwritten shows up in the comparisons
    scales = torch.full((max(svdq.scales_bytes(M, K), 16),), 0xFF, dtype=torch.uint8, device="cuda")
    r_pad = layer.info.r_pad
    T = torch.empty((max(M, 1), max(r_pad, 8)), dtype=torch.int16, device="cuda") if layer.rank else None
    Xd = gh.dev_u16(X)
    layer.quantize_act(Xd, M, codes, scales, T)
    torch.cuda.synchronize()
    layer.check_error()
    c = gh.unpack_codes(codes.cpu().numpy()[:M])
    s = gh.untile_scales(scales.cpu().numpy(), M, K)
    t = None if T is None else sq.bf16_to_f64(gh.host_u16(T)[:M])
    return c, s, t, scales.cpu().numpy()


def run_forward(layer, X, M):
    Xd = gh.dev_u16(X)
    Y = torch.empty((M, layer.N), dtype=torch.bfloat16, device="cuda")
    layer.forward(Xd, Y, M)
    torch.cuda.synchronize()
    layer.check_error()
    return sq.bf16_to_f64(gh.host_u16(Y.view(torch.int16)))


PARITY = synthetic.parity_cases()


@pytest.mark.parametrize("w", PARITY, ids=lambda w: w.name)
def test_k1_codes_scales_bitexact(w):
    d, layer, exp = case(w)
    c, s, t, raw = run_k1(layer, d["X"], w.M)
    rc, rs, xh = sq.quantize_act(d["X"], exp["inv_lambda"], exp["s_gX"])
    assert np.array_equal(s, rs), f"scale mismatches: {np.sum(s != rs)}"
    assert np.array_equal(c, rc), f"code mismatches: {np.sum(c != rc)}"
    # rows past M in the last 128-row tile hold zero scales
    full = gh.untile_scales(raw, ((w.M + 127) // 128) * 128, w.K)
    assert np.all(full[w.M:] == 0)
    if w.rank:
        Tref = sq.lowrank_down(xh, exp["L1"])
        T = t[:, : w.rank] * np.float64(exp["alpha"])
        rel = np.linalg.norm(T - Tref) / np.linalg.norm(Tref)
        assert rel < 4e-3, rel
        assert np.all(t[:, w.rank:] == 0)


def test_k1_rounding_edges():
    """Exact E2M1 ties, -0, negative values that round to zero, saturation and zero blocks.
    lambda = 1 and s_gX = 1 make x^ = x and, for an amax of 6, d = 1 so q = x exactly."""
    K, N = 256, 64
    ties = [6.0, 0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, -0.25, -0.75, -1.25, -1.75, -2.5, -3.5, -5.0, -0.0]
    rows = [ties * (K // 16),
            [6.0, -0.1, -0.2, 0.1, -0.0, 0.0, -1e-3, 5.9, -6.0, 0.24, -0.26, 0.74, -0.76, 4.9, -5.1, 3.0] * (K // 16),
            [0.0] * K,
            [-0.0] * K,
            [3000.0] + [1.0] * (K - 1),              # scale saturates at 448
            [1e-4] * K]                               # scale underflows to 0
    rng = np.random.default_rng(5)
    rows += [list(rng.standard_normal(K) * 10 ** rng.uniform(-2, 2)) for _ in range(26)]
    X = synthetic.f64_to_bf16_bits(np.array(rows))
    W = synthetic.f64_to_bf16_bits(rng.standard_normal((N, K)) / 16)
    layer = svdq.Layer(W, 0, smooth=False, s_gX=1.0, M_max=len(rows))
    exp = layer.export()
    assert exp["s_gX"] == 1.0
    c, s, _, _ = run_k1(layer, X, len(rows))
    rc, rs, _ = sq.quantize_act(X, exp["inv_lambda"], exp["s_gX"])
    assert np.array_equal(s, rs)
    bad = np.argwhere(c != rc)
    assert bad.size == 0, [(int(i), int(j), float(sq.bf16_to_f64(X[i, j])), int(c[i, j]), int(rc[i, j])) for i, j in bad[:8]]
    assert np.all(rc[0, :16] == nvfp4.e2m1_encode(np.float32(ties)))


def test_k1_scale_code_boundaries():
    """Block maxima exactly at every E4M3 rounding midpoint (times 6, so that with s_gX = 1 the
    raw scale amax / 6 is the midpoint itself) and one bf16 step to either side."""
    from oracle import nvfp4 as nv
    vals = nv.e4m3_decode(np.arange(0, 127, dtype=np.uint8))
    mids = (vals[:-1] + vals[1:]) / 2
    amax = np.concatenate([6 * mids, 6 * vals[1:]])
    bits = synthetic.f64_to_bf16_bits(amax)
    cand = np.concatenate([bits, bits + np.uint16(1), bits - np.uint16(1)])
    amaxv = sq.bf16_to_f64(cand)
    amaxv = amaxv[(amaxv > 0) & (amaxv < 6 * 448)]
    rng = np.random.default_rng(9)
    K = 256
    nblk = len(amaxv)
    rows = int(np.ceil(nblk / (K // 16)))
    X = np.zeros((rows, K))
    for b, am in enumerate(amaxv):
        r, j = divmod(b, K // 16)
        blk = rng.uniform(-1, 1, 16) * am * 0.9
        blk[rng.integers(16)] = am if rng.random() < 0.5 else -am
        X[r, 16 * j:16 * j + 16] = blk
    Xb = synthetic.f64_to_bf16_bits(X)
    W = synthetic.f64_to_bf16_bits(rng.standard_normal((64, K)) / 16)
    layer = svdq.Layer(W, 0, smooth=False, s_gX=1.0, M_max=rows)
    exp = layer.export()
    c, s, _, _ = run_k1(layer, Xb, rows)
    rc, rs, _ = sq.quantize_act(Xb, exp["inv_lambda"], exp["s_gX"])
    assert np.array_equal(s, rs), f"scale mismatches {np.sum(s != rs)}"
    assert np.array_equal(c, rc)


@pytest.mark.parametrize("w", PARITY, ids=lambda w: w.name)
def test_forward_matches_oracle(w):
    d, layer, exp = case(w)
    Y = run_forward(layer, d["X"], w.M)
    ref = sq.forward(d["X"], gh.oracle_packed(exp))
    gh.assert_y_close(Y, ref, w.name)


@pytest.mark.parametrize("M", [1, 7, 64, 127, 129, 300])
def test_ragged_m(M):
    w = PARITY[1]
    d, layer, exp = case(w)
    X = d["X"][:M]
    Y = run_forward(layer, X, M)
    ref = sq.forward(X, gh.oracle_packed(exp))
    gh.assert_y_close(Y, ref, f"M={M}")


def test_m_zero_is_noop():
    w = PARITY[0]
    d, layer, exp = case(w)
    Y = torch.full((4, layer.N), 7.0, dtype=torch.bfloat16, device="cuda")
    layer.forward(gh.dev_u16(d["X"]), Y, 0)
    torch.cuda.synchronize()
    assert torch.all(Y == 7.0)


def test_gemm_on_oracle_operands():
    """Kernel 2 alone, fed the oracle's quantised activations and T."""
    w = PARITY[1]
    d, layer, exp = case(w)
    M, K = w.M, w.K
    p = gh.oracle_packed(exp)
    cx, sx, xh = sq.quantize_act(d["X"], p["inv_lambda"], p["s_gX"])
    packed = (cx[:, 0::2] | (cx[:, 1::2] << 4)).astype(np.uint8)
    Tref = sq.lowrank_down(xh, p["L1"]) / np.float64(exp["alpha"])
    r_pad = layer.info.r_pad
    Tp = np.zeros((M, r_pad))
    Tp[:, : w.rank] = Tref
    codes = torch.from_numpy(packed).cuda()
    scales = torch.from_numpy(gh.tile_scales(sx, M, K)).cuda()
    T = gh.dev_u16(sq.f64_to_bf16(Tp))
    Y = torch.empty((M, layer.N), dtype=torch.bfloat16, device="cuda")
    layer.gemm_quantized(codes, scales, T, Y, M)
    torch.cuda.synchronize()
    layer.check_error()
    got = sq.bf16_to_f64(gh.host_u16(Y.view(torch.int16)))
    ref = sq.forward(d["X"], p)
    gh.assert_y_close(got, ref, "gemm_quantized")


def test_fp4_product_within_fp32_summation_bound():
    """rank 0: Y = alpha * (exact sum of E2M1 x E4M3 products) + b; the FP32 tensor-core
    accumulator must stay within the FP32 summation bound of the exact sum."""
    w = synthetic.scaled(synthetic.QKV, name="r0", M=256, K=1024, N=512, rank=0, n_outlier=4)
    d = synthetic.make(w)
    layer = svdq.Layer(d["W"], 0, bias=d["bias"], Xcal=d["X"], M_max=w.M)
    exp = layer.export()
    Y = run_forward(layer, d["X"], w.M)
    p = gh.oracle_packed(exp)
    cx, sx, _ = sq.quantize_act(d["X"], p["inv_lambda"], p["s_gX"])
    Xd = nvfp4.dequantize_blocks(cx, sx)
    Rd = nvfp4.dequantize_blocks(p["R_codes"], p["R_scales"])
    a = np.float64(sq.alpha(p))
    exact = a * (Xd @ Rd.T) + sq.bf16_to_f64(p["bias"])[None, :]
    bound = a * (np.abs(Xd) @ np.abs(Rd).T) * (w.K * 2.0 ** -24) + np.abs(exact) * 2.0 ** -8
    assert np.all(np.abs(Y - exact) <= bound + 1e-30)


def test_two_calls_identical_and_host_entry():
    w = PARITY[1]
    d, layer, exp = case(w)
    Y1 = run_forward(layer, d["X"], w.M)
    Y2 = run_forward(layer, d["X"], w.M)
    assert np.array_equal(Y1, Y2)
    layer.reserve(w.M, host_staging=True)
    Xh = torch.from_numpy(d["X"].view(np.int16)).pin_memory()
    Yh = torch.empty((w.M, layer.N), dtype=torch.int16).pin_memory()
    layer.forward_host(Xh, Yh, w.M)
    assert np.array_equal(sq.bf16_to_f64(Yh.numpy().view(np.uint16)), Y1)


def test_caller_workspace():
    w = PARITY[0]
    d = synthetic.make(w)
    layer = svdq.Layer(d["W"], w.rank, bias=d["bias"], Xcal=d["X"])
    with pytest.raises(svdq.SvdqError) as e:
        run_forward(layer, d["X"], w.M)
    assert e.value.status == svdq.ERR_WORKSPACE
    nbytes = layer.workspace_size(w.M)
    buf = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    layer.set_workspace(buf, w.M)
    Y = run_forward(layer, d["X"], w.M)
    gh.assert_y_close(Y, sq.forward(d["X"], gh.oracle_packed(layer.export())), "caller workspace")
    with pytest.raises(svdq.SvdqError) as e:
        run_forward(layer, np.concatenate([d["X"], d["X"]]), 2 * w.M)
    assert e.value.status == svdq.ERR_WORKSPACE


def test_error_statuses():
    rng = np.random.default_rng(0)
    W = synthetic.f64_to_bf16_bits(rng.standard_normal((64, 96)))
    with pytest.raises(svdq.SvdqError) as e:
        svdq.Layer(W, 16)                                  # K % 64 != 0
    assert e.value.status == svdq.ERR_UNSUPPORTED_SHAPE
    W = synthetic.f64_to_bf16_bits(rng.standard_normal((64, 128)))
    with pytest.raises(svdq.SvdqError) as e:
        svdq.Layer(W, 24)                                  # rank % 16 != 0
    assert e.value.status == svdq.ERR_UNSUPPORTED_SHAPE
    layer = svdq.Layer(W, 16, M_max=8)
    X = torch.zeros((9, 128), dtype=torch.int16, device="cuda")
    Y = torch.zeros((9, 64), dtype=torch.int16, device="cuda")
    with pytest.raises(svdq.SvdqError) as e:
        layer.forward(X[1:].view(-1)[1:], Y, 4)            # misaligned pointer
    assert e.value.status == svdq.ERR_INVALID_ARG
    with pytest.raises(svdq.SvdqError) as e:
        layer.forward(X, X, 8)                             # aliasing
    assert e.value.status == svdq.ERR_INVALID_ARG
    with pytest.raises(svdq.SvdqError) as e:
        layer.forward(X, X.view(-1)[256:], 4)              # Y starts inside X's first 4 rows
    assert e.value.status == svdq.ERR_INVALID_ARG and b"overlap" in svdq.LIB.svdq_last_error()
    layer.forward(X, X.view(-1)[512:], 4)                  # Y right after X's 4 rows: allowed
    with pytest.raises(svdq.SvdqError) as e:
        layer.forward(X, Y, 9)                             # above the workspace
    assert e.value.status == svdq.ERR_WORKSPACE
    layer.check_error()


def test_ragged_n_and_k():
    """N not a multiple of the 256-wide tile and K not a multiple of the 256-wide stage."""
    w = synthetic.scaled(synthetic.QKV, name="ragged", M=200, K=320, N=272, rank=16, n_outlier=3)
    d, layer, exp = case(w)
    c, s, _, raw = run_k1(layer, d["X"], w.M)
    rc, rs, _ = sq.quantize_act(d["X"], exp["inv_lambda"], exp["s_gX"])
    assert np.array_equal(c, rc) and np.array_equal(s, rs)
    # scale groups past K (K = 320: groups 5..7 of each 128-row tile) must be zero scales
    KG = 4 * -(-w.K // 256)
    tiles = raw[: -(-w.M // 128) * KG * 512].reshape(-1, KG, 512)
    assert np.all(tiles[:, w.K // 64:, :] == 0)
    Y = run_forward(layer, d["X"], w.M)
    gh.assert_y_close(Y, sq.forward(d["X"], gh.oracle_packed(exp)), "ragged")


@pytest.mark.parametrize("rank", [16, 32, 48, 64, 96])
def test_tall_path_ragged_m_and_odd_chunk_count(rank):
    """M large enough for the whole-K 32-row kernel, M % 32 != 0, K with an odd number of
    64-column chunks (the last stage's later chunks are past K) and K % 256 != 0; ranks on
    both down-projection forms (four chunks in one product for r <= 64, one per chunk above)."""
    w = synthetic.scaled(synthetic.QKV, name="tall_ragged", M=2413, K=576, N=256, rank=rank, n_outlier=6)
    d, layer, exp = case(w)
    c, s, t, raw = run_k1(layer, d["X"], w.M)
    rc, rs, xh = sq.quantize_act(d["X"], exp["inv_lambda"], exp["s_gX"])
    assert np.array_equal(c, rc) and np.array_equal(s, rs)
    KG = 4 * -(-w.K // 256)
    tiles = raw[: -(-w.M // 128) * KG * 512].reshape(-1, KG, 512)
    assert np.all(tiles[:, w.K // 64:, :] == 0)
    # T' = (X^ L1) / alpha against the oracle's float64 down-projection
    tref = sq.lowrank_down(xh, exp["L1"]) / float(exp["alpha"])
    assert np.max(np.abs(t[:, :w.rank] - tref)) <= 2e-2 * np.max(np.abs(tref))
    assert np.all(t[:, w.rank:] == 0)
    Y = run_forward(layer, d["X"], w.M)
    gh.assert_y_close(Y, sq.forward(d["X"], gh.oracle_packed(exp)), "tall ragged")


@pytest.mark.parametrize("w", [synthetic.QKV, synthetic.scaled(synthetic.MLP_DOWN, name="down_m1024", M=1024)],
                         ids=lambda w: w.name)
def test_k1_bitexact_on_repeated_launches(w):
    """Kernel 1 run back to back (whole-K 32-row kernel for QKV, split-K kernel for 1024
    tokens of the MLP down-projection, K = 12288): every launch is bit-exact.  A missing
    ordering between the quantiser's reads of a stage and the copies that refill it shows up
    here as a few blocks read from the wrong step."""
    d, layer, exp = case(w)
    rc, rs, _ = sq.quantize_act(d["X"], exp["inv_lambda"], exp["s_gX"])
    for i in range(6):
        c, s, _, _ = run_k1(layer, d["X"], w.M)
        assert np.array_equal(s, rs), f"launch {i}: scale mismatches {np.sum(s != rs)}"
        assert np.array_equal(c, rc), f"launch {i}: code mismatches {np.sum(c != rc)}"


# ------------------------------------------------------------------ full FLUX-shaped sizes
FULL = [synthetic.QKV, synthetic.MLP_UP, synthetic.MLP_DOWN, *synthetic.OPROJ_M, *synthetic.OPROJ_R]


@pytest.mark.parametrize("w", FULL, ids=lambda w: w.name)
def test_full_size(w):
    d, layer, exp = case(w)
    # kernel 1 on every row, bit-exact
    c, s, t, _ = run_k1(layer, d["X"], w.M)
    rc, rs, xh = sq.quantize_act(d["X"], exp["inv_lambda"], exp["s_gX"])
    assert np.array_equal(s, rs), f"scale mismatches {np.sum(s != rs)}"
    assert np.array_equal(c, rc), f"code mismatches {np.sum(c != rc)}"
    del c, rc, s, rs, t, xh
    # Y on every element, plus every 256 x 256 output tile on its own
    Y = run_forward(layer, d["X"], w.M)
    ref = sq.forward(d["X"], gh.oracle_packed(exp))
    gh.assert_y_close(Y, ref, w.name)
    gh.assert_tiles_close(Y, ref, w.name)
