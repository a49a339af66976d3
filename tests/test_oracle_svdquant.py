"""Pins for the oracle's SVDQuant pipeline (CPU only).

The pages print no worked example, so the oracle is pinned by what the method
and the mathematics fix: the smoothing identity, Eckart-Young, the full-rank and
zero-rank special cases, a pure-Python loop evaluation of the forward on a tiny
problem, and the method's claim that the low-rank branch makes 4-bit
quantisation more accurate on outlier-heavy inputs.
"""
import numpy as np
import pytest

from oracle import nvfp4
from oracle import svdquant as sq
from w4a4_rank_corrected_e2m1_b300 import synthetic


@pytest.fixture(scope="module")
def tiny():
    w = synthetic.TINY
    d = synthetic.make(w)
    return w, d


def test_bf16_rounding_matches_torch():
    """float64 -> bf16 with one rounding: torch on float32-exact inputs (where its
    float32 intermediate is exact), and nearest-neighbour brute force on float64 inputs."""
    import torch
    rng = np.random.default_rng(4)
    a = (rng.standard_normal(100000) * np.exp2(rng.uniform(-30, 30, 100000)))
    a32 = a.astype(np.float32).astype(np.float64)
    ours = sq.f64_to_bf16(a32)
    theirs = torch.from_numpy(a32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, theirs)
    b = sq.f64_to_bf16(a)
    v = sq.bf16_to_f64(b)
    up = sq.bf16_to_f64(b + np.uint16(1))        # neighbours in magnitude on the bf16 grid
    dn = sq.bf16_to_f64(b - np.uint16(1))
    assert np.all(np.abs(a - v) <= np.abs(a - up)) and np.all(np.abs(a - v) <= np.abs(a - dn))


def test_smoothing_identity(tiny):
    w, d = tiny
    lam, inv = sq.smoothing_factors(d["X"], d["W"])
    Xh = sq.smooth_act(d["X"], inv).astype(np.float64)
    Wh = sq.smooth_weight(d["W"], lam)
    ref = sq.bf16_to_f64(d["X"]) @ sq.bf16_to_f64(d["W"]).T
    # x^ carries one fp32 rounding and inv_lambda is fl32(1/lambda): error ~ 2^-23
    assert sq.rel_fro(Xh @ Wh.T, ref) < 1e-6
    # outlier channels get the largest lambda (outliers move into the weights)
    top = np.argsort(lam)[-len(d["outlier_channels"]):]
    assert set(top) == set(d["outlier_channels"])
    # lambda follows its closed form on one channel, computed by hand
    c = int(d["outlier_channels"][0])
    xm = np.max(np.abs(sq.bf16_to_f64(d["X"][:, c])))
    wm = np.max(np.abs(sq.bf16_to_f64(d["W"][:, c])))
    assert lam[c] == np.float32(np.sqrt(xm / wm))


def test_smoothing_zero_guard_and_hand_values():
    """lambda_c = sqrt(max|X_c| / max|W_c|); a channel whose activation or weight column is all
    zero keeps lambda = 1 (inv_lambda = 1).  Hand values: max|X| = 4, max|W| = 1 gives lambda 2,
    inv 0.5; max|X| = 1, max|W| = 4 gives 0.5, inv 2."""
    bf = lambda a: sq.f64_to_bf16(np.asarray(a, np.float64))
    X = bf([[4.0, 0.0, 1.0, 3.0, 0.0],
            [-2.0, 0.0, -1.0, 1.0, 0.0]])
    W = bf([[1.0, 5.0, 4.0, 0.0, 0.0],
            [-0.5, -2.0, 0.25, 0.0, 0.0]])
    lam, inv = sq.smoothing_factors(X, W)
    assert lam.dtype == np.float32 and inv.dtype == np.float32
    assert list(lam) == [2.0, 1.0, 0.5, 1.0, 1.0]
    assert list(inv) == [0.5, 1.0, 2.0, 1.0, 1.0]


def test_eckart_young(tiny):
    w, d = tiny
    lam, _ = sq.smoothing_factors(d["X"], d["W"])
    Wh = sq.smooth_weight(d["W"], lam)
    for r in (0, 4, 16, 64):
        L1, L2, _ = sq.lowrank_factors(Wh, r)
        res = np.sum((Wh.T - L1 @ L2) ** 2)
        ev = np.sort(np.linalg.eigvalsh(Wh.T @ Wh))[::-1]       # sigma^2, independent route
        tail = np.sum(np.clip(ev[r:], 0, None))
        assert abs(res - tail) <= 1e-9 * np.sum(ev)
        if r:
            assert np.allclose(L1.T @ L1, np.eye(r), atol=1e-12)   # L1 orthonormal


def test_full_rank_leaves_zero_residual(tiny):
    w, d = tiny
    lam, inv = sq.smoothing_factors(d["X"], d["W"])
    Wh = sq.smooth_weight(d["W"], lam)
    L1, L2, _ = sq.lowrank_factors(Wh, w.K)
    assert np.linalg.norm(Wh - (L1 @ L2).T) <= 1e-12 * np.linalg.norm(Wh)
    p = sq.pack(d["W"], d["bias"], w.K, Xcal_bits=d["X"])
    # only the bf16 rounding of the factors is left in R
    assert np.linalg.norm(p["R"]) < 2 ** -7 * np.linalg.norm(Wh)
    Y = sq.forward(d["X"], p)
    ref = sq.exact_product(d["X"], d["W"], d["bias"])
    assert sq.rel_fro(Y, ref) < 2e-3


def test_unsmoothed_rank0_is_plain_w4a4(tiny):
    w, d = tiny
    p = sq.pack(d["W"], d["bias"], 0, Xcal_bits=None, smooth=False)
    wf = sq.bf16_to_f32(d["W"])
    cw, sw = nvfp4.quantize_blocks(wf, nvfp4.global_scale(np.max(np.abs(wf))))
    assert np.array_equal(p["R_codes"], cw) and np.array_equal(p["R_scales"], sw)
    assert np.array_equal(p["R"], wf)
    x = sq.bf16_to_f32(d["X"])
    p["s_gX"] = nvfp4.global_scale(np.max(np.abs(x)))
    cx, sx, _ = sq.quantize_act(d["X"], p["inv_lambda"], p["s_gX"])
    cx2, sx2 = nvfp4.quantize_blocks(x, p["s_gX"])
    assert np.array_equal(cx, cx2) and np.array_equal(sx, sx2)
    assert np.allclose(sq.forward(d["X"], p), sq.naive_w4a4(d["X"], d["W"], d["bias"]), rtol=0, atol=1e-12)


def test_forward_against_python_loops():
    """4 x 16 x 16 (and 3 x 32 x 5): the forward written as explicit scalar loops."""
    for (M, K, N, r) in [(4, 16, 16, 4), (3, 32, 5, 2)]:
        w = synthetic.scaled(synthetic.TINY, M=M, K=K, N=N, rank=r, n_outlier=1, spike_rank=1)
        d = synthetic.make(w, seed=7)
        p = sq.pack(d["W"], d["bias"], r, Xcal_bits=d["X"])
        Y = sq.forward(d["X"], p)
        cx, sx, xh = sq.quantize_act(d["X"], p["inv_lambda"], p["s_gX"])
        L1 = sq.bf16_to_f64(p["L1"])
        L2 = sq.bf16_to_f64(p["L2"])
        b = sq.bf16_to_f64(p["bias"])
        a = float(np.float32(p["s_gX"]) * np.float32(p["s_gW"]))
        for m in range(M):
            for n in range(N):
                acc = 0.0
                for k in range(K):
                    xv = float(nvfp4.e2m1_decode(cx[m, k])) * float(nvfp4.e4m3_decode(sx[m, k // 16]))
                    wv = float(nvfp4.e2m1_decode(p["R_codes"][n, k])) * float(nvfp4.e4m3_decode(p["R_scales"][n, k // 16]))
                    acc += xv * wv
                lr = 0.0
                for j in range(r):
                    t = 0.0
                    for k in range(K):
                        t += float(xh[m, k]) * L1[k, j]
                    lr += t * L2[j, n]
                assert abs(a * acc + lr + b[n] - Y[m, n]) <= 1e-9 * (1 + abs(Y[m, n]))


@pytest.mark.parametrize("name", ["tiny", "qkv_small"])
def test_svdquant_beats_naive_w4a4_on_outliers(name):
    w = {c.name: c for c in synthetic.parity_cases()}[name]
    d = synthetic.make(w)
    ref = sq.exact_product(d["X"], d["W"], d["bias"])
    p = sq.pack(d["W"], d["bias"], w.rank, Xcal_bits=d["X"])
    e_svdq = sq.rel_fro(sq.forward(d["X"], p), ref)
    e_naive = sq.rel_fro(sq.naive_w4a4(d["X"], d["W"], d["bias"]), ref)
    assert e_svdq < e_naive, (e_svdq, e_naive)


def test_residual_against_rounded_factors(tiny):
    w, d = tiny
    p = sq.pack(d["W"], d["bias"], w.rank, Xcal_bits=d["X"])
    Wh = sq.smooth_weight(d["W"], p["lam"])
    LL = sq.bf16_to_f64(p["L1"]) @ sq.bf16_to_f64(p["L2"])
    assert np.array_equal(p["R"], (Wh - LL.T).astype(np.float32))
    # the rank-r branch carries the spike: the residual is much smaller than W^
    assert np.linalg.norm(p["R"]) < 0.8 * np.linalg.norm(Wh)


# ------------------------------------------------------------------ LoRA term
def _lora_case(seed, M=6, K=16, N=12, r=3):
    rng = np.random.default_rng(seed)
    X = sq.f64_to_bf16(rng.standard_normal((M, K)))
    A = sq.f64_to_bf16(rng.standard_normal((K, r)))
    B = sq.f64_to_bf16(rng.standard_normal((r, N)))
    return X, A, B


def test_lora_delta_against_python_loops():
    """Brute force on a tiny case: sum_j sum_k x_ik a_kj b_jn, written as loops."""
    X, A, B = _lora_case(11)
    x, a, b = sq.bf16_to_f64(X), sq.bf16_to_f64(A), sq.bf16_to_f64(B)
    M, K = x.shape
    r, N = b.shape
    ref = np.zeros((M, N))
    for i in range(M):
        for n in range(N):
            acc = 0.0
            for j in range(r):
                t = 0.0
                for k in range(K):
                    t += x[i, k] * a[k, j]
                acc += t * b[j, n]
            ref[i, n] = 0.75 * acc
    got = sq.lora_delta(X, A, B, 0.75)
    assert np.allclose(got, ref, rtol=1e-13, atol=1e-12)


def test_lora_delta_zero_and_linear_in_scale():
    X, A, B = _lora_case(12)
    assert np.all(sq.lora_delta(X, A, np.zeros_like(B), 3.0) == 0.0)
    assert np.all(sq.lora_delta(X, A, B, 0.0) == 0.0)
    d1 = sq.lora_delta(X, A, B, 1.0)
    assert np.allclose(sq.lora_delta(X, A, B, -2.5), -2.5 * d1, rtol=1e-14, atol=1e-14)


def test_lora_delta_rows_subset_matches_full():
    X, A, B = _lora_case(13, M=9)
    full = sq.lora_delta(X, A, B, 0.5)
    rows = np.array([0, 4, 8])
    assert np.array_equal(sq.lora_delta(X, A, B, 0.5, rows=rows), full[rows])


# ----------------------------------------------------------------------------- INT4 variant
def _naive_int4(X_bits, W_bits, bias_bits):
    """Plain INT4 W4A4 (64-element groups) without smoothing or low-rank branch."""
    from oracle import int4
    cx, sx = int4.quantize_groups(sq.bf16_to_f32(X_bits))
    cw, sw = int4.quantize_groups(sq.bf16_to_f32(W_bits))
    return int4.dequantize_groups(cx, sx) @ int4.dequantize_groups(cw, sw).T + sq.bf16_to_f64(bias_bits)[None, :]


def test_int4_unsmoothed_rank0_is_plain_int4(tiny):
    from oracle import int4
    w, d = tiny
    p = sq.pack_int4(d["W"], d["bias"], 0, Xcal_bits=None, smooth=False)
    wf = sq.bf16_to_f32(d["W"])
    cw, sw = int4.quantize_groups(wf)
    assert np.array_equal(p["R"], wf)
    assert np.array_equal(p["R_codes"], cw) and np.array_equal(p["R_scales"], sw)
    assert np.allclose(sq.forward_int4(d["X"], p), _naive_int4(d["X"], d["W"], d["bias"]), rtol=0, atol=1e-12)


def test_int4_forward_against_python_loops():
    """3 x 128 x 5 and 2 x 64 x 4: the INT4 forward as explicit scalar loops, group by group:
    the integer dot product of each 64-element group scaled by its two scales."""
    for (M, K, N, r) in [(3, 128, 5, 2), (2, 64, 4, 1)]:
        w = synthetic.scaled(synthetic.TINY, M=M, K=K, N=N, rank=r, n_outlier=1, spike_rank=1)
        d = synthetic.make(w, seed=9)
        p = sq.pack_int4(d["W"], d["bias"], r, Xcal_bits=d["X"])
        Y = sq.forward_int4(d["X"], p)
        cx, sx, xh = sq.quantize_act_int4(d["X"], p["inv_lambda"])
        L1 = sq.bf16_to_f64(p["L1"])
        L2 = sq.bf16_to_f64(p["L2"])
        b = sq.bf16_to_f64(p["bias"])
        for m in range(M):
            for n in range(N):
                acc = 0.0
                for g in range(K // 64):
                    isum = 0
                    for k in range(64 * g, 64 * g + 64):
                        isum += (int(cx[m, k]) - 8) * (int(p["R_codes"][n, k]) - 8)
                    acc += float(sx[m, g]) * float(p["R_scales"][n, g]) * isum
                lr = 0.0
                for j in range(r):
                    t = 0.0
                    for k in range(K):
                        t += float(xh[m, k]) * L1[k, j]
                    lr += t * L2[j, n]
                assert abs(acc + lr + b[n] - Y[m, n]) <= 1e-9 * (1 + abs(Y[m, n]))


def test_int4_full_rank_reproduces_product(tiny):
    w, d = tiny
    p = sq.pack_int4(d["W"], d["bias"], w.K, Xcal_bits=d["X"])
    Y = sq.forward_int4(d["X"], p)
    assert sq.rel_fro(Y, sq.exact_product(d["X"], d["W"], d["bias"])) < 2e-3


@pytest.mark.parametrize("name", ["tiny", "qkv_small"])
def test_int4_svdquant_beats_naive_int4_on_outliers(name):
    w = {c.name: c for c in synthetic.parity_cases()}[name]
    d = synthetic.make(w)
    ref = sq.exact_product(d["X"], d["W"], d["bias"])
    p = sq.pack_int4(d["W"], d["bias"], w.rank, Xcal_bits=d["X"])
    e_svdq = sq.rel_fro(sq.forward_int4(d["X"], p), ref)
    e_naive = sq.rel_fro(_naive_int4(d["X"], d["W"], d["bias"]), ref)
    assert e_svdq < e_naive, (e_svdq, e_naive)


# ----------------------------------------------------------------------------- MLP pair
def test_gelu_hand_values_and_limits():
    """GELU(y) = y Phi(y): Phi(1) = 0.8413447460685429, Phi(-1) = 0.15865525393145707,
    Phi(2) = 0.9772498680518208, Phi(-10) = 7.619853024160527e-24 (standard normal tail value);
    0 at 0; y for large y; odd part y/2 (GELU(y) - GELU(-y) = y).  The Phi(-10) pin fails for the
    1 + erf form, which cancels to 0 there."""
    g = sq.gelu(np.array([0.0, 1.0, -1.0, 2.0, 40.0, -40.0, 0.5, -0.5, -10.0]))
    assert g[0] == 0.0
    assert abs(g[1] - 0.8413447460685429) < 1e-15 and abs(g[2] + 0.15865525393145707) < 1e-15
    assert abs(g[3] - 2 * 0.9772498680518208) < 1e-15
    assert g[4] == 40.0 and g[5] <= 0.0 and abs(g[5]) < 1e-300
    assert abs((g[6] - g[7]) - 0.5) < 1e-15
    assert abs(g[8] / (-10.0 * 7.619853024160527e-24) - 1.0) < 1e-12


def test_mlp_pair_is_the_composition_of_the_pinned_steps(tiny):
    """The pair's forward equals the down layer's forward on bf16(GELU(bf16(up forward))); the down
    input's codes are the down layer's quantiser applied to that G; T = x^ L1."""
    w, d = tiny
    up = sq.pack(d["W"], d["bias"], w.rank, Xcal_bits=d["X"])
    rng = np.random.default_rng(3)
    Wd = synthetic.f64_to_bf16_bits(rng.standard_normal((64, w.N)) / np.sqrt(w.N))
    Yup = sq.f64_to_bf16(sq.forward(d["X"], up))
    Gref = sq.f64_to_bf16(sq.gelu(sq.bf16_to_f64(Yup)))
    down = sq.pack(Wd, None, 16, Xcal_bits=Gref)
    G, c, s, xh, T = sq.mlp_down_input(Yup, down)
    assert np.array_equal(G, Gref)
    c2, s2, xh2 = sq.quantize_act(Gref, down["inv_lambda"], down["s_gX"])
    assert np.array_equal(c, c2) and np.array_equal(s, s2)
    assert np.allclose(T, xh2.astype(np.float64) @ sq.bf16_to_f64(down["L1"]), rtol=1e-12, atol=0)
    Y = sq.mlp_pair_forward(d["X"], up, down)
    assert np.array_equal(Y, sq.forward(Gref, down))
