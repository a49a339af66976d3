"""SVDQuant W4A4 linear layer, restated step by step on the CPU (test infrastructure only).

What the method computes, as the Nunchaku/SVDQuant pages describe it
("What SVDQuant actually does" and "How Nunchaku four bit quantization actually
works", aiflownews article; "How Nunchaku Works: W4A8 and SVD-Quant", n1n.ai
article):

  1. smoothing: move activation outliers into the weights,
         X^ = X diag(lambda)^-1,   W^ = W diag(lambda)
  2. low rank: SVD of the smoothed weight, the top-r part kept in 16 bit,
         W^T ~= L1 L2  (L1: K x r, L2: r x N, both bfloat16)
  3. residual: R = W^ - (L1 L2)^T, quantised to 4 bit (NVFP4); activations
     X^ are quantised to 4 bit at run time
  4. two-branch forward: a small 16-bit low-rank branch that absorbs the
     hardest part of the weight distribution, summed with a 4-bit branch that
     does most of the arithmetic:
         Y = Q4(X^) Q4(R)^T + (X^ L1) L2 + b

Readings where the pages are silent (each also listed in the design notes):
  * lambda_c = sqrt(max_m |X_mc| / max_n |W_nc|) from calibration activations
    (float64, stored as float32; 1 where either maximum is 0); inv_lambda is the
    float32 quotient 1/lambda.
  * Sigma goes entirely onto L2 (L1 = U_r orthonormal); both factors rounded to
    bfloat16 (RNE); R is taken against the rounded factors, in float64, then
    cast to float32.
  * NVFP4 two-level scaling with static global scales s_gW = amax|R|/2688 and
    s_gX = amax|X^_cal|/2688 (see oracle.nvfp4).
  * the 4-bit product is scaled by alpha = fl32(s_gX * s_gW).

Products and sums here are float64 (numpy BLAS for the matmuls, LAPACK for the
SVD); the quantiser is float32 IEEE as fixed in oracle.nvfp4.

Pins (tests/test_oracle_svdquant.py): the smoothing identity X^ W^T = X W^T;
Eckart-Young (residual energy equals the tail of the spectrum computed through
an eigen-decomposition); full rank leaves R = 0; lambda = 1 with r = 0 equals
plain W4A4 quantisation of X and W; a pure-Python loop evaluation of the
forward on 4 x 16 x 16; SVDQuant beats naive W4A4 on outlier-heavy inputs.
The MLP pair (gelu, mlp_down_input, mlp_pair_forward) composes two layers through the
activation; gelu is pinned to hand values of y * Phi(y) and its limits.
The INT4 variant (pack_int4, quantize_act_int4, forward_int4) shares every step up to the
residual and quantises with oracle.int4 instead; its pins mirror the NVFP4 ones (reduction to
plain INT4 W4A4 at lambda = 1 and r = 0, loops on a tiny case, the method claim on outliers).
Image-quality and end-to-end speed claims of the pages: parity unpinned (they
need trained models).
"""
from __future__ import annotations

import numpy as np

from . import int4, nvfp4


# ----------------------------------------------------------------------------- formats
def bf16_to_f64(bits) -> np.ndarray:
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    return b.view(np.float32).astype(np.float64)


def bf16_to_f32(bits) -> np.ndarray:
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    return b.view(np.float32)


def f64_to_bf16(a) -> np.ndarray:
    """float64 -> bfloat16 bits, one rounding (nearest, ties to even); finite inputs."""
    a = np.asarray(a, dtype=np.float64)
    _, ex = np.frexp(a)
    ex = np.maximum(ex, -125)                 # below 2^-126: bf16 subnormal spacing 2^-133
    q = np.ldexp(1.0, ex - 8)                 # 8 significant bits
    v = (np.rint(a / q) * q).astype(np.float32)
    return (v.view(np.uint32) >> 16).astype(np.uint16)


# ----------------------------------------------------------------------------- step 1
def smoothing_factors(Xcal_bits, W_bits):
    """lambda (float32, K) and inv_lambda = fl32(1/lambda)."""
    xmax = np.max(np.abs(bf16_to_f64(Xcal_bits)), axis=0)
    wmax = np.max(np.abs(bf16_to_f64(W_bits)), axis=0)
    ok = (xmax > 0) & (wmax > 0)
    lam = np.ones_like(xmax)
    lam[ok] = np.sqrt(xmax[ok] / wmax[ok])
    lam32 = lam.astype(np.float32)
    inv32 = (np.float32(1.0) / lam32).astype(np.float32)
    return lam32, inv32


def smooth_weight(W_bits, lam32) -> np.ndarray:
    """W^ = W diag(lambda) in float64 (exact: bf16 x fp32 fits in 53 bits)."""
    return bf16_to_f64(W_bits) * lam32.astype(np.float64)[None, :]


def smooth_act(X_bits, inv32) -> np.ndarray:
    """x^ = fl32(x * inv_lambda), float32."""
    return (bf16_to_f32(X_bits) * inv32[None, :]).astype(np.float32)


# ----------------------------------------------------------------------------- step 2
def lowrank_factors(What, rank):
    """Top-r SVD of W^T (K x N): L1 = U_r, L2 = Sigma_r V_r^T (float64, before rounding)."""
    K = What.shape[1]
    N = What.shape[0]
    if rank == 0:
        return np.zeros((K, 0)), np.zeros((0, N)), np.linalg.svd(What.T, compute_uv=False)
    U, S, Vt = np.linalg.svd(What.T, full_matrices=False)
    return U[:, :rank], S[:rank, None] * Vt[:rank, :], S


# ----------------------------------------------------------------------------- step 3
def residual(What, L1_bits, L2_bits) -> np.ndarray:
    """R = W^ - (L1 L2)^T against the bf16 factors, float64 -> float32."""
    L1 = bf16_to_f64(L1_bits)
    L2 = bf16_to_f64(L2_bits)
    return (What - (L1 @ L2).T).astype(np.float32)


def split(W_bits, rank, Xcal_bits=None, smooth=True, L1_bits=None, L2_bits=None):
    """Stages one to three up to the residual: lambda, inv_lambda, the bf16 factors and the
    float32 residual R (shared by the NVFP4 and the INT4 variants)."""
    N, K = W_bits.shape
    if smooth and Xcal_bits is not None:
        lam, inv = smoothing_factors(Xcal_bits, W_bits)
    else:
        lam = np.ones(K, np.float32)
        inv = np.ones(K, np.float32)
    What = smooth_weight(W_bits, lam)
    if L1_bits is None:
        L1, L2, _ = lowrank_factors(What, rank)
        L1_bits, L2_bits = f64_to_bf16(L1), f64_to_bf16(L2)
    R = residual(What, L1_bits, L2_bits)
    return lam, inv, np.asarray(L1_bits, np.uint16), np.asarray(L2_bits, np.uint16), R


def pack(W_bits, bias_bits, rank, Xcal_bits=None, smooth=True, L1_bits=None, L2_bits=None):
    """Offline step: smoothing, low-rank split, residual quantisation.

    Returns a dict of the packed layer in canonical layouts:
      inv_lambda (K fp32), lam (K fp32), L1 (K x r bf16 bits), L2 (r x N bf16 bits),
      R_codes (N x K uint8 nibbles), R_scales (N x K/16 E4M3 bits), s_gW, s_gX (fp32),
      bias (N bf16 bits), R (N x K fp32).
    """
    N, K = W_bits.shape
    lam, inv, L1_bits, L2_bits, R = split(W_bits, rank, Xcal_bits, smooth, L1_bits, L2_bits)
    s_gW = nvfp4.global_scale(np.max(np.abs(R)) if R.size else 0.0)
    codes, scales = nvfp4.quantize_blocks(R, s_gW)
    if Xcal_bits is not None:
        s_gX = nvfp4.global_scale(np.max(np.abs(smooth_act(Xcal_bits, inv))))
    else:
        s_gX = np.float32(1.0)
    if bias_bits is None:
        bias_bits = np.zeros(N, np.uint16)
    return dict(lam=lam, inv_lambda=inv, L1=L1_bits, L2=L2_bits, R=R, R_codes=codes, R_scales=scales,
                s_gW=np.float32(s_gW), s_gX=np.float32(s_gX), bias=np.asarray(bias_bits, np.uint16),
                rank=int(rank))


def pack_int4(W_bits, bias_bits, rank, Xcal_bits=None, smooth=True, L1_bits=None, L2_bits=None):
    """The INT4 variant's offline step: the same smoothing, low-rank split and residual, then R
    quantised to INT4 groups (oracle.int4): R_codes (N x K nibbles q + 8), R_scales (N x K/64
    float32).  No global scales."""
    N, K = W_bits.shape
    lam, inv, L1_bits, L2_bits, R = split(W_bits, rank, Xcal_bits, smooth, L1_bits, L2_bits)
    codes, scales = int4.quantize_groups(R)
    if bias_bits is None:
        bias_bits = np.zeros(N, np.uint16)
    return dict(fmt="int4", lam=lam, inv_lambda=inv, L1=L1_bits, L2=L2_bits, R=R, R_codes=codes,
                R_scales=scales, bias=np.asarray(bias_bits, np.uint16), rank=int(rank))


# ----------------------------------------------------------------------------- step 4
def quantize_act(X_bits, inv32, s_gX):
    """Run-time activation quantisation: x^ = fl32(x inv_lambda), then Qz(x^, s_gX)."""
    xh = smooth_act(X_bits, inv32)
    codes, scales = nvfp4.quantize_blocks(xh, s_gX)
    return codes, scales, xh


def lowrank_down(xhat32, L1_bits) -> np.ndarray:
    """T = X^ L1 in float64."""
    return xhat32.astype(np.float64) @ bf16_to_f64(L1_bits)


def alpha(p) -> np.float32:
    return np.float32(np.float32(p["s_gX"]) * np.float32(p["s_gW"]))


def forward(X_bits, p):
    """Y = alpha * deq(Q4(X^)) deq(Q4(R))^T + (X^ L1) L2 + b in float64."""
    Xb = np.asarray(X_bits)
    cx, sx, xh = quantize_act(Xb, p["inv_lambda"], p["s_gX"])
    Xdq = nvfp4.dequantize_blocks(cx, sx)
    Rdq = nvfp4.dequantize_blocks(p["R_codes"], p["R_scales"])
    Y = np.float64(alpha(p)) * (Xdq @ Rdq.T)
    if p["rank"]:
        Y += lowrank_down(xh, p["L1"]) @ bf16_to_f64(p["L2"])
    return Y + bf16_to_f64(p["bias"])[None, :]


def quantize_act_int4(X_bits, inv32):
    """The INT4 variant's run-time activation quantisation: x^ = fl32(x inv_lambda), then INT4
    groups of 64 with a float32 scale each (oracle.int4)."""
    xh = smooth_act(X_bits, inv32)
    codes, scales = int4.quantize_groups(xh)
    return codes, scales, xh


def forward_int4(X_bits, p):
    """Y = deq(Q4i(X^)) deq(Q4i(R))^T + (X^ L1) L2 + b in float64 for the INT4 variant."""
    cx, sx, xh = quantize_act_int4(np.asarray(X_bits), p["inv_lambda"])
    Y = int4.dequantize_groups(cx, sx) @ int4.dequantize_groups(p["R_codes"], p["R_scales"]).T
    if p["rank"]:
        Y += lowrank_down(xh, p["L1"]) @ bf16_to_f64(p["L2"])
    return Y + bf16_to_f64(p["bias"])[None, :]


def lora_delta(X_bits, A_bits, B_bits, scale, rows=None):
    """The LoRA adapter's contribution scale * (X A) B in float64, X in bf16 values.

    The pages note that SVDQuant keeps working with existing LoRA adapters without
    re-quantising the residual (aiflownews article on Nunchaku, "What SVDQuant actually
    does"), i.e. the adapter is a further 16-bit branch beside the low-rank one; it acts on
    the layer's input X, which is what the adapter was trained against.
    """
    Xb = np.asarray(X_bits)
    if rows is not None:
        Xb = Xb[rows]
    return float(scale) * ((bf16_to_f64(Xb) @ bf16_to_f64(A_bits)) @ bf16_to_f64(B_bits))


# ----------------------------------------------------------------------------- MLP pair
def gelu(y) -> np.ndarray:
    """GELU(y) = y * Phi(y), Phi the standard normal CDF, in float64 (the pages name the MLP's
    activation without a formula; this is GELU's definition, not the tanh approximation).
    Phi(y) = erfc(-y / sqrt(2)) / 2 (scipy.special.erfc): the same function as (1 + erf(y/sqrt(2)))/2,
    but without the cancellation that rounds Phi to 0 for y below about -8.3."""
    from scipy.special import erfc
    y = np.asarray(y, np.float64)
    return y * (0.5 * erfc(-y / np.sqrt(2.0)))


def mlp_down_input(Y_up_bits, p_down):
    """What the MLP-down layer receives from MLP-up in an MLP pair: G = bf16(GELU(Y_up)) with Y_up
    the up layer's bf16 output, then the down layer's run-time quantisation of G (smoothing by its
    inv_lambda, NVFP4 blocks with its s_gX) and its down-projection T = G^ L1_down (float64).
    Returns (G bits, codes, scales, x^ float32, T)."""
    G = f64_to_bf16(gelu(bf16_to_f64(Y_up_bits)))
    codes, scales, xh = quantize_act(G, p_down["inv_lambda"], p_down["s_gX"])
    T = lowrank_down(xh, p_down["L1"]) if p_down["rank"] else np.zeros((G.shape[0], 0))
    return G, codes, scales, xh, T


def mlp_pair_forward(X_bits, p_up, p_down):
    """The MLP pair: Y_up = forward(X, up) rounded to bf16, G = bf16(GELU(Y_up)), Y = forward(G, down)
    in float64."""
    Y_up = f64_to_bf16(forward(X_bits, p_up))
    G = f64_to_bf16(gelu(bf16_to_f64(Y_up)))
    return forward(G, p_down)


# ----------------------------------------------------------------------------- references
def exact_product(X_bits, W_bits, bias_bits) -> np.ndarray:
    """The unquantised layer X W^T + b on the bf16 inputs, float64."""
    return bf16_to_f64(X_bits) @ bf16_to_f64(W_bits).T + bf16_to_f64(bias_bits)[None, :]


def naive_w4a4(X_bits, W_bits, bias_bits) -> np.ndarray:
    """Plain NVFP4 W4A4 without smoothing or low-rank branch."""
    x = bf16_to_f32(X_bits)
    w = bf16_to_f32(W_bits)
    sx = nvfp4.global_scale(np.max(np.abs(x)))
    sw = nvfp4.global_scale(np.max(np.abs(w)))
    cx, bx = nvfp4.quantize_blocks(x, sx)
    cw, bw = nvfp4.quantize_blocks(w, sw)
    a = np.float64(np.float32(sx * sw))
    return a * (nvfp4.dequantize_blocks(cx, bx) @ nvfp4.dequantize_blocks(cw, bw).T) \
        + bf16_to_f64(bias_bits)[None, :]


def rel_fro(a, b) -> float:
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-300))
