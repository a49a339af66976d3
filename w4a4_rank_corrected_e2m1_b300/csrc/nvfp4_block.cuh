// Device routines shared by the kernels that quantise activations to NVFP4 (kernel 1, and
// kernel 2's fused MLP epilogue, which quantises the next layer's input): the 16-element block
// quantiser, the tiled activation-scale layout, and the MLP activation.
#pragma once
#include <cuda_runtime.h>
#include <stdint.h>

#include "ptx.cuh"

namespace svdq {

// One 16-element NVFP4 block of a row: w holds its 16 bf16 values (8 words, low half first),
// il their 1/lambda.  x^ = fl32(x * inv_lambda); scale code s8 = E4M3(fl32(amax / fl32(6 s_gX)))
// from one product with the reciprocal, settled by the thresholds; codes = E2M1(fl32(x^ * rcp)).
// Returns s8 and the 16 codes as two words (element 2j in the low nibble of byte j).
__device__ __forceinline__ uint32_t quant_block(const uint32_t* w, const float* il, float inv_six, const float* s_thr,
                                                const float* s_rcp, uint32_t* code0, uint32_t* code1) {
  // straight-line code with short dependency chains (a pairwise max tree, no branch): the
  // quantiser warps are few, so their throughput is set by latency, not by issue slots
  float2 xh[8];
  float a8[8];
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    const float2 xv = make_float2(__uint_as_float(w[k] << 16), __uint_as_float(w[k] & 0xFFFF0000u));
    xh[k] = ptx::mul2_rn(xv, make_float2(il[2 * k], il[2 * k + 1]));
    a8[k] = fmaxf(fabsf(xh[k].x), fabsf(xh[k].y));
  }
  const float m = fmaxf(fmaxf(fmaxf(fmaxf(a8[0], a8[1]), fmaxf(a8[2], a8[3])),
                              fmaxf(fmaxf(a8[4], a8[5]), fmaxf(a8[6], a8[7]))),
                        0.f);
  int code = int(ptx::cvt_e4m3x2(0.f, __fmul_rn(m, inv_six)) & 0xFF);
  code = code - (m < s_thr[code] ? 1 : 0) + (m >= s_thr[code + 1] ? 1 : 0);
  const float rcp = s_rcp[code];
  const float2 r2 = make_float2(rcp, rcp);
  float2 q[8];
#pragma unroll
  for (int k = 0; k < 8; ++k) q[k] = ptx::mul2_rn(xh[k], r2);
  const uint32_t c0 = ptx::cvt_e2m1x8(q[0].x, q[0].y, q[1].x, q[1].y, q[2].x, q[2].y, q[3].x, q[3].y);
  const uint32_t c1 = ptx::cvt_e2m1x8(q[4].x, q[4].y, q[5].x, q[5].y, q[6].x, q[6].y, q[7].x, q[7].y);
  // a zero scale gives zero codes (x * 0 may be -0, whose E2M1 code is not 0)
  *code0 = code != 0 ? c0 : 0u;
  *code1 = code != 0 ? c1 : 0u;
  return uint32_t(code);
}

// Byte offset of the 32-bit word holding row `row`'s four scales of 64-column chunk c in the
// tiled activation-scale layout.
__device__ __forceinline__ int64_t scale_word_offset(int64_t row, int64_t c, int64_t KG) {
  return ((row >> 7) * KG + c) * 512 + (row & 31) * 16 + ((row >> 5) & 3) * 4;
}

// GELU(y) = y * Phi(y), Phi the standard normal CDF (GELU's definition, not the tanh
// approximation), in float32.  With Q(u) = erfc(u / sqrt(2)) / 2 the upper normal tail,
// GELU(y) = y Q(|y|) for y <= 0 and y (1 - Q(y)) for y > 0, so the small values of large negative
// y keep their relative accuracy (no 1 + erf cancellation).  erfc comes from the Chebyshev fit of
// Numerical Recipes (Press et al., 2nd ed., section 6.2, routine erfcc), whose fractional error is
// below 1.2e-7 for every argument z >= 0:
//   erfc(z) = t exp(-z^2 + P(t)),  t = 1 / (1 + z/2),  P the fit's degree-9 polynomial in t.
// The reciprocal and the exponential (as 2^(u log2 e)) come from the special-function unit, so
// GELU costs about 20 instructions (erfcf about 70).  The relative error of the float32 result
// stays below 2^-19 (y >= 0) and 2^-19 + y^2 2^-22 (y < 0, where the rounding of z^2 and of the
// exponent grows with y^2); results below the float32 normal range flush to a zero of y's sign.
// The GPU tests check this over every bf16 input.
__device__ __forceinline__ float gelu_f32(float y) {
  const float z = fabsf(y) * 0.70710678118654752f;
  const float t = ptx::rcp_approx(fmaf(0.5f, z, 1.0f));
  float p = 0.17087277f;
  p = fmaf(p, t, -0.82215223f);
  p = fmaf(p, t, 1.48851587f);
  p = fmaf(p, t, -1.13520398f);
  p = fmaf(p, t, 0.27886807f);
  p = fmaf(p, t, -0.18628806f);
  p = fmaf(p, t, 0.09678418f);
  p = fmaf(p, t, 0.37409196f);
  p = fmaf(p, t, 1.00002368f);
  p = fmaf(p, t, -1.26551223f);
  const float q = (0.5f * t) * ptx::ex2_approx(fmaf(-z, z, p) * 1.44269504088896341f);   // Q(|y|)
  return y <= 0.0f ? y * q : y * (1.0f - q);
}

// bf16 pair (low half first) -> bf16(GELU) pair: gelu_f32 on both halves with packed float32
// operations (two IEEE operations per instruction), bit for bit the same values.  The exponent
// is formed negated, z^2 - P(t) from the negated polynomial, and scaled by -log2 e: negation
// commutes with rounding to nearest even, so every rounded value is gelu_f32's up to sign.
__device__ __forceinline__ uint32_t gelu_bf16x2(uint32_t w) {
  const float2 y = make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xFFFF0000u));
  const float2 nz = ptx::mul2_rn(make_float2(fabsf(y.x), fabsf(y.y)),
                                 make_float2(-0.70710678118654752f, -0.70710678118654752f));   // -z
  const float2 d = ptx::fma2_rn(make_float2(-0.5f, -0.5f), nz, make_float2(1.0f, 1.0f));     // 1 + z/2
  const float2 t = make_float2(ptx::rcp_approx(d.x), ptx::rcp_approx(d.y));
  auto c2 = [](float c) { return make_float2(c, c); };
  float2 pn = ptx::fma2_rn(c2(-0.17087277f), t, c2(0.82215223f));                             // -P(t)
  pn = ptx::fma2_rn(pn, t, c2(-1.48851587f));
  pn = ptx::fma2_rn(pn, t, c2(1.13520398f));
  pn = ptx::fma2_rn(pn, t, c2(-0.27886807f));
  pn = ptx::fma2_rn(pn, t, c2(0.18628806f));
  pn = ptx::fma2_rn(pn, t, c2(-0.09678418f));
  pn = ptx::fma2_rn(pn, t, c2(-0.37409196f));
  pn = ptx::fma2_rn(pn, t, c2(-1.00002368f));
  pn = ptx::fma2_rn(pn, t, c2(1.26551223f));
  const float2 u = ptx::mul2_rn(ptx::fma2_rn(nz, nz, pn), c2(-1.44269504088896341f));        // (-z^2 + P) log2 e
  const float2 e = make_float2(ptx::ex2_approx(u.x), ptx::ex2_approx(u.y));
  const float2 q = ptx::mul2_rn(ptx::mul2_rn(c2(0.5f), t), e);                                 // Q(|y|)
  const float2 om = ptx::fma2_rn(q, c2(-1.0f), c2(1.0f));                                     // 1 - Q
  const float2 g = ptx::mul2_rn(y, make_float2(y.x <= 0.0f ? q.x : om.x, y.y <= 0.0f ? q.y : om.y));
  return ptx::pack_bf16x2(g.x, g.y);
}

}  // namespace svdq
