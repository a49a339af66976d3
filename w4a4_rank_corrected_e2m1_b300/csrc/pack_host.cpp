// Offline packing of an SVDQuant layer on the CPU.
//
// The three stages of SVDQuant ("What SVDQuant actually does", aiflownews article on
// Nunchaku in Diffusers): move activation outliers into the weights (smoothing), split
// the smoothed weight by SVD into a 16-bit low-rank part and a residual, quantise the
// residual to 4 bit (NVFP4 on Blackwell).  Readings where the pages are silent:
//   lambda_c = sqrt(max_m |X_mc| / max_n |W_nc|), 1 where either maximum is 0;
//   Sigma goes onto L2, L1 = U_r; factors rounded to bfloat16;
//   R = W diag(lambda) - (L1 L2)^T against the rounded factors (float64, then float32);
//   NVFP4: E4M3 scale per 16 elements, s_gW = amax|R| / (6 * 448), round to nearest even.
//
// The top-r SVD is a randomized range finder with subspace iteration (Halko, Martinsson,
// Tropp, "Finding structure with randomness", SIAM Review 2011, Algorithms 4.4 and 5.1),
// followed by a cyclic Jacobi eigen-decomposition of the small projected Gram matrix.
#include <algorithm>
#include <cmath>
#include <cstring>
#include <limits>
#include <new>

#include "svdq_internal.h"

#ifdef _OPENMP
#include <omp.h>
#endif

namespace svdq {

// ------------------------------------------------------------------ formats
float bf16_to_f32(uint16_t b) {
  uint32_t u = uint32_t(b) << 16;
  float f;
  std::memcpy(&f, &u, 4);
  return f;
}

uint16_t f64_to_bf16(double a) {
  // One rounding to 8 significant bits, nearest-even (the default FP rounding mode).
  if (a == 0.0) return std::signbit(a) ? 0x8000 : 0;
  int ex;
  std::frexp(a, &ex);
  if (ex < -125) ex = -125;
  const double q = std::ldexp(1.0, ex - 8);
  const float v = float(std::nearbyint(a / q) * q);
  uint32_t u;
  std::memcpy(&u, &v, 4);
  return uint16_t(u >> 16);
}

// Unsigned E4M3 (bias 7, max 448), round to nearest even on the float32 bit pattern,
// saturating.
uint8_t e4m3_encode_nonneg(float s) {
  if (!(s < 448.0f)) return 0x7E;
  if (s <= 0.0f) return 0;
  uint32_t u;
  std::memcpy(&u, &s, 4);
  const int biased = int((u >> 23) & 0xFF);
  if (biased == 0) return 0;                       // float32 subnormal: far below 2^-10
  int e = biased - 127;
  if (e >= -6) {
    uint32_t mant = u & 0x7FFFFF;
    uint32_t keep = mant >> 20, rem = mant & 0xFFFFF;
    if (rem > 0x80000u || (rem == 0x80000u && (keep & 1u))) ++keep;
    if (keep == 8) { keep = 0; ++e; }
    return uint8_t(((e + 7) << 3) | int(keep));
  }
  // E4M3 subnormal range: value = n * 2^-9 (n = 8 is the smallest normal, same bits)
  const float n = std::nearbyint(s * 512.0f);
  return uint8_t(n);
}

float e4m3_decode(uint8_t b) {
  const int e = (b >> 3) & 0xF, m = b & 7;
  float v = (e == 0) ? std::ldexp(float(m), -9) : std::ldexp(1.0f + float(m) / 8.0f, e - 7);
  return (b & 0x80) ? -v : v;
}

// E2M1 by decision thresholds (midpoints go to the even code), saturating at 6;
// the sign bit follows the float's sign bit.
uint8_t e2m1_encode(float v) {
  const float a = std::fabs(v);
  uint8_t c;
  if (a <= 0.25f) c = 0;
  else if (a < 0.75f) c = 1;
  else if (a <= 1.25f) c = 2;
  else if (a < 1.75f) c = 3;
  else if (a <= 2.5f) c = 4;
  else if (a < 3.5f) c = 5;
  else if (a <= 5.0f) c = 6;
  else c = 7;
  return uint8_t(c | (std::signbit(v) ? 8 : 0));
}

// Qz on one row of K float32 values: codes (K/2 bytes, even k in the low nibble) and
// K/16 E4M3 scales.  Every step is a single float32 operation (compiled without
// contraction).
static void quantize_row(const float* v, int64_t K, float s_g, uint8_t* codes, uint8_t* scales) {
  const float six_sg = 6.0f * s_g;
  for (int64_t b = 0; b < K / 16; ++b) {
    const float* x = v + b * 16;
    float amax = 0.f;
    for (int i = 0; i < 16; ++i) amax = std::max(amax, std::fabs(x[i]));
    const float s_raw = amax / six_sg;
    const uint8_t s8 = e4m3_encode_nonneg(s_raw);
    scales[b] = s8;
    uint8_t* c = codes + b * 8;
    if (s8 == 0) {
      std::memset(c, 0, 8);
      continue;
    }
    const float d = e4m3_decode(s8) * s_g;
    const float rcp = 1.0f / d;
    for (int i = 0; i < 8; ++i) {
      const uint8_t lo = e2m1_encode(x[2 * i] * rcp);
      const uint8_t hi = e2m1_encode(x[2 * i + 1] * rcp);
      c[i] = uint8_t(lo | (hi << 4));
    }
  }
}

void act_quant_tables(float s_g, float* thr, float* rcp) {
  const float six = 6.0f * s_g;
  auto code_of = [&](uint32_t bits) {
    float a;
    std::memcpy(&a, &bits, 4);
    return int(e4m3_encode_nonneg(a / six));
  };
  thr[0] = 0.f;
  for (int c = 1; c < 127; ++c) {
    uint32_t lo = 0, hi = 0x7F800000u;              // +inf saturates to the top code
    while (lo < hi) {                               // smallest bit pattern whose code is >= c
      const uint32_t mid = lo + (hi - lo) / 2;
      if (code_of(mid) >= c) hi = mid;
      else lo = mid + 1;
    }
    std::memcpy(&thr[c], &lo, 4);
  }
  thr[127] = std::numeric_limits<float>::infinity();
  rcp[0] = 0.f;
  for (int c = 1; c < 128; ++c) {
    const float d = e4m3_decode(uint8_t(c)) * s_g;
    rcp[c] = 1.0f / d;
  }
}

static float global_scale(float amax) {
  if (amax == 0.f) return 1.f;
  return amax / 2688.0f;
}

// ------------------------------------------------------------------ randomized SVD
namespace {

struct Rng {  // splitmix64 + Box-Muller
  uint64_t s;
  explicit Rng(uint64_t seed) : s(seed ^ 0x9E3779B97F4A7C15ull) {}
  uint64_t next() {
    uint64_t z = (s += 0x9E3779B97F4A7C15ull);
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
  }
  double uniform() { return (double(next() >> 11) + 0.5) * (1.0 / 9007199254740992.0); }
  double gauss() {
    const double u1 = uniform(), u2 = uniform();
    return std::sqrt(-2.0 * std::log(u1)) * std::cos(6.283185307179586 * u2);
  }
};

// Y (K x l) = What^T Omega, What: N x K row-major, Omega: N x l.
void mul_wt(const double* What, int64_t N, int64_t K, const double* Om, int64_t l, double* Y) {
  const int64_t KB = 256;
#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t k0 = 0; k0 < K; k0 += KB) {
    const int64_t k1 = std::min(K, k0 + KB);
    std::fill(Y + k0 * l, Y + k1 * l, 0.0);
    for (int64_t n = 0; n < N; ++n) {
      const double* w = What + n * K;
      const double* o = Om + n * l;
      for (int64_t k = k0; k < k1; ++k) {
        const double a = w[k];
        double* y = Y + k * l;
        for (int64_t j = 0; j < l; ++j) y[j] += a * o[j];
      }
    }
  }
}

// Z (N x l) = What Q, Q: K x l.
void mul_w(const double* What, int64_t N, int64_t K, const double* Q, int64_t l, double* Z) {
#pragma omp parallel for schedule(static)
  for (int64_t n = 0; n < N; ++n) {
    double* z = Z + n * l;
    std::fill(z, z + l, 0.0);
    const double* w = What + n * K;
    for (int64_t k = 0; k < K; ++k) {
      const double a = w[k];
      const double* q = Q + k * l;
      for (int64_t j = 0; j < l; ++j) z[j] += a * q[j];
    }
  }
}

// Orthonormalise the l columns of a rows x l row-major matrix (Gram-Schmidt, two passes).
void orthonormalize(double* A, int64_t rows, int64_t l) {
  std::vector<double> dots(l);
  for (int pass = 0; pass < 2; ++pass) {
    for (int64_t j = 0; j < l; ++j) {
      // project out columns 0..j-1
      if (j > 0) {
        std::fill(dots.begin(), dots.begin() + j, 0.0);
        for (int64_t r = 0; r < rows; ++r) {
          const double* a = A + r * l;
          for (int64_t i = 0; i < j; ++i) dots[i] += a[i] * a[j];
        }
        for (int64_t r = 0; r < rows; ++r) {
          double* a = A + r * l;
          double s = 0.0;
          for (int64_t i = 0; i < j; ++i) s += dots[i] * a[i];
          a[j] -= s;
        }
      }
      double nrm = 0.0;
      for (int64_t r = 0; r < rows; ++r) nrm += A[r * l + j] * A[r * l + j];
      nrm = std::sqrt(nrm);
      const double inv = nrm > 0 ? 1.0 / nrm : 0.0;
      for (int64_t r = 0; r < rows; ++r) A[r * l + j] *= inv;
    }
  }
}

// Cyclic Jacobi eigen-decomposition of a symmetric n x n matrix G (destroyed).
// Eigenvalues in w, eigenvectors in the columns of V (row-major n x n).
void jacobi_eig(std::vector<double>& G, int64_t n, std::vector<double>& w, std::vector<double>& V) {
  V.assign(n * n, 0.0);
  for (int64_t i = 0; i < n; ++i) V[i * n + i] = 1.0;
  for (int sweep = 0; sweep < 60; ++sweep) {
    double off = 0.0, diag = 0.0;
    for (int64_t i = 0; i < n; ++i)
      for (int64_t j = 0; j < n; ++j) (i == j ? diag : off) += G[i * n + j] * G[i * n + j];
    if (off <= 1e-30 * diag || off == 0.0) break;
    for (int64_t p = 0; p < n - 1; ++p)
      for (int64_t q = p + 1; q < n; ++q) {
        const double apq = G[p * n + q];
        if (apq == 0.0) continue;
        const double app = G[p * n + p], aqq = G[q * n + q];
        const double theta = (aqq - app) / (2.0 * apq);
        const double t = (theta >= 0 ? 1.0 : -1.0) / (std::fabs(theta) + std::sqrt(theta * theta + 1.0));
        const double c = 1.0 / std::sqrt(t * t + 1.0), s = t * c;
        for (int64_t k = 0; k < n; ++k) {  // G = J^T G J
          const double gkp = G[k * n + p], gkq = G[k * n + q];
          G[k * n + p] = c * gkp - s * gkq;
          G[k * n + q] = s * gkp + c * gkq;
        }
        for (int64_t k = 0; k < n; ++k) {
          const double gpk = G[p * n + k], gqk = G[q * n + k];
          G[p * n + k] = c * gpk - s * gqk;
          G[q * n + k] = s * gpk + c * gqk;
        }
        for (int64_t k = 0; k < n; ++k) {
          const double vkp = V[k * n + p], vkq = V[k * n + q];
          V[k * n + p] = c * vkp - s * vkq;
          V[k * n + q] = s * vkp + c * vkq;
        }
      }
  }
  w.resize(n);
  for (int64_t i = 0; i < n; ++i) w[i] = G[i * n + i];
}

// Top-r factors of What^T (K x N): L1 = U_r (K x r), L2 = U_r^T What^T (r x N).
void randomized_lowrank(const double* What, int64_t N, int64_t K, int64_t r, int q, int p,
                        uint64_t seed, std::vector<double>& L1, std::vector<double>& L2) {
  const int64_t l = std::min<int64_t>(std::min(N, K), r + p);
  std::vector<double> Om(N * l), Y(K * l), Z(N * l);
  Rng rng(seed);
  for (auto& x : Om) x = rng.gauss();
  mul_wt(What, N, K, Om.data(), l, Y.data());
  orthonormalize(Y.data(), K, l);
  for (int it = 0; it < q; ++it) {
    mul_w(What, N, K, Y.data(), l, Z.data());
    orthonormalize(Z.data(), N, l);
    mul_wt(What, N, K, Z.data(), l, Y.data());
    orthonormalize(Y.data(), K, l);
  }
  // B^T = What Q (N x l); G = B B^T (l x l)
  mul_w(What, N, K, Y.data(), l, Z.data());
  std::vector<double> G(l * l, 0.0);
  for (int64_t n = 0; n < N; ++n) {
    const double* z = Z.data() + n * l;
    for (int64_t i = 0; i < l; ++i)
      for (int64_t j = 0; j < l; ++j) G[i * l + j] += z[i] * z[j];
  }
  std::vector<double> w, V;
  jacobi_eig(G, l, w, V);
  std::vector<int64_t> order(l);
  for (int64_t i = 0; i < l; ++i) order[i] = i;
  std::sort(order.begin(), order.end(), [&](int64_t a, int64_t b) { return w[a] > w[b]; });
  L1.assign(K * r, 0.0);
  L2.assign(r * N, 0.0);
#pragma omp parallel for schedule(static)
  for (int64_t k = 0; k < K; ++k)
    for (int64_t j = 0; j < r; ++j) {
      const int64_t c = order[j];
      double s = 0.0;
      for (int64_t i = 0; i < l; ++i) s += Y[k * l + i] * V[i * l + c];
      L1[k * r + j] = s;
    }
#pragma omp parallel for schedule(static)
  for (int64_t n = 0; n < N; ++n)
    for (int64_t j = 0; j < r; ++j) {
      const int64_t c = order[j];
      double s = 0.0;
      for (int64_t i = 0; i < l; ++i) s += V[i * l + c] * Z[n * l + i];
      L2[j * N + n] = s;
    }
}

}  // namespace

// ------------------------------------------------------------------ pack
// INT4 group quantiser of the INT4 variant, per 64 elements: s = fl32(amax / 7), q =
// clamp(rint(fl32(v * fl32(1 / s))), -7, 7) (ties to even), stored as the nibble q + 8 (element
// k in byte k / 2, low nibble for even k); an all-zero group has s = 0 and q = 0.
void int4_quantize_row(const float* v, int64_t K, uint8_t* codes, float* scales) {
  for (int64_t g = 0; g < K / 64; ++g) {
    float amax = 0.f;
    for (int i = 0; i < 64; ++i) amax = std::max(amax, std::fabs(v[64 * g + i]));
    const float s = amax / 7.0f;
    scales[g] = s;
    const float rcp = s > 0.f ? 1.0f / s : 0.f;
    for (int i = 0; i < 64; i += 2) {
      uint8_t byte = 0;
      for (int h = 0; h < 2; ++h) {
        int q = 0;
        if (s > 0.f) {
          const float t = v[64 * g + i + h] * rcp;
          q = int(std::nearbyint(t));
          q = q < -7 ? -7 : (q > 7 ? 7 : q);
        }
        byte |= uint8_t(q + 8) << (4 * h);
      }
      codes[(64 * g + i) / 2] = byte;
    }
  }
}

svdq_status_t pack_on_host(const svdq_pack_params_t* p, HostPack* out, std::string* err, std::vector<float>* R_keep) {
  if (!p || !out) { *err = "null argument"; return SVDQ_ERR_INVALID_ARG; }
  const int64_t N = p->N, K = p->K, r = p->rank;
  if (N <= 0 || K <= 0 || r < 0 || !p->W_bf16) { *err = "N, K must be > 0, rank >= 0, W required"; return SVDQ_ERR_INVALID_ARG; }
  if (K % 16 != 0) { *err = "K must be a multiple of 16"; return SVDQ_ERR_UNSUPPORTED_SHAPE; }
  if (r > std::min(N, K)) { *err = "rank must not exceed min(N, K)"; return SVDQ_ERR_UNSUPPORTED_SHAPE; }
  if ((p->L1_bf16 == nullptr) != (p->L2_bf16 == nullptr)) { *err = "L1 and L2 overrides go together"; return SVDQ_ERR_INVALID_ARG; }
  if (p->Xcal_bf16 && p->Mcal <= 0) { *err = "Mcal must be > 0 with Xcal"; return SVDQ_ERR_INVALID_ARG; }
  try {
    HostPack& o = *out;
    o.N = N; o.K = K; o.rank = r;
    o.lambda.assign(K, 1.f);
    o.inv_lambda.assign(K, 1.f);
    // stage one: smoothing factors
    if (!(p->flags & SVDQ_NO_SMOOTH)) {
      if (p->lambda) {
        for (int64_t k = 0; k < K; ++k) {
          if (!(p->lambda[k] > 0.f) || !std::isfinite(p->lambda[k])) { *err = "lambda must be positive and finite"; return SVDQ_ERR_INVALID_ARG; }
          o.lambda[k] = p->lambda[k];
        }
      } else if (p->Xcal_bf16) {
        std::vector<double> xmax(K, 0.0), wmax(K, 0.0);
        for (int64_t m = 0; m < p->Mcal; ++m)
          for (int64_t k = 0; k < K; ++k)
            xmax[k] = std::max(xmax[k], std::fabs(double(bf16_to_f32(p->Xcal_bf16[m * K + k]))));
        for (int64_t n = 0; n < N; ++n)
          for (int64_t k = 0; k < K; ++k)
            wmax[k] = std::max(wmax[k], std::fabs(double(bf16_to_f32(p->W_bf16[n * K + k]))));
        for (int64_t k = 0; k < K; ++k)
          o.lambda[k] = (xmax[k] > 0 && wmax[k] > 0) ? float(std::sqrt(xmax[k] / wmax[k])) : 1.f;
      }
      for (int64_t k = 0; k < K; ++k) o.inv_lambda[k] = 1.0f / o.lambda[k];
    }
    // W^ = W diag(lambda), float64
    std::vector<double> What(size_t(N) * K);
#pragma omp parallel for schedule(static)
    for (int64_t n = 0; n < N; ++n)
      for (int64_t k = 0; k < K; ++k)
        What[n * K + k] = double(bf16_to_f32(p->W_bf16[n * K + k])) * double(o.lambda[k]);
    // stage two: low-rank factors in bfloat16
    o.L1.assign(K * r, 0);
    o.L2.assign(r * N, 0);
    if (r > 0) {
      if (p->L1_bf16) {
        std::memcpy(o.L1.data(), p->L1_bf16, sizeof(uint16_t) * K * r);
        std::memcpy(o.L2.data(), p->L2_bf16, sizeof(uint16_t) * r * N);
      } else {
        std::vector<double> L1, L2;
        const int q = p->svd_power_iters > 0 ? p->svd_power_iters : 6;
        const int ov = p->svd_oversample > 0 ? p->svd_oversample : 16;
        randomized_lowrank(What.data(), N, K, r, q, ov, p->svd_seed, L1, L2);
        for (int64_t i = 0; i < K * r; ++i) o.L1[i] = f64_to_bf16(L1[i]);
        for (int64_t i = 0; i < r * N; ++i) o.L2[i] = f64_to_bf16(L2[i]);
      }
    }
    // stage three: residual against the rounded factors, then NVFP4
    std::vector<float> R(size_t(N) * K);
    {
      std::vector<double> L1d(K * r), L2t(N * r);
      for (int64_t i = 0; i < K * r; ++i) L1d[i] = bf16_to_f32(o.L1[i]);
      for (int64_t j = 0; j < r; ++j)
        for (int64_t n = 0; n < N; ++n) L2t[n * r + j] = bf16_to_f32(o.L2[j * N + n]);
#pragma omp parallel for schedule(static)
      for (int64_t n = 0; n < N; ++n)
        for (int64_t k = 0; k < K; ++k) {
          double s = 0.0;
          for (int64_t j = 0; j < r; ++j) s += L1d[k * r + j] * L2t[n * r + j];
          R[n * K + k] = float(What[n * K + k] - s);
        }
    }
    float amax = 0.f;
    for (float x : R) amax = std::max(amax, std::fabs(x));
    o.s_gW = global_scale(amax);
    o.R_codes.assign(size_t(N) * K / 2, 0);
    o.R_scales.assign(size_t(N) * K / 16, 0);
#pragma omp parallel for schedule(static)
    for (int64_t n = 0; n < N; ++n)
      quantize_row(R.data() + n * K, K, o.s_gW, o.R_codes.data() + n * K / 2, o.R_scales.data() + n * K / 16);
    if (R_keep) R_keep->swap(R);
    // activation global scale
    if (p->Xcal_bf16) {
      float xa = 0.f;
      for (int64_t m = 0; m < p->Mcal; ++m)
        for (int64_t k = 0; k < K; ++k)
          xa = std::max(xa, std::fabs(bf16_to_f32(p->Xcal_bf16[m * K + k]) * o.inv_lambda[k]));
      o.s_gX = global_scale(xa);
    } else {
      o.s_gX = p->s_gX > 0.f ? p->s_gX : 1.f;
    }
    o.alpha = o.s_gX * o.s_gW;
    o.bias.assign(N, 0);
    if (p->bias_bf16) std::memcpy(o.bias.data(), p->bias_bf16, sizeof(uint16_t) * N);
  } catch (const std::bad_alloc&) {
    *err = "host allocation failed";
    return SVDQ_ERR_OOM;
  }
  return SVDQ_OK;
}

}  // namespace svdq
