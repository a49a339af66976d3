// Offline step of the AWQ-style W4A16 layer, on the host: activation-aware per-channel
// scales (exponent picked by a grid search on calibration activations), then asymmetric
// 4-bit quantisation of W diag(s) in groups of 64 input channels with a float32 scale and an
// integer zero point.  The pages keep 16-bit activations and AWQ-style 4-bit weights for the
// adaptive-normalisation and modulation layers (aiflownews article on Nunchaku, "How Nunchaku
// four bit quantization actually works"); the group size, scale format and search rule are
// readings of ours:
//   s = fl32(max(w_max - w_min, 1e-5) / 15),  z = clamp(rint(-w_min / s), 0, 15),
//   q = clamp(rint(w / s) + z, 0, 15)                          (float32, ties to even)
//   s_c = a_c^alpha / sqrt(max s * min s),  a_c = mean |Xcal_c|,  alpha in {0, 0.05, .., 0.95}
#include <cmath>
#include <cstring>
#include <limits>
#include <string>
#include <vector>

#include "svdq_internal.h"

namespace svdq {

namespace {

constexpr int kGroup = 64;

// float32 group quantiser over rows of w (N x K) -> codes (N x K, one per byte), scales and
// zeros (N x K/64)
void quantize_groups(const float* w, int64_t N, int64_t K, uint8_t* q, float* s, uint8_t* z) {
  const int64_t KG = K / kGroup;
#pragma omp parallel for schedule(static)
  for (int64_t n = 0; n < N; ++n) {
    for (int64_t g = 0; g < KG; ++g) {
      const float* v = w + n * K + g * kGroup;
      float mn = v[0], mx = v[0];
      for (int i = 1; i < kGroup; ++i) {
        mn = std::fmin(mn, v[i]);
        mx = std::fmax(mx, v[i]);
      }
      volatile float range = mx - mn;                         // float32 rounding, no contraction
      const float r = std::fmax(range, 1e-5f);
      volatile float sc_v = r / 15.0f;
      const float sc = sc_v;
      volatile float zq = -mn / sc;
      float zr = std::nearbyint(float(zq));
      zr = zr < 0.f ? 0.f : (zr > 15.f ? 15.f : zr);
      s[n * KG + g] = sc;
      z[n * KG + g] = uint8_t(zr);
      for (int i = 0; i < kGroup; ++i) {
        volatile float t = v[i] / sc;
        float c = std::nearbyint(float(t)) + zr;
        c = c < 0.f ? 0.f : (c > 15.f ? 15.f : c);
        q[n * K + g * kGroup + i] = uint8_t(c);
      }
    }
  }
}

std::vector<float> scales_for(const std::vector<double>& a, double alpha) {
  const int64_t K = int64_t(a.size());
  std::vector<double> v(K, 1.0);
  double vmax = 0.0, vmin = std::numeric_limits<double>::infinity();
  bool any = false;
  for (int64_t c = 0; c < K; ++c)
    if (a[c] > 0) {
      v[c] = std::pow(a[c], alpha);
      vmax = std::fmax(vmax, v[c]);
      vmin = std::fmin(vmin, v[c]);
      any = true;
    }
  std::vector<float> s(K, 1.0f);
  if (any) {
    const double norm = std::sqrt(vmax * vmin);
    for (int64_t c = 0; c < K; ++c) s[c] = a[c] > 0 ? float(v[c] / norm) : 1.0f;
  }
  return s;
}

void scaled_weight(const uint16_t* W, int64_t N, int64_t K, const float* s, float* out) {
#pragma omp parallel for schedule(static)
  for (int64_t n = 0; n < N; ++n)
    for (int64_t k = 0; k < K; ++k) {
      volatile float p = bf16_to_f32(W[n * K + k]) * s[k];
      out[n * K + k] = p;
    }
}

}  // namespace

svdq_status_t awq_pack_host(const svdq_awq_params_t* p, AwqHostPack* out, std::string* err) {
  const int64_t N = p->N, K = p->K;
  if (N <= 0 || K <= 0 || !p->W_bf16) {
    *err = "N, K must be > 0 and W is required";
    return SVDQ_ERR_INVALID_ARG;
  }
  if (K % kGroup != 0) {
    *err = "K must be a multiple of 64 (the weight group size)";
    return SVDQ_ERR_UNSUPPORTED_SHAPE;
  }
  if (p->Xcal_bf16 && p->Mcal <= 0) {
    *err = "Mcal must be > 0 when Xcal is given";
    return SVDQ_ERR_INVALID_ARG;
  }
  const int64_t KG = K / kGroup;
  out->N = N;
  out->K = K;
  out->alpha = -1.f;
  out->s.assign(K, 1.0f);
  std::vector<float> ws(size_t(N) * K);
  std::vector<uint8_t> q(size_t(N) * K);
  out->scales.assign(size_t(N) * KG, 0.f);
  out->zeros.assign(size_t(N) * KG, 0);
  if (p->s) {
    std::memcpy(out->s.data(), p->s, size_t(K) * sizeof(float));
  } else if (p->Xcal_bf16) {
    // grid search: the alpha whose quantised layer reproduces Xcal W^T best (float64 error)
    const int64_t Mc = p->Mcal;
    std::vector<double> a(K, 0.0), X(size_t(Mc) * K), ref(size_t(Mc) * N, 0.0);
    for (int64_t m = 0; m < Mc; ++m)
      for (int64_t k = 0; k < K; ++k) {
        X[m * K + k] = bf16_to_f32(p->Xcal_bf16[m * K + k]);
        a[k] += std::fabs(X[m * K + k]);
      }
    for (int64_t k = 0; k < K; ++k) a[k] /= double(Mc);
#pragma omp parallel for schedule(static)
    for (int64_t n = 0; n < N; ++n)
      for (int64_t m = 0; m < Mc; ++m) {
        double acc = 0.0;
        for (int64_t k = 0; k < K; ++k) acc += X[m * K + k] * double(bf16_to_f32(p->W_bf16[n * K + k]));
        ref[m * N + n] = acc;
      }
    double best = std::numeric_limits<double>::infinity();
    for (int i = 0; i < 20; ++i) {
      const double alpha = i / 20.0;
      const std::vector<float> s = scales_for(a, alpha);
      scaled_weight(p->W_bf16, N, K, s.data(), ws.data());
      quantize_groups(ws.data(), N, K, q.data(), out->scales.data(), out->zeros.data());
      std::vector<float> xs(size_t(Mc) * K);
      for (int64_t m = 0; m < Mc; ++m)
        for (int64_t k = 0; k < K; ++k) {
          volatile float inv = 1.0f / s[k];
          volatile float v = bf16_to_f32(p->Xcal_bf16[m * K + k]) * inv;
          xs[m * K + k] = v;
        }
      double e = 0.0;
#pragma omp parallel for schedule(static) reduction(+ : e)
      for (int64_t n = 0; n < N; ++n)
        for (int64_t m = 0; m < Mc; ++m) {
          double acc = 0.0;
          for (int64_t k = 0; k < K; ++k) {
            const int64_t g = k / kGroup;
            const double d = (double(q[n * K + k]) - double(out->zeros[n * KG + g])) * double(out->scales[n * KG + g]);
            acc += double(xs[m * K + k]) * d;
          }
          const double diff = acc - ref[m * N + n];
          e += diff * diff;
        }
      if (e < best) {
        best = e;
        out->alpha = float(alpha);
        out->s = s;
      }
    }
  }
  scaled_weight(p->W_bf16, N, K, out->s.data(), ws.data());
  quantize_groups(ws.data(), N, K, q.data(), out->scales.data(), out->zeros.data());
  out->codes.assign(size_t(N) * K / 2, 0);
  for (int64_t n = 0; n < N; ++n)
    for (int64_t k = 0; k < K; k += 2)
      out->codes[(n * K + k) / 2] = uint8_t(q[n * K + k] | (q[n * K + k + 1] << 4));
  out->inv_s.resize(K);
  for (int64_t k = 0; k < K; ++k) {
    volatile float inv = 1.0f / out->s[k];
    out->inv_s[k] = inv;
  }
  out->bias.assign(N, 0);
  if (p->bias_bf16) std::memcpy(out->bias.data(), p->bias_bf16, size_t(N) * 2);
  return SVDQ_OK;
}

}  // namespace svdq
