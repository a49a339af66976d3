// C-ABI entry points of the SVDQuant layer's INT4 variant (declared in include/svdq.h).
//
// The handle owns the packed INT4 layer on one device: the residual's INT4 codes and group
// scales, the folded down-projection factor (diag(1 / lambda) L1)^T for kernel int4_k1, L2^T
// and the bias for kernel int4_k2, 1/lambda, a device error word and the workspace (activation
// codes, activation group scales, T).  The forward is the two launches of int4_path.cu.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstring>
#include <new>
#include <string>
#include <vector>

#include "abi_util.cuh"
#include "svdq_internal.h"

using namespace svdq;

struct svdq_int4_layer {
  HostPack host;                 // lambda, inv_lambda, L1, L2, bias (the NVFP4 fields are unused)
  std::vector<uint8_t> codes;    // N x K/2, nibble q + 8
  std::vector<float> scales;     // N x K/64, row-major
  int device = 0;
  int64_t r_pad = 0;
  uint8_t* d_codes = nullptr;
  float* d_scales = nullptr;     // [K/64][round_up(N, 128)]
  float* d_inv_lambda = nullptr;
  uint16_t* d_L1t = nullptr;     // r_pad x K: bf16(inv_lambda[k] L1[k][j]) at [j][k]
  uint16_t* d_L2t = nullptr;     // N x r_pad
  uint16_t* d_bias = nullptr;
  int* d_err = nullptr;
  Int4K1Maps k1maps{};           // L1t filled at pack
  Int4K2Maps k2maps{};           // B, SB and L2 filled at pack
  unsigned char* ws = nullptr;   // activation codes, scales, T for M <= ws_M
  int64_t ws_M = 0;
  uint64_t wait_ns = kDefaultWaitNs;
};

namespace {

int64_t scale_ld(int64_t M) { return round_up(std::max<int64_t>(M, 1), 128); }

struct I4Ws {
  size_t codes, scales, T, total;
};
I4Ws i4_ws(const svdq_int4_layer* h, int64_t M) {
  const int64_t K = h->host.K;
  I4Ws w{};
  size_t off = 0;
  w.codes = off; off += (size_t(M) * K / 2 + 255) & ~size_t(255);
  w.scales = off; off += (size_t(K / 64) * scale_ld(M) * 4 + 255) & ~size_t(255);
  w.T = off; off += (size_t(M) * h->r_pad * 2 + 255) & ~size_t(255);
  w.total = off;
  return w;
}

void free_i4(svdq_int4_layer* h) {
  cudaFree(h->d_codes);
  cudaFree(h->d_scales);
  cudaFree(h->d_inv_lambda);
  cudaFree(h->d_L1t);
  cudaFree(h->d_L2t);
  cudaFree(h->d_bias);
  cudaFree(h->d_err);
  cudaFree(h->ws);
}

svdq_status_t i4_check_shape(const svdq_pack_params_t* p) {
  if (p->K % 64 != 0 || p->N % 16 != 0 || p->rank < 0 || p->rank > 128 || p->rank % 16 != 0 ||
      p->rank > std::min(p->N, p->K))
    return fail(SVDQ_ERR_UNSUPPORTED_SHAPE,
                "INT4 path needs K % 64 == 0, N % 16 == 0, rank % 16 == 0, 0 <= rank <= min(128, N, K)");
  return SVDQ_OK;
}

// Offline step on the host: the shared smoothing, low-rank split and residual, then INT4 groups.
svdq_status_t i4_pack_host(const svdq_pack_params_t* p, svdq_int4_layer* h) {
  std::string err;
  std::vector<float> R;
  svdq_status_t s = pack_on_host(p, &h->host, &err, &R);
  if (s != SVDQ_OK) return fail(s, err);
  const int64_t N = p->N, K = p->K;
  try {
    h->codes.assign(size_t(N) * K / 2, 0);
    h->scales.assign(size_t(N) * (K / 64), 0.f);
  } catch (const std::bad_alloc&) {
    return fail(SVDQ_ERR_OOM, "host allocation failed");
  }
#pragma omp parallel for schedule(static)
  for (int64_t n = 0; n < N; ++n)
    int4_quantize_row(R.data() + n * K, K, h->codes.data() + n * K / 2, h->scales.data() + n * (K / 64));
  return SVDQ_OK;
}

void copy_out(const svdq_int4_layer* h, svdq_int4_host_t* out) {
  const HostPack& hp = h->host;
  const int64_t N = hp.N, K = hp.K, r = hp.rank;
  if (out->lambda) std::memcpy(out->lambda, hp.lambda.data(), sizeof(float) * K);
  if (out->inv_lambda) std::memcpy(out->inv_lambda, hp.inv_lambda.data(), sizeof(float) * K);
  if (out->L1_bf16 && r) std::memcpy(out->L1_bf16, hp.L1.data(), sizeof(uint16_t) * K * r);
  if (out->L2_bf16 && r) std::memcpy(out->L2_bf16, hp.L2.data(), sizeof(uint16_t) * r * N);
  if (out->R_codes) std::memcpy(out->R_codes, h->codes.data(), h->codes.size());
  if (out->R_scales) std::memcpy(out->R_scales, h->scales.data(), sizeof(float) * h->scales.size());
  if (out->bias_bf16) std::memcpy(out->bias_bf16, hp.bias.data(), sizeof(uint16_t) * N);
}

// Kernel int4_k1 on caller buffers (codes M x K/2, scales [K/64][ld], T M x r_pad).
svdq_status_t i4_launch_k1(svdq_int4_layer* h, const void* X, int64_t M, void* codes, float* scales, int64_t ld,
                           void* T, cudaStream_t s) {
  const int64_t K = h->host.K;
  Int4K1Maps maps = h->k1maps;
  std::string err;
  if (!encode_map_2d(maps.X, 2, X, K, M, K * 2, 64, 32, 1, &err)) return fail(SVDQ_ERR_CUDA, err);
  Int4K1Args a{};
  a.inv_lambda = h->d_inv_lambda;
  a.codes = static_cast<uint8_t*>(codes);
  a.scales = scales;
  a.T = static_cast<uint16_t*>(T);
  a.M = M;
  a.K = K;
  a.scale_ld = ld;
  a.r_pad = int(h->r_pad);
  a.err = h->d_err;
  a.wait_ns = h->wait_ns;
  const int e = int4_k1_launch(maps, a, s);
  return e ? cuda_fail(cudaError_t(e), "INT4 kernel 1 launch") : SVDQ_OK;
}

svdq_status_t i4_launch_k2(svdq_int4_layer* h, const void* codes, const float* scales, int64_t ld, const void* T,
                           void* Y, int64_t M, cudaStream_t s) {
  const int64_t K = h->host.K, N = h->host.N;
  Int4K2Maps maps = h->k2maps;
  std::string err;
  if (!encode_map_2d(maps.A, 1, codes, K / 2, M, K / 2, 32, 128, 0, &err) ||
      !encode_map_2d(maps.SA, 4, scales, ld, K / 64, ld * 4, 128, 1, 0, &err))
    return fail(SVDQ_ERR_CUDA, err);
  if (h->r_pad && !encode_map_2d(maps.T, 2, T, h->r_pad, M, h->r_pad * 2, 64, 128, 1, &err))
    return fail(SVDQ_ERR_CUDA, err);
  Int4K2Args a{};
  a.bias = h->d_bias;
  a.Y = static_cast<uint16_t*>(Y);
  a.M = M;
  a.N = N;
  a.K = K;
  a.r_pad = int(h->r_pad);
  a.err = h->d_err;
  a.wait_ns = h->wait_ns;
  const int e = int4_k2_launch(maps, a, s);
  return e ? cuda_fail(cudaError_t(e), "INT4 kernel 2 launch") : SVDQ_OK;
}

}  // namespace

extern "C" {

int64_t svdq_int4_scale_ld(int64_t M) { return M < 0 ? 0 : scale_ld(M); }

svdq_status_t svdq_int4_pack_host(const svdq_pack_params_t* p, svdq_int4_host_t* out) {
  if (!p || !out) return fail(SVDQ_ERR_INVALID_ARG, "null argument");
  svdq_status_t s = i4_check_shape(p);
  if (s != SVDQ_OK) return s;
  svdq_int4_layer* h = new (std::nothrow) svdq_int4_layer();
  if (!h) return fail(SVDQ_ERR_OOM, "host allocation failed");
  s = i4_pack_host(p, h);
  if (s == SVDQ_OK) copy_out(h, out);
  delete h;
  return s;
}

svdq_status_t svdq_int4_pack(const svdq_pack_params_t* p, svdq_int4_handle_t* out) {
  if (!p || !out) return fail(SVDQ_ERR_INVALID_ARG, "null argument");
  *out = nullptr;
  svdq_status_t s = i4_check_shape(p);
  if (s != SVDQ_OK) return s;
  if (p->M_max < 0) return fail(SVDQ_ERR_INVALID_ARG, "M_max must be >= 0");
  int ndev = 0;
  cudaError_t e = cudaGetDeviceCount(&ndev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDeviceCount");
  if (p->device < 0 || p->device >= ndev) return fail(SVDQ_ERR_INVALID_ARG, "no such device");
  s = check_arch(p->device);
  if (s != SVDQ_OK) return s;
  svdq_int4_layer* h = new (std::nothrow) svdq_int4_layer();
  if (!h) return fail(SVDQ_ERR_OOM, "host allocation failed");
  s = i4_pack_host(p, h);
  if (s != SVDQ_OK) {
    delete h;
    return s;
  }
  DeviceGuard guard(p->device);
  cudaStream_t stream = static_cast<cudaStream_t>(p->stream);
  h->device = p->device;
  const HostPack& hp = h->host;
  const int64_t N = hp.N, K = hp.K, r = hp.rank, G = K / 64, ldn = scale_ld(N);
  h->r_pad = rank_pad(r);
  const int64_t rp = h->r_pad;
  // device layouts
  std::vector<float> sc(size_t(G) * ldn, 0.f);
  for (int64_t n = 0; n < N; ++n)
    for (int64_t g = 0; g < G; ++g) sc[g * ldn + n] = h->scales[n * G + g];
  std::vector<uint16_t> l1t(size_t(std::max<int64_t>(rp, 1)) * K, 0), l2t(size_t(N) * std::max<int64_t>(rp, 1), 0);
  for (int64_t j = 0; j < r; ++j)
    for (int64_t k = 0; k < K; ++k)
      l1t[j * K + k] = f64_to_bf16(double(hp.inv_lambda[k]) * double(bf16_to_f32(hp.L1[k * r + j])));
  for (int64_t n = 0; n < N; ++n)
    for (int64_t j = 0; j < r; ++j) l2t[n * rp + j] = hp.L2[j * N + n];
  auto up = [&](void** dst, const void* src, size_t bytes) -> cudaError_t {
    cudaError_t ee;
    *dst = dalloc(bytes, &ee);
    if (ee != cudaSuccess) return ee;
    if (bytes) ee = cudaMemcpyAsync(*dst, src, bytes, cudaMemcpyHostToDevice, stream);
    return ee;
  };
  e = up(reinterpret_cast<void**>(&h->d_codes), h->codes.data(), h->codes.size());
  if (e == cudaSuccess) e = up(reinterpret_cast<void**>(&h->d_scales), sc.data(), sc.size() * 4);
  if (e == cudaSuccess) e = up(reinterpret_cast<void**>(&h->d_inv_lambda), hp.inv_lambda.data(), K * 4);
  if (e == cudaSuccess) e = up(reinterpret_cast<void**>(&h->d_L1t), l1t.data(), l1t.size() * 2);
  if (e == cudaSuccess) e = up(reinterpret_cast<void**>(&h->d_L2t), l2t.data(), l2t.size() * 2);
  if (e == cudaSuccess) e = up(reinterpret_cast<void**>(&h->d_bias), hp.bias.data(), N * 2);
  if (e == cudaSuccess) {
    h->d_err = static_cast<int*>(dalloc(sizeof(int), &e));
    if (e == cudaSuccess) e = cudaMemsetAsync(h->d_err, 0, sizeof(int), stream);
  }
  if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
  std::string err;
  bool ok = e == cudaSuccess;
  if (ok) {
    ok = encode_map_2d(h->k2maps.B, 1, h->d_codes, K / 2, N, K / 2, 32, 128, 0, &err) &&
         encode_map_2d(h->k2maps.SB, 4, h->d_scales, ldn, G, ldn * 4, 128, 1, 0, &err);
    if (ok && rp)
      ok = encode_map_2d(h->k1maps.L1t, 2, h->d_L1t, K, rp, K * 2, 64, uint32_t(rp), 1, &err) &&
           encode_map_2d(h->k2maps.L2, 2, h->d_L2t, rp, N, rp * 2, 64, 128, 1, &err);
  }
  if (!ok) {
    free_i4(h);
    delete h;
    if (e == cudaErrorMemoryAllocation) return fail(SVDQ_ERR_OOM, "device allocation failed");
    return e != cudaSuccess ? cuda_fail(e, "uploading the INT4 layer") : fail(SVDQ_ERR_CUDA, err);
  }
  if (p->M_max > 0) {
    s = svdq_int4_reserve(h, p->M_max);
    if (s != SVDQ_OK) {
      free_i4(h);
      delete h;
      return s;
    }
  }
  *out = h;
  return SVDQ_OK;
}

svdq_status_t svdq_int4_export(svdq_int4_handle_t h, svdq_int4_host_t* out) {
  if (!h || !out) return fail(SVDQ_ERR_INVALID_ARG, "null argument");
  copy_out(h, out);
  return SVDQ_OK;
}

svdq_status_t svdq_int4_reserve(svdq_int4_handle_t h, int64_t M_max) {
  if (!h || M_max < 0) return fail(SVDQ_ERR_INVALID_ARG, "null handle or negative M_max");
  DeviceGuard guard(h->device);
  cudaError_t e;
  void* p = dalloc(i4_ws(h, M_max).total, &e);
  if (e != cudaSuccess) return fail(SVDQ_ERR_OOM, "workspace allocation failed");
  cudaFree(h->ws);
  h->ws = static_cast<unsigned char*>(p);
  h->ws_M = M_max;
  return SVDQ_OK;
}

svdq_status_t svdq_int4_quantize_act(svdq_int4_handle_t h, const void* X, int64_t M, void* x_codes, float* x_scales,
                                     void* T, void* stream) {
  if (!h || M < 0) return fail(SVDQ_ERR_INVALID_ARG, "null handle or negative M");
  if (M == 0) return SVDQ_OK;
  if (!X || !x_codes || !x_scales || (h->r_pad && !T)) return fail(SVDQ_ERR_INVALID_ARG, "null buffer");
  if (!aligned16(X) || !aligned16(x_codes) || !aligned16(x_scales) || (T && !aligned16(T)))
    return fail(SVDQ_ERR_INVALID_ARG, "buffers must be 16-byte aligned");
  DeviceGuard guard(h->device);
  return i4_launch_k1(h, X, M, x_codes, x_scales, scale_ld(M), T, static_cast<cudaStream_t>(stream));
}

svdq_status_t svdq_int4_forward(svdq_int4_handle_t h, const void* X, void* Y, int64_t M, void* stream) {
  if (!h || M < 0) return fail(SVDQ_ERR_INVALID_ARG, "null handle or negative M");
  if (M == 0) return SVDQ_OK;
  if (!X || !Y) return fail(SVDQ_ERR_INVALID_ARG, "null buffer");
  if (!aligned16(X) || !aligned16(Y)) return fail(SVDQ_ERR_INVALID_ARG, "buffers must be 16-byte aligned");
  if (!h->ws || h->ws_M < M) return fail(SVDQ_ERR_WORKSPACE, "no workspace for this M (svdq_int4_reserve)");
  const size_t xb = size_t(M) * h->host.K * 2, yb = size_t(M) * h->host.N * 2;
  const I4Ws w = i4_ws(h, h->ws_M);
  if (overlaps(X, xb, Y, yb) || overlaps(X, xb, h->ws, w.total) || overlaps(Y, yb, h->ws, w.total))
    return fail(SVDQ_ERR_INVALID_ARG, "X, Y and the workspace must not overlap");
  DeviceGuard guard(h->device);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  void* codes = h->ws + w.codes;
  float* scales = reinterpret_cast<float*>(h->ws + w.scales);
  void* T = h->r_pad ? h->ws + w.T : nullptr;
  const int64_t ld = scale_ld(h->ws_M);
  svdq_status_t st = i4_launch_k1(h, X, M, codes, scales, ld, T, s);
  if (st != SVDQ_OK) return st;
  return i4_launch_k2(h, codes, scales, ld, T, Y, M, s);
}

svdq_status_t svdq_int4_check_error(svdq_int4_handle_t h) {
  if (!h) return fail(SVDQ_ERR_INVALID_ARG, "null handle");
  DeviceGuard guard(h->device);
  cudaError_t e = cudaDeviceSynchronize();
  if (e != cudaSuccess) return cuda_fail(e, "device synchronisation");
  int v = 0;
  e = cudaMemcpy(&v, h->d_err, sizeof(int), cudaMemcpyDeviceToHost);
  if (e == cudaSuccess) e = cudaMemset(h->d_err, 0, sizeof(int));
  if (e != cudaSuccess) return cuda_fail(e, "reading the device error word");
  if (v) return fail(SVDQ_ERR_TIMEOUT, "an INT4 kernel gave up a bounded wait");
  return SVDQ_OK;
}

svdq_status_t svdq_int4_destroy(svdq_int4_handle_t h) {
  if (!h) return SVDQ_OK;
  DeviceGuard guard(h->device);
  cudaDeviceSynchronize();
  free_i4(h);
  delete h;
  return SVDQ_OK;
}

}  // extern "C"
