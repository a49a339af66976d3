// C-ABI entry points of the SVDQuant W4A4 linear layer (declared in include/svdq.h).
//
// The handle owns the packed layer on one device: the tiled NVFP4 residual, the folded and
// permuted L1 for kernel 1, L2^T for kernel 2, 1/lambda, the bias, a device error word and
// (optionally) a workspace.  The forward is two launches on the caller's stream: kernel 1
// (smoothing + NVFP4 quantisation + down-projection, one read of X) and kernel 2 (block-scaled
// FP4 tensor-core GEMM + up-projection + bias, one write of Y).
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <cmath>
#include <cstring>
#include <atomic>
#include <mutex>
#include <new>
#include <string>
#include <vector>

#include "abi_util.cuh"
#include "svdq_internal.h"

using namespace svdq;

namespace {

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

}  // namespace

namespace svdq {

std::string& last_error_slot() {
  thread_local std::string msg;
  return msg;
}

svdq_status_t check_arch(int device) {
  cudaDeviceProp prop;
  cudaError_t e = cudaGetDeviceProperties(&prop, device);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDeviceProperties");
  if (!(prop.major == 10 && prop.minor == 3))
    return fail(SVDQ_ERR_ARCH, "device " + std::to_string(device) + " is sm_" + std::to_string(prop.major) +
                                   std::to_string(prop.minor) + ", this library is built for sm_103a (B300)");
  return SVDQ_OK;
}

bool encode_map_2d(void* map, int dtype_bytes, const void* base, uint64_t inner, uint64_t outer,
                   uint64_t row_stride_bytes, uint32_t box_inner, uint32_t box_outer, int swizzle128,
                   std::string* err) {
  std::call_once(g_encode_once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  });
  if (!g_encode) {
    *err = "cuTensorMapEncodeTiled is not available from the driver";
    return false;
  }
  const CUtensorMapDataType dt = dtype_bytes == 1   ? CU_TENSOR_MAP_DATA_TYPE_UINT8
                                 : dtype_bytes == 4 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32
                                                    : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  cuuint64_t dims[2] = {inner, outer < 1 ? 1 : outer};
  cuuint64_t strides[1] = {row_stride_bytes};
  cuuint32_t box[2] = {box_inner, box_outer};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = g_encode(reinterpret_cast<CUtensorMap*>(map), dt, 2, const_cast<void*>(base), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE,
                        swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    *err = "cuTensorMapEncodeTiled failed with CUresult " + std::to_string(int(r));
    return false;
  }
  return true;
}

}  // namespace svdq

struct svdq_layer {
  HostPack host;
  int device = 0;
  int sm_count = 0;
  int64_t r_pad = 0;
  // device copies
  uint8_t* d_wt = nullptr;         // kernel 2's weight blocks: codes and scales per pair tile, K step, half
  uint16_t* d_L2t = nullptr;       // N x r_pad
  unsigned char* d_LI = nullptr;   // groups of four chunks: folded + permuted L1 slices, then 1/lambda
  float* d_inv_lambda = nullptr;
  float* d_qtab = nullptr;         // activation quantiser tables (thresholds, reciprocals)
  uint16_t* d_bias = nullptr;
  int* d_err = nullptr;
  K2Maps maps{};                   // L2 filled at pack
  // LoRA factors appended to the low-rank branch (svdq_attach_lora): r_lora columns of
  // bf16(scale * A) after L1's columns, r_lora rows of B after L2's rows
  int64_t r_lora = 0;
  std::vector<uint16_t> lora_A;    // K x r_lora (bf16 bits, scale applied)
  std::vector<uint16_t> lora_B;    // r_lora x N (bf16 bits)
  int64_t rank_k() const { return host.rank + r_lora; }   // rank the kernels run with
  // workspace
  unsigned char* ws = nullptr;
  size_t ws_bytes = 0;
  bool ws_owned = false;
  int64_t ws_M = 0;
  int ws_staging = 0;              // device staging slots for host X / Y (0, 1 or 2)
  // pipelined host calls (svdq_linear_forward_host_batch): copy streams and slot events,
  // created on first use
  cudaStream_t pipe_in = nullptr, pipe_out = nullptr;
  cudaEvent_t ev_in[2] = {nullptr, nullptr}, ev_comp[2] = {nullptr, nullptr}, ev_out[2] = {nullptr, nullptr};
  float inv_six = 1.f / 6.f, inv_alpha = 1.f;
  // failure-detection tests (svdq_set_wait_limit): limit of the kernels' bounded waits, and
  // which kernel's MMA warp waits on a barrier nothing completes (0 none, 1 kernel 1, 2 kernel 2)
  uint64_t wait_ns = kDefaultWaitNs;
  int stall = 0;
  uint64_t low_rank_gen = 0;       // counts uploads of the low-rank factors (MLP pairs check it)
};

namespace {

struct WsLayout {
  size_t codes, scales, T, partial, arrivals, Xs[2], Ys[2], total;
};

// host_staging argument -> number of staging slots
int staging_slots(int32_t host_staging) { return host_staging <= 0 ? 0 : (host_staging >= 2 ? 2 : 1); }

WsLayout ws_layout(const svdq_layer* h, int64_t M, int staging) {
  WsLayout w{};
  const int64_t K = h->host.K, N = h->host.N, r = h->rank_k();
  size_t off = 0;
  w.codes = off; off += align256(size_t(M) * K / 2);
  w.scales = off; off += align256(size_t(svdq_scales_bytes(M, K)));
  w.T = off; off += align256(size_t(M) * h->r_pad * 2);
  w.partial = off; off += align256(k1_partial_bytes(M, int(r)));
  w.arrivals = off; off += align256(r ? k1_arrival_bytes(M) : 0);
  for (int i = 0; i < 2; ++i) {
    w.Xs[i] = off; off += i < staging ? align256(size_t(M) * K * 2) : 0;
    w.Ys[i] = off; off += i < staging ? align256(size_t(M) * N * 2) : 0;
  }
  w.total = off;
  return w;
}


svdq_status_t check_shape(int64_t N, int64_t K, int64_t r) {
  if (K % 64 != 0 || N % 16 != 0 || r < 0 || r > 128 || r % 16 != 0 || r > std::min(N, K))
    return fail(SVDQ_ERR_UNSUPPORTED_SHAPE,
                "CUDA path needs K % 64 == 0, N % 16 == 0, rank % 16 == 0, 0 <= rank <= min(128, N, K)");
  return SVDQ_OK;
}

void free_layer(svdq_layer* h) {
  cudaFree(h->d_wt);
  cudaFree(h->d_L2t);
  cudaFree(h->d_LI);
  cudaFree(h->d_inv_lambda);
  cudaFree(h->d_qtab);
  cudaFree(h->d_bias);
  cudaFree(h->d_err);
  if (h->ws_owned) cudaFree(h->ws);
  if (h->pipe_in) cudaStreamDestroy(h->pipe_in);
  if (h->pipe_out) cudaStreamDestroy(h->pipe_out);
  for (int i = 0; i < 2; ++i) {
    if (h->ev_in[i]) cudaEventDestroy(h->ev_in[i]);
    if (h->ev_comp[i]) cudaEventDestroy(h->ev_comp[i]);
    if (h->ev_out[i]) cudaEventDestroy(h->ev_out[i]);
  }
}

// Device layouts of the low-rank branch for the handle's kernel rank (SVD rank plus any LoRA
// rank), uploaded into fresh buffers that replace the old ones:
//   LI   per group of four 64-column chunks: the chunks' slices of L1' (rank_k rows of 64
//        K-values, bf16, K-major, 128-byte rows with the 128-byte swizzle the tensor cores
//        read: 16-byte unit u of row j stored at unit u ^ (j % 8)), then the chunks' 64 values
//        of 1/lambda each (fp32, in the bank-spread order described where they are written).
//        L1' = diag(1/lambda) L1 for the SVD columns (kernel 1 multiplies raw X by it, which
//        is X^ L1), and bf16(scale * A) for the LoRA columns (X A needs no smoothing)
//   L2t  N x r_pad bf16: L2 transposed, then B transposed, zero padding
// Column j of L1' at row k (bf16 bits): bf16(1/lambda_k * L1[k][j]) for an SVD column, the
// scaled LoRA A for a LoRA column.
uint16_t l1_prime(const svdq_layer* h, int64_t k, int64_t j) {
  const HostPack& hp = h->host;
  const int64_t r = hp.rank;
  return j < r ? f64_to_bf16(double(hp.inv_lambda[k]) * double(bf16_to_f32(hp.L1[k * r + j])))
               : h->lora_A[k * h->r_lora + (j - r)];
}

svdq_status_t upload_low_rank(svdq_layer* h, cudaStream_t stream) {
  const HostPack& hp = h->host;
  const int64_t N = hp.N, K = hp.K, r = hp.rank, rl = h->r_lora, rk = r + rl;
  const int64_t r_pad = rank_pad(rk);
  std::vector<uint16_t> l2t(size_t(N) * std::max<int64_t>(r_pad, 1), 0);
  for (int64_t n = 0; n < N; ++n) {
    for (int64_t j = 0; j < r; ++j) l2t[n * r_pad + j] = hp.L2[j * N + n];
    for (int64_t j = 0; j < rl; ++j) l2t[n * r_pad + r + j] = h->lora_B[j * N + n];
  }
  // groups of four chunks (4g .. 4g + 3): [the four slices][the four 1/lambda parts]; a chunk
  // past K stays zero
  const int64_t nch = K / 64, ngroups = (nch + 3) / 4;
  const int64_t li_group = 4 * (rk * 128 + 256);
  std::vector<unsigned char> li(size_t(ngroups) * li_group, 0);
  for (int64_t c = 0; c < nch; ++c) {
    unsigned char* grp = li.data() + (c / 4) * li_group;
    unsigned char* slice = grp + (c % 4) * rk * 128;
    for (int64_t j = 0; j < rk; ++j)
      for (int i = 0; i < 64; ++i) {
        const int64_t k = 64 * c + i;
        const uint16_t v = l1_prime(h, k, j);
        const int unit = (i / 8) ^ int(j % 8);
        reinterpret_cast<uint16_t*>(slice + j * 128 + unit * 16)[i % 8] = v;
      }
    // 1/lambda part: thread t of a quantiser quad reads floats 16 t .. 16 t + 15 as four 16-byte
    // loads k = 0..3; load k of thread t sits in 16-byte unit 4 t + (k ^ (t >> 1)), so the four
    // threads' k-th loads fall in four different bank groups
    for (int tt = 0; tt < 4; ++tt)
      for (int kk = 0; kk < 4; ++kk)
        std::memcpy(grp + 4 * rk * 128 + (c % 4) * 256 + 16 * (4 * tt + (kk ^ (tt >> 1))),
                    hp.inv_lambda.data() + 64 * c + 16 * tt + 4 * kk, 16);
  }
  cudaError_t e;
  uint16_t* d_l2t = static_cast<uint16_t*>(dalloc(l2t.size() * 2, &e));
  unsigned char* d_li = nullptr;
  if (e == cudaSuccess) d_li = static_cast<unsigned char*>(dalloc(li.size(), &e));
  if (e == cudaSuccess) e = cudaMemcpyAsync(d_l2t, l2t.data(), l2t.size() * 2, cudaMemcpyHostToDevice, stream);
  if (e == cudaSuccess) e = cudaMemcpyAsync(d_li, li.data(), li.size(), cudaMemcpyHostToDevice, stream);
  if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
  K2Maps maps = h->maps;
  std::string err;
  if (e == cudaSuccess && rk > 0 && !encode_map_2d(maps.L2, 2, d_l2t, r_pad, N, r_pad * 2, 64, 128, 1, &err)) {
    cudaFree(d_l2t);
    cudaFree(d_li);
    return fail(SVDQ_ERR_CUDA, err);
  }
  if (e != cudaSuccess) {
    cudaFree(d_l2t);
    cudaFree(d_li);
    return e == cudaErrorMemoryAllocation ? fail(SVDQ_ERR_OOM, "device allocation failed")
                                          : cuda_fail(e, "uploading the low-rank branch");
  }
  cudaFree(h->d_L2t);
  cudaFree(h->d_LI);
  h->d_L2t = d_l2t;
  h->d_LI = d_li;
  h->maps = maps;
  h->r_pad = r_pad;
  ++h->low_rank_gen;
  return SVDQ_OK;
}

svdq_status_t attach_workspace(svdq_layer* h, void* ptr, size_t bytes, int64_t M_max, int staging, bool owned,
                               cudaStream_t stream) {
  if (h->ws_owned && h->ws) cudaFree(h->ws);
  h->ws = static_cast<unsigned char*>(ptr);
  h->ws_bytes = bytes;
  h->ws_owned = owned;
  h->ws_M = ptr ? M_max : 0;
  h->ws_staging = ptr ? staging : 0;
  (void)stream;
  return SVDQ_OK;
}

// Kernel 1 launches draw a process-wide unique epoch for their split-K arrival words.
std::atomic<unsigned long long> g_k1_epoch{1};

void k1_scratch(K1Args* a, unsigned char* ws, const WsLayout& w) {
  a->partial = reinterpret_cast<float*>(ws + w.partial);
  a->arrivals = reinterpret_cast<unsigned long long*>(ws + w.arrivals);
  a->epoch = g_k1_epoch.fetch_add(1) & ((1ull << 56) - 1);
}

svdq_status_t launch_k1(svdq_layer* h, const void* X, int64_t M, void* codes, void* scales, void* T,
                        cudaStream_t stream) {
  K1Args a{};
  k1_scratch(&a, h->ws, ws_layout(h, h->ws_M, h->ws_staging));
  a.X = static_cast<const uint16_t*>(X);
  a.LI = h->d_LI;
  a.x_codes = static_cast<uint8_t*>(codes);
  a.x_scales = static_cast<uint8_t*>(scales);
  a.T = static_cast<uint16_t*>(T);
  a.M = M;
  a.K = h->host.K;
  a.rank = int(h->rank_k());
  a.r_pad = int(h->r_pad);
  a.s_gX = h->host.s_gX;
  a.inv_six = h->inv_six;
  a.inv_alpha = h->inv_alpha;
  a.qtab = h->d_qtab;
  a.err = h->d_err;
  a.wait_ns = h->wait_ns;
  a.stall = h->stall == 1;
  const K1Plan plan = k1_plan(M, a.K, a.rank, h->sm_count);
  std::string err;
  const int e = k1_launch(a, plan, stream, &err);
  if (e == -1) return fail(SVDQ_ERR_CUDA, err);
  if (e != 0) return cuda_fail(cudaError_t(e), "kernel 1 launch");
  return SVDQ_OK;
}

svdq_status_t launch_k2(svdq_layer* h, const void* codes, const void* scales, const void* T, void* Y, int64_t M,
                        cudaStream_t stream) {
  const int64_t K = h->host.K, N = h->host.N;
  K2Maps maps = h->maps;
  std::string err;
  if (!encode_map_2d(maps.A, 1, codes, K / 2, M, K / 2, 128, 128, 1, &err) ||
      !encode_map_2d(maps.SFA, 1, scales, 256, svdq_scales_bytes(M, K) / 256, 256, 256, 8, 0, &err) ||
      !encode_map_2d(maps.Y, 2, Y, N, M, N * 2, 64, 32, 1, &err))
    return fail(SVDQ_ERR_CUDA, err);
  if (h->rank_k() > 0 && !encode_map_2d(maps.T, 2, T, h->r_pad, M, h->r_pad * 2, 64, 128, 1, &err))
    return fail(SVDQ_ERR_CUDA, err);
  K2Args a{};
  a.bias = h->d_bias;
  a.wt = h->d_wt;
  a.err = h->d_err;
  a.M = M;
  a.N = N;
  a.K = K;
  a.rank = int(h->rank_k());
  a.alpha = h->host.alpha;
  a.wait_ns = h->wait_ns;
  a.stall = h->stall == 2;
  const int e = k2_launch(maps, a, h->sm_count, stream);
  if (e != 0) return cuda_fail(cudaError_t(e), "kernel 2 launch");
  return SVDQ_OK;
}


}  // namespace

extern "C" {

const char* svdq_status_string(svdq_status_t s) {
  switch (s) {
    case SVDQ_OK: return "ok";
    case SVDQ_ERR_INVALID_ARG: return "invalid argument";
    case SVDQ_ERR_UNSUPPORTED_SHAPE: return "unsupported shape";
    case SVDQ_ERR_ARCH: return "unsupported device architecture";
    case SVDQ_ERR_OOM: return "out of memory";
    case SVDQ_ERR_CUDA: return "CUDA error";
    case SVDQ_ERR_TIMEOUT: return "kernel wait timed out";
    case SVDQ_ERR_WORKSPACE: return "workspace missing or too small";
  }
  return "unknown status";
}

const char* svdq_last_error(void) { return last_error_slot().c_str(); }

int64_t svdq_scales_bytes(int64_t M, int64_t K) {
  if (M < 0 || K < 0) return 0;
  return ceil_div(M, 128) * scale_groups(K) * 512;
}

svdq_status_t svdq_pack_host(const svdq_pack_params_t* p, svdq_packed_host_t* out) {
  if (!p || !out) return fail(SVDQ_ERR_INVALID_ARG, "null argument");
  HostPack hp;
  std::string err;
  svdq_status_t s = pack_on_host(p, &hp, &err);
  if (s != SVDQ_OK) return fail(s, err);
  const int64_t N = hp.N, K = hp.K, r = hp.rank;
  if (out->lambda) std::memcpy(out->lambda, hp.lambda.data(), sizeof(float) * K);
  if (out->inv_lambda) std::memcpy(out->inv_lambda, hp.inv_lambda.data(), sizeof(float) * K);
  if (out->L1_bf16 && r) std::memcpy(out->L1_bf16, hp.L1.data(), sizeof(uint16_t) * K * r);
  if (out->L2_bf16 && r) std::memcpy(out->L2_bf16, hp.L2.data(), sizeof(uint16_t) * r * N);
  if (out->R_codes) std::memcpy(out->R_codes, hp.R_codes.data(), hp.R_codes.size());
  if (out->R_scales) std::memcpy(out->R_scales, hp.R_scales.data(), hp.R_scales.size());
  if (out->bias_bf16) std::memcpy(out->bias_bf16, hp.bias.data(), sizeof(uint16_t) * N);
  out->s_gW = hp.s_gW;
  out->s_gX = hp.s_gX;
  out->alpha = hp.alpha;
  return SVDQ_OK;
}

svdq_status_t svdq_pack_weights(const svdq_pack_params_t* p, svdq_handle_t* out) {
  if (!p || !out) return fail(SVDQ_ERR_INVALID_ARG, "null argument");
  *out = nullptr;
  svdq_status_t s = check_shape(p->N, p->K, p->rank);
  if (s != SVDQ_OK) return s;
  if (p->M_max < 0) return fail(SVDQ_ERR_INVALID_ARG, "M_max must be >= 0");
  int ndev = 0;
  cudaError_t e = cudaGetDeviceCount(&ndev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDeviceCount");
  if (p->device < 0 || p->device >= ndev) return fail(SVDQ_ERR_INVALID_ARG, "no such device");
  s = check_arch(p->device);
  if (s != SVDQ_OK) return s;

  svdq_layer* h = new (std::nothrow) svdq_layer();
  if (!h) return fail(SVDQ_ERR_OOM, "host allocation failed");
  std::string err;
  s = pack_on_host(p, &h->host, &err);
  if (s != SVDQ_OK) {
    delete h;
    return fail(s, err);
  }
  DeviceGuard guard(p->device);
  cudaStream_t stream = static_cast<cudaStream_t>(p->stream);
  h->device = p->device;
  cudaDeviceGetAttribute(&h->sm_count, cudaDevAttrMultiProcessorCount, p->device);
  const int64_t N = p->N, K = p->K;
  const HostPack& hp = h->host;
  h->inv_six = 1.0f / (6.0f * hp.s_gX);
  h->inv_alpha = 1.0f / hp.alpha;
  std::vector<float> qtab(256);
  act_quant_tables(hp.s_gX, qtab.data(), qtab.data() + 128);

  // ---- device layouts on the host
  const int64_t KG = scale_groups(K);
  const int64_t Npad = round_up(N, 256);
  // kernel 2's weight blocks: per 256-row pair tile, 256-wide K step and 128-row half one
  // contiguous block, so a CTA takes a stage's weights with one bulk copy.
  //  - codes: row r of the half, 16-byte chunk c of the step at r * 128 + 16 (c ^ (r % 8)), the
  //    128-byte swizzle the MMA's shared-memory descriptor reads;
  //  - then the pair tile's 4 KB scale block of the step, the same in both halves: for each of the
  //    step's four 64-column groups, the two halves' 512-byte tiles side by side (row r of a half
  //    at 16 (r % 32) + 4 ((r % 128) / 32), group element j % 4).
  const int64_t n_k = KG / 4;
  std::vector<uint8_t> wt(size_t(Npad / 128) * n_k * kK2WeightBlock, 0);
  auto block = [&](int64_t n, int64_t kq) {
    return wt.data() + (((n / 256) * n_k + kq) * 2 + (n / 128) % 2) * kK2WeightBlock;
  };
  for (int64_t n = 0; n < N; ++n) {
    const int64_t r = n % 128;
    for (int64_t kb = 0; kb < K / 2; kb += 16) {
      const int64_t c = (kb % 128) / 16;
      std::memcpy(block(n, kb / 128) + r * 128 + 16 * (c ^ (r % 8)), hp.R_codes.data() + n * (K / 2) + kb, 16);
    }
    for (int64_t j = 0; j < K / 16; ++j) {
      const int64_t g = j / 4, kq = g / 4, kk = g % 4, h = (n / 128) % 2;
      const int64_t at = 128 * 128 + kk * 1024 + h * 512 + (n % 32) * 16 + ((n % 128) / 32) * 4 + (j % 4);
      block(n, kq)[at] = hp.R_scales[n * (K / 16) + j];   // this half's copy of the block
      block(n ^ 128, kq)[at] = hp.R_scales[n * (K / 16) + j];   // the other half's copy
    }
  }
  // ---- upload
  auto up = [&](void** dst, const void* src, size_t bytes) -> cudaError_t {
    cudaError_t ee;
    *dst = dalloc(bytes, &ee);
    if (ee != cudaSuccess) return ee;
    if (bytes) ee = cudaMemcpyAsync(*dst, src, bytes, cudaMemcpyHostToDevice, stream);
    return ee;
  };
  e = up(reinterpret_cast<void**>(&h->d_wt), wt.data(), wt.size());
  if (e == cudaSuccess) e = up(reinterpret_cast<void**>(&h->d_inv_lambda), hp.inv_lambda.data(), K * 4);
  if (e == cudaSuccess) e = up(reinterpret_cast<void**>(&h->d_qtab), qtab.data(), qtab.size() * 4);
  if (e == cudaSuccess) e = up(reinterpret_cast<void**>(&h->d_bias), hp.bias.data(), N * 2);
  if (e == cudaSuccess) {
    h->d_err = static_cast<int*>(dalloc(sizeof(int), &e));
    if (e == cudaSuccess) e = cudaMemsetAsync(h->d_err, 0, sizeof(int), stream);
  }
  if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
  if (e != cudaSuccess) {
    free_layer(h);
    delete h;
    return e == cudaErrorMemoryAllocation ? fail(SVDQ_ERR_OOM, "device allocation failed")
                                          : cuda_fail(e, "uploading the packed layer");
  }
  s = upload_low_rank(h, stream);
  if (s != SVDQ_OK) {
    free_layer(h);
    delete h;
    return s;
  }
  if (p->M_max > 0) {
    s = svdq_reserve(h, p->M_max, 0);
    if (s != SVDQ_OK) {
      free_layer(h);
      delete h;
      return s;
    }
  }
  *out = h;
  return SVDQ_OK;
}

svdq_status_t svdq_destroy(svdq_handle_t h) {
  if (!h) return SVDQ_OK;
  DeviceGuard guard(h->device);
  cudaDeviceSynchronize();
  free_layer(h);
  delete h;
  return SVDQ_OK;
}

svdq_status_t svdq_get_info(svdq_handle_t h, svdq_info_t* info) {
  if (!h || !info) return fail(SVDQ_ERR_INVALID_ARG, "null argument");
  info->N = h->host.N;
  info->K = h->host.K;
  info->rank = h->host.rank;
  info->lora_rank = h->r_lora;
  info->r_pad = h->r_pad;
  info->M_max = h->ws_M;
  info->s_gW = h->host.s_gW;
  info->s_gX = h->host.s_gX;
  info->alpha = h->host.alpha;
  info->device = h->device;
  info->sm_count = h->sm_count;
  return SVDQ_OK;
}

svdq_status_t svdq_export(svdq_handle_t h, svdq_packed_host_t* out) {
  if (!h || !out) return fail(SVDQ_ERR_INVALID_ARG, "null argument");
  const HostPack& hp = h->host;
  const int64_t N = hp.N, K = hp.K, r = hp.rank;
  if (out->lambda) std::memcpy(out->lambda, hp.lambda.data(), sizeof(float) * K);
  if (out->inv_lambda) std::memcpy(out->inv_lambda, hp.inv_lambda.data(), sizeof(float) * K);
  if (out->L1_bf16 && r) std::memcpy(out->L1_bf16, hp.L1.data(), sizeof(uint16_t) * K * r);
  if (out->L2_bf16 && r) std::memcpy(out->L2_bf16, hp.L2.data(), sizeof(uint16_t) * r * N);
  if (out->R_codes) std::memcpy(out->R_codes, hp.R_codes.data(), hp.R_codes.size());
  if (out->R_scales) std::memcpy(out->R_scales, hp.R_scales.data(), hp.R_scales.size());
  if (out->bias_bf16) std::memcpy(out->bias_bf16, hp.bias.data(), sizeof(uint16_t) * N);
  out->s_gW = hp.s_gW;
  out->s_gX = hp.s_gX;
  out->alpha = hp.alpha;
  return SVDQ_OK;
}

svdq_status_t svdq_workspace_size(svdq_handle_t h, int64_t M, int32_t host_staging, size_t* bytes) {
  if (!h || !bytes || M < 0) return fail(SVDQ_ERR_INVALID_ARG, "null argument or negative M");
  *bytes = ws_layout(h, M, staging_slots(host_staging)).total;
  return SVDQ_OK;
}

svdq_status_t svdq_attach_lora(svdq_handle_t h, const uint16_t* A_bf16, const uint16_t* B_bf16, int64_t r_lora,
                               float scale, void* stream) {
  if (!h || r_lora < 0) return fail(SVDQ_ERR_INVALID_ARG, "null handle or negative LoRA rank");
  if (r_lora > 0 && (!A_bf16 || !B_bf16)) return fail(SVDQ_ERR_INVALID_ARG, "null LoRA factor");
  if (!std::isfinite(scale)) return fail(SVDQ_ERR_INVALID_ARG, "LoRA scale must be finite");
  const int64_t K = h->host.K, N = h->host.N, rk = h->host.rank + r_lora;
  if (r_lora % 16 != 0 || rk > 128)
    return fail(SVDQ_ERR_UNSUPPORTED_SHAPE, "LoRA rank must be a multiple of 16 with rank + LoRA rank <= 128");
  DeviceGuard guard(h->device);
  cudaError_t e = cudaDeviceSynchronize();                 // no kernel still reads the old buffers
  if (e != cudaSuccess) return cuda_fail(e, "device synchronisation");
  std::vector<uint16_t> A(size_t(K) * r_lora), B(B_bf16 ? B_bf16 : nullptr, B_bf16 ? B_bf16 + size_t(r_lora) * N : nullptr);
  for (size_t i = 0; i < A.size(); ++i) A[i] = f64_to_bf16(double(scale) * double(bf16_to_f32(A_bf16[i])));
  // the workspace layout depends on the kernel rank: a lent workspace must already be big enough
  const int64_t old_rl = h->r_lora, old_pad = h->r_pad;
  h->r_lora = r_lora;
  h->r_pad = rank_pad(rk);
  const size_t need = h->ws ? ws_layout(h, h->ws_M, h->ws_staging).total : 0;
  h->r_lora = old_rl;
  h->r_pad = old_pad;
  if (h->ws && !h->ws_owned && h->ws_bytes < need)
    return fail(SVDQ_ERR_WORKSPACE, "the lent workspace is too small for the rank with LoRA (svdq_workspace_size)");
  std::vector<uint16_t> oldA, oldB;
  oldA.swap(h->lora_A);
  oldB.swap(h->lora_B);
  h->lora_A.swap(A);
  h->lora_B.swap(B);
  h->r_lora = r_lora;
  svdq_status_t st = upload_low_rank(h, static_cast<cudaStream_t>(stream));
  if (st != SVDQ_OK) {                                      // the device buffers are unchanged
    h->lora_A.swap(oldA);
    h->lora_B.swap(oldB);
    h->r_lora = old_rl;
    return st;
  }
  if (h->ws && h->ws_owned && h->ws_bytes < need) return svdq_reserve(h, h->ws_M, h->ws_staging);
  return SVDQ_OK;
}

svdq_status_t svdq_reserve(svdq_handle_t h, int64_t M_max, int32_t host_staging) {
  if (!h || M_max < 0) return fail(SVDQ_ERR_INVALID_ARG, "null handle or negative M_max");
  DeviceGuard guard(h->device);
  const size_t bytes = ws_layout(h, M_max, staging_slots(host_staging)).total;
  cudaError_t e;
  void* p = dalloc(bytes, &e);
  if (e != cudaSuccess) return fail(SVDQ_ERR_OOM, "workspace allocation failed");
  return attach_workspace(h, p, bytes, M_max, staging_slots(host_staging), true, nullptr);
}

svdq_status_t svdq_set_workspace(svdq_handle_t h, void* dev_ptr, size_t bytes, int64_t M_max, int32_t host_staging) {
  if (!h || M_max < 0) return fail(SVDQ_ERR_INVALID_ARG, "null handle or negative M_max");
  DeviceGuard guard(h->device);
  if (dev_ptr == nullptr) return attach_workspace(h, nullptr, 0, 0, 0, false, nullptr);
  if (reinterpret_cast<uintptr_t>(dev_ptr) & 255u) return fail(SVDQ_ERR_INVALID_ARG, "workspace must be 256-byte aligned");
  if (bytes < ws_layout(h, M_max, staging_slots(host_staging)).total)
    return fail(SVDQ_ERR_WORKSPACE, "workspace smaller than svdq_workspace_size");
  return attach_workspace(h, dev_ptr, bytes, M_max, staging_slots(host_staging), false, nullptr);
}

svdq_status_t svdq_quantize_act(svdq_handle_t h, const void* X, int64_t M, void* x_codes, void* x_scales, void* T,
                                void* stream) {
  if (!h || M < 0) return fail(SVDQ_ERR_INVALID_ARG, "null handle or negative M");
  if (M == 0) return SVDQ_OK;
  if (!X || !x_codes || !x_scales || (h->rank_k() > 0 && !T)) return fail(SVDQ_ERR_INVALID_ARG, "null buffer");
  if (!aligned16(X) || !aligned16(x_codes) || !aligned16(x_scales) || (T && !aligned16(T)))
    return fail(SVDQ_ERR_INVALID_ARG, "buffers must be 16-byte aligned");
  if (!h->ws || h->ws_M < M) return fail(SVDQ_ERR_WORKSPACE, "no workspace for this M (svdq_reserve)");
  DeviceGuard guard(h->device);
  return launch_k1(h, X, M, x_codes, x_scales, T, static_cast<cudaStream_t>(stream));
}

svdq_status_t svdq_gemm_quantized(svdq_handle_t h, const void* x_codes, const void* x_scales, const void* T, void* Y,
                                  int64_t M, void* stream) {
  if (!h || M < 0) return fail(SVDQ_ERR_INVALID_ARG, "null handle or negative M");
  if (M == 0) return SVDQ_OK;
  if (!x_codes || !x_scales || !Y || (h->rank_k() > 0 && !T)) return fail(SVDQ_ERR_INVALID_ARG, "null buffer");
  if (!aligned16(x_codes) || !aligned16(x_scales) || !aligned16(Y) || (T && !aligned16(T)))
    return fail(SVDQ_ERR_INVALID_ARG, "buffers must be 16-byte aligned");
  DeviceGuard guard(h->device);
  return launch_k2(h, x_codes, x_scales, T, Y, M, static_cast<cudaStream_t>(stream));
}

svdq_status_t svdq_linear_forward(svdq_handle_t h, const void* X, void* Y, int64_t M, void* stream) {
  if (!h || M < 0) return fail(SVDQ_ERR_INVALID_ARG, "null handle or negative M");
  if (M == 0) return SVDQ_OK;
  if (!X || !Y) return fail(SVDQ_ERR_INVALID_ARG, "null buffer");
  if (!aligned16(X) || !aligned16(Y)) return fail(SVDQ_ERR_INVALID_ARG, "buffers must be 16-byte aligned");
  if (!h->ws || h->ws_M < M) return fail(SVDQ_ERR_WORKSPACE, "no workspace for this M (svdq_reserve)");
  const size_t xb = size_t(M) * h->host.K * 2, yb = size_t(M) * h->host.N * 2;
  if (overlaps(X, xb, Y, yb)) return fail(SVDQ_ERR_INVALID_ARG, "X and Y must not overlap");
  const WsLayout w = ws_layout(h, h->ws_M, h->ws_staging);
  // the kernels' scratch part of the workspace (the host staging slots after it are X and Y of
  // the host-buffer entry points)
  if (overlaps(X, xb, h->ws, w.Xs[0]) || overlaps(Y, yb, h->ws, w.Xs[0]))
    return fail(SVDQ_ERR_INVALID_ARG, "X and Y must not overlap the workspace");
  DeviceGuard guard(h->device);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  void* codes = h->ws + w.codes;
  void* scales = h->ws + w.scales;
  void* T = h->rank_k() ? h->ws + w.T : nullptr;
  svdq_status_t st = launch_k1(h, X, M, codes, scales, T, s);
  if (st != SVDQ_OK) return st;
  return launch_k2(h, codes, scales, T, Y, M, s);
}

svdq_status_t svdq_linear_forward_host(svdq_handle_t h, const uint16_t* X_host, uint16_t* Y_host, int64_t M,
                                       void* stream) {
  if (!h || M < 0) return fail(SVDQ_ERR_INVALID_ARG, "null handle or negative M");
  if (M == 0) return SVDQ_OK;
  if (!X_host || !Y_host) return fail(SVDQ_ERR_INVALID_ARG, "null buffer");
  if (!h->ws || !h->ws_staging || h->ws_M < M)
    return fail(SVDQ_ERR_WORKSPACE, "needs a workspace reserved with host staging for this M");
  DeviceGuard guard(h->device);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const WsLayout w = ws_layout(h, h->ws_M, h->ws_staging);
  void* Xd = h->ws + w.Xs[0];
  void* Yd = h->ws + w.Ys[0];
  cudaError_t e = cudaMemcpyAsync(Xd, X_host, size_t(M) * h->host.K * 2, cudaMemcpyHostToDevice, s);
  if (e != cudaSuccess) return cuda_fail(e, "copying X to the device");
  svdq_status_t st = svdq_linear_forward(h, Xd, Yd, M, stream);
  if (st != SVDQ_OK) return st;
  e = cudaMemcpyAsync(Y_host, Yd, size_t(M) * h->host.N * 2, cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return cuda_fail(e, "copying Y to the host");
  return SVDQ_OK;
}

svdq_status_t svdq_linear_forward_host_batch(svdq_handle_t h, const uint16_t* const* X_host, uint16_t* const* Y_host,
                                             int32_t B, int64_t M, void* stream) {
  if (!h || M < 0 || B < 0) return fail(SVDQ_ERR_INVALID_ARG, "null handle, negative M or negative batch count");
  if (M == 0 || B == 0) return SVDQ_OK;
  if (!X_host || !Y_host) return fail(SVDQ_ERR_INVALID_ARG, "null buffer list");
  for (int32_t b = 0; b < B; ++b)
    if (!X_host[b] || !Y_host[b]) return fail(SVDQ_ERR_INVALID_ARG, "null buffer");
  if (!h->ws || h->ws_staging < 2 || h->ws_M < M)
    return fail(SVDQ_ERR_WORKSPACE, "needs a workspace reserved with two host staging slots for this M");
  DeviceGuard guard(h->device);
  cudaError_t e = cudaSuccess;
  if (!h->pipe_in) {
    if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&h->pipe_in, cudaStreamNonBlocking);
    if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&h->pipe_out, cudaStreamNonBlocking);
    for (int i = 0; i < 2 && e == cudaSuccess; ++i) {
      e = cudaEventCreateWithFlags(&h->ev_in[i], cudaEventDisableTiming);
      if (e == cudaSuccess) e = cudaEventCreateWithFlags(&h->ev_comp[i], cudaEventDisableTiming);
      if (e == cudaSuccess) e = cudaEventCreateWithFlags(&h->ev_out[i], cudaEventDisableTiming);
    }
    if (e != cudaSuccess) return cuda_fail(e, "creating the copy streams and events");
  }
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const WsLayout w = ws_layout(h, h->ws_M, h->ws_staging);
  const size_t xb = size_t(M) * h->host.K * 2, yb = size_t(M) * h->host.N * 2;
  // everything already queued on the caller's stream comes first
  e = cudaEventRecord(h->ev_comp[0], s);
  if (e == cudaSuccess) e = cudaEventRecord(h->ev_comp[1], s);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(h->pipe_in, h->ev_comp[0], 0);
  if (e == cudaSuccess) e = cudaEventRecord(h->ev_out[0], s);
  if (e == cudaSuccess) e = cudaEventRecord(h->ev_out[1], s);
  for (int32_t b = 0; b < B && e == cudaSuccess; ++b) {
    const int k = b & 1;
    void* Xd = h->ws + w.Xs[k];
    void* Yd = h->ws + w.Ys[k];
    // upload of step b once step b - 2's kernels no longer read the slot's X
    e = cudaStreamWaitEvent(h->pipe_in, h->ev_comp[k], 0);
    if (e == cudaSuccess) e = cudaMemcpyAsync(Xd, X_host[b], xb, cudaMemcpyHostToDevice, h->pipe_in);
    if (e == cudaSuccess) e = cudaEventRecord(h->ev_in[k], h->pipe_in);
    // kernels of step b once its X is in and step b - 2's Y has left the slot
    if (e == cudaSuccess) e = cudaStreamWaitEvent(s, h->ev_in[k], 0);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(s, h->ev_out[k], 0);
    if (e != cudaSuccess) break;
    svdq_status_t st = svdq_linear_forward(h, Xd, Yd, M, stream);
    if (st != SVDQ_OK) {
      cudaStreamSynchronize(h->pipe_in);
      cudaStreamSynchronize(h->pipe_out);
      return st;
    }
    e = cudaEventRecord(h->ev_comp[k], s);
    // download of step b
    if (e == cudaSuccess) e = cudaStreamWaitEvent(h->pipe_out, h->ev_comp[k], 0);
    if (e == cudaSuccess) e = cudaMemcpyAsync(Y_host[b], Yd, yb, cudaMemcpyDeviceToHost, h->pipe_out);
    if (e == cudaSuccess) e = cudaEventRecord(h->ev_out[k], h->pipe_out);
  }
  const cudaError_t e_in = cudaStreamSynchronize(h->pipe_in);
  const cudaError_t e_out = cudaStreamSynchronize(h->pipe_out);
  const cudaError_t e_s = cudaStreamSynchronize(s);
  if (e == cudaSuccess) e = e_in != cudaSuccess ? e_in : (e_out != cudaSuccess ? e_out : e_s);
  if (e != cudaSuccess) return cuda_fail(e, "pipelined host forward");
  return SVDQ_OK;
}

svdq_status_t svdq_set_wait_limit(svdq_handle_t h, uint64_t wait_ns, int32_t stall_kernel) {
  if (!h) return fail(SVDQ_ERR_INVALID_ARG, "null handle");
  if (stall_kernel < 0 || stall_kernel > 2) return fail(SVDQ_ERR_INVALID_ARG, "stall_kernel must be 0, 1 or 2");
  h->wait_ns = wait_ns ? wait_ns : kDefaultWaitNs;
  h->stall = stall_kernel;
  return SVDQ_OK;
}

svdq_status_t svdq_check_error(svdq_handle_t h) {
  if (!h) return fail(SVDQ_ERR_INVALID_ARG, "null handle");
  DeviceGuard guard(h->device);
  cudaError_t e = cudaDeviceSynchronize();
  if (e != cudaSuccess) return cuda_fail(e, "device synchronisation");
  int v = 0;
  e = cudaMemcpy(&v, h->d_err, sizeof(int), cudaMemcpyDeviceToHost);
  if (e == cudaSuccess) e = cudaMemset(h->d_err, 0, sizeof(int));
  if (e != cudaSuccess) return cuda_fail(e, "reading the device error word");
  if (v) return fail(SVDQ_ERR_TIMEOUT, "a kernel gave up a bounded wait (error word " + std::to_string(v) + ")");
  return SVDQ_OK;
}

}  // extern "C"

// ------------------------------------------------------------------ forward without allocation
// Some callers cannot allocate device memory at the point where they run a layer: code running
// under a framework's memory pool or budget (where a library-owned cudaMalloc would bypass the
// pool and may not fit), or latency-critical loops where cudaMalloc's implicit device
// synchronisation is not acceptable.  svdq_linear_forward_noalloc serves them: its scratch
// (quantised activations, T and kernel 1's split-K partial sums and arrival words) lives in one
// statically sized device array that the library holds on every device it is loaded on, so the
// call itself allocates nothing.  Nothing in it needs clearing between calls: kernel 2 reads
// only bytes kernel 1 wrote earlier in the same call, and the arrival words carry a per-launch
// epoch that makes stale contents (another layer's, or an aborted call's) restart the count.
namespace {

constexpr size_t kStaticScratchBytes = size_t(32) << 20;   // 32 MiB per device
static __device__ __align__(256) unsigned char g_static_scratch[kStaticScratchBytes];

std::mutex g_static_mu;
void* g_static_ptr[64] = {nullptr};

// Device address of g_static_scratch on the current device.  In host code the array's name is
// only a host-side stand-in, so the address comes from cudaGetSymbolAddress with the device
// current.  Outside stream capture it is looked up on every call (cheap), so an address made
// stale by a device reset is never used; inside a capture the address cached by the last call
// outside one is used, since the capture must not be disturbed by a first-time module load.
svdq_status_t static_scratch(int device, cudaStream_t stream, unsigned char** out) {
  if (device < 0 || device >= 64) return fail(SVDQ_ERR_INVALID_ARG, "device ordinal out of range");
  cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(stream, &cap) != cudaSuccess) {
    cudaGetLastError();                       // not sticky: clear it and take the cached address
    cap = cudaStreamCaptureStatusActive;
  }
  std::lock_guard<std::mutex> lock(g_static_mu);
  if (cap == cudaStreamCaptureStatusNone) {
    void* p = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&p, g_static_scratch);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress of the static scratch");
    g_static_ptr[device] = p;
  } else if (!g_static_ptr[device]) {
    return fail(SVDQ_ERR_INVALID_ARG,
                "the first svdq_linear_forward_noalloc call on a device must come before any stream capture");
  }
  *out = static_cast<unsigned char*>(g_static_ptr[device]);
  return SVDQ_OK;
}

}  // namespace

extern "C" svdq_status_t svdq_linear_forward_noalloc(svdq_handle_t h, const void* X, void* Y, int64_t M,
                                                     void* stream) {
  if (!h || M < 0) return fail(SVDQ_ERR_INVALID_ARG, "null handle or negative M");
  if (M == 0) return SVDQ_OK;
  if (!X || !Y) return fail(SVDQ_ERR_INVALID_ARG, "null buffer");
  if (!aligned16(X) || !aligned16(Y)) return fail(SVDQ_ERR_INVALID_ARG, "buffers must be 16-byte aligned");
  const WsLayout w = ws_layout(h, M, 0);
  if (w.total > kStaticScratchBytes)
    return fail(SVDQ_ERR_WORKSPACE, "M = " + std::to_string(M) + " needs " + std::to_string(w.total) +
                                        " bytes of scratch; the static scratch holds " +
                                        std::to_string(kStaticScratchBytes) + " bytes");
  const size_t xb = size_t(M) * h->host.K * 2, yb = size_t(M) * h->host.N * 2;
  if (overlaps(X, xb, Y, yb)) return fail(SVDQ_ERR_INVALID_ARG, "X and Y must not overlap");
  DeviceGuard guard(h->device);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  unsigned char* ws = nullptr;
  svdq_status_t st = static_scratch(h->device, s, &ws);
  if (st != SVDQ_OK) return st;
  if (overlaps(X, xb, ws, kStaticScratchBytes) || overlaps(Y, yb, ws, kStaticScratchBytes))
    return fail(SVDQ_ERR_INVALID_ARG, "X and Y must not overlap the static scratch");
  K1Args a{};
  k1_scratch(&a, ws, w);
  a.X = static_cast<const uint16_t*>(X);
  a.LI = h->d_LI;
  a.x_codes = ws + w.codes;
  a.x_scales = ws + w.scales;
  a.T = h->rank_k() ? reinterpret_cast<uint16_t*>(ws + w.T) : nullptr;
  a.M = M;
  a.K = h->host.K;
  a.rank = int(h->rank_k());
  a.r_pad = int(h->r_pad);
  a.s_gX = h->host.s_gX;
  a.inv_six = h->inv_six;
  a.inv_alpha = h->inv_alpha;
  a.qtab = h->d_qtab;
  a.err = h->d_err;
  a.wait_ns = h->wait_ns;
  a.stall = h->stall == 1;
  std::string err;
  const int e1 = k1_launch(a, k1_plan(M, a.K, a.rank, h->sm_count), s, &err);
  if (e1 == -1) return fail(SVDQ_ERR_CUDA, err);
  if (e1 != 0) return cuda_fail(cudaError_t(e1), "kernel 1 launch");
  return launch_k2(h, a.x_codes, a.x_scales, a.T, Y, M, s);
}

// ------------------------------------------------------------------ MLP pair (fused epilogue)
// The up layer's kernel 2 writes the down layer's kernel-1 outputs for G = bf16(GELU(Y_up))
// (codes, scales and partial sums of G L1'), so Y_up is never written to memory and the down
// layer's kernel 1 does not run.  The pair owns the down layer's L1' in warp-MMA fragment order
// and the partial sums; the activations pass through the two layers' workspaces.
struct svdq_mlp {
  svdq_layer* up = nullptr;
  svdq_layer* down = nullptr;
  int device = 0;
  int rd = 0;                       // the down layer's kernel rank
  uint64_t down_gen = 0;            // its low-rank upload the fragments were built from
  int pairs = 0;                    // CTA pairs of the fused kernel on this device
  int64_t M_max = 0;
  uint16_t* d_l1f = nullptr;        // N_up x rd bf16 in fragment order
  float* d_part = nullptr;          // partial sums
  size_t part_bytes = 0;
};

namespace {

// Bytes of partial sums the fused epilogue writes for M rows.
size_t mlp_part_bytes(const svdq_mlp* p, int64_t M) {
  if (p->rd == 0 || M == 0) return 0;
  const int64_t N = p->up->host.N;
  const int U = k2_fused_unit_len(M, N, p->pairs);
  return size_t(k2_fused_partials(M, N, U)) * size_t(M) * size_t(p->rd) * 4;
}

void free_mlp(svdq_mlp* p) {
  cudaFree(p->d_l1f);
  cudaFree(p->d_part);
}

// Kernel 1 of the up layer on X, then its kernel 2 with the fused epilogue writing the down
// layer's codes, scales and T (through the partial sums and their reduction).
svdq_status_t mlp_up(svdq_mlp* p, const void* X, int64_t M, void* codes, void* scales, void* T, cudaStream_t stream) {
  svdq_layer* up = p->up;
  svdq_layer* dn = p->down;
  const WsLayout w = ws_layout(up, up->ws_M, up->ws_staging);
  void* ucodes = up->ws + w.codes;
  void* uscales = up->ws + w.scales;
  void* uT = up->rank_k() ? up->ws + w.T : nullptr;
  svdq_status_t st = launch_k1(up, X, M, ucodes, uscales, uT, stream);
  if (st != SVDQ_OK) return st;
  const int64_t K = up->host.K, N = up->host.N;
  K2Maps maps = up->maps;
  std::string err;
  if (!encode_map_2d(maps.A, 1, ucodes, K / 2, M, K / 2, 128, 128, 1, &err) ||
      !encode_map_2d(maps.SFA, 1, uscales, 256, svdq_scales_bytes(M, K) / 256, 256, 256, 8, 0, &err))
    return fail(SVDQ_ERR_CUDA, err);
  if (up->rank_k() > 0 && !encode_map_2d(maps.T, 2, uT, up->r_pad, M, up->r_pad * 2, 64, 128, 1, &err))
    return fail(SVDQ_ERR_CUDA, err);
  K2Args a{};
  a.bias = up->d_bias;
  a.wt = up->d_wt;
  a.err = up->d_err;
  a.M = M;
  a.N = N;
  a.K = K;
  a.rank = int(up->rank_k());
  a.alpha = up->host.alpha;
  a.wait_ns = up->wait_ns;
  a.stall = up->stall == 2;
  a.unit_len = k2_fused_unit_len(M, N, p->pairs);
  a.fuse.inv_lambda = dn->d_inv_lambda;
  a.fuse.qtab = dn->d_qtab;
  a.fuse.inv_six = dn->inv_six;
  a.fuse.x_codes = static_cast<uint8_t*>(codes);
  a.fuse.x_scales = static_cast<uint8_t*>(scales);
  a.fuse.l1f = p->d_l1f;
  a.fuse.part = p->d_part;
  a.fuse.rd = p->rd;
  int e = k2_fused_launch(maps, a, up->sm_count, stream);
  if (e != 0) return cuda_fail(cudaError_t(e), "fused kernel 2 launch");
  if (p->rd > 0) {
    e = k2_t_reduce_launch(p->d_part, k2_fused_partials(M, N, a.unit_len), M, p->rd, int(dn->r_pad), dn->inv_alpha,
                           static_cast<uint16_t*>(T), stream);
    if (e != 0) return cuda_fail(cudaError_t(e), "partial-sum reduction launch");
  }
  return SVDQ_OK;
}

svdq_status_t mlp_check(const svdq_mlp* p, int64_t M) {
  if (p->down->low_rank_gen != p->down_gen)
    return fail(SVDQ_ERR_INVALID_ARG, "the down layer's low-rank factors changed after svdq_mlp_create");
  if (p->up->host.N != p->down->host.K) return fail(SVDQ_ERR_INVALID_ARG, "layer shapes changed");
  if (M > p->M_max) return fail(SVDQ_ERR_WORKSPACE, "M is larger than the pair's M_max");
  if (!p->up->ws || p->up->ws_M < M) return fail(SVDQ_ERR_WORKSPACE, "no up-layer workspace for this M (svdq_reserve)");
  return SVDQ_OK;
}

}  // namespace

extern "C" {

svdq_status_t svdq_mlp_create(svdq_handle_t up, svdq_handle_t down, int64_t M_max, svdq_mlp_t* out) {
  if (!up || !down || !out || M_max < 0) return fail(SVDQ_ERR_INVALID_ARG, "null argument or negative M_max");
  if (up == down) return fail(SVDQ_ERR_INVALID_ARG, "the up and down layers must be different handles");
  if (up->device != down->device) return fail(SVDQ_ERR_INVALID_ARG, "the layers live on different devices");
  if (up->host.N != down->host.K)
    return fail(SVDQ_ERR_INVALID_ARG, "the up layer's N must equal the down layer's K");
  const int64_t rd = down->rank_k();
  if (rd > kFuseMaxRank)
    return fail(SVDQ_ERR_UNSUPPORTED_SHAPE, "the fused epilogue supports a down-layer rank (with LoRA) of at most 64");
  svdq_mlp* p = new (std::nothrow) svdq_mlp();
  if (!p) return fail(SVDQ_ERR_OOM, "host allocation failed");
  DeviceGuard guard(up->device);
  p->up = up;
  p->down = down;
  p->device = up->device;
  p->rd = int(rd);
  p->down_gen = down->low_rank_gen;
  p->pairs = k2_fused_pairs(up->sm_count);
  p->M_max = M_max;
  const int64_t N = up->host.N;
  // the largest partial-sum buffer any M <= M_max needs (the schedule depends on M's row blocks)
  size_t part = 0;
  for (int64_t mb = 1; mb <= ceil_div(M_max, 256); ++mb)
    part = std::max(part, mlp_part_bytes(p, std::min<int64_t>(mb * 256, M_max)));
  cudaError_t e = cudaSuccess;
  if (rd > 0) {
    std::vector<uint16_t> l1(size_t(N) * rd), frag(size_t(N) * rd);
    for (int64_t k = 0; k < N; ++k)
      for (int64_t j = 0; j < rd; ++j) l1[k * rd + j] = l1_prime(down, k, j);
    k2_l1_fragments(l1.data(), N, int(rd), frag.data());
    p->d_l1f = static_cast<uint16_t*>(dalloc(frag.size() * 2, &e));
    if (e == cudaSuccess) e = cudaMemcpy(p->d_l1f, frag.data(), frag.size() * 2, cudaMemcpyHostToDevice);
    if (e == cudaSuccess && part) p->d_part = static_cast<float*>(dalloc(part, &e));
  }
  if (e != cudaSuccess) {
    free_mlp(p);
    delete p;
    return e == cudaErrorMemoryAllocation ? fail(SVDQ_ERR_OOM, "device allocation failed")
                                          : cuda_fail(e, "uploading the pair's fragments");
  }
  p->part_bytes = part;
  *out = p;
  return SVDQ_OK;
}

svdq_status_t svdq_mlp_destroy(svdq_mlp_t p) {
  if (!p) return SVDQ_OK;
  DeviceGuard guard(p->device);
  cudaDeviceSynchronize();
  free_mlp(p);
  delete p;
  return SVDQ_OK;
}

svdq_status_t svdq_mlp_up_quantize(svdq_mlp_t p, const void* X, int64_t M, void* x_codes, void* x_scales, void* T,
                                   void* stream) {
  if (!p || M < 0) return fail(SVDQ_ERR_INVALID_ARG, "null pair or negative M");
  if (M == 0) return SVDQ_OK;
  if (!X || !x_codes || !x_scales || (p->rd > 0 && !T)) return fail(SVDQ_ERR_INVALID_ARG, "null buffer");
  if (!aligned16(X) || !aligned16(x_codes) || !aligned16(x_scales) || (T && !aligned16(T)))
    return fail(SVDQ_ERR_INVALID_ARG, "buffers must be 16-byte aligned");
  svdq_status_t st = mlp_check(p, M);
  if (st != SVDQ_OK) return st;
  const int64_t K = p->up->host.K, N = p->up->host.N;
  const size_t xb = size_t(M) * K * 2, cb = size_t(M) * N / 2, sb = size_t(svdq_scales_bytes(M, N)),
               tb = size_t(M) * p->down->r_pad * 2;
  if (overlaps(X, xb, x_codes, cb) || overlaps(X, xb, x_scales, sb) || overlaps(x_codes, cb, x_scales, sb) ||
      (T && (overlaps(T, tb, X, xb) || overlaps(T, tb, x_codes, cb) || overlaps(T, tb, x_scales, sb))))
    return fail(SVDQ_ERR_INVALID_ARG, "X and the outputs must not overlap");
  DeviceGuard guard(p->device);
  return mlp_up(p, X, M, x_codes, x_scales, T, static_cast<cudaStream_t>(stream));
}

svdq_status_t svdq_mlp_forward(svdq_mlp_t p, const void* X, void* Y, int64_t M, void* stream) {
  if (!p || M < 0) return fail(SVDQ_ERR_INVALID_ARG, "null pair or negative M");
  if (M == 0) return SVDQ_OK;
  if (!X || !Y) return fail(SVDQ_ERR_INVALID_ARG, "null buffer");
  if (!aligned16(X) || !aligned16(Y)) return fail(SVDQ_ERR_INVALID_ARG, "buffers must be 16-byte aligned");
  svdq_status_t st = mlp_check(p, M);
  if (st != SVDQ_OK) return st;
  svdq_layer* dn = p->down;
  if (!dn->ws || dn->ws_M < M) return fail(SVDQ_ERR_WORKSPACE, "no down-layer workspace for this M (svdq_reserve)");
  const size_t xb = size_t(M) * p->up->host.K * 2, yb = size_t(M) * dn->host.N * 2;
  if (overlaps(X, xb, Y, yb)) return fail(SVDQ_ERR_INVALID_ARG, "X and Y must not overlap");
  const WsLayout wu = ws_layout(p->up, p->up->ws_M, p->up->ws_staging);
  const WsLayout wd = ws_layout(dn, dn->ws_M, dn->ws_staging);
  if (overlaps(X, xb, p->up->ws, wu.Xs[0]) || overlaps(Y, yb, p->up->ws, wu.Xs[0]) ||
      overlaps(X, xb, dn->ws, wd.Xs[0]) || overlaps(Y, yb, dn->ws, wd.Xs[0]))
    return fail(SVDQ_ERR_INVALID_ARG, "X and Y must not overlap the layers' workspaces");
  DeviceGuard guard(p->device);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  void* codes = dn->ws + wd.codes;
  void* scales = dn->ws + wd.scales;
  void* T = p->rd ? dn->ws + wd.T : nullptr;
  st = mlp_up(p, X, M, codes, scales, T, s);
  if (st != SVDQ_OK) return st;
  return launch_k2(dn, codes, scales, T, Y, M, s);
}

svdq_status_t svdq_mlp_check_error(svdq_mlp_t p) {
  if (!p) return fail(SVDQ_ERR_INVALID_ARG, "null pair");
  const svdq_status_t a = svdq_check_error(p->up);
  const svdq_status_t b = svdq_check_error(p->down);
  return a != SVDQ_OK ? a : b;
}

svdq_status_t svdq_gelu_bf16(const void* Y, void* G, int64_t n, void* stream) {
  if (n < 0 || (n > 0 && (!Y || !G))) return fail(SVDQ_ERR_INVALID_ARG, "null buffer or negative n");
  if (n % 8) return fail(SVDQ_ERR_INVALID_ARG, "n must be a multiple of 8");
  if (n == 0) return SVDQ_OK;
  if (!aligned16(Y) || !aligned16(G)) return fail(SVDQ_ERR_INVALID_ARG, "buffers must be 16-byte aligned");
  if (Y != G && overlaps(Y, size_t(n) * 2, G, size_t(n) * 2))
    return fail(SVDQ_ERR_INVALID_ARG, "Y and G must be the same buffer or not overlap");
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int e = gelu_launch(static_cast<const uint16_t*>(Y), static_cast<uint16_t*>(G), n, sms, stream);
  if (e != 0) return cuda_fail(cudaError_t(e), "GELU kernel launch");
  return SVDQ_OK;
}

}  // extern "C"

// ------------------------------------------------------------------ AWQ-style W4A16 layer
struct svdq_awq_layer {
  AwqHostPack host;
  int device = 0;
  int sm_count = 0;
  uint8_t* d_codes = nullptr;
  float* d_sz = nullptr;            // N x K/64 (scale, zero point) pairs, 16 bytes of padding
  float* d_inv_s = nullptr;
  uint16_t* d_bias = nullptr;
  int* d_err = nullptr;
};

namespace {

void free_awq(svdq_awq_layer* h) {
  cudaFree(h->d_codes);
  cudaFree(h->d_sz);
  cudaFree(h->d_inv_s);
  cudaFree(h->d_bias);
  cudaFree(h->d_err);
}

void copy_awq_out(const AwqHostPack& hp, svdq_awq_host_t* out) {
  const int64_t N = hp.N, K = hp.K, KG = K / 64;
  if (out->s) std::memcpy(out->s, hp.s.data(), size_t(K) * 4);
  if (out->inv_s) std::memcpy(out->inv_s, hp.inv_s.data(), size_t(K) * 4);
  if (out->codes) std::memcpy(out->codes, hp.codes.data(), hp.codes.size());
  if (out->scales) std::memcpy(out->scales, hp.scales.data(), size_t(N) * KG * 4);
  if (out->zeros) std::memcpy(out->zeros, hp.zeros.data(), size_t(N) * KG);
  if (out->bias_bf16) std::memcpy(out->bias_bf16, hp.bias.data(), size_t(N) * 2);
  out->alpha = hp.alpha;
}

}  // namespace

extern "C" {

svdq_status_t svdq_awq_pack_host(const svdq_awq_params_t* p, svdq_awq_host_t* out) {
  if (!p || !out) return fail(SVDQ_ERR_INVALID_ARG, "null argument");
  AwqHostPack hp;
  std::string err;
  const svdq_status_t s = awq_pack_host(p, &hp, &err);
  if (s != SVDQ_OK) return fail(s, err);
  copy_awq_out(hp, out);
  return SVDQ_OK;
}

svdq_status_t svdq_awq_pack(const svdq_awq_params_t* p, svdq_awq_handle_t* out) {
  if (!p || !out) return fail(SVDQ_ERR_INVALID_ARG, "null argument");
  int ndev = 0;
  if (cudaGetDeviceCount(&ndev) != cudaSuccess || p->device < 0 || p->device >= ndev)
    return fail(SVDQ_ERR_INVALID_ARG, "no such device");
  svdq_status_t s = check_arch(p->device);
  if (s != SVDQ_OK) return s;
  svdq_awq_layer* h = new (std::nothrow) svdq_awq_layer();
  if (!h) return fail(SVDQ_ERR_OOM, "host allocation failed");
  std::string err;
  s = awq_pack_host(p, &h->host, &err);
  if (s != SVDQ_OK) {
    delete h;
    return fail(s, err);
  }
  DeviceGuard guard(p->device);
  h->device = p->device;
  cudaDeviceGetAttribute(&h->sm_count, cudaDevAttrMultiProcessorCount, p->device);
  cudaStream_t stream = static_cast<cudaStream_t>(p->stream);
  const AwqHostPack& hp = h->host;
  auto up = [&](void** dst, const void* src, size_t bytes) -> cudaError_t {
    cudaError_t ee;
    *dst = dalloc(bytes, &ee);
    if (ee != cudaSuccess) return ee;
    if (bytes) ee = cudaMemcpyAsync(*dst, src, bytes, cudaMemcpyHostToDevice, stream);
    return ee;
  };
  std::vector<float> sz(hp.scales.size() * 2 + 4, 0.f);
  for (size_t i = 0; i < hp.scales.size(); ++i) {
    sz[2 * i] = hp.scales[i];
    sz[2 * i + 1] = float(hp.zeros[i]);
  }
  cudaError_t e = up(reinterpret_cast<void**>(&h->d_codes), hp.codes.data(), hp.codes.size());
  if (e == cudaSuccess) e = up(reinterpret_cast<void**>(&h->d_sz), sz.data(), sz.size() * 4);
  if (e == cudaSuccess) e = up(reinterpret_cast<void**>(&h->d_inv_s), hp.inv_s.data(), hp.inv_s.size() * 4);
  if (e == cudaSuccess) e = up(reinterpret_cast<void**>(&h->d_bias), hp.bias.data(), hp.bias.size() * 2);
  if (e == cudaSuccess) {
    h->d_err = static_cast<int*>(dalloc(sizeof(int), &e));
    if (e == cudaSuccess) e = cudaMemsetAsync(h->d_err, 0, sizeof(int), stream);
  }
  if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
  if (e != cudaSuccess) {
    free_awq(h);
    delete h;
    return e == cudaErrorMemoryAllocation ? fail(SVDQ_ERR_OOM, "device allocation failed")
                                          : cuda_fail(e, "uploading the AWQ layer");
  }
  *out = h;
  return SVDQ_OK;
}

svdq_status_t svdq_awq_destroy(svdq_awq_handle_t h) {
  if (!h) return SVDQ_OK;
  DeviceGuard guard(h->device);
  cudaDeviceSynchronize();
  free_awq(h);
  delete h;
  return SVDQ_OK;
}

svdq_status_t svdq_awq_check_error(svdq_awq_handle_t h) {
  if (!h) return fail(SVDQ_ERR_INVALID_ARG, "null handle");
  DeviceGuard guard(h->device);
  cudaError_t e = cudaDeviceSynchronize();
  if (e != cudaSuccess) return cuda_fail(e, "device synchronisation");
  int v = 0;
  e = cudaMemcpy(&v, h->d_err, sizeof(int), cudaMemcpyDeviceToHost);
  if (e == cudaSuccess) e = cudaMemset(h->d_err, 0, sizeof(int));
  if (e != cudaSuccess) return cuda_fail(e, "reading the device error word");
  if (v) return fail(SVDQ_ERR_TIMEOUT, "the AWQ kernel gave up a bounded wait");
  return SVDQ_OK;
}

svdq_status_t svdq_awq_export(svdq_awq_handle_t h, svdq_awq_host_t* out) {
  if (!h || !out) return fail(SVDQ_ERR_INVALID_ARG, "null argument");
  copy_awq_out(h->host, out);
  return SVDQ_OK;
}

svdq_status_t svdq_awq_forward(svdq_awq_handle_t h, const void* X, void* Y, int64_t M, void* stream) {
  if (!h || M < 0) return fail(SVDQ_ERR_INVALID_ARG, "null handle or negative M");
  if (M == 0) return SVDQ_OK;
  if (!X || !Y) return fail(SVDQ_ERR_INVALID_ARG, "null buffer");
  if (!aligned16(X) || !aligned16(Y)) return fail(SVDQ_ERR_INVALID_ARG, "buffers must be 16-byte aligned");
  if (overlaps(X, size_t(M) * h->host.K * 2, Y, size_t(M) * h->host.N * 2))
    return fail(SVDQ_ERR_INVALID_ARG, "X and Y must not overlap");
  DeviceGuard guard(h->device);
  AwqArgs a{};
  a.X = static_cast<const uint16_t*>(X);
  a.inv_s = h->d_inv_s;
  a.codes = h->d_codes;
  a.sz = h->d_sz;
  a.bias = h->d_bias;
  a.err = h->d_err;
  a.Y = static_cast<uint16_t*>(Y);
  a.M = M;
  a.N = h->host.N;
  a.K = h->host.K;
  const int e = awq_launch(a, h->sm_count, stream);
  if (e != 0) return cuda_fail(cudaError_t(e), "AWQ kernel launch");
  return SVDQ_OK;
}

}  // extern "C"
