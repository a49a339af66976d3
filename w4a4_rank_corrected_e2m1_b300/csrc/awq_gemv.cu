// AWQ-style W4A16 linear layer for the modulation / adaptive-normalisation shapes (a few rows
// of activations against a wide weight): Y = x' W'^T + b with x' = fl32(x * fl32(1 / s_c)) and
// W' dequantised from asymmetric 4-bit codes in groups of 64 input channels,
// w' = (q - z) * sc.  The pages keep these layers at 16-bit activations with AWQ-style 4-bit
// weights (aiflownews article on Nunchaku, "How Nunchaku four bit quantization actually
// works").
//
// The work is one pass over the packed weights (HBM-bound: 0.5 byte per weight plus 5 bytes
// per group), so the design keeps the ALU cost per weight small:
//   * the block's rows of x' sit in shared memory in 32-element segments padded by 4 floats,
//     so the eight 16-byte reads a lane makes for its 32 channels are conflict-free;
//   * a lane takes 16 bytes of codes (32 weights, half a group) at a time and turns a code q
//     into the exact float 1 + q/16 with one shift and one LOP3 (exponent of 1.0, q in the
//     top mantissa bits); two products accumulate per packed fma.rn.f32x2;
//   * the zero point and scale are applied once per 32 weights through
//       sum_k x'_k (q_k - z) = 16 sum_k x'_k (1 + q_k/16) - (16 + z) sum_k x'_k,
//     with the 32-channel sums of x' precomputed per block;
//   * each warp owns whole output rows (grid-strided), reduces its lanes with shuffles and
//     writes bf16(acc + b).
// Codes are read with non-allocating 16-byte loads; a warp issues all of two rows' loads (up
// to four per lane per row) before using any.
#include <cuda_runtime.h>

#include "ptx.cuh"
#include "svdq_internal.h"

namespace svdq {

namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;

__host__ __device__ constexpr int64_t padded(int64_t k) { return k + (k >> 5) * 4; }   // 32 floats + 4 pad

__device__ __forceinline__ float2 fma2_rn(float2 a, float2 b, float2 c) {
  uint64_t d, x, y, z;
  asm("mov.b64 %0, {%1, %2};" : "=l"(x) : "f"(a.x), "f"(a.y));
  asm("mov.b64 %0, {%1, %2};" : "=l"(y) : "f"(b.x), "f"(b.y));
  asm("mov.b64 %0, {%1, %2};" : "=l"(z) : "f"(c.x), "f"(c.y));
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(x), "l"(y), "l"(z));
  float2 r;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(r.x), "=f"(r.y) : "l"(d));
  return r;
}

// 1 + q/16 for nibble i of w (exact: exponent of 1.0, q in mantissa bits 22..19)
template <int I>
__device__ __forceinline__ float nib(uint32_t w) {
  constexpr int sh = 4 * I - 19;
  const uint32_t v = sh >= 0 ? (w >> sh) : (w << -sh);
  return __uint_as_float((v & 0x00780000u) | 0x3F800000u);
}

template <int MB>
__global__ void __launch_bounds__(kThreads) awq_gemv_kernel(AwqArgs a, int64_t m0) {
  extern __shared__ __align__(16) float sm[];
  const int64_t K = a.K, N = a.N;
  const int64_t KP = padded(K);
  const int nseg = int(K / 32);
  float* xs = sm;                       // [MB][KP]: x' in padded 32-float segments
  float* seg_sum = sm + MB * KP;        // [MB][K / 32]: sum of each segment of x'
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

#pragma unroll
  for (int m = 0; m < MB; ++m) {
    const bool live = m0 + m < a.M;
    for (int64_t k = threadIdx.x; k < K; k += blockDim.x) {
      float v = 0.f;
      if (live) v = __fmul_rn(__uint_as_float(uint32_t(a.X[(m0 + m) * K + k]) << 16), a.inv_s[k]);
      xs[m * KP + padded(k)] = v;
    }
  }
  __syncthreads();
  for (int i = threadIdx.x; i < MB * nseg; i += blockDim.x) {
    const int m = i / nseg, sgi = i - m * nseg;
    const float* p = xs + m * KP + int64_t(sgi) * 36;
    float s = 0.f;
#pragma unroll 8
    for (int j = 0; j < 32; ++j) s += p[j];
    seg_sum[m * nseg + sgi] = s;
  }
  __syncthreads();

  const int64_t KG = K / 64;
  const int64_t nwarps = int64_t(gridDim.x) * kWarps;
  // two output rows per warp at a time, and up to kBatch 16-byte code loads per row per lane
  // issued before any of them is used, so that enough bytes are in flight to cover HBM latency
  constexpr int kRowsInFlight = 2, kBatch = 4;
  for (int64_t n0 = int64_t(blockIdx.x) * kWarps + warp; n0 < N; n0 += nwarps * kRowsInFlight) {
    float part[kRowsInFlight][MB];
#pragma unroll
    for (int r = 0; r < kRowsInFlight; ++r)
#pragma unroll
      for (int m = 0; m < MB; ++m) part[r][m] = 0.f;
    for (int sb = 0; sb < nseg; sb += 32 * kBatch) {
      uint4 c[kRowsInFlight][kBatch];
      float sc[kRowsInFlight][kBatch], zf[kRowsInFlight][kBatch];
#pragma unroll
      for (int r = 0; r < kRowsInFlight; ++r) {
        const int64_t n = n0 + r * nwarps;
#pragma unroll
        for (int i = 0; i < kBatch; ++i) {
          const int sgi = sb + lane + 32 * i;
          if (n < N && sgi < nseg) {
            c[r][i] = ptx::ld_stream_v4(a.codes + n * (K / 2) + int64_t(sgi) * 16);
            sc[r][i] = __ldg(a.scales + n * KG + (sgi >> 1));
            zf[r][i] = float(__ldg(a.zeros + n * KG + (sgi >> 1)));
          } else {
            c[r][i] = make_uint4(0, 0, 0, 0);
            sc[r][i] = 0.f;
            zf[r][i] = 0.f;
          }
        }
      }
#pragma unroll
      for (int i = 0; i < kBatch; ++i) {
        const int sgi = sb + lane + 32 * i;
        if (sgi >= nseg) break;
#pragma unroll
        for (int m = 0; m < MB; ++m) {
          const float4* xp = reinterpret_cast<const float4*>(xs + m * KP + int64_t(sgi) * 36);
          float4 xv[8];
#pragma unroll
          for (int v = 0; v < 8; ++v) xv[v] = xp[v];                  // channels 4v .. 4v + 3
          const float ssum = seg_sum[m * nseg + sgi];
#pragma unroll
          for (int r = 0; r < kRowsInFlight; ++r) {
            float2 acc = make_float2(0.f, 0.f);
            const uint32_t cw[4] = {c[r][i].x, c[r][i].y, c[r][i].z, c[r][i].w};
#pragma unroll
            for (int u = 0; u < 4; ++u) {                              // channels 8u .. 8u + 7
              const uint32_t w = cw[u];                                // element 2j in the low nibble
              const float4 x0 = xv[2 * u], x1 = xv[2 * u + 1];
              acc = fma2_rn(make_float2(x0.x, x0.y), make_float2(nib<0>(w), nib<1>(w)), acc);
              acc = fma2_rn(make_float2(x0.z, x0.w), make_float2(nib<2>(w), nib<3>(w)), acc);
              acc = fma2_rn(make_float2(x1.x, x1.y), make_float2(nib<4>(w), nib<5>(w)), acc);
              acc = fma2_rn(make_float2(x1.z, x1.w), make_float2(nib<6>(w), nib<7>(w)), acc);
            }
            const float t = acc.x + acc.y;                             // sum x' (1 + q/16)
            part[r][m] = fmaf(sc[r][i], fmaf(16.f, t, -(16.f + zf[r][i]) * ssum), part[r][m]);
          }
        }
      }
    }
#pragma unroll
    for (int r = 0; r < kRowsInFlight; ++r) {
      const int64_t n = n0 + r * nwarps;
#pragma unroll
      for (int m = 0; m < MB; ++m) {
        float v = part[r][m];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
        if (lane == 0 && n < N && m0 + m < a.M) {
          const float b = __uint_as_float(uint32_t(a.bias[n]) << 16);
          a.Y[(m0 + m) * N + n] = uint16_t(ptx::pack_bf16x2(v + b, 0.f) & 0xFFFFu);
        }
      }
    }
  }
}

template <int MB>
int launch_mb(const AwqArgs& a, int sm_count, cudaStream_t s) {
  const size_t smem = (size_t(MB) * padded(a.K) + size_t(MB) * (a.K / 32)) * sizeof(float);
  static int attr_done[64] = {0};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 64 && !attr_done[dev]) {
    cudaError_t e = cudaFuncSetAttribute(awq_gemv_kernel<MB>, cudaFuncAttributeMaxDynamicSharedMemorySize, 220 * 1024);
    if (e != cudaSuccess) return int(e);
    attr_done[dev] = 1;
  }
  const int64_t rows_per_block = kWarps;
  int64_t blocks = (a.N + rows_per_block - 1) / rows_per_block;
  const int64_t cap = int64_t(sm_count) * (smem <= 100 * 1024 ? 2 : 1) * 2;   // a couple of waves of rows each
  if (blocks > cap) blocks = cap;
  for (int64_t m0 = 0; m0 < a.M; m0 += MB) {
    awq_gemv_kernel<MB><<<unsigned(blocks), kThreads, smem, s>>>(a, m0);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return int(e);
  }
  return 0;
}

}  // namespace

size_t awq_smem_bytes(int64_t K, int mb) { return (size_t(mb) * padded(K) + size_t(mb) * (K / 32)) * sizeof(float); }

int awq_launch(const AwqArgs& a, int sm_count, void* stream) {
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // rows of X per pass: as many as the shared memory for x' allows, at most 8
  int mb = a.M >= 8 ? 8 : (a.M >= 4 ? 4 : (a.M >= 2 ? 2 : 1));
  while (mb > 1 && awq_smem_bytes(a.K, mb) > 200 * 1024) mb >>= 1;
  if (awq_smem_bytes(a.K, mb) > 200 * 1024) return int(cudaErrorInvalidValue);
  switch (mb) {
    case 8: return launch_mb<8>(a, sm_count, s);
    case 4: return launch_mb<4>(a, sm_count, s);
    case 2: return launch_mb<2>(a, sm_count, s);
    default: return launch_mb<1>(a, sm_count, s);
  }
}

}  // namespace svdq
