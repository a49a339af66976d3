// The INT4 variant of the SVDQuant layer.  The pages say SVDQuant supports both INT4 and FP4
// and that Nunchaku runs INT4 kernels on hardware older than Blackwell (aiflownews article on
// Nunchaku, "What SVDQuant actually does", "How Nunchaku four bit quantization actually works").
// Here the residual and the smoothed activations are quantised to symmetric INT4 groups: codes
// q in [-7, 7] (stored as the nibble q + 8), one float32 scale s = fl32(amax / 7) per 64
// elements along K, q = clamp(rint(fl32(v * fl32(1 / s))), -7, 7):
//
//   Y = sum_g sX[m, g] sW[n, g] * (sum_{k in g} qx[m, k] qw[n, k])  +  (X^ L1) L2  +  b
//
// The per-group scales sit inside the K sum, so the integer dot product of every 64-element
// group has to be finished, and scaled, before the next group is added.  tcgen05 has no integer
// kind on this part (ptxas rejects kind::i8 for sm_103a) and keeps its accumulator in TMEM, out of
// reach of a per-group rescale; the legacy warp MMA keeps it in registers.  Measured on this part:
// mma.sync s4 runs at ~51 TOPS, s8 at ~143 TOPS, bf16 at ~572 TFLOP/s.  So the codes are unpacked
// to bf16 in registers (exact: integers -7..7) and each group's four 16-deep bf16 MMAs add the
// integer products exactly in float32 (|sum| <= 64 * 49 < 2^24), after which the group partial is
// multiplied by sX * sW and added to the float32 accumulator.
//
// Kernel int4_k1: per 32 rows, one pass over X in 64-column groups through a TMA ring: the
// quantiser (x^ = fl32(x inv_lambda), group maximum, scale, codes) and the down-projection
// T = X (diag(inv_lambda) L1) on bf16 warp MMAs from the same shared-memory tile.
// Kernel int4_k2: per 128 x 128 output tile, a TMA ring of one group per stage (the two tiles'
// codes and group scales); then T L2 on bf16 warp MMAs into the same accumulator, the bias, and
// bf16 Y.  Every wait is bounded; on expiry the error word is set and the kernel finishes what
// it started.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "ptx.cuh"
#include "svdq_internal.h"

namespace svdq {

namespace {

constexpr uint64_t kDrainNs = 2000000000ull;

__device__ bool i4_wait(uint64_t* bar, uint32_t parity, volatile int* abort_flag, int* err, uint64_t limit_ns) {
  if (ptx::mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = ptx::globaltimer();
  for (uint32_t i = 1;; ++i) {
    if (ptx::mbar_try_wait(bar, parity)) return true;
    if ((i & 31u) == 0u) {
      if (*abort_flag) return false;
      if (ptx::globaltimer() - t0 > limit_ns) {
        *abort_flag = 1;
        atomicOr(err, 32);
        return false;
      }
    }
  }
}
// Waits for copies already started (ignores the abort flag; bounded).
__device__ void i4_drain(uint64_t* bar, uint32_t parity) {
  const uint64_t t0 = ptx::globaltimer();
  while (!ptx::mbar_try_wait(bar, parity))
    if (ptx::globaltimer() - t0 > kDrainNs) return;
}

// Byte of two INT4 nibbles (c_lo, c_hi; code = q + 8) -> bf16x2 (q_lo, q_hi), exact: the bf16
// with bits 0x4300 | c is 128 + c, and 128 + c - 136 = q.
__device__ __forceinline__ uint32_t i4pair_bf16(uint32_t byte) {
  uint32_t v = (byte & 0xFu) | ((byte & 0xF0u) << 12) | 0x43004300u;
  const __nv_bfloat162 r = __hsub2(*reinterpret_cast<const __nv_bfloat162*>(&v), __floats2bfloat162_rn(136.f, 136.f));
  return *reinterpret_cast<const uint32_t*>(&r);
}

// ------------------------------------------------------------------ kernel int4_k1
constexpr int kK1Rows = 32;
constexpr int kK1Consumers = 8;                      // warps: quantiser + down-projection
constexpr int kK1Threads = 32 * (kK1Consumers + 1);  // + producer warp

template <int RP>   // r_pad: 0, 64 or 128
struct K1I4 {
  static constexpr int X_BYTES = kK1Rows * 128;      // 32 rows x 64 bf16, 128-byte swizzle
  static constexpr int L_BYTES = RP * 128;           // r_pad rows x 64 bf16 of (diag(inv_lambda) L1)^T
  static constexpr int STAGE = X_BYTES + L_BYTES;
  static constexpr int STAGES = (192 * 1024) / STAGE > 12 ? 12 : (192 * 1024) / STAGE;
  static constexpr int NT = RP / 32;                 // n8 tiles of T per warp (4 warps share a m16 tile)
  static constexpr int SMEM = STAGES * STAGE + 1024;
  static_assert(STAGE % 1024 == 0, "stage alignment");
};

template <int RP>
__global__ void __launch_bounds__(kK1Threads, 1) int4_k1_kernel(const __grid_constant__ Int4K1Maps maps, Int4K1Args a) {
  using C = K1I4<RP>;
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* ring = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  __shared__ uint64_t full[C::STAGES], empty[C::STAGES];
  __shared__ volatile int abort_flag;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t M = a.M, K = a.K;
  const int G = int(K / 64);
  const int64_t row0 = int64_t(blockIdx.x) * kK1Rows;

  ptx::griddep_launch_dependents();
  if (threadIdx.x == 0) {
    for (int i = 0; i < C::STAGES; ++i) {
      ptx::mbar_init(&full[i], 1);
      ptx::mbar_init(&empty[i], kK1Consumers);
    }
    abort_flag = 0;
    ptx::fence_barrier_init();
  }
  __syncthreads();
  ptx::griddep_wait();                               // X may come from the previous kernel

  if (warp == kK1Consumers) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      ptx::prefetch_tmap(&maps.X);
      if (RP) ptx::prefetch_tmap(&maps.L1t);
      int issued = 0;
      for (int g = 0; g < G; ++g, ++issued) {
        const int stage = g % C::STAGES;
        if (g >= C::STAGES) {
          if (!i4_wait(&empty[stage], uint32_t((g / C::STAGES) - 1) & 1u, &abort_flag, a.err, a.wait_ns)) break;
          ptx::fence_proxy_async_smem();             // the consumers' ordinary loads before the refill
        }
        unsigned char* st = ring + stage * C::STAGE;
        ptx::mbar_arrive_expect_tx(&full[stage], C::STAGE);
        ptx::tma_load_2d(st, &maps.X, &full[stage], 64 * g, int(row0));
        if (RP) ptx::tma_load_2d(st + C::X_BYTES, &maps.L1t, &full[stage], 64 * g, 0);
      }
      for (int i = 0; i < C::STAGES; ++i) {          // every copy issued has landed
        const int uses = issued > i ? (issued - i + C::STAGES - 1) / C::STAGES : 0;
        if (uses > 0) i4_drain(&full[i], uint32_t(uses - 1) & 1u);
      }
    }
  } else {
    // ------------------------------------------------------------ quantiser + down-projection
    const int tq = threadIdx.x;                      // 0..255
    const int qrow = tq >> 3, qc = tq & 7;           // row of the tile, 16-byte chunk (8 channels)
    const int64_t grow = row0 + qrow;
    const int mi = warp & 1, nq = warp >> 1;         // T: m16 tile, first n8 tile (n8 tiles nq + 4u)
    float acc[C::NT > 0 ? C::NT : 1][4];
#pragma unroll
    for (int u = 0; u < (C::NT > 0 ? C::NT : 1); ++u) acc[u][0] = acc[u][1] = acc[u][2] = acc[u][3] = 0.f;
    for (int g = 0; g < G; ++g) {
      const int stage = g % C::STAGES;
      if (!i4_wait(&full[stage], uint32_t(g / C::STAGES) & 1u, &abort_flag, a.err, a.wait_ns)) break;
      const uint32_t xs = ptx::smem_u32(ring + stage * C::STAGE);
      // quantiser: x^ = fl32(x inv_lambda) for 8 channels; the group (64 channels of this row)
      // is spread over the 8 lanes with the same qrow
      {
        const uint4 xv = ptx::lds_v4(xs + uint32_t(qrow) * 128u + (uint32_t(qc ^ (qrow & 7)) << 4));
        const float4 i0 = __ldg(reinterpret_cast<const float4*>(a.inv_lambda + 64 * int64_t(g) + 8 * qc));
        const float4 i1 = __ldg(reinterpret_cast<const float4*>(a.inv_lambda + 64 * int64_t(g) + 8 * qc + 4));
        const float inv[8] = {i0.x, i0.y, i0.z, i0.w, i1.x, i1.y, i1.z, i1.w};
        const uint32_t xw[4] = {xv.x, xv.y, xv.z, xv.w};
        float xh[8];
        float amax = 0.f;
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const uint32_t bits = (e & 1) ? (xw[e >> 1] & 0xFFFF0000u) : (xw[e >> 1] << 16);
          xh[e] = __fmul_rn(__uint_as_float(bits), inv[e]);
          amax = fmaxf(amax, fabsf(xh[e]));
        }
        amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, 1));
        amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, 2));
        amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, 4));
        const float s = __fdiv_rn(amax, 7.f);
        uint32_t word = 0x88888888u;                 // all-zero group: q = 0
        if (s > 0.f) {
          const float rcp = __frcp_rn(s);
          word = 0u;
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            int q = __float2int_rn(__fmul_rn(xh[e], rcp));
            q = q < -7 ? -7 : (q > 7 ? 7 : q);
            word |= uint32_t(q + 8) << (4 * e);
          }
        }
        if (grow < M) {
          *reinterpret_cast<uint32_t*>(a.codes + grow * (K / 2) + 32 * int64_t(g) + 4 * qc) = word;
          if (qc == 0) a.scales[int64_t(g) * a.scale_ld + grow] = s;
        }
      }
      // down-projection: T += X (64 channels) L1'^T slice, bf16 warp MMAs
      if constexpr (RP > 0) {
        const uint32_t ls = xs + C::X_BYTES;
#pragma unroll
        for (int s4 = 0; s4 < 4; ++s4) {
          uint32_t af[4];
          const int r = 16 * mi + (lane & 15), ch = 2 * s4 + (lane >> 4);
          ptx::ldmatrix_x4(xs + uint32_t(r) * 128u + (uint32_t(ch ^ (r & 7)) << 4), af);
#pragma unroll
          for (int u = 0; u < C::NT; ++u) {
            uint32_t bf[2];
            const int rn = 8 * (nq + 4 * u) + (lane & 7), chb = 2 * s4 + ((lane >> 3) & 1);
            ptx::ldmatrix_x2(ls + uint32_t(rn) * 128u + (uint32_t(chb ^ (rn & 7)) << 4), bf);
            ptx::mma_bf16_16816(acc[u], af[0], af[1], af[2], af[3], bf[0], bf[1]);
          }
        }
      }
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(&empty[stage]);
    }
    if constexpr (RP > 0) {
      const int64_t r0 = row0 + 16 * mi + (lane >> 2), r1 = r0 + 8;
#pragma unroll
      for (int u = 0; u < C::NT; ++u) {
        const int col = 8 * (nq + 4 * u) + 2 * (lane & 3);
        if (r0 < M) *reinterpret_cast<uint32_t*>(a.T + r0 * RP + col) = ptx::pack_bf16x2(acc[u][0], acc[u][1]);
        if (r1 < M) *reinterpret_cast<uint32_t*>(a.T + r1 * RP + col) = ptx::pack_bf16x2(acc[u][2], acc[u][3]);
      }
    }
  }
}

template <int RP>
int launch_k1(const Int4K1Maps& maps, const Int4K1Args& a, cudaStream_t s) {
  using C = K1I4<RP>;
  static int attr_done[64] = {0};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 64 && !attr_done[dev]) {
    const cudaError_t e = cudaFuncSetAttribute(int4_k1_kernel<RP>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
    if (e != cudaSuccess) return int(e);
    attr_done[dev] = 1;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(unsigned(ceil_div(a.M, kK1Rows)), 1, 1);
  cfg.blockDim = dim3(kK1Threads, 1, 1);
  cfg.dynamicSmemBytes = C::SMEM;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return int(cudaLaunchKernelEx(&cfg, int4_k1_kernel<RP>, maps, a));
}

// ------------------------------------------------------------------ kernel int4_k2
constexpr int kK2Tile = 128;
constexpr int kK2Consumers = 8;                      // 4 (rows) x 2 (columns) warps of 32 x 64
constexpr int kK2Threads = 32 * (kK2Consumers + 1);
constexpr int kK2Stages = 8;
constexpr int kCodeBytes = kK2Tile * 32;             // 128 rows x 64 codes
constexpr int kK2Stage = 2 * kCodeBytes + 2 * kK2Tile * 4;   // codes of both tiles + their group scales
static_assert(kK2Stage % 1024 == 0, "stage alignment");

template <int RP>
struct K2I4 {
  static constexpr int LR_BYTES = RP * kK2Tile * 2;  // T or L2^T of the tile: r_pad / 64 boxes of 16 KB
  static constexpr int SMEM = kK2Stages * kK2Stage + 2 * LR_BYTES + 1024;
};

template <int RP>
__global__ void __launch_bounds__(kK2Threads, 1) int4_k2_kernel(const __grid_constant__ Int4K2Maps maps, Int4K2Args a) {
  using C = K2I4<RP>;
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* ring = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  unsigned char* t_s = ring + kK2Stages * kK2Stage;  // T tile (r_pad / 64 swizzled 128 x 64 boxes)
  unsigned char* l_s = t_s + C::LR_BYTES;            // L2^T tile, same
  __shared__ uint64_t full[kK2Stages], empty[kK2Stages], lr_full;
  __shared__ volatile int abort_flag;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t M = a.M, N = a.N, K = a.K;
  const int G = int(K / 64);
  const int m0 = int(blockIdx.y) * kK2Tile, n0 = int(blockIdx.x) * kK2Tile;

  ptx::griddep_launch_dependents();
  if (threadIdx.x == 0) {
    for (int i = 0; i < kK2Stages; ++i) {
      ptx::mbar_init(&full[i], 1);
      ptx::mbar_init(&empty[i], kK2Consumers);
    }
    ptx::mbar_init(&lr_full, 1);
    abort_flag = 0;
    ptx::fence_barrier_init();
  }
  __syncthreads();
  ptx::griddep_wait();

  if (warp == kK2Consumers) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      ptx::prefetch_tmap(&maps.A);
      ptx::prefetch_tmap(&maps.B);
      ptx::prefetch_tmap(&maps.SA);
      ptx::prefetch_tmap(&maps.SB);
      if (RP) {
        ptx::mbar_arrive_expect_tx(&lr_full, 2 * C::LR_BYTES);
        for (int c = 0; c < RP / 64; ++c) {
          ptx::tma_load_2d(t_s + c * 16384, &maps.T, &lr_full, 64 * c, m0);
          ptx::tma_load_2d(l_s + c * 16384, &maps.L2, &lr_full, 64 * c, n0);
        }
      }
      int issued = 0;
      for (int g = 0; g < G; ++g, ++issued) {
        const int stage = g % kK2Stages;
        if (g >= kK2Stages) {
          if (!i4_wait(&empty[stage], uint32_t((g / kK2Stages) - 1) & 1u, &abort_flag, a.err, a.wait_ns)) break;
          ptx::fence_proxy_async_smem();             // the consumers' ordinary loads before the refill
        }
        unsigned char* st = ring + stage * kK2Stage;
        ptx::mbar_arrive_expect_tx(&full[stage], kK2Stage);
        ptx::tma_load_2d(st, &maps.A, &full[stage], 32 * g, m0);
        ptx::tma_load_2d(st + kCodeBytes, &maps.B, &full[stage], 32 * g, n0);
        ptx::tma_load_2d(st + 2 * kCodeBytes, &maps.SA, &full[stage], m0, g);
        ptx::tma_load_2d(st + 2 * kCodeBytes + kK2Tile * 4, &maps.SB, &full[stage], n0, g);
      }
      for (int i = 0; i < kK2Stages; ++i) {          // every copy issued has landed
        const int uses = issued > i ? (issued - i + kK2Stages - 1) / kK2Stages : 0;
        if (uses > 0) i4_drain(&full[i], uint32_t(uses - 1) & 1u);
      }
      if (RP) i4_drain(&lr_full, 0);
    }
  } else {
    // ------------------------------------------------------------ MMA warps (32 x 64 each)
    const int wm = warp & 3, wn = warp >> 2;
    const int gq = lane >> 2, tq = lane & 3;
    float acc[2][8][4];
#pragma unroll
    for (int i = 0; i < 2; ++i)
#pragma unroll
      for (int j = 0; j < 8; ++j) acc[i][j][0] = acc[i][j][1] = acc[i][j][2] = acc[i][j][3] = 0.f;
    for (int g = 0; g < G; ++g) {
      const int stage = g % kK2Stages;
      if (!i4_wait(&full[stage], uint32_t(g / kK2Stages) & 1u, &abort_flag, a.err, a.wait_ns)) break;
      const uint32_t a_s = ptx::smem_u32(ring + stage * kK2Stage);
      const uint32_t b_s = a_s + kCodeBytes;
      const float* sa = reinterpret_cast<const float*>(ring + stage * kK2Stage + 2 * kCodeBytes);
      const float* sb = sa + kK2Tile;
      float part[2][8][4];
#pragma unroll
      for (int s4 = 0; s4 < 4; ++s4) {
        // A fragments: rows 32 wm + 16 i + gq (+ 8), k = 16 s4 + 2 tq (+ 8): bytes 8 s4 + tq and
        // 8 s4 + 4 + tq of the row's 32 code bytes
        uint32_t af[2][4];
#pragma unroll
        for (int i = 0; i < 2; ++i)
#pragma unroll
          for (int hr = 0; hr < 2; ++hr) {
            const int row = 32 * wm + 16 * i + gq + 8 * hr;
            const uint2 w = ptx::lds_v2(a_s + uint32_t(row) * 32u + 8u * uint32_t(s4));
            af[i][hr] = i4pair_bf16((w.x >> (8 * tq)) & 0xFFu);
            af[i][2 + hr] = i4pair_bf16((w.y >> (8 * tq)) & 0xFFu);
          }
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const int col = 64 * wn + 8 * j + gq;
          const uint2 w = ptx::lds_v2(b_s + uint32_t(col) * 32u + 8u * uint32_t(s4));
          const uint32_t b0 = i4pair_bf16((w.x >> (8 * tq)) & 0xFFu), b1 = i4pair_bf16((w.y >> (8 * tq)) & 0xFFu);
#pragma unroll
          for (int i = 0; i < 2; ++i) {
            if (s4 == 0) part[i][j][0] = part[i][j][1] = part[i][j][2] = part[i][j][3] = 0.f;
            ptx::mma_bf16_16816(part[i][j], af[i][0], af[i][1], af[i][2], af[i][3], b0, b1);
          }
        }
      }
      // the group's exact integer sums, scaled by sX[row] * sW[col]
      float sxr[2][2];
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        sxr[i][0] = sa[32 * wm + 16 * i + gq];
        sxr[i][1] = sa[32 * wm + 16 * i + gq + 8];
      }
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const float2 swc = *reinterpret_cast<const float2*>(sb + 64 * wn + 8 * j + 2 * tq);
#pragma unroll
        for (int i = 0; i < 2; ++i) {
          acc[i][j][0] = fmaf(part[i][j][0], sxr[i][0] * swc.x, acc[i][j][0]);
          acc[i][j][1] = fmaf(part[i][j][1], sxr[i][0] * swc.y, acc[i][j][1]);
          acc[i][j][2] = fmaf(part[i][j][2], sxr[i][1] * swc.x, acc[i][j][2]);
          acc[i][j][3] = fmaf(part[i][j][3], sxr[i][1] * swc.y, acc[i][j][3]);
        }
      }
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(&empty[stage]);
    }
    // low-rank branch: acc += T L2 (bf16 warp MMAs, K = r_pad)
    if constexpr (RP > 0) {
      if (i4_wait(&lr_full, 0, &abort_flag, a.err, a.wait_ns)) {
        const uint32_t ts = ptx::smem_u32(t_s), l2s = ptx::smem_u32(l_s);
#pragma unroll
        for (int c = 0; c < RP / 16; ++c) {
          const uint32_t box = uint32_t(c >> 2) * 16384u;
          const int s4 = c & 3;
          uint32_t af[2][4];
#pragma unroll
          for (int i = 0; i < 2; ++i) {
            const int r = 32 * wm + 16 * i + (lane & 15), ch = 2 * s4 + (lane >> 4);
            ptx::ldmatrix_x4(ts + box + uint32_t(r) * 128u + (uint32_t(ch ^ (r & 7)) << 4), af[i]);
          }
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            uint32_t bf[2];
            const int rn = 64 * wn + 8 * j + (lane & 7), chb = 2 * s4 + ((lane >> 3) & 1);
            ptx::ldmatrix_x2(l2s + box + uint32_t(rn) * 128u + (uint32_t(chb ^ (rn & 7)) << 4), bf);
#pragma unroll
            for (int i = 0; i < 2; ++i) ptx::mma_bf16_16816(acc[i][j], af[i][0], af[i][1], af[i][2], af[i][3], bf[0], bf[1]);
          }
        }
      }
    }
    // epilogue: + bias, bf16 Y
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int64_t col = n0 + 64 * wn + 8 * j + 2 * tq;
      if (col >= N) continue;
      const uint32_t bb = *reinterpret_cast<const uint32_t*>(a.bias + col);
      const float b0 = __uint_as_float(bb << 16), b1 = __uint_as_float(bb & 0xFFFF0000u);
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        const int64_t r0 = m0 + 32 * wm + 16 * i + gq, r1 = r0 + 8;
        if (r0 < M) *reinterpret_cast<uint32_t*>(a.Y + r0 * N + col) = ptx::pack_bf16x2(acc[i][j][0] + b0, acc[i][j][1] + b1);
        if (r1 < M) *reinterpret_cast<uint32_t*>(a.Y + r1 * N + col) = ptx::pack_bf16x2(acc[i][j][2] + b0, acc[i][j][3] + b1);
      }
    }
  }
}

template <int RP>
int launch_k2(const Int4K2Maps& maps, const Int4K2Args& a, cudaStream_t s) {
  using C = K2I4<RP>;
  static int attr_done[64] = {0};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 64 && !attr_done[dev]) {
    const cudaError_t e = cudaFuncSetAttribute(int4_k2_kernel<RP>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
    if (e != cudaSuccess) return int(e);
    attr_done[dev] = 1;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(unsigned(ceil_div(a.N, kK2Tile)), unsigned(ceil_div(a.M, kK2Tile)), 1);
  cfg.blockDim = dim3(kK2Threads, 1, 1);
  cfg.dynamicSmemBytes = C::SMEM;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return int(cudaLaunchKernelEx(&cfg, int4_k2_kernel<RP>, maps, a));
}

}  // namespace

int int4_k1_launch(const Int4K1Maps& maps, const Int4K1Args& a, void* stream) {
  if (a.M == 0) return 0;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  switch (a.r_pad) {
    case 0: return launch_k1<0>(maps, a, s);
    case 64: return launch_k1<64>(maps, a, s);
    case 128: return launch_k1<128>(maps, a, s);
    default: return int(cudaErrorInvalidValue);
  }
}

int int4_k2_launch(const Int4K2Maps& maps, const Int4K2Args& a, void* stream) {
  if (a.M == 0) return 0;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  switch (a.r_pad) {
    case 0: return launch_k2<0>(maps, a, s);
    case 64: return launch_k2<64>(maps, a, s);
    case 128: return launch_k2<128>(maps, a, s);
    default: return int(cudaErrorInvalidValue);
  }
}

}  // namespace svdq
