// Kernel 1: one pass over the bf16 activations X that
//   (a) smooths them, x^ = fl32(x * inv_lambda)            (stage one of SVDQuant),
//   (b) quantises x^ to NVFP4: one E4M3 scale per 16 elements, E2M1 codes (stage three),
//   (c) computes the low-rank down-projection T = X^ L1 of the 16-bit branch (stage two),
// so X is read from HBM exactly once ("the low rank branch and the 4 bit branch ... share
// inputs", Nunchaku section of the aiflownews article on Nunchaku in Diffusers).
//
// Work decomposition: a CTA owns a tile of rows (128, or 64 for rank > 64) and a range of
// 64-column chunks; splitting K across CTAs keeps all SMs busy at small M.  A warp owns
// 16*MT rows.  Thread (g = lane/4, t = lane%4) loads, for each of its rows, the 16
// consecutive bf16 at columns 16t..16t+15 of the chunk (two 16-byte loads): exactly one
// NVFP4 block, so the block maximum needs no shuffles, and a quad writes 32 contiguous
// bytes of codes per row.  The E2M1 conversion (cvt.rn.satfinite.e2m1x2) rounds to nearest
// even and keeps the sign of a negative value that rounds to zero, which is the format rule
// the codes follow.
//
// Down-projection on the warp MMA (m16n8k16, bf16 in, f32 accumulate).  The registers a
// thread already holds are used directly as A fragments: the k order inside each 16-wide
// MMA step is permuted so that thread t's A elements are its own columns
//   step s: logical k {2t, 2t+1, 2t+8, 2t+9}  <->  chunk columns 16t + 4s + {0, 1, 2, 3},
// and the B operand (L1 with 1/lambda folded in, prepared at pack time) is stored in the
// same permuted order ("Lperm": for chunk c, n-tile j, lane l = 4g + t, the 16 values
// L1'[64c + 16t + i][8j + g], i = 0..15), one 32-byte load per thread and n-tile.
// With K split over several CTAs, partial sums go to a float32 workspace and the last CTA
// of a row tile to finish adds them in split order (deterministic), scales by 1/alpha and
// writes T in bfloat16.
#include <cuda_runtime.h>

#include "ptx.cuh"
#include "svdq_internal.h"

namespace svdq {

namespace {

constexpr int kWarps = 4;
constexpr uint32_t kFull = 0xFFFFFFFFu;

template <int NT, int MT>
__global__ void __launch_bounds__(kWarps * 32) k1_kernel(K1Args a, int chunks_per_split, int nsplit) {
  constexpr int ROWS = kWarps * 16 * MT;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, t = lane & 3;
  const int tile = blockIdx.x, split = blockIdx.y;
  const int64_t M = a.M, K = a.K;
  const int64_t KG = scale_groups(K);
  const int nchunks = int(K / 64);
  const int c0 = split * chunks_per_split;
  const int c1 = min(nchunks, c0 + chunks_per_split);
  const int64_t row_base = int64_t(tile) * ROWS + warp * 16 * MT;

  float acc[MT][NT > 0 ? NT : 1][4];
#pragma unroll
  for (int i = 0; i < MT; ++i)
#pragma unroll
    for (int j = 0; j < (NT > 0 ? NT : 1); ++j) acc[i][j][0] = acc[i][j][1] = acc[i][j][2] = acc[i][j][3] = 0.f;

  for (int c = c0; c < c1; ++c) {
    const int64_t col = int64_t(c) * 64 + 16 * t;
    // raw bf16 of the thread's rows: w[r][0..7], rows r = 2*mt (+g) and 2*mt+1 (+g+8)
    uint32_t w[2 * MT][8];
#pragma unroll
    for (int r = 0; r < 2 * MT; ++r) {
      const int64_t row = row_base + 16 * (r >> 1) + g + 8 * (r & 1);
      if (row < M) {
        const uint16_t* src = a.X + row * K + col;
        const uint4 u0 = ptx::ld_stream_v4(src);
        const uint4 u1 = ptx::ld_stream_v4(src + 8);
        w[r][0] = u0.x; w[r][1] = u0.y; w[r][2] = u0.z; w[r][3] = u0.w;
        w[r][4] = u1.x; w[r][5] = u1.y; w[r][6] = u1.z; w[r][7] = u1.w;
      } else {
#pragma unroll
        for (int i = 0; i < 8; ++i) w[r][i] = 0u;
      }
    }
    float il[16];
    {
      const float4* p = reinterpret_cast<const float4*>(a.inv_lambda + col);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float4 v = __ldg(p + i);
        il[4 * i] = v.x; il[4 * i + 1] = v.y; il[4 * i + 2] = v.z; il[4 * i + 3] = v.w;
      }
    }
    // ---- NVFP4 quantisation, two rows at a time (the E4M3 conversions go in pairs)
#pragma unroll
    for (int rp = 0; rp < MT; ++rp) {
      float xh[2][16];
      float amax[2];
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int r = 2 * rp + h;
        float m = 0.f;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const float lo = __uint_as_float(w[r][i] << 16);
          const float hi = __uint_as_float(w[r][i] & 0xFFFF0000u);
          xh[h][2 * i] = __fmul_rn(lo, il[2 * i]);
          xh[h][2 * i + 1] = __fmul_rn(hi, il[2 * i + 1]);
          m = fmaxf(m, fmaxf(fabsf(xh[h][2 * i]), fabsf(xh[h][2 * i + 1])));
        }
        amax[h] = m;
      }
      const float s0 = __fdiv_rn(amax[0], a.six_sgX);
      const float s1 = __fdiv_rn(amax[1], a.six_sgX);
      const uint16_t s8 = ptx::cvt_e4m3x2(s1, s0);          // row h=0 in the low byte
      const float2 dec = ptx::e4m3x2_to_f32x2(s8);
      uint32_t sc[2] = {uint32_t(s8 & 0xFF), uint32_t(s8 >> 8)};
      float dd[2] = {dec.x, dec.y};
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int r = 2 * rp + h;
        const int64_t row = row_base + 16 * rp + g + 8 * h;
        uint32_t code0 = 0u, code1 = 0u;
        if (sc[h] != 0u) {
          const float d = __fmul_rn(dd[h], a.s_gX);
          const float rcp = __frcp_rn(d);
          float q[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) q[i] = __fmul_rn(xh[h][i], rcp);
          code0 = ptx::cvt_e2m1x8(q[0], q[1], q[2], q[3], q[4], q[5], q[6], q[7]);
          code1 = ptx::cvt_e2m1x8(q[8], q[9], q[10], q[11], q[12], q[13], q[14], q[15]);
        }
        if (row < M) {
          uint2* dst = reinterpret_cast<uint2*>(a.x_codes + row * (K / 2) + col / 2);
          *dst = make_uint2(code0, code1);
        }
        // the quad's four scale bytes of this row form one 32-bit word of the tiled layout
        uint32_t word = sc[h] << (8 * t);
        word |= __shfl_xor_sync(kFull, word, 1);
        word |= __shfl_xor_sync(kFull, word, 2);
        if (t == ((2 * rp + h) & 3)) {
          const int64_t off = ((row >> 7) * KG + c) * 512 + (row & 31) * 16 + ((row >> 5) & 3) * 4;
          *reinterpret_cast<uint32_t*>(a.x_scales + off) = word;
        }
      }
    }
    // ---- down-projection: 4 MMA k-steps per chunk
    if constexpr (NT > 0) {
      const uint4* lp = reinterpret_cast<const uint4*>(a.Lperm) + (int64_t(c) * NT * 32 + lane) * 2;
#pragma unroll
      for (int j = 0; j < NT; ++j) {
        const uint4 b0 = __ldg(lp + j * 64);
        const uint4 b1 = __ldg(lp + j * 64 + 1);
        const uint32_t bw[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
#pragma unroll
        for (int mt = 0; mt < MT; ++mt)
#pragma unroll
          for (int s = 0; s < 4; ++s)
            ptx::mma_bf16_16816(acc[mt][j], w[2 * mt][2 * s], w[2 * mt + 1][2 * s], w[2 * mt][2 * s + 1],
                                w[2 * mt + 1][2 * s + 1], bw[2 * s], bw[2 * s + 1]);
      }
    }
  }

  if constexpr (NT > 0) {
    const int rank = a.rank, r_pad = a.r_pad;
    const int64_t rows_pad = int64_t(gridDim.x) * ROWS;
    if (nsplit == 1) {
#pragma unroll
      for (int mt = 0; mt < MT; ++mt)
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int64_t row = row_base + 16 * mt + g + 8 * h;
          if (row >= M) continue;
          uint32_t* dst = reinterpret_cast<uint32_t*>(a.T + row * r_pad);
#pragma unroll
          for (int j = 0; j < NT; ++j)
            dst[(8 * j + 2 * t) / 2] = ptx::pack_bf16x2(acc[mt][j][2 * h] * a.inv_alpha,
                                                         acc[mt][j][2 * h + 1] * a.inv_alpha);
          for (int j = NT; j < r_pad / 8; ++j) dst[(8 * j + 2 * t) / 2] = 0u;
        }
    } else {
      float* part = a.partial + int64_t(split) * rows_pad * rank;
#pragma unroll
      for (int mt = 0; mt < MT; ++mt)
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int64_t row = row_base + 16 * mt + g + 8 * h;
#pragma unroll
          for (int j = 0; j < NT; ++j)
            *reinterpret_cast<float2*>(part + row * rank + 8 * j + 2 * t) =
                make_float2(acc[mt][j][2 * h], acc[mt][j][2 * h + 1]);
        }
      __threadfence();
      __syncthreads();
      __shared__ unsigned int s_last;
      if (threadIdx.x == 0) s_last = (atomicAdd(a.counters + tile, 1u) == unsigned(nsplit - 1));
      __syncthreads();
      if (s_last) {
        __threadfence();
#pragma unroll
        for (int mt = 0; mt < MT; ++mt)
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const int64_t row = row_base + 16 * mt + g + 8 * h;
            float sum[NT][2];
#pragma unroll
            for (int j = 0; j < NT; ++j) sum[j][0] = sum[j][1] = 0.f;
            for (int s = 0; s < nsplit; ++s) {
              const float* ps = a.partial + int64_t(s) * rows_pad * rank + row * rank + 2 * t;
#pragma unroll
              for (int j = 0; j < NT; ++j) {
                const float2 v = __ldcg(reinterpret_cast<const float2*>(ps + 8 * j));
                sum[j][0] += v.x;
                sum[j][1] += v.y;
              }
            }
            if (row >= M) continue;
            uint32_t* dst = reinterpret_cast<uint32_t*>(a.T + row * r_pad);
#pragma unroll
            for (int j = 0; j < NT; ++j)
              dst[(8 * j + 2 * t) / 2] = ptx::pack_bf16x2(sum[j][0] * a.inv_alpha, sum[j][1] * a.inv_alpha);
            for (int j = NT; j < r_pad / 8; ++j) dst[(8 * j + 2 * t) / 2] = 0u;
          }
        if (threadIdx.x == 0) a.counters[tile] = 0u;
      }
    }
  }
}

template <int NT, int MT>
int launch_t(const K1Args& a, const K1Plan& p, cudaStream_t s) {
  dim3 grid(p.row_tiles, p.nsplit);
  k1_kernel<NT, MT><<<grid, kWarps * 32, 0, s>>>(a, p.chunks_per_split, p.nsplit);
  return int(cudaGetLastError());
}

int rows_per_cta(int rank) { return rank > 64 ? kWarps * 16 : kWarps * 32; }

}  // namespace

K1Plan k1_plan(int64_t M, int64_t K, int rank, int sm_count) {
  K1Plan p;
  const int rows = rows_per_cta(rank);
  p.row_tiles = int(ceil_div(M, rows));
  const int nchunks = int(K / 64);
  const int target = 3 * sm_count;
  int nsplit = p.row_tiles > 0 ? int(ceil_div(target, p.row_tiles)) : 1;
  nsplit = nsplit < 1 ? 1 : (nsplit > nchunks ? nchunks : nsplit);
  p.chunks_per_split = int(ceil_div(nchunks, nsplit));
  p.nsplit = int(ceil_div(nchunks, p.chunks_per_split));
  return p;
}

size_t k1_partial_bytes(int64_t M, int64_t K, int rank, int sm_count) {
  if (rank == 0) return 0;
  const K1Plan p = k1_plan(M, K, rank, sm_count);
  if (p.nsplit == 1) return 0;
  return size_t(p.nsplit) * size_t(p.row_tiles) * size_t(rows_per_cta(rank)) * size_t(rank) * sizeof(float);
}

int k1_launch(const K1Args& a, const K1Plan& p, void* stream) {
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int nt = a.rank / 8;
  switch (nt) {
    case 0: return launch_t<0, 2>(a, p, s);
    case 2: return launch_t<2, 2>(a, p, s);
    case 4: return launch_t<4, 2>(a, p, s);
    case 6: return launch_t<6, 2>(a, p, s);
    case 8: return launch_t<8, 2>(a, p, s);
    case 10: return launch_t<10, 1>(a, p, s);
    case 12: return launch_t<12, 1>(a, p, s);
    case 14: return launch_t<14, 1>(a, p, s);
    case 16: return launch_t<16, 1>(a, p, s);
    default: return int(cudaErrorInvalidValue);
  }
}

}  // namespace svdq
