// AWQ-style W4A16 linear layer for the modulation / adaptive-normalisation shapes (a few rows
// of activations against a wide weight): Y = x' W'^T + b with x' = fl32(x * fl32(1 / s_c)) and
// W' dequantised from asymmetric 4-bit codes in groups of 64 input channels,
// w' = (q - z) * sc.  The pages keep these layers at 16-bit activations with AWQ-style 4-bit
// weights (aiflownews article on Nunchaku, "How Nunchaku four bit quantization actually
// works").
//
// The work is one pass over the packed weights (HBM-bound: 0.5 byte per weight plus 8 bytes
// per group of 64), streamed by one block per SM: a producer warp moves the block's
// contiguous run of weight rows (codes, then the rows' (scale, zero point) pairs) through a
// shared-memory ring with bulk copies, and sixteen warps consume it (two weight rows each per
// stage where three stages of that size fit: two independent chains per warp, one read of x'
// for both), keeping the ALU cost per weight small:
//   * the block's rows of x' sit in shared memory in fp16, 32-channel segments padded to 80
//     bytes so that a warp's 16-byte reads are conflict-free;
//   * a lane takes 16 bytes of codes (32 weights, half a group) at a time; LOP3s turn two codes
//     into the fp16 pair (1024 + q) (or (1024 + 16 q) for the odd nibbles, which need no
//     shift), one HSUB2 subtracts (1024 + z) or (1024 + 16 z) (exact: the differences are small
//     integers), and HFMA2 multiplies by the paired x' values;
//   * two 16-byte words' products (eight per half) are summed in fp16 and added into a float32
//     total, which the group scale multiplies once per 32 weights;
//   * the warp reduces its lanes with shuffles and writes bf16(acc + b).
// fp16 keeps 11 bits of the products; longer sums are float32.  A half2 lane sums four products
// x' (q - z) with |q - z| <= 15, so a row of x' whose largest magnitude exceeds 512 is first
// scaled by an exact power of two 2^-s (s chosen per row from that magnitude) and its sums
// multiplied back by 2^s: every fp16 sum then stays below 4 * 512 * 15 = 30720 < 65504, for any
// input, and rows within 512 (s = 0) are computed exactly as without the scaling.
// Every wait is bounded (about two seconds; on expiry the error word is set and the block
// returns).
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "ptx.cuh"
#include "svdq_internal.h"

namespace svdq {

namespace {

constexpr int kThreads = 512;              // compute warps (a producer warp comes on top)
constexpr int kWarps = kThreads / 32;

// x' is kept in fp16 in shared memory, one 80-byte slot per 32-channel segment (64 bytes of
// data, 16 of padding so that the four 16-byte reads of a warp quarter hit distinct banks).
// Inside a segment, word u (channels 8u .. 8u + 7) holds the pairs (8u + p, 8u + p + 4),
// p = 0..3, matching the order in which one LOP3 pulls two codes out of a 32-bit word.
constexpr int kSegBytes = 80;
__host__ __device__ constexpr int64_t xs_bytes_per_row(int64_t K) { return (K / 32) * kSegBytes; }


constexpr uint64_t kTimeoutNs = 2000000000ull;

// Bounded mbarrier wait: about two seconds, then the block gives up (flag + error word).
__device__ bool bounded_wait(uint64_t* bar, uint32_t parity, volatile int* abort_flag) {
  if (ptx::mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = ptx::globaltimer();
  for (uint32_t i = 1;; ++i) {
    if (ptx::mbar_try_wait(bar, parity)) return true;
    if ((i & 31u) == 0u) {
      if (*abort_flag) return false;
      if (ptx::globaltimer() - t0 > kTimeoutNs) {
        *abort_flag = 1;
        return false;
      }
    }
  }
}

// Two codes of a 32-bit word as fp16 (1024 + q): nibbles at bits 4p and 4p + 16 go into the
// low and high mantissas of the exponent of 1024 (one LOP3 after the shift).
template <int P>
__device__ __forceinline__ __half2 codes_pair(uint32_t w) {
  uint32_t v = (w >> (4 * P)) & 0x000F000Fu;
  v |= 0x64006400u;
  return *reinterpret_cast<__half2*>(&v);
}

// Rows per stage and ring depth for a K (codes 0.5 B and scale/zero pairs 8 B / 64 per weight)
struct AwqPlan {
  int rs, stages, mb;
  size_t stage_bytes, xs_bytes, smem;
};

__host__ __device__ constexpr int64_t stage_rows_for(int64_t K) {
  return K <= 3072 ? 32 : (K <= 6144 ? 16 : (K <= 12288 ? 8 : 4));   // two rows a warp where three stages still fit
}

__device__ __forceinline__ unsigned char* xs_row(unsigned char* xs, int m, int64_t K) {
  return xs + size_t(m) * xs_bytes_per_row(K);
}

template <int MB>
__global__ void __launch_bounds__(kThreads + 32, 1) awq_gemv_kernel(AwqArgs a, int64_t m0, int rs, int stages,
                                                                   int stage_bytes) {
  extern __shared__ __align__(128) unsigned char smem_raw[];
  __shared__ uint64_t full[8], empty[8];
  __shared__ volatile int abort_flag;
  __shared__ unsigned int row_max_bits[MB];
  const int64_t K = a.K, N = a.N;
  const int nseg = int(K / 32);
  const int64_t KG = K / 64;
  unsigned char* xs = smem_raw;                                     // [MB] rows of x' (fp16, paired segments)
  unsigned char* ring = smem_raw + ((size_t(MB) * xs_bytes_per_row(K) + 127) / 128) * 128;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int codes_row = int(K / 2), sz_row = int(KG * 8);

  // rows [r_begin, r_end) of this block: a contiguous run of the packed weights
  const int64_t per_block = ((N + gridDim.x - 1) / gridDim.x + rs - 1) / rs * rs;
  const int64_t r_begin = int64_t(blockIdx.x) * per_block;
  const int64_t r_end = r_begin + per_block < N ? r_begin + per_block : N;
  const int nst = r_begin < r_end ? int((r_end - r_begin + rs - 1) / rs) : 0;

  if (threadIdx.x == 0) {
    for (int i = 0; i < stages; ++i) {
      ptx::mbar_init(&full[i], 1);
      ptx::mbar_init(&empty[i], kWarps);
    }
    for (int m = 0; m < MB; ++m) row_max_bits[m] = 0u;
    abort_flag = 0;
    ptx::fence_barrier_init();
  }
  __syncthreads();

  if (warp == kWarps) {
    // ------------------------------------------------------------ producer (bulk copies)
    if (lane == 0) {
      int stage = 0, issued = 0;
      uint32_t phase = 0;
      for (int j = 0; j < nst; ++j, ++issued) {
        if (j >= stages) {
          if (!bounded_wait(&empty[stage], phase ^ 1u, &abort_flag)) break;
          ptx::fence_proxy_async_smem();   // the compute warps' ordinary loads before the refill
        }
        const int64_t row = r_begin + int64_t(j) * rs;
        const int nrows = int(r_end - row < rs ? r_end - row : rs);
        unsigned char* st = ring + size_t(stage) * stage_bytes;
        // the pair copy is rounded up to 16 bytes (the device array carries 16 bytes of padding)
        const uint32_t cb = uint32_t(nrows * codes_row), zb = (uint32_t(nrows * sz_row) + 15u) & ~15u;
        ptx::mbar_arrive_expect_tx(&full[stage], cb + zb);
        ptx::bulk_load(st, a.codes + row * codes_row, cb, &full[stage]);
        ptx::bulk_load(st + size_t(rs) * codes_row, reinterpret_cast<const unsigned char*>(a.sz) + row * sz_row, zb,
                       &full[stage]);
        if (++stage == stages) { stage = 0; phase ^= 1u; }
      }
      for (int i = 0; i < stages; ++i) {       // every copy issued has landed, also after an abort
        const int used = issued - i;
        if (used <= 0) continue;
        const uint64_t t0 = ptx::globaltimer();
        while (!ptx::mbar_try_wait(&full[i], uint32_t(((used - 1) / stages) & 1)))
          if (ptx::globaltimer() - t0 > kTimeoutNs) break;
      }
    }
  } else {
    // ------------------------------------------------------------ compute warps
    // largest |x'| of each row, then the row's power-of-two scaling 2^-shift[m] (see the header)
    {
      float mx[MB];
#pragma unroll
      for (int m = 0; m < MB; ++m) mx[m] = 0.f;
      for (int64_t k8 = threadIdx.x; k8 < K / 8; k8 += kThreads) {
        const int64_t k = 8 * k8;
        const float4 i0 = *reinterpret_cast<const float4*>(a.inv_s + k);
        const float4 i1 = *reinterpret_cast<const float4*>(a.inv_s + k + 4);
        const float inv[8] = {i0.x, i0.y, i0.z, i0.w, i1.x, i1.y, i1.z, i1.w};
#pragma unroll
        for (int m = 0; m < MB; ++m) {
          if (m0 + m >= a.M) continue;
          const uint4 xr = *reinterpret_cast<const uint4*>(a.X + (m0 + m) * K + k);
          const uint32_t xw[4] = {xr.x, xr.y, xr.z, xr.w};
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            const uint32_t bits = (e & 1) ? (xw[e >> 1] & 0xFFFF0000u) : (xw[e >> 1] << 16);
            mx[m] = fmaxf(mx[m], fabsf(__fmul_rn(__uint_as_float(bits), inv[e])));
          }
        }
      }
#pragma unroll
      for (int m = 0; m < MB; ++m) {
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) mx[m] = fmaxf(mx[m], __shfl_xor_sync(0xFFFFFFFFu, mx[m], o));
        if (lane == 0) atomicMax(&row_max_bits[m], __float_as_uint(mx[m]));   // non-negative: bit order = value order
      }
    }
    asm volatile("bar.sync 1, %0;" ::"r"(kThreads));
    float row_down[MB], row_up[MB];
#pragma unroll
    for (int m = 0; m < MB; ++m) {
      // smallest shift with max * 2^-shift <= 512: shift = max(0, floor(log2 max) - 8)
      const int ex = int((row_max_bits[m] >> 23) & 0xFFu) - 127;
      const int shift = ex > 8 ? (ex - 8 < 120 ? ex - 8 : 120) : 0;
      row_down[m] = __uint_as_float(uint32_t(127 - shift) << 23);   // 2^-shift
      row_up[m] = __uint_as_float(uint32_t(127 + shift) << 23);     // 2^shift
    }
    // x' = fl32(x * fl32(1 / s)) (times 2^-shift) rounded to fp16, in the paired segment order:
    // a thread takes 8 channels (one 16-byte load of X) and writes them as one 16-byte word of
    // a segment
    for (int64_t k8 = threadIdx.x; k8 < K / 8; k8 += kThreads) {
      const int64_t k = 8 * k8;
      const float4 i0 = *reinterpret_cast<const float4*>(a.inv_s + k);
      const float4 i1 = *reinterpret_cast<const float4*>(a.inv_s + k + 4);
      const float inv[8] = {i0.x, i0.y, i0.z, i0.w, i1.x, i1.y, i1.z, i1.w};
      uint4 xr[MB];
#pragma unroll
      for (int m = 0; m < MB; ++m)
        xr[m] = m0 + m < a.M ? *reinterpret_cast<const uint4*>(a.X + (m0 + m) * K + k) : make_uint4(0, 0, 0, 0);
      const int64_t sgi = k >> 5;
      const int u = int(k & 31) >> 3;
#pragma unroll
      for (int m = 0; m < MB; ++m) {
        const uint32_t xw[4] = {xr[m].x, xr[m].y, xr[m].z, xr[m].w};
        float v[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const uint32_t bits = (e & 1) ? (xw[e >> 1] & 0xFFFF0000u) : (xw[e >> 1] << 16);
          v[e] = __fmul_rn(__fmul_rn(__uint_as_float(bits), inv[e]), row_down[m]);
        }
        // pairs (e, e + 4), e = 0..3; the odd pairs meet codes read as 16 q, so they are stored
        // divided by 16 (exact power-of-two scaling) to keep every product x' (q - z)
        uint4 out;
        __half2 h;
        h = __floats2half2_rn(v[0], v[4]); out.x = *reinterpret_cast<uint32_t*>(&h);
        h = __floats2half2_rn(0.0625f * v[1], 0.0625f * v[5]); out.y = *reinterpret_cast<uint32_t*>(&h);
        h = __floats2half2_rn(v[2], v[6]); out.z = *reinterpret_cast<uint32_t*>(&h);
        h = __floats2half2_rn(0.0625f * v[3], 0.0625f * v[7]); out.w = *reinterpret_cast<uint32_t*>(&h);
        *reinterpret_cast<uint4*>(xs_row(xs, m, K) + sgi * kSegBytes + u * 16) = out;
      }
    }
    asm volatile("bar.sync 1, %0;" ::"r"(kThreads));

    int stage = 0;
    uint32_t phase = 0;
    for (int j = 0; j < nst; ++j) {
      if (!bounded_wait(&full[stage], phase, &abort_flag)) break;
      const unsigned char* st = ring + size_t(stage) * stage_bytes;
      const int64_t row0 = r_begin + int64_t(j) * rs;
      // two weight rows per warp at a time (rr and rr + kWarps): two independent chains, and each
      // x' read from shared memory serves both
      for (int rr = warp; rr < rs; rr += 2 * kWarps) {
        const int64_t n0 = row0 + rr;
        if (n0 >= r_end) break;
        const bool two = rr + kWarps < rs && n0 + kWarps < r_end;
        const int rb = two ? rr + kWarps : rr;     // the second row (the first again when absent)
        uint32_t crow[2], szrow[2];
        crow[0] = ptx::smem_u32(st + size_t(rr) * codes_row);
        crow[1] = ptx::smem_u32(st + size_t(rb) * codes_row);
        szrow[0] = ptx::smem_u32(st + size_t(rs) * codes_row + size_t(rr) * sz_row);
        szrow[1] = ptx::smem_u32(st + size_t(rs) * codes_row + size_t(rb) * sz_row);
        float part[2][MB];
#pragma unroll
        for (int h = 0; h < 2; ++h)
#pragma unroll
          for (int m = 0; m < MB; ++m) part[h][m] = 0.f;
        // three 32-weight chunks per lane at a time (K = 3072 in one pass), all loaded first
        constexpr int kU = 3;
        for (int sg0 = lane; sg0 < nseg; sg0 += 32 * kU) {
          uint4 c[2][kU];
          float2 sz[2][kU];
#pragma unroll
          for (int i = 0; i < kU; ++i) {
            const int sgi = sg0 + 32 * i;
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              if (sgi < nseg) {
                c[h][i] = ptx::lds_v4(crow[h] + uint32_t(sgi) * 16u);
                sz[h][i] = ptx::lds_f32x2(szrow[h] + uint32_t(sgi >> 1) * 8u);    // scale, zero point
              } else {
                c[h][i] = make_uint4(0x64646464u, 0x64646464u, 0x64646464u, 0x64646464u);
                sz[h][i] = make_float2(0.f, 0.f);
              }
            }
          }
#pragma unroll
          for (int i = 0; i < kU; ++i) {
            const int sgi = sg0 + 32 * i;
            // codes 8u + p (low half) and 8u + p + 4 (high half): for p = 0, 2 as fp16 (1024 + q),
            // for p = 1, 3 straight from bits 4..7 as (1024 + 16 q) (exact: multiples of 16 below
            // 1024); subtracting (1024 + z), resp. (1024 + 16 z), leaves q - z, resp. 16 (q - z)
            __half2 qz[2][4][4];
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              const __half2 zz = __float2half2_rn(1024.f + sz[h][i].y);
              const __half2 zz16 = __float2half2_rn(1024.f + 16.f * sz[h][i].y);
              const uint32_t cw[4] = {c[h][i].x, c[h][i].y, c[h][i].z, c[h][i].w};
#pragma unroll
              for (int u = 0; u < 4; ++u) {
                const uint32_t w = cw[u], w8 = cw[u] >> 8;
                uint32_t v0 = (w & 0x000F000Fu) | 0x64006400u, v1 = (w & 0x00F000F0u) | 0x64006400u;
                uint32_t v2 = (w8 & 0x000F000Fu) | 0x64006400u, v3 = (w8 & 0x00F000F0u) | 0x64006400u;
                qz[h][u][0] = __hsub2(*reinterpret_cast<__half2*>(&v0), zz);
                qz[h][u][1] = __hsub2(*reinterpret_cast<__half2*>(&v1), zz16);
                qz[h][u][2] = __hsub2(*reinterpret_cast<__half2*>(&v2), zz);
                qz[h][u][3] = __hsub2(*reinterpret_cast<__half2*>(&v3), zz16);
              }
            }
#pragma unroll
            for (int m = 0; m < MB; ++m) {
              const uint32_t xp = ptx::smem_u32(xs_row(xs, m, K)) + uint32_t(sgi < nseg ? sgi : 0) * kSegBytes;
              // products of pairs 0, 2 and of pairs 1, 3 in two fp16 sums per two words (eight
              // products per half), then float32
              float t[2] = {0.f, 0.f};
#pragma unroll
              for (int uu = 0; uu < 4; uu += 2) {
                const uint4 xa = ptx::lds_v4(xp + 16u * uu), xb = ptx::lds_v4(xp + 16u * (uu + 1));
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                  __half2 e = __hmul2(*reinterpret_cast<const __half2*>(&xa.x), qz[h][uu][0]);
                  e = __hfma2(*reinterpret_cast<const __half2*>(&xa.z), qz[h][uu][2], e);
                  e = __hfma2(*reinterpret_cast<const __half2*>(&xb.x), qz[h][uu + 1][0], e);
                  e = __hfma2(*reinterpret_cast<const __half2*>(&xb.z), qz[h][uu + 1][2], e);
                  __half2 o = __hmul2(*reinterpret_cast<const __half2*>(&xa.y), qz[h][uu][1]);
                  o = __hfma2(*reinterpret_cast<const __half2*>(&xa.w), qz[h][uu][3], o);
                  o = __hfma2(*reinterpret_cast<const __half2*>(&xb.y), qz[h][uu + 1][1], o);
                  o = __hfma2(*reinterpret_cast<const __half2*>(&xb.w), qz[h][uu + 1][3], o);
                  const float2 fe = __half22float2(e), fo = __half22float2(o);
                  t[h] += (fe.x + fe.y) + (fo.x + fo.y);
                }
              }
#pragma unroll
              for (int h = 0; h < 2; ++h) part[h][m] = fmaf(sz[h][i].x, t[h], part[h][m]);   // sum x' (q - z) * sc
            }
          }
        }
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          if (h == 1 && !two) break;
          const int64_t n = n0 + h * kWarps;
#pragma unroll
          for (int m = 0; m < MB; ++m) {
            float v = part[h][m];
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
            if (lane == 0 && m0 + m < a.M) {
              const float b = __uint_as_float(uint32_t(a.bias[n]) << 16);
              a.Y[(m0 + m) * N + n] = uint16_t(ptx::pack_bf16x2(fmaf(v, row_up[m], b), 0.f) & 0xFFFFu);
            }
          }
        }
      }
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(&empty[stage]);
      if (++stage == stages) { stage = 0; phase ^= 1u; }
    }
  }
  if (abort_flag && threadIdx.x == 0) atomicOr(a.err, 16);
}

AwqPlan awq_plan(int64_t K, int64_t M) {
  AwqPlan p{};
  p.rs = int(stage_rows_for(K));
  p.stage_bytes = ((size_t(p.rs) * (K / 2 + (K / 64) * 8)) + 16 + 127) / 128 * 128;
  p.mb = M >= 8 ? 8 : (M >= 4 ? 4 : (M >= 2 ? 2 : 1));
  for (;; p.mb >>= 1) {
    p.xs_bytes = (size_t(p.mb) * xs_bytes_per_row(K) + 127) / 128 * 128;
    const size_t room = size_t(210) * 1024 > p.xs_bytes ? size_t(210) * 1024 - p.xs_bytes : 0;
    p.stages = int(room / p.stage_bytes);
    if (p.stages > 8) p.stages = 8;
    if (p.stages >= 3 || p.mb == 1) break;
  }
  p.smem = p.xs_bytes + size_t(p.stages) * p.stage_bytes;
  return p;
}

template <int MB>
int launch_mb(const AwqArgs& a, const AwqPlan& p, int sm_count, cudaStream_t s) {
  static int attr_done[64] = {0};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 64 && !attr_done[dev]) {
    cudaError_t e = cudaFuncSetAttribute(awq_gemv_kernel<MB>, cudaFuncAttributeMaxDynamicSharedMemorySize, 220 * 1024);
    if (e != cudaSuccess) return int(e);
    attr_done[dev] = 1;
  }
  // one block per SM, each streaming a contiguous run of rows
  const int64_t blocks = sm_count < a.N ? sm_count : a.N;
  for (int64_t m0 = 0; m0 < a.M; m0 += MB) {
    awq_gemv_kernel<MB><<<unsigned(blocks), kThreads + 32, p.smem, s>>>(a, m0, p.rs, p.stages, int(p.stage_bytes));
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return int(e);
  }
  return 0;
}

}  // namespace

int awq_launch(const AwqArgs& a, int sm_count, void* stream) {
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const AwqPlan p = awq_plan(a.K, a.M);
  if (p.stages < 2) return int(cudaErrorInvalidValue);
  switch (p.mb) {
    case 8: return launch_mb<8>(a, p, sm_count, s);
    case 4: return launch_mb<4>(a, p, sm_count, s);
    case 2: return launch_mb<2>(a, p, sm_count, s);
    default: return launch_mb<1>(a, p, sm_count, s);
  }
}

}  // namespace svdq
