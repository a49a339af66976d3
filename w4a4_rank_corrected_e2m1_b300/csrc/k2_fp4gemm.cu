// Kernel 2: the "dominant 4 bit path" of SVDQuant plus the low-rank up-projection, as one
// tensor-core GEMM per 128 x 256 output tile (aiflownews article on Nunchaku, "What SVDQuant
// actually does": a compact high-precision low-rank path and a 4-bit path whose results are
// summed; Nunchaku section: the two branches share outputs).
//
//   acc  = sum_k  sX * sW * e2m1(x) * e2m1(w)      tcgen05.mma kind::mxf4nvf4, UE4M3 scales
//                                                  per 16 K (scale_vec::4X), E2M1 operands
//   acc += T' * L2                                 tcgen05.mma kind::f16 (bf16), K = rank,
//                                                  T' = X^ L1 / alpha from kernel 1
//   Y    = bf16( alpha * acc + b )                 written once, by TMA
//
// Because kernel 1 stores T already divided by alpha, both branches accumulate into one
// FP32 TMEM tile and the epilogue is a single scale-and-bias.
//
// Persistent, warp-specialised CTA (one per SM, 192 threads):
//   warp 0      TMA producer: operand tiles (128-byte swizzle) and scale blocks into a
//               3-stage shared-memory ring guarded by mbarriers
//   warp 1      TMEM owner and MMA issuer (one lane): copies the stage's scales to TMEM
//               (tcgen05.cp 32x128b.warpx4) and issues the MMAs; tcgen05.commit frees the
//               stage and, at the end of a tile, hands the accumulator to the epilogue
//   warps 2..5  epilogue: tcgen05.ld of their 32-lane quarter, alpha/bias, bf16, swizzled
//               staging and a TMA store per 32 x 64 box
// Every mbarrier wait is bounded (about two seconds); on expiry the CTA records
// SVDQ_ERR_TIMEOUT in the error word, drains what it started and exits.
#include <cuda.h>
#include <cuda_runtime.h>

#include "ptx.cuh"
#include "svdq_internal.h"

namespace svdq {

namespace {

constexpr int BM = 128, BN = 256;
constexpr int STAGES = 3;
constexpr int A_BYTES = BM * 128;                 // 128 rows x 256 fp4
constexpr int B_BYTES = BN * 128;                 // 256 rows x 256 fp4
constexpr int SFA_BYTES = 4 * 512;                // 4 k64-groups x (128 rows x 4 scales)
constexpr int SFB_BYTES = 2 * 4 * 512;            // two 128-row halves
constexpr int STAGE_BYTES = A_BYTES + B_BYTES + SFA_BYTES + SFB_BYTES;
constexpr int EPI_WARPS = 4;
constexpr int STG_BYTES = 32 * 128;               // one 32-row x 64-col bf16 box
constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + EPI_WARPS * 2 * STG_BYTES + 1024 /*bars*/ + 1024 /*align*/;
constexpr int THREADS = 64 + EPI_WARPS * 32;
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t SF_COL0 = 256;                 // scale columns: 48 per stage after the accumulator
constexpr uint32_t SF_COLS_PER_STAGE = 48;
constexpr uint64_t kTimeoutNs = 2000000000ull;

static_assert(STAGE_BYTES % 1024 == 0, "stage alignment");
static_assert(SF_COL0 + STAGES * SF_COLS_PER_STAGE <= TMEM_COLS, "TMEM budget");

// Instruction descriptors (tcgen05 instruction-descriptor bit layout):
//   [4,6) D type / B scale id  [7,10) A type  [10,13) B type  [15] A major  [16] B major
//   [17,23) N >> 3  [23] scale type (mxf4nvf4: 0 = UE4M3)  [24,29) M >> 4
constexpr uint32_t IDESC_NVFP4 = (1u << 7) | (1u << 10) | (uint32_t(BN >> 3) << 17) | (uint32_t(BM >> 4) << 24);
constexpr uint32_t IDESC_BF16 = (1u << 4) | (1u << 7) | (1u << 10) | (uint32_t(BN >> 3) << 17) | (uint32_t(BM >> 4) << 24);

struct Smem {
  uint64_t full[STAGES];
  uint64_t empty[STAGES];
  uint64_t acc_full;
  uint64_t acc_empty;
  uint64_t drain;
  uint32_t tmem_base;
  volatile int abort_flag;
};

__device__ bool wait_bounded(uint64_t* bar, uint32_t parity, Smem* s, int* err) {
  if (ptx::mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = ptx::globaltimer();
  for (uint32_t i = 1;; ++i) {
    if (ptx::mbar_try_wait(bar, parity)) return true;
    if ((i & 31u) == 0u) {
      if (s->abort_flag) return false;
      if (ptx::globaltimer() - t0 > kTimeoutNs) {
        s->abort_flag = 1;
        atomicOr(err, 1);
        return false;
      }
    }
  }
}
// Same, but ignores the abort flag: used to drain work already started.
__device__ void wait_drain(uint64_t* bar, uint32_t parity, int* err) {
  const uint64_t t0 = ptx::globaltimer();
  while (!ptx::mbar_try_wait(bar, parity)) {
    if (ptx::globaltimer() - t0 > kTimeoutNs) {
      atomicOr(err, 2);
      return;
    }
  }
}

__global__ void __launch_bounds__(THREADS, 1) k2_kernel(const __grid_constant__ K2Maps maps, K2Args a) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* base = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  unsigned char* stages = base;
  unsigned char* stg = base + STAGES * STAGE_BYTES;
  Smem* s = reinterpret_cast<Smem*>(stg + EPI_WARPS * 2 * STG_BYTES);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t M = a.M, N = a.N, K = a.K;
  const int num_m = int(ceil_div(M, BM)), num_n = int(ceil_div(N, BN));
  const int num_tiles = num_m * num_n;
  const int n_lr = a.rank > 0 ? int(ceil_div(a.rank, 64)) : 0;
  const int n_k = int(ceil_div(K, 256));
  const int iters = n_lr + n_k;
  const int64_t KG = scale_groups(K);

  if (threadIdx.x == 0) {
    for (int i = 0; i < STAGES; ++i) {
      ptx::mbar_init(&s->full[i], 1);
      ptx::mbar_init(&s->empty[i], 1);
    }
    ptx::mbar_init(&s->acc_full, 1);
    ptx::mbar_init(&s->acc_empty, EPI_WARPS);
    ptx::mbar_init(&s->drain, 1);
    s->abort_flag = 0;
    ptx::fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    ptx::prefetch_tmap(&maps.A);
    ptx::prefetch_tmap(&maps.B);
    ptx::prefetch_tmap(&maps.Y);
    if (n_lr) {
      ptx::prefetch_tmap(&maps.T);
      ptx::prefetch_tmap(&maps.L2);
    }
  }
  if (warp == 1) {
    ptx::tmem_alloc(&s->tmem_base, TMEM_COLS);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = s->tmem_base;

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      uint32_t last_parity[STAGES];
      bool used[STAGES];
      for (int i = 0; i < STAGES; ++i) used[i] = false;
      bool ok = true;
      for (int tile = blockIdx.x; tile < num_tiles && ok; tile += gridDim.x) {
        const int m0 = (tile / num_n) * BM, n0 = (tile % num_n) * BN;
        for (int it = 0; it < iters; ++it) {
          if (!wait_bounded(&s->empty[stage], phase ^ 1u, s, a.err)) { ok = false; break; }
          unsigned char* st = stages + stage * STAGE_BYTES;
          uint64_t* fb = &s->full[stage];
          if (it < n_lr) {
            ptx::mbar_arrive_expect_tx(fb, A_BYTES + B_BYTES);
            ptx::tma_load_2d(st, &maps.T, fb, 64 * it, m0);
            ptx::tma_load_2d(st + A_BYTES, &maps.L2, fb, 64 * it, n0);
          } else {
            const int kq = it - n_lr;
            ptx::mbar_arrive_expect_tx(fb, STAGE_BYTES);
            ptx::tma_load_2d(st, &maps.A, fb, 128 * kq, m0);
            ptx::tma_load_2d(st + A_BYTES, &maps.B, fb, 128 * kq, n0);
            ptx::bulk_load(st + A_BYTES + B_BYTES, a.sfa + ((int64_t(m0) / 128) * KG + 4 * kq) * 512, SFA_BYTES, fb);
            unsigned char* sfb = st + A_BYTES + B_BYTES + SFA_BYTES;
            ptx::bulk_load(sfb, a.sfb + ((int64_t(n0) / 128) * KG + 4 * kq) * 512, SFA_BYTES, fb);
            ptx::bulk_load(sfb + SFA_BYTES, a.sfb + ((int64_t(n0) / 128 + 1) * KG + 4 * kq) * 512, SFA_BYTES, fb);
          }
          used[stage] = true;
          last_parity[stage] = phase;
          if (++stage == STAGES) { stage = 0; phase ^= 1u; }
        }
      }
      // every copy this CTA started has landed before shared memory is released
      for (int i = 0; i < STAGES; ++i)
        if (used[i]) wait_drain(&s->full[i], last_parity[i], a.err);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      int local = 0;
      for (int tile = blockIdx.x; tile < num_tiles && ok; tile += gridDim.x, ++local) {
        if (!wait_bounded(&s->acc_empty, (uint32_t(local) & 1u) ^ 1u, s, a.err)) break;
        ptx::tc_fence_after();
        uint32_t accumulate = 0;
        for (int it = 0; it < iters; ++it) {
          if (!wait_bounded(&s->full[stage], phase, s, a.err)) { ok = false; break; }
          ptx::tc_fence_after();
          const uint32_t a_s = ptx::smem_u32(stages + stage * STAGE_BYTES);
          const uint32_t b_s = a_s + A_BYTES;
          if (it < n_lr) {
            const int ksteps = min(4, (a.rank - 64 * it) / 16);
            for (int kk = 0; kk < ksteps; ++kk) {
              ptx::mma_bf16(tmem, ptx::desc_sw128(a_s + 32 * kk), ptx::desc_sw128(b_s + 32 * kk), IDESC_BF16,
                            accumulate);
              accumulate = 1;
            }
          } else {
            const int kq = it - n_lr;
            const int64_t krem = (K - 256 * int64_t(kq)) / 64;
            const int ksteps = krem < 4 ? int(krem) : 4;
            const uint32_t sfa_s = b_s + B_BYTES, sfb_s = sfa_s + SFA_BYTES;
            const uint32_t sfa_t = tmem + SF_COL0 + stage * SF_COLS_PER_STAGE;
            const uint32_t sfb_t = sfa_t + 16;
            for (int kk = 0; kk < ksteps; ++kk) {
              ptx::tmem_cp_32x128b_warpx4(sfa_t + 4 * kk, ptx::desc_sf(sfa_s + 512 * kk));
              ptx::tmem_cp_32x128b_warpx4(sfb_t + 8 * kk, ptx::desc_sf(sfb_s + 512 * kk));
              ptx::tmem_cp_32x128b_warpx4(sfb_t + 8 * kk + 4, ptx::desc_sf(sfb_s + 2048 + 512 * kk));
            }
            for (int kk = 0; kk < ksteps; ++kk) {
              ptx::mma_nvfp4(tmem, ptx::desc_sw128(a_s + 32 * kk), ptx::desc_sw128(b_s + 32 * kk), IDESC_NVFP4,
                             sfa_t + 4 * kk, sfb_t + 8 * kk, accumulate);
              accumulate = 1;
            }
          }
          ptx::tc_commit(&s->empty[stage]);
          if (++stage == STAGES) { stage = 0; phase ^= 1u; }
        }
        if (!ok) break;
        ptx::tc_commit(&s->acc_full);
      }
      // all MMAs this thread issued have finished before TMEM is released
      ptx::tc_commit(&s->drain);
      wait_drain(&s->drain, 0, a.err);
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;                        // TMEM lane quarter this warp may access
    unsigned char* my_stg = stg + (warp - 2) * 2 * STG_BYTES;
    int local = 0, buf = 0;
    for (int tile = blockIdx.x; tile < num_tiles; tile += gridDim.x, ++local) {
      const int m0 = (tile / num_n) * BM, n0 = (tile % num_n) * BN;
      if (!wait_bounded(&s->acc_full, uint32_t(local) & 1u, s, a.err)) break;
      ptx::tc_fence_after();
      for (int c = 0; c < BN / 64; ++c) {
        uint32_t r[64];
        const uint32_t taddr = tmem + (uint32_t(32 * q) << 16) + uint32_t(64 * c);
        ptx::tmem_ld_32x32b_x32(taddr, r);
        ptx::tmem_ld_32x32b_x32(taddr + 32, r + 32);
        ptx::tmem_wait_ld();
        if (c == BN / 64 - 1) {
          ptx::tc_fence_before();
          __syncwarp();
          if (lane == 0) ptx::mbar_arrive(&s->acc_empty);
        }
        const int64_t ncol = int64_t(n0) + 64 * c;
        if (ncol >= N) continue;
        uint32_t outw[32];
#pragma unroll
        for (int v = 0; v < 8; ++v) {
          uint4 bb = make_uint4(0, 0, 0, 0);
          if (ncol + 8 * v < N) bb = __ldg(reinterpret_cast<const uint4*>(a.bias + ncol + 8 * v));
          const uint32_t bw[4] = {bb.x, bb.y, bb.z, bb.w};
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const float b0 = __uint_as_float(bw[u] << 16), b1 = __uint_as_float(bw[u] & 0xFFFF0000u);
            const float y0 = fmaf(a.alpha, __uint_as_float(r[8 * v + 2 * u]), b0);
            const float y1 = fmaf(a.alpha, __uint_as_float(r[8 * v + 2 * u + 1]), b1);
            outw[4 * v + u] = ptx::pack_bf16x2(y0, y1);
          }
        }
        unsigned char* sb = my_stg + buf * STG_BYTES;
        if (lane == 0) ptx::bulk_wait_read<1>();
        __syncwarp();
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          uint4* dst = reinterpret_cast<uint4*>(sb + lane * 128 + ((j ^ (lane & 7)) << 4));
          *dst = make_uint4(outw[4 * j], outw[4 * j + 1], outw[4 * j + 2], outw[4 * j + 3]);
        }
        ptx::fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          ptx::tma_store_2d(&maps.Y, sb, int(ncol), m0 + 32 * q);
          ptx::bulk_commit();
        }
        buf ^= 1;
      }
    }
    if (lane == 0) ptx::bulk_wait<0>();
    __syncwarp();
  }

  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, TMEM_COLS);
  }
}

}  // namespace

size_t k2_smem_bytes() { return SMEM_BYTES; }

int k2_launch(const K2Maps& maps, const K2Args& a, int sm_count, void* stream) {
  static bool attr_done = false;
  if (!attr_done) {
    cudaError_t e = cudaFuncSetAttribute(k2_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
    if (e != cudaSuccess) return int(e);
    attr_done = true;
  }
  const int64_t tiles = ceil_div(a.M, BM) * ceil_div(a.N, BN);
  const int grid = int(tiles < sm_count ? tiles : sm_count);
  if (grid == 0) return 0;
  k2_kernel<<<grid, THREADS, SMEM_BYTES, static_cast<cudaStream_t>(stream)>>>(maps, a);
  return int(cudaGetLastError());
}

}  // namespace svdq
