// Kernel 2: the 4-bit branch of SVDQuant, which carries most of the arithmetic, plus the
// low-rank up-projection, as one tensor-core GEMM per 256 x 256 output tile.  The layer's
// output is the sum of the two branches (aiflownews article on Nunchaku, "What SVDQuant
// actually does"), and the Nunchaku section fuses them so the output is written once.
//
//   acc  = sum_k  sX * sW * e2m1(x) * e2m1(w)      tcgen05.mma kind::mxf4nvf4, UE4M3 scales
//                                                  per 16 K (scale_vec::4X), E2M1 operands
//   acc += T' * L2                                 tcgen05.mma kind::f16 (bf16), K = rank,
//                                                  T' = X^ L1 / alpha from kernel 1
//   Y    = bf16( alpha * acc + b )                 written once, by TMA
//
// Because kernel 1 stores T already divided by alpha, both branches accumulate into one FP32
// TMEM tile and the epilogue is a single scale-and-bias.
//
// Each tile is computed by a CTA pair (cluster of 2, tcgen05 cta_group::2): CTA r of the pair
// owns rows m0 + 128 r .. +127 of the tile and holds them (A) plus half of the tile's 256
// weight rows (B, rows n0 + 128 r ..) in shared memory; the pair's tensor cores exchange the
// B halves, so each SM streams 8 KB instead of 12 KB per 64-wide K step.  The even CTA issues
// every MMA for the pair.
//
// Block scales reach TMEM through tcgen05.st by four "scale warps" per CTA instead of
// tcgen05.cp.  For the activation scales the MMA reads the four scales of row m from TMEM lane
// m, column base + m / 32 (base a multiple of 4), so each warp writes, for its 32-lane
// quarter, the one word per row and K step that the MMA reads.  The weight scales are read by
// every lane quarter for all 256 weight rows (column base + 4 h + j, lane i: row 128 h + 32 j
// + i), so each warp copies the whole block into its quarter.  Copies through tcgen05.cp
// occupied the tensor pipe between MMAs; the stores run on the warps' own datapath.
//
// Persistent, warp-specialised CTA (one per SM, 448 threads):
//   warp 0       TMA producer: A, B, scale tiles into a 5-stage ring (local "full" barrier)
//   warp 1       TMEM owner; in the even CTA lane 0 issues the MMAs for the pair once the
//                stage is "ready" in both CTAs; tcgen05.commit (multicast to both CTAs) frees
//                each stage and hands the accumulator to both epilogues
//   warps 2..5   scale warps: per stage, wait for the local loads, write the stage's scales
//                to TMEM, then arrive on the even CTA's "ready" barrier (8 arrivals per stage)
//   warps 6..13  epilogue: each warp drains 32 lanes x 128 columns of the accumulator (two
//                64-column halves), releases it to the MMA warp, applies alpha and the bias,
//                converts to bf16 and writes Y through swizzled staging and TMA stores
// Every mbarrier wait is bounded (about two seconds); on expiry the CTA records
// SVDQ_ERR_TIMEOUT in the error word, drains what it started and exits.
#include <cuda.h>
#include <cuda_runtime.h>

#include "ptx.cuh"
#include "svdq_internal.h"

namespace svdq {

namespace {

constexpr int BM = 128;                            // rows per CTA (pair tile: 256)
constexpr int BN = 256;                            // columns per pair tile
constexpr int STAGES = 5;
constexpr int A_BYTES = BM * 128;                  // 128 rows x 256 fp4
constexpr int B_BYTES = (BN / 2) * 128;            // this CTA's 128 weight rows x 256 fp4
constexpr int SFA_BYTES = 4 * 512;                 // 4 k64-groups x (128 rows x 4 scales)
constexpr int SFB_BYTES = 2 * 4 * 512;             // both 128-row halves of the tile's weights
constexpr int STAGE_BYTES = A_BYTES + B_BYTES + SFA_BYTES + SFB_BYTES;
constexpr int SCALE_WARP0 = 2;
constexpr int EPI_WARP0 = 6;
constexpr int EPI_WARPS = 8;
constexpr int STG_BYTES = 32 * 128;                // one 32-row x 64-col bf16 box per warp
constexpr int BIAS_BYTES = 128 * 2;                // per warp: its 128 columns of bias
constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + EPI_WARPS * (STG_BYTES + BIAS_BYTES) + 1024 + 1024;
constexpr int THREADS = 32 * (EPI_WARP0 + EPI_WARPS);
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t SF_COL0 = 256;                  // scale columns after the accumulator
constexpr uint32_t SF_COLS_PER_STAGE = 48;         // A: 4 k-steps x 4, B: 4 k-steps x 8
constexpr uint64_t kTimeoutNs = 2000000000ull;
constexpr uint16_t kPairMask = 0x3;

static_assert(STAGE_BYTES % 1024 == 0, "stage alignment");
static_assert(SF_COL0 + STAGES * SF_COLS_PER_STAGE <= TMEM_COLS, "TMEM budget");
static_assert(SMEM_BYTES <= 232448, "shared memory budget");

// Instruction descriptors (tcgen05 instruction-descriptor bit layout):
//   [4,6) D type / B scale id  [7,10) A type  [10,13) B type  [15] A major  [16] B major
//   [17,23) N >> 3  [23] scale type (mxf4nvf4: 0 = UE4M3)  [24,29) M >> 4
// The pair computes M = 256 (128 per CTA).
constexpr uint32_t IDESC_NVFP4 = (1u << 7) | (1u << 10) | (uint32_t(BN >> 3) << 17) | (uint32_t(256 >> 4) << 24);
constexpr uint32_t IDESC_BF16 =
    (1u << 4) | (1u << 7) | (1u << 10) | (uint32_t(BN >> 3) << 17) | (uint32_t(256 >> 4) << 24);

struct Smem {
  uint64_t full[STAGES];     // this CTA's loads of a stage landed (producer arrive + bytes)
  uint64_t empty[STAGES];    // this CTA's stage may be refilled (MMA commit, multicast)
  uint64_t ready[STAGES];    // even CTA: both CTAs' stage landed and its scales are in TMEM
  uint64_t acc_full;         // accumulator ready for this CTA's epilogue (MMA commit, multicast)
  uint64_t acc_empty;        // even CTA: both epilogues drained the accumulator (16 warps)
  uint64_t drain;            // even CTA: every MMA issued has completed
  uint64_t never;            // arrived at by nothing (the failure-detection stall waits on it)
  uint32_t tmem_base;
  volatile int abort_flag;
};

__device__ bool wait_bounded(uint64_t* bar, uint32_t parity, Smem* s, int* err, uint64_t limit_ns) {
  if (ptx::mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = ptx::globaltimer();
  for (uint32_t i = 1;; ++i) {
    if (ptx::mbar_try_wait(bar, parity)) return true;
    if ((i & 31u) == 0u) {
      if (s->abort_flag) return false;
      if (ptx::globaltimer() - t0 > limit_ns) {
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

// alpha * acc + bias -> 32 packed bf16 pairs for 64 columns
__device__ __forceinline__ void convert64(const uint32_t* r, const uint16_t* bias, float alpha, uint32_t* out) {
#pragma unroll
  for (int v = 0; v < 8; ++v) {
    const uint4 bb = *reinterpret_cast<const uint4*>(bias + 8 * v);
    const uint32_t bw[4] = {bb.x, bb.y, bb.z, bb.w};
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const float b0 = __uint_as_float(bw[u] << 16), b1 = __uint_as_float(bw[u] & 0xFFFF0000u);
      const float y0 = fmaf(alpha, __uint_as_float(r[8 * v + 2 * u]), b0);
      const float y1 = fmaf(alpha, __uint_as_float(r[8 * v + 2 * u + 1]), b1);
      out[4 * v + u] = ptx::pack_bf16x2(y0, y1);
    }
  }
}

__device__ __forceinline__ void store64(const void* map, unsigned char* stg, const uint32_t* w, int lane, int x,
                                        int y) {
  if (lane == 0) ptx::bulk_wait_read<0>();
  __syncwarp();
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    uint4* dst = reinterpret_cast<uint4*>(stg + lane * 128 + ((j ^ (lane & 7)) << 4));
    *dst = make_uint4(w[4 * j], w[4 * j + 1], w[4 * j + 2], w[4 * j + 3]);
  }
  ptx::fence_proxy_async_smem();
  __syncwarp();
  if (lane == 0) {
    ptx::tma_store_2d(map, stg, x, y);
    ptx::bulk_commit();
  }
}

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(THREADS, 1)
    k2_kernel(const __grid_constant__ K2Maps maps, K2Args a) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* base = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  unsigned char* stages = base;
  unsigned char* stg = base + STAGES * STAGE_BYTES;
  unsigned char* bias_s = stg + EPI_WARPS * STG_BYTES;
  Smem* s = reinterpret_cast<Smem*>(bias_s + EPI_WARPS * BIAS_BYTES);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = ptx::cluster_ctarank();
  const bool leader = rank == 0;
  const int64_t M = a.M, N = a.N, K = a.K;
  const int num_mp = int(ceil_div(M, 2 * BM)), num_n = int(ceil_div(N, BN));
  const int num_tiles = num_mp * num_n;
  const int pair = blockIdx.x >> 1, num_pairs = gridDim.x >> 1;
  const int n_lr = a.rank > 0 ? int(ceil_div(a.rank, 64)) : 0;
  const int n_k = int(ceil_div(K, 256));
  const int iters = n_lr + n_k;
  const int64_t KG = scale_groups(K);

  ptx::griddep_launch_dependents();
  if (threadIdx.x == 0) {
    for (int i = 0; i < STAGES; ++i) {
      ptx::mbar_init(&s->full[i], 1);
      ptx::mbar_init(&s->empty[i], 1);
      ptx::mbar_init(&s->ready[i], 8);
    }
    ptx::mbar_init(&s->acc_full, 1);
    ptx::mbar_init(&s->acc_empty, 2 * EPI_WARPS);
    ptx::mbar_init(&s->drain, 1);
    ptx::mbar_init(&s->never, 1);
    s->abort_flag = 0;
    ptx::fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    ptx::prefetch_tmap(&maps.A);
    ptx::prefetch_tmap(&maps.B);
    ptx::prefetch_tmap(&maps.SFA);
    ptx::prefetch_tmap(&maps.SFB);
    ptx::prefetch_tmap(&maps.Y);
    if (n_lr) {
      ptx::prefetch_tmap(&maps.T);
      ptx::prefetch_tmap(&maps.L2);
    }
  }
  if (warp == 1) {
    ptx::tmem_alloc2(&s->tmem_base, TMEM_COLS);   // collective over the pair: same columns in both
    ptx::tmem_relinquish2();
  }
  ptx::tc_fence_before();
  ptx::cluster_sync();                            // barriers of both CTAs initialised, TMEM allocated
  ptx::tc_fence_after();
  const uint32_t tmem = s->tmem_base;
  // every role's bounded waits start once the previous grid is done (the producer first
  // issues the weight loads of its first ring pass, then waits)
  if (warp != 0) ptx::griddep_wait();

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer (both CTAs)
    if (lane == 0) {
      // Weight-side loads (L2, R codes and scales) depend on nothing kernel 1 writes: those of
      // the first tile's first ring pass are issued before waiting for the previous grid, so
      // they overlap its tail when this grid is launched as its programmatic dependent.
      const int pre = pair < num_tiles ? (iters < STAGES ? iters : STAGES) : 0;
      auto weight_loads = [&](int it, int n0, int nb, unsigned char* st, uint64_t* fb) {
        if (it < n_lr) {
          ptx::mbar_arrive_expect_tx(fb, A_BYTES + B_BYTES);
          ptx::tma_load_2d(st + A_BYTES, &maps.L2, fb, 64 * it, nb);
        } else {
          const int kq = it - n_lr;
          ptx::mbar_arrive_expect_tx(fb, STAGE_BYTES);
          ptx::tma_load_2d(st + A_BYTES, &maps.B, fb, 128 * kq, nb);
          // scales: 2 KB chunks = 8 rows of the 256-byte-wide view of the tiled buffers
          unsigned char* sfb = st + A_BYTES + B_BYTES + SFA_BYTES;
          ptx::tma_load_2d(sfb, &maps.SFB, fb, 0, int(((int64_t(n0) / 128) * KG + 4 * kq) * 2));
          ptx::tma_load_2d(sfb + SFA_BYTES, &maps.SFB, fb, 0, int(((int64_t(n0) / 128 + 1) * KG + 4 * kq) * 2));
        }
      };
      auto act_loads = [&](int it, int m0, unsigned char* st, uint64_t* fb) {
        if (it < n_lr) {
          ptx::tma_load_2d(st, &maps.T, fb, 64 * it, m0);
        } else {
          const int kq = it - n_lr;
          ptx::tma_load_2d(st, &maps.A, fb, 128 * kq, m0);
          ptx::tma_load_2d(st + A_BYTES + B_BYTES, &maps.SFA, fb, 0, int(((int64_t(m0) / 128) * KG + 4 * kq) * 2));
        }
      };
      if (pre > 0) {
        const int n0 = (pair % num_n) * BN;
        for (int it = 0; it < pre; ++it)   // stages start empty: no wait
          weight_loads(it, n0, n0 + int(rank) * (BN / 2), stages + it * STAGE_BYTES, &s->full[it]);
      }
      ptx::griddep_wait();
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      for (int tile = pair; tile < num_tiles && ok; tile += num_pairs) {
        const int m0 = (tile / num_n) * 2 * BM + int(rank) * BM;
        const int n0 = (tile % num_n) * BN;
        const int nb = n0 + int(rank) * (BN / 2);   // this CTA's half of the weight rows
        for (int it = 0; it < iters; ++it) {
          unsigned char* st = stages + stage * STAGE_BYTES;
          uint64_t* fb = &s->full[stage];
          if (!(tile == pair && it < pre)) {
            if (!wait_bounded(&s->empty[stage], phase ^ 1u, s, a.err, a.wait_ns)) { ok = false; break; }
            // No proxy fence is needed before overwriting the stage: the scale warps' ordinary
            // loads of its scales have completed before the stage is released (their values
            // went into tcgen05.st and tcgen05.wait::st returned before the warps arrived on
            // "ready", which precedes the MMAs whose commit frees the stage).
            weight_loads(it, n0, nb, st, fb);
          }
          act_loads(it, m0, st, fb);
          if (++stage == STAGES) { stage = 0; phase ^= 1u; }
        }
      }
      // every copy this CTA started has landed before shared memory is released
      // (the scale warps consume every full phase; waiting here covers an abort)
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer (even CTA)
    if (leader && lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      bool ok = !(a.stall && !wait_bounded(&s->never, 0, s, a.err, a.wait_ns));
      int local = 0;
      for (int tile = pair; tile < num_tiles && ok; tile += num_pairs, ++local) {
        if (!wait_bounded(&s->acc_empty, (uint32_t(local) & 1u) ^ 1u, s, a.err, a.wait_ns)) break;
        ptx::tc_fence_after();
        uint32_t accumulate = 0;
        for (int it = 0; it < iters; ++it) {
          if (!wait_bounded(&s->ready[stage], phase, s, a.err, a.wait_ns)) { ok = false; break; }
          ptx::tc_fence_after();
          const uint32_t a_s = ptx::smem_u32(stages + stage * STAGE_BYTES);
          const uint32_t b_s = a_s + A_BYTES;
          if (it < n_lr) {
            const int ksteps = min(4, (a.rank - 64 * it) / 16);
            for (int kk = 0; kk < ksteps; ++kk) {
              ptx::mma2_bf16(tmem, ptx::desc_sw128(a_s + 32 * kk), ptx::desc_sw128(b_s + 32 * kk), IDESC_BF16,
                             accumulate);
              accumulate = 1;
            }
          } else {
            const int kq = it - n_lr;
            const int64_t krem = (K - 256 * int64_t(kq)) / 64;
            const int ksteps = krem < 4 ? int(krem) : 4;
            const uint32_t sfa_t = tmem + SF_COL0 + stage * SF_COLS_PER_STAGE;
            const uint32_t sfb_t = sfa_t + 16;
            if (ksteps == 4) {
              // full 256-wide K step: descriptors built once, the k-slices 32 bytes apart
              // (start-address field in 16-byte units)
              const uint64_t ad = ptx::desc_sw128(a_s), bd = ptx::desc_sw128(b_s);
#pragma unroll
              for (int kk = 0; kk < 4; ++kk)
                ptx::mma2_nvfp4(tmem, ad + uint64_t(2 * kk), bd + uint64_t(2 * kk), IDESC_NVFP4, sfa_t + 4 * kk,
                                sfb_t + 8 * kk, kk == 0 ? accumulate : 1u);
              accumulate = 1;
            } else {
              for (int kk = 0; kk < ksteps; ++kk) {
                ptx::mma2_nvfp4(tmem, ptx::desc_sw128(a_s + 32 * kk), ptx::desc_sw128(b_s + 32 * kk), IDESC_NVFP4,
                                sfa_t + 4 * kk, sfb_t + 8 * kk, accumulate);
                accumulate = 1;
              }
            }
          }
          ptx::tc_commit2_mc(&s->empty[stage], kPairMask);
          if (++stage == STAGES) { stage = 0; phase ^= 1u; }
        }
        if (!ok) break;
        ptx::tc_commit2_mc(&s->acc_full, kPairMask);
      }
      // every MMA issued for the pair has finished before TMEM is released
      ptx::tc_commit2_mc(&s->drain, 0x1);
      wait_drain(&s->drain, 0, a.err);
    }
  } else if (warp < EPI_WARP0) {
    // ------------------------------------------------------------ scale warps (both CTAs)
    const uint32_t q = uint32_t(warp & 3);         // TMEM lane quarter this warp may access
    const uint32_t lane_off = (32u * q) << 16;
    const uint32_t ready_c = ptx::mapa(ptx::smem_u32(&s->ready[0]), 0);
    int stage = 0;
    uint32_t phase = 0;
    bool ok = true;
    for (int tile = pair; tile < num_tiles && ok; tile += num_pairs) {
      for (int it = 0; it < iters; ++it) {
        if (!wait_bounded(&s->full[stage], phase, s, a.err, a.wait_ns)) { ok = false; break; }
        if (it >= n_lr) {
          // A scales: the MMA reads row 32q + lane from this lane, column base + 4 kk + q; the
          // row's four scales of k-step kk are the word at kk * 512 + lane * 16 + q * 4 of the
          // 128 x 4 tile layout (the value goes to all four columns of the group).
          const uint32_t* sfa = reinterpret_cast<const uint32_t*>(stages + stage * STAGE_BYTES + A_BYTES + B_BYTES);
          const int w = lane * 4 + int(q);
          const uint32_t sfa_t = tmem + lane_off + SF_COL0 + stage * SF_COLS_PER_STAGE;
          ptx::tmem_st_32x32b_x16_rep4(sfa_t, sfa[w], sfa[128 + w], sfa[256 + w], sfa[384 + w]);
          // B scales: every lane quarter holds all 256 weight rows; column 8 kk + 4 h + j of
          // lane i is weight row 128 h + 32 j + i, i.e. 16-byte row i of the (h, kk) tile.
          const uint4* sfb = reinterpret_cast<const uint4*>(sfa + SFA_BYTES / 4);
          uint32_t vb[32];
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              const uint4 t = sfb[h * 128 + kk * 32 + lane];
              vb[8 * kk + 4 * h] = t.x;
              vb[8 * kk + 4 * h + 1] = t.y;
              vb[8 * kk + 4 * h + 2] = t.z;
              vb[8 * kk + 4 * h + 3] = t.w;
            }
          ptx::tmem_st_32x32b_x32(sfa_t + 16, vb);
          ptx::tmem_wait_st();
        }
        // tcgen05.wait::st has completed the stores; the fence orders them before the arrive
        // (a release at cluster scope here stalled the warp for a microsecond per stage)
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive_cluster(ready_c + 8u * uint32_t(stage));
        if (++stage == STAGES) { stage = 0; phase ^= 1u; }
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue (both CTAs)
    const int e = warp - EPI_WARP0;
    const int q = warp & 3;                         // TMEM lane quarter this warp may access
    const int half = e >> 2;                        // which 128 of the 256 columns
    unsigned char* my_stg = stg + e * STG_BYTES;
    uint16_t* my_bias = reinterpret_cast<uint16_t*>(bias_s + e * BIAS_BYTES);
    const uint32_t acc_empty_c = ptx::mapa(ptx::smem_u32(&s->acc_empty), 0);
    int local = 0;
    for (int tile = pair; tile < num_tiles; tile += num_pairs, ++local) {
      const int m0 = (tile / num_n) * 2 * BM + int(rank) * BM;
      const int ncol0 = (tile % num_n) * BN + 128 * half;
      // this warp's 128 bias values, staged while the MMAs run
      {
        const int64_t c = ncol0 + 4 * lane;
        uint2 v = make_uint2(0, 0);
        if (c < N) v = __ldg(reinterpret_cast<const uint2*>(a.bias + c));
        *reinterpret_cast<uint2*>(my_bias + 4 * lane) = v;
        __syncwarp();
      }
      if (!wait_bounded(&s->acc_full, uint32_t(local) & 1u, s, a.err, a.wait_ns)) break;
      ptx::tc_fence_after();
      const uint32_t taddr = tmem + (uint32_t(32 * q) << 16) + uint32_t(128 * half);
      uint32_t r[64], o[32];
      ptx::tmem_ld_32x32b_x32(taddr, r);
      ptx::tmem_ld_32x32b_x32(taddr + 32, r + 32);
      ptx::tmem_wait_ld();
      convert64(r, my_bias, a.alpha, o);
      if (ncol0 < N) store64(&maps.Y, my_stg, o, lane, ncol0, m0 + 32 * q);
      ptx::tmem_ld_32x32b_x32(taddr + 64, r);
      ptx::tmem_ld_32x32b_x32(taddr + 96, r + 32);
      ptx::tmem_wait_ld();
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive_cluster(acc_empty_c);   // accumulator free for the next tile
      convert64(r, my_bias + 64, a.alpha, o);
      if (ncol0 + 64 < N) store64(&maps.Y, my_stg, o, lane, ncol0 + 64, m0 + 32 * q);
    }
    if (lane == 0) ptx::bulk_wait<0>();
    __syncwarp();
  }

  // copies still in flight after an abort land well within this delay
  if (s->abort_flag) {
    const uint64_t t0 = ptx::globaltimer();
    while (ptx::globaltimer() - t0 < 20000000ull) {
    }
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::cluster_sync();                            // the pair's MMAs and epilogues are done
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc2(tmem, TMEM_COLS);
  }
}

}  // namespace

size_t k2_smem_bytes() { return SMEM_BYTES; }

int k2_launch(const K2Maps& maps, const K2Args& a, int sm_count, void* stream) {
  static int attr_done[64] = {0};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 64 && !attr_done[dev]) {
    cudaError_t e = cudaFuncSetAttribute(k2_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
    if (e != cudaSuccess) return int(e);
    attr_done[dev] = 1;
  }
  const int64_t tiles = ceil_div(a.M, 2 * BM) * ceil_div(a.N, BN);
  if (tiles == 0) return 0;
  // as many co-resident CTA pairs as the GPU holds, never more than there are tiles
  static int max_pairs[64] = {0};
  if (dev < 64 && max_pairs[dev] == 0) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * (sm_count / 2), 1, 1);
    cfg.blockDim = dim3(THREADS, 1, 1);
    cfg.dynamicSmemBytes = SMEM_BYTES;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, k2_kernel, &cfg) != cudaSuccess || n <= 0) {
      cudaGetLastError();
      n = sm_count / 2;
    }
    max_pairs[dev] = n;
  }
  const int pairs = int(tiles < max_pairs[dev] ? tiles : max_pairs[dev]);
  // launched as a programmatic dependent of the previous kernel in the stream: the prologue
  // and the first weight loads run while that kernel drains (only the TMA producer waits on it)
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * pairs, 1, 1);
  cfg.blockDim = dim3(THREADS, 1, 1);
  cfg.dynamicSmemBytes = SMEM_BYTES;
  cfg.stream = static_cast<cudaStream_t>(stream);
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return int(cudaLaunchKernelEx(&cfg, k2_kernel, maps, a));
}

}  // namespace svdq
