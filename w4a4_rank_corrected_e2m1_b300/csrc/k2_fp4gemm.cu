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

#include <algorithm>
#include <climits>

#include "nvfp4_block.cuh"
#include "ptx.cuh"
#include "svdq_internal.h"

namespace svdq {

namespace {

constexpr int BM = 128;                            // rows per CTA (pair tile: 256)
constexpr int BN = 256;                            // columns per pair tile
constexpr int A_BYTES = BM * 128;                  // 128 rows x 256 fp4
constexpr int B_BYTES = (BN / 2) * 128;            // this CTA's 128 weight rows x 256 fp4
constexpr int SFB_BYTES = 2 * 4 * 512;             // both 128-row halves of the tile's weights
constexpr int SFA_BYTES = 4 * 512;                 // 4 k64-groups x (128 rows x 4 scales)
// stage: A codes | B codes | B scales | A scales (B codes and scales are one weight block)
constexpr int SFB_OFF = A_BYTES + B_BYTES;
constexpr int SFA_OFF = SFB_OFF + SFB_BYTES;
constexpr int STAGE_BYTES = SFA_OFF + SFA_BYTES;
static_assert(B_BYTES + SFB_BYTES == kK2WeightBlock, "a weight block fills a stage's B codes and scales");
constexpr int SCALE_WARP0 = 2;
constexpr int EPI_WARP0 = 6;
constexpr int EPI_WARPS = 8;
constexpr int BIAS_BYTES = 128 * 2;                // per warp: its 128 columns of bias
constexpr int THREADS = 32 * (EPI_WARP0 + EPI_WARPS);
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t SF_COL0 = 256;                  // scale columns after the accumulator
constexpr uint32_t SF_COLS_PER_STAGE = 48;         // A: 4 k-steps x 4, B: 4 k-steps x 8
constexpr uint64_t kTimeoutNs = 2000000000ull;
constexpr uint16_t kPairMask = 0x3;

// Shared-memory plan.  The plain layer: a 5-stage ring and one 32-row x 64-column bf16 box per
// epilogue warp (staging of the TMA stores of Y).  The fused MLP epilogue: a 4-stage ring, so
// that each epilogue warp can hold its whole 32 x 128 slice of y (two boxes) and release the
// accumulator before the slow part of its work, plus its 128 values of the next layer's
// 1/lambda and the next layer's quantiser tables.
template <bool FUSED>
struct Cfg {
  static constexpr int STAGES = FUSED ? 4 : 5;
  static constexpr int STG_BYTES = (FUSED ? 2 : 1) * 32 * 128;
  static constexpr int IL_BYTES = FUSED ? 128 * 4 : 0;
  static constexpr int QTAB_BYTES = FUSED ? 256 * 4 : 0;
  static constexpr int EPI_BYTES = EPI_WARPS * (STG_BYTES + BIAS_BYTES + IL_BYTES) + QTAB_BYTES;
  static constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + EPI_BYTES + 1024 + 1024;
  static_assert(SF_COL0 + STAGES * SF_COLS_PER_STAGE <= TMEM_COLS, "TMEM budget");
  static_assert(SMEM_BYTES <= 232448, "shared memory budget");
};

static_assert(STAGE_BYTES % 1024 == 0, "stage alignment");

// Instruction descriptors (tcgen05 instruction-descriptor bit layout):
//   [4,6) D type / B scale id  [7,10) A type  [10,13) B type  [15] A major  [16] B major
//   [17,23) N >> 3  [23] scale type (mxf4nvf4: 0 = UE4M3)  [24,29) M >> 4
// The pair computes M = 256 (128 per CTA).
constexpr uint32_t IDESC_NVFP4 = (1u << 7) | (1u << 10) | (uint32_t(BN >> 3) << 17) | (uint32_t(256 >> 4) << 24);
constexpr uint32_t IDESC_BF16 =
    (1u << 4) | (1u << 7) | (1u << 10) | (uint32_t(BN >> 3) << 17) | (uint32_t(256 >> 4) << 24);

constexpr int kMaxStages = 5;
struct Smem {
  uint64_t full[kMaxStages];    // this CTA's loads of a stage landed (producer arrive + bytes)
  uint64_t empty[kMaxStages];   // this CTA's stage may be refilled (MMA commit, multicast)
  uint64_t ready[kMaxStages];   // even CTA: both CTAs' stage landed and its scales are in TMEM
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

// alpha * acc + bias -> 16 packed bf16 pairs for 32 columns (convert64's arithmetic, two fused
// multiply-adds per packed instruction)
__device__ __forceinline__ void convert32(const uint32_t* r, const uint16_t* bias, float alpha, uint32_t* out) {
  const float2 a2 = make_float2(alpha, alpha);
#pragma unroll
  for (int v = 0; v < 4; ++v) {
    const uint4 bb = *reinterpret_cast<const uint4*>(bias + 8 * v);
    const uint32_t bw[4] = {bb.x, bb.y, bb.z, bb.w};
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const float2 b = make_float2(__uint_as_float(bw[u] << 16), __uint_as_float(bw[u] & 0xFFFF0000u));
      const float2 y = ptx::fma2_rn(a2, make_float2(__uint_as_float(r[8 * v + 2 * u]), __uint_as_float(r[8 * v + 2 * u + 1])), b);
      out[4 * v + u] = ptx::pack_bf16x2(y.x, y.y);
    }
  }
}

// Address of 16-byte unit j (8 bf16) of row r in a 32 x 64 bf16 staging box: unit j of row r is
// stored at unit j ^ (r % 8), so a warp writing one unit of 32 rows, or ldmatrix reading 8 rows
// of one unit, touches every bank once per 128 bytes.
__device__ __forceinline__ int box_off(int r, int j) { return r * 128 + ((j ^ (r & 7)) << 4); }
__device__ __forceinline__ unsigned char* box_unit(unsigned char* box, int r, int j) { return box + box_off(r, j); }

// Tile order.  Tiles (row block of 256, column tile of 256) are taken in units of unit_len
// consecutive column tiles of one row block; unit u covers row block u / S and column tiles
// (u % S) unit_len .. + unit_len - 1 (S units per row block), and CTA pair p takes units p,
// p + pairs, ...  The plain layer uses unit_len = 1, so pair p takes tiles p, p + pairs, ...
// The fused MLP epilogue sums its partial down-projections over a unit, so longer units mean
// fewer partial sums to write and add.
//
// Fused MLP epilogue (FUSED, RD = the next layer's kernel rank).  Each epilogue warp turns its
// 32 rows x 128 columns of the accumulator into the next layer's kernel-1 outputs:
//   y = bf16(alpha acc + b)              exactly the plain layer's Y, into two staging boxes;
//                                        then the accumulator is released to the MMA warp
//   G = bf16(GELU(y))                    in place (thread = row, as the accumulator lanes)
//   codes, scales of G                   the next layer's smoothing and NVFP4 block quantiser
//                                        (one thread holds whole 16-element blocks of its row),
//                                        stored straight to global memory: 32 bytes of codes
//                                        and one scale word per row and 64 columns
//   part += G L1'                        bf16 warp MMAs (ldmatrix from the boxes, L1' fragments
//                                        from global memory), summed over the unit in registers
// and at the end of each unit writes its 32 x RD partial sum of G L1' for its column half;
// k2_t_reduce_kernel adds the 2 S partials of every row in a fixed order.
template <bool FUSED, int RD>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(THREADS, 1)
    k2_kernel(const __grid_constant__ K2Maps maps, K2Args a) {
  using C = Cfg<FUSED>;
  constexpr int STAGES = C::STAGES;
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* base = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  unsigned char* stages = base;
  unsigned char* stg = base + STAGES * STAGE_BYTES;
  unsigned char* bias_s = stg + EPI_WARPS * C::STG_BYTES;
  unsigned char* il_s = bias_s + EPI_WARPS * BIAS_BYTES;
  float* qtab_s = reinterpret_cast<float*>(il_s + EPI_WARPS * C::IL_BYTES);
  Smem* s = reinterpret_cast<Smem*>(reinterpret_cast<unsigned char*>(qtab_s) + C::QTAB_BYTES);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = ptx::cluster_ctarank();
  const bool leader = rank == 0;
  const int64_t M = a.M, N = a.N, K = a.K;
  const int num_mp = int(ceil_div(M, 2 * BM)), num_n = int(ceil_div(N, BN));
  const int U = FUSED ? a.unit_len : 1, S = (num_n + U - 1) / U;   // the plain layer: one tile a unit
  const int num_units = num_mp * S;
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
  if constexpr (FUSED) {
    // the next layer's quantiser tables (constant layer data)
    if (threadIdx.x < 256) qtab_s[threadIdx.x] = __ldg(a.fuse.qtab + threadIdx.x);
  }
  if (warp == 0 && lane == 0) {
    ptx::prefetch_tmap(&maps.A);
    ptx::prefetch_tmap(&maps.SFA);
    if (!FUSED) ptx::prefetch_tmap(&maps.Y);
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
      const int pre = pair < num_units ? (iters < STAGES ? iters : STAGES) : 0;
      auto weight_loads = [&](int it, int n0, int nb, unsigned char* st, uint64_t* fb) {
        if (it < n_lr) {
          ptx::mbar_arrive_expect_tx(fb, A_BYTES + B_BYTES);
          ptx::tma_load_2d(st + A_BYTES, &maps.L2, fb, 64 * it, nb);
        } else {
          const int kq = it - n_lr;
          ptx::mbar_arrive_expect_tx(fb, STAGE_BYTES);
          // this half's weight block of the step: codes already in swizzled order, then the
          // pair tile's scales
          const uint8_t* wb = a.wt + ((int64_t(n0 / 256) * n_k + kq) * 2 + int64_t(rank)) * kK2WeightBlock;
          ptx::bulk_load(st + A_BYTES, wb, kK2WeightBlock, fb);
        }
      };
      auto act_loads = [&](int it, int m0, unsigned char* st, uint64_t* fb) {
        if (it < n_lr) {
          ptx::tma_load_2d(st, &maps.T, fb, 64 * it, m0);
        } else {
          const int kq = it - n_lr;
          ptx::tma_load_2d(st, &maps.A, fb, 128 * kq, m0);
          ptx::tma_load_2d(st + SFA_OFF, &maps.SFA, fb, 0, int(((int64_t(m0) / 128) * KG + 4 * kq) * 2));
        }
      };
      if (pre > 0) {
        const int n0 = ((pair % S) * U) * BN;     // the first tile's column tile
        for (int it = 0; it < pre; ++it)   // stages start empty: no wait
          weight_loads(it, n0, n0 + int(rank) * (BN / 2), stages + it * STAGE_BYTES, &s->full[it]);
      }
      ptx::griddep_wait();
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true, first = true;
      for (int u = pair; u < num_units && ok; u += num_pairs) {
        const int nb_t = (u % S) * U, ne_t = min(nb_t + U, num_n);
        for (int nt = nb_t; nt < ne_t && ok; ++nt, first = false) {
          const int m0 = (u / S) * 2 * BM + int(rank) * BM;
          const int n0 = nt * BN;
          const int nb = n0 + int(rank) * (BN / 2);   // this CTA's half of the weight rows
          for (int it = 0; it < iters; ++it) {
            unsigned char* st = stages + stage * STAGE_BYTES;
            uint64_t* fb = &s->full[stage];
            if (!(first && it < pre)) {
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
      for (int u = pair; u < num_units && ok; u += num_pairs) {
        const int nb_t = (u % S) * U, ne_t = min(nb_t + U, num_n);
        for (int nt = nb_t; nt < ne_t && ok; ++nt, ++local) {
          if (!wait_bounded(&s->acc_empty, (uint32_t(local) & 1u) ^ 1u, s, a.err, a.wait_ns)) { ok = false; break; }
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
    for (int u = pair; u < num_units && ok; u += num_pairs) {
      const int nb_t = (u % S) * U, ne_t = min(nb_t + U, num_n);
      for (int nt = nb_t; nt < ne_t && ok; ++nt) {
        for (int it = 0; it < iters; ++it) {
          if (!wait_bounded(&s->full[stage], phase, s, a.err, a.wait_ns)) { ok = false; break; }
          if (it >= n_lr) {
            // A scales: the MMA reads row 32q + lane from this lane, column base + 4 kk + q; the
            // row's four scales of k-step kk are the word at kk * 512 + lane * 16 + q * 4 of the
            // 128 x 4 tile layout (the value goes to all four columns of the group).
            const uint32_t* sfa = reinterpret_cast<const uint32_t*>(stages + stage * STAGE_BYTES + SFA_OFF);
            const int w = lane * 4 + int(q);
            const uint32_t sfa_t = tmem + lane_off + SF_COL0 + stage * SF_COLS_PER_STAGE;
            ptx::tmem_st_32x32b_x16_rep4(sfa_t, sfa[w], sfa[128 + w], sfa[256 + w], sfa[384 + w]);
            // B scales: every lane quarter holds all 256 weight rows; column 8 kk + 4 h + j of
            // lane i is weight row 128 h + 32 j + i, i.e. 16-byte row i of the (kk, h) tile.
            const uint4* sfb = reinterpret_cast<const uint4*>(stages + stage * STAGE_BYTES + SFB_OFF);
            uint32_t vb[32];
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
#pragma unroll
              for (int h = 0; h < 2; ++h) {
                const uint4 t = sfb[(kk * 2 + h) * 32 + lane];
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
    }
  } else {
    // ------------------------------------------------------------ epilogue (both CTAs)
    const int e = warp - EPI_WARP0;
    const int q = warp & 3;                         // TMEM lane quarter this warp may access
    const int half = e >> 2;                        // which 128 of the 256 columns
    unsigned char* my_stg = stg + e * C::STG_BYTES;
    uint16_t* my_bias = reinterpret_cast<uint16_t*>(bias_s + e * BIAS_BYTES);
    const uint32_t acc_empty_c = ptx::mapa(ptx::smem_u32(&s->acc_empty), 0);
    int local = 0;
    bool ok = true;
    if constexpr (!FUSED) {
      for (int u = pair; u < num_units && ok; u += num_pairs) {
        const int nb_t = (u % S) * U, ne_t = min(nb_t + U, num_n);
        for (int nt = nb_t; nt < ne_t; ++nt, ++local) {
          const int m0 = (u / S) * 2 * BM + int(rank) * BM;
          const int ncol0 = nt * BN + 128 * half;
          // this warp's 128 bias values, staged while the MMAs run
          {
            const int64_t c = ncol0 + 4 * lane;
            uint2 v = make_uint2(0, 0);
            if (c < N) v = __ldg(reinterpret_cast<const uint2*>(a.bias + c));
            *reinterpret_cast<uint2*>(my_bias + 4 * lane) = v;
            __syncwarp();
          }
          if (!wait_bounded(&s->acc_full, uint32_t(local) & 1u, s, a.err, a.wait_ns)) { ok = false; break; }
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
      }
      if (lane == 0) ptx::bulk_wait<0>();
      __syncwarp();
    } else {
      float* my_il = reinterpret_cast<float*>(il_s + e * C::IL_BYTES);
      const float* s_thr = qtab_s;
      const float* s_rcp = qtab_s + 128;
      const int64_t M_pad = round_up(M, 128);       // rows of the tiled scale layout
      const int64_t KGn = scale_groups(N);          // its 64-column groups (the next layer's K = N)
      constexpr int NT = RD / 8 > 0 ? RD / 8 : 1;   // 8-column groups of the partial down-projection
      const int g = lane >> 2, t = lane & 3;
      float part[2][NT][4];
      // bias and the next layer's 1/lambda of this warp's 128 columns, loaded one tile ahead
      uint2 pf_b = make_uint2(0, 0);
      float4 pf_il = make_float4(0.f, 0.f, 0.f, 0.f);
      auto prefetch = [&](int nt) {
        const int64_t c = int64_t(nt) * BN + 128 * half + 4 * lane;
        pf_b = make_uint2(0, 0);
        pf_il = make_float4(0.f, 0.f, 0.f, 0.f);
        if (nt >= 0 && c < N) {
          pf_b = __ldg(reinterpret_cast<const uint2*>(a.bias + c));
          pf_il = __ldg(reinterpret_cast<const float4*>(a.fuse.inv_lambda + c));
        }
      };
      if (pair < num_units) prefetch((pair % S) * U);
      for (int u = pair; u < num_units && ok; u += num_pairs) {
        const int nb_t = (u % S) * U, ne_t = min(nb_t + U, num_n);
        const int m0 = (u / S) * 2 * BM + int(rank) * BM;
        const int64_t row = m0 + 32 * q + lane;
#pragma unroll
        for (int i = 0; i < 2; ++i)
#pragma unroll
          for (int j = 0; j < NT; ++j)
#pragma unroll
            for (int k = 0; k < 4; ++k) part[i][j][k] = 0.f;
        for (int nt = nb_t; nt < ne_t; ++nt, ++local) {
          const int64_t ncol0 = int64_t(nt) * BN + 128 * half;
          *reinterpret_cast<uint2*>(my_bias + 4 * lane) = pf_b;
          *reinterpret_cast<float4*>(my_il + 4 * lane) = pf_il;
          __syncwarp();
          {
            // the next tile of this pair: the next of this unit, else the first of its next unit
            const int un = u + num_pairs;
            prefetch(nt + 1 < ne_t ? nt + 1 : (un < num_units ? (un % S) * U : -1));
          }
          if (!wait_bounded(&s->acc_full, uint32_t(local) & 1u, s, a.err, a.wait_ns)) { ok = false; break; }
          ptx::tc_fence_after();
          const uint32_t taddr = tmem + (uint32_t(32 * q) << 16) + uint32_t(128 * half);
          // y = bf16(alpha acc + b) into the two boxes (row = lane), then free the accumulator
#pragma unroll 1
          for (int c = 0; c < 4; ++c) {
            uint32_t r[32], o[16];
            ptx::tmem_ld_32x32b_x32(taddr + 32 * c, r);
            ptx::tmem_wait_ld();
            if (c == 3) {
              ptx::tc_fence_before();
              __syncwarp();
              if (lane == 0) ptx::mbar_arrive_cluster(acc_empty_c);
            }
            convert32(r, my_bias + 32 * c, a.alpha, o);
            unsigned char* box = my_stg + (c >> 1) * 4096;
#pragma unroll
            for (int j = 0; j < 4; ++j)
              *reinterpret_cast<uint4*>(box_unit(box, lane, 4 * (c & 1) + j)) =
                  make_uint4(o[4 * j], o[4 * j + 1], o[4 * j + 2], o[4 * j + 3]);
          }
#pragma unroll 1
          for (int h = 0; h < 2; ++h) {
            const int64_t col = ncol0 + 64 * h;     // first of the 64 columns (a whole scale group)
            unsigned char* box = my_stg + h * 4096;
            if (col >= N) {
              // scale groups past N (N not a multiple of 256) read as zero scales by the next GEMM
              if (row < M_pad) *reinterpret_cast<uint32_t*>(a.fuse.x_scales + scale_word_offset(row, col / 64, KGn)) = 0u;
              continue;
            }
            uint32_t cw[8], sword = 0;
#pragma unroll
            for (int b = 0; b < 4; ++b) {
              uint4* p0 = reinterpret_cast<uint4*>(box_unit(box, lane, 2 * b));
              uint4* p1 = reinterpret_cast<uint4*>(box_unit(box, lane, 2 * b + 1));
              const uint4 u0 = *p0, u1 = *p1;
              uint32_t w[8] = {gelu_bf16x2(u0.x), gelu_bf16x2(u0.y), gelu_bf16x2(u0.z), gelu_bf16x2(u0.w),
                               gelu_bf16x2(u1.x), gelu_bf16x2(u1.y), gelu_bf16x2(u1.z), gelu_bf16x2(u1.w)};
              *p0 = make_uint4(w[0], w[1], w[2], w[3]);
              *p1 = make_uint4(w[4], w[5], w[6], w[7]);
              const uint32_t s8 = quant_block(w, my_il + 64 * h + 16 * b, a.fuse.inv_six, s_thr, s_rcp, &cw[2 * b],
                                              &cw[2 * b + 1]);
              sword |= s8 << (8 * b);
            }
            if (row < M) {
              uint4* cp = reinterpret_cast<uint4*>(a.fuse.x_codes + row * (N / 2) + col / 2);
              cp[0] = make_uint4(cw[0], cw[1], cw[2], cw[3]);
              cp[1] = make_uint4(cw[4], cw[5], cw[6], cw[7]);
            }
            // rows from M to the end of their 128-row scale tile get zero scales, as kernel 1 writes
            if (row < M_pad)
              *reinterpret_cast<uint32_t*>(a.fuse.x_scales + scale_word_offset(row, col / 64, KGn)) = row < M ? sword : 0u;
            if constexpr (RD > 0) {
              __syncwarp();                         // G of all 32 rows is in the box
              const uint32_t box_s = ptx::smem_u32(box);
#pragma unroll
              for (int kk = 0; kk < 4; ++kk) {
                // A: matrices (rows 0-7 | 8-15) x (k 0-7 | 8-15) of the two 16 x 16 row tiles
                const int mi = lane >> 3;
                uint32_t af[2][4];
#pragma unroll
                for (int mt = 0; mt < 2; ++mt) {
                  const int rr = 16 * mt + (mi & 1) * 8 + (lane & 7);
                  ptx::ldmatrix_x4(box_s + uint32_t(box_off(rr, 2 * kk + (mi >> 1))), af[mt]);
                }
                const uint4* bp = static_cast<const uint4*>(a.fuse.l1f) + ((col / 16 + kk) * (RD / 16)) * 32 + lane;
#pragma unroll
                for (int np = 0; np < RD / 16; ++np) {
                  const uint4 v = __ldg(bp + np * 32);   // B of 8-column groups 2 np and 2 np + 1
#pragma unroll
                  for (int mt = 0; mt < 2; ++mt) {
                    ptx::mma_bf16_16816(part[mt][2 * np], af[mt][0], af[mt][1], af[mt][2], af[mt][3], v.x, v.y);
                    ptx::mma_bf16_16816(part[mt][2 * np + 1], af[mt][0], af[mt][1], af[mt][2], af[mt][3], v.z, v.w);
                  }
                }
              }
            }
          }
          __syncwarp();                             // the boxes are free for the next tile
        }
        if constexpr (RD > 0) {
          if (ok) {
            // this unit's partial G L1' over this warp's column half: C fragment (g, t) holds
            // rows g and g + 8 of each 16-row tile, columns 2 t and 2 t + 1 of each 8-column group
            float* pp = a.fuse.part + (int64_t(2 * (u % S) + half) * M) * RD;
#pragma unroll
            for (int mt = 0; mt < 2; ++mt)
#pragma unroll
              for (int hh = 0; hh < 2; ++hh) {
                const int64_t rw = m0 + 32 * q + 16 * mt + 8 * hh + g;
                if (rw < M) {
#pragma unroll
                  for (int j = 0; j < NT; ++j)
                    *reinterpret_cast<float2*>(pp + rw * RD + 8 * j + 2 * t) =
                        make_float2(part[mt][j][2 * hh], part[mt][j][2 * hh + 1]);
                }
              }
          }
        }
      }
    }
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

// Sum of the fused epilogue's partial down-projections, in partial order.
__global__ void __launch_bounds__(256) k2_t_reduce_kernel(const float* __restrict__ part, int64_t P, int64_t M, int rd,
                                                          int r_pad, float inv_alpha, uint16_t* __restrict__ T) {
  ptx::griddep_wait();
  const int64_t n = M * (r_pad / 2);
  for (int64_t i = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; i < n; i += int64_t(gridDim.x) * blockDim.x) {
    const int64_t row = i / (r_pad / 2);
    const int j = 2 * int(i % (r_pad / 2));
    uint32_t o = 0;
    if (j < rd) {
      float s0 = 0.f, s1 = 0.f;
      for (int64_t p = 0; p < P; ++p) {
        const float2 v = __ldg(reinterpret_cast<const float2*>(part + (p * M + row) * rd + j));
        s0 += v.x;
        s1 += v.y;
      }
      o = ptx::pack_bf16x2(s0 * inv_alpha, s1 * inv_alpha);
    }
    reinterpret_cast<uint32_t*>(T + row * r_pad)[j / 2] = o;
  }
}

// G = bf16(GELU(y)), eight elements per thread and step
__global__ void __launch_bounds__(256) gelu_kernel(const uint4* __restrict__ Y, uint4* __restrict__ G, int64_t n8) {
  for (int64_t i = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; i < n8; i += int64_t(gridDim.x) * blockDim.x) {
    const uint4 v = __ldg(Y + i);
    G[i] = make_uint4(gelu_bf16x2(v.x), gelu_bf16x2(v.y), gelu_bf16x2(v.z), gelu_bf16x2(v.w));
  }
}

template <bool FUSED, int RD>
int max_pairs_for(int sm_count) {
  static int cache[64] = {0};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 64 && cache[dev] > 0) return cache[dev];
  cudaError_t e = cudaFuncSetAttribute(k2_kernel<FUSED, RD>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       Cfg<FUSED>::SMEM_BYTES);
  if (e != cudaSuccess) return -int(e);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * (sm_count / 2), 1, 1);
  cfg.blockDim = dim3(THREADS, 1, 1);
  cfg.dynamicSmemBytes = Cfg<FUSED>::SMEM_BYTES;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, k2_kernel<FUSED, RD>, &cfg) != cudaSuccess || n <= 0) {
    cudaGetLastError();
    n = sm_count / 2;
  }
  if (dev < 64) cache[dev] = n;
  return n;
}

// Launched as a programmatic dependent of the previous kernel in the stream: the prologue and
// the first weight loads run while that kernel drains (only the TMA producer waits on it).
template <bool FUSED, int RD>
int launch(const K2Maps& maps, const K2Args& a, int sm_count, void* stream) {
  const int max_pairs = max_pairs_for<FUSED, RD>(sm_count);
  if (max_pairs < 0) return -max_pairs;
  const int64_t num_n = ceil_div(a.N, BN);
  const int64_t units = ceil_div(a.M, 2 * BM) * ceil_div(num_n, a.unit_len);
  if (units == 0) return 0;
  const int pairs = int(units < max_pairs ? units : max_pairs);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * pairs, 1, 1);
  cfg.blockDim = dim3(THREADS, 1, 1);
  cfg.dynamicSmemBytes = Cfg<FUSED>::SMEM_BYTES;
  cfg.stream = static_cast<cudaStream_t>(stream);
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return int(cudaLaunchKernelEx(&cfg, k2_kernel<FUSED, RD>, maps, a));
}

}  // namespace

size_t k2_smem_bytes() { return Cfg<false>::SMEM_BYTES; }

int k2_launch(const K2Maps& maps, const K2Args& a, int sm_count, void* stream) {
  if (a.unit_len != 1) return int(cudaErrorInvalidValue);
  return launch<false, 0>(maps, a, sm_count, stream);
}

int k2_fused_pairs(int sm_count) {
  const int n = max_pairs_for<true, 0>(sm_count);
  return n > 0 ? n : sm_count / 2;
}

// Unit length with the shortest schedule (whole rounds of units over the pairs, in tiles);
// ties go to the longer unit, which has fewer partial sums.
int k2_fused_unit_len(int64_t M, int64_t N, int pairs) {
  const int64_t num_mp = ceil_div(M, 2 * BM), num_n = ceil_div(N, BN);
  if (num_mp == 0 || num_n == 0 || pairs <= 0) return 1;
  int64_t best_u = 1, best = INT64_MAX;
  for (int64_t u = 1; u <= num_n; ++u) {
    const int64_t units = num_mp * ceil_div(num_n, u);
    const int64_t span = ceil_div(units, pairs) * u;
    if (span <= best) {
      best = span;
      best_u = u;
    }
  }
  return int(best_u);
}

int64_t k2_fused_partials(int64_t M, int64_t N, int unit_len) {
  (void)M;
  return 2 * ceil_div(ceil_div(N, BN), unit_len);
}

int k2_fused_launch(const K2Maps& maps, const K2Args& a, int sm_count, void* stream) {
  switch (a.fuse.rd) {
    case 0: return launch<true, 0>(maps, a, sm_count, stream);
    case 16: return launch<true, 16>(maps, a, sm_count, stream);
    case 32: return launch<true, 32>(maps, a, sm_count, stream);
    case 48: return launch<true, 48>(maps, a, sm_count, stream);
    case 64: return launch<true, 64>(maps, a, sm_count, stream);
    default: return int(cudaErrorInvalidValue);
  }
}

int k2_t_reduce_launch(const float* part, int64_t P, int64_t M, int rd, int r_pad, float inv_alpha, uint16_t* T,
                       void* stream) {
  const int64_t n = M * (r_pad / 2);
  if (n == 0) return 0;
  const int64_t blocks = std::min<int64_t>(ceil_div(n, 256), 148 * 8);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(unsigned(blocks), 1, 1);
  cfg.blockDim = dim3(256, 1, 1);
  cfg.stream = static_cast<cudaStream_t>(stream);
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return int(cudaLaunchKernelEx(&cfg, k2_t_reduce_kernel, part, P, M, rd, r_pad, inv_alpha, T));
}

int gelu_launch(const uint16_t* Y, uint16_t* G, int64_t n, int sm_count, void* stream) {
  const int64_t n8 = n / 8;
  if (n8 == 0) return 0;
  const int64_t blocks = std::min<int64_t>(ceil_div(n8, 256), int64_t(sm_count) * 8);
  gelu_kernel<<<unsigned(blocks), 256, 0, static_cast<cudaStream_t>(stream)>>>(
      reinterpret_cast<const uint4*>(Y), reinterpret_cast<uint4*>(G), n8);
  return int(cudaGetLastError());
}

void k2_l1_fragments(const uint16_t* L1p, int64_t K, int rd, uint16_t* out) {
  const int np_n = rd / 16;
  for (int64_t st = 0; st < K / 16; ++st)
    for (int np = 0; np < np_n; ++np)
      for (int l = 0; l < 32; ++l) {
        const int g = l / 4, t = l % 4;
        uint16_t* o = out + ((st * np_n + np) * 32 + l) * 8;
        for (int gi = 0; gi < 2; ++gi) {
          const int n = 16 * np + 8 * gi + g;
          const int64_t k0 = 16 * st + 2 * t;
          o[4 * gi + 0] = L1p[(k0)*rd + n];
          o[4 * gi + 1] = L1p[(k0 + 1) * rd + n];
          o[4 * gi + 2] = L1p[(k0 + 8) * rd + n];
          o[4 * gi + 3] = L1p[(k0 + 9) * rd + n];
        }
      }
}

}  // namespace svdq
