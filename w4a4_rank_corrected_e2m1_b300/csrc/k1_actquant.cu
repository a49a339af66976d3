// Kernel 1: one pass over the bf16 activations X that
//   (a) smooths them, x^ = fl32(x * inv_lambda)            (stage one of SVDQuant),
//   (b) quantises x^ to NVFP4: one E4M3 scale per 16 elements, E2M1 codes (stage three),
//   (c) computes the low-rank down-projection T = X^ L1 of the 16-bit branch (stage two),
// so X is read from HBM exactly once: both branches of the layer consume the same smoothed
// input, which the Nunchaku section of the aiflownews article on Nunchaku in Diffusers gives
// as the reason to fuse them.
//
// Two kernels do this.  k1_tall_kernel (further down) takes 32 rows and the whole of K per CTA;
// it runs when M fills the GPU with 32-row tiles or K <= 6144.  k1_kernel, described here, splits
// K for long K at small M.
//
// Work decomposition (k1_kernel).  A CTA owns a tile of 128 rows and every nsplit-th 64-column
// chunk of K (a K split).  At the end each CTA writes its partial down-projection (float32) to
// the workspace; the last CTA of the row tile to arrive adds the partials in split order
// (deterministic whatever the arrival order), scales by 1/alpha and writes T in bfloat16.
// Arrival is counted in one 64-bit word per row tile holding (launch epoch << 8) | count,
// updated by compare-and-swap: a word left by an earlier launch (finished, aborted, or another
// layer's use of the same memory) carries another epoch and restarts the count, so the
// workspace needs no clearing; the last CTA puts the word back to zero, so a replayed launch
// with the same epoch starts clean as well.
//
// Data movement.  The kernel is bound by HBM bandwidth, and each SM's TMA unit takes a copy
// instruction every few tens of nanoseconds whatever its size, so a stage is two large copies:
// the 128 x 64 bf16 X tile (one tensor copy, 128-byte swizzle) and the chunk's slice of L1
// (with 1/lambda folded in, transposed and pre-swizzled at pack time) followed by its 64
// values of 1/lambda (one bulk copy).
//
// Roles of k1_kernel (320 threads):
//   warps 0..7  quantisers: each takes 16 rows of the tile; thread (g = lane/4, t = lane%4)
//               takes rows g and g+8 and the 16 bf16 at columns 16t..16t+15 of the chunk:
//               exactly one NVFP4 block, so the block maximum needs no shuffles and a quad
//               writes 32 contiguous bytes of codes per row
//   warp 8      TMA producer
//   warp 9      TMEM owner and MMA issuer: the X tile in shared memory is the A operand of
//               tcgen05.mma kind::f16 (M = 128, K = 16, bf16), the L1 slice the B operand
//               (N = rank); T accumulates in TMEM across the CTA's chunks
// The E2M1 conversion (cvt.rn.satfinite.e2m1x2) rounds to nearest even and keeps the sign of
// a negative value that rounds to zero, which is the format rule the codes follow.  Block
// scale code: s8 = E4M3(fl32(amax / fl32(6 s_gX))); one product with the reciprocal lands
// within one code of it and host-built thresholds (thr[c] = smallest amax whose code is >= c)
// settle the code exactly; the element scale 1/d comes from a host-built table of
// fl32(1 / fl32(E4M3value(c) * s_gX)).
#include <cuda.h>
#include <cuda_runtime.h>

#include "nvfp4_block.cuh"
#include "ptx.cuh"
#include "svdq_internal.h"

namespace svdq {

namespace {

constexpr int kQWarps = 8;                // quantiser warps
constexpr int kProducer = kQWarps;        // warp 8
constexpr int kMma = kQWarps + 1;         // warp 9
constexpr int kThreads = 32 * (kQWarps + 2);
constexpr int kRows = 128;                // rows per CTA (TMEM lanes)
constexpr uint32_t kFull = 0xFFFFFFFFu;
constexpr uint64_t kTimeoutNs = 2000000000ull;

struct alignas(64) XMap {
  unsigned char m[128];
};

template <int R>   // R = rank (0 or a multiple of 16, <= 128)
struct Cfg {
  static constexpr int X_BYTES = kRows * 128;              // 128 rows x 64 bf16
  static constexpr int L_BYTES = R * 128;                  // R rows x 64 bf16 (L1 slice, transposed)
  static constexpr int LI_BYTES = L_BYTES + 256;           // + 64 floats of 1/lambda
  static constexpr int STAGE_BYTES = ((X_BYTES + LI_BYTES + 1023) / 1024) * 1024;
  static constexpr int STAGES = R > 64 ? 3 : 4;              // two CTAs per SM at every rank
  static constexpr int RING_BYTES = STAGES * STAGE_BYTES;
  static constexpr int RED_BYTES = kRows * (R > 0 ? R : 1) * 4;   // this CTA's partial T
  static constexpr int SMEM = (RING_BYTES > RED_BYTES ? RING_BYTES : RED_BYTES) + 1024;
  static constexpr uint32_t TMEM_COLS = R <= 32 ? 32 : (R <= 64 ? 64 : 128);
  // kind::f16, D f32, A/B bf16, K-major, N = R, M = 128
  static constexpr uint32_t IDESC = (1u << 4) | (1u << 7) | (1u << 10) | (uint32_t(R >> 3) << 17) | (uint32_t(128 >> 4) << 24);
};

// The L1 / 1/lambda buffer comes in groups of four 64-column chunks (4g .. 4g + 3):
//   [L1' slices of the four chunks][1/lambda of the four chunks]
// each slice R rows x 128 bytes (bf16, K-major, 128-byte swizzle), each 1/lambda part 64 fp32.
constexpr int kLIGroup = 4;
__host__ __device__ constexpr int64_t li_group_bytes(int R) { return int64_t(kLIGroup) * (R * 128 + 256); }

// Split kernel: chunk c's slice and 1/lambda values into the stage, after its X tile.
template <int R>
__device__ __forceinline__ void li_loads(unsigned char* st, const unsigned char* LI, int c, uint64_t* bar) {
  const unsigned char* g = LI + int64_t(c / kLIGroup) * li_group_bytes(R);
  const int i = c % kLIGroup;
  constexpr int X_BYTES = 128 * 128, L_BYTES = R * 128;
  if (R > 0) ptx::bulk_load(st + X_BYTES, g + i * L_BYTES, L_BYTES, bar);
  ptx::bulk_load(st + X_BYTES + L_BYTES, g + kLIGroup * L_BYTES + i * 256, 256, bar);
}

__device__ bool k1_wait(uint64_t* bar, uint32_t parity, volatile int* abort_flag, int* err, uint64_t limit_ns) {
  if (ptx::mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = ptx::globaltimer();
  for (uint32_t i = 1;; ++i) {
    if (ptx::mbar_try_wait(bar, parity)) return true;
    if ((i & 31u) == 0u) {
      if (*abort_flag) return false;
      if (ptx::globaltimer() - t0 > limit_ns) {
        *abort_flag = 1;
        atomicOr(err, 4);
        return false;
      }
    }
  }
}
// Waits for work already started (ignores the abort flag; gives up after the default limit).
__device__ void k1_drain(uint64_t* bar, uint32_t parity, int* err) {
  const uint64_t t0 = ptx::globaltimer();
  while (!ptx::mbar_try_wait(bar, parity)) {
    if (ptx::globaltimer() - t0 > kTimeoutNs) {
      atomicOr(err, 4);
      return;
    }
  }
}

template <int R>
__global__ void __launch_bounds__(kThreads, 2)
    k1_kernel(const __grid_constant__ XMap xmap, K1Args a) {
  using C = Cfg<R>;
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* ring = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  __shared__ uint64_t full[C::STAGES], empty[C::STAGES], done, never;
  __shared__ volatile int abort_flag;
  __shared__ uint32_t tmem_slot;
  __shared__ float s_thr[128], s_rcp[128];

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, t = lane & 3;
  const int64_t M = a.M, K = a.K;
  const int64_t KG = scale_groups(K);
  const int nchunks = int(K / 64);
  const int split = blockIdx.y, nsplit = gridDim.y;
  // split s takes chunks s, s + nsplit, s + 2 nsplit, ...: the splits of a row tile read
  // neighbouring column ranges at the same time
  const int c0 = split;
  const int64_t row0 = int64_t(blockIdx.x) * kRows;

  ptx::griddep_launch_dependents();
  // the quantiser tables (pack-time constants) are loaded into registers here and stored after
  // the block barrier, so that no role waits for this load before its first step: threads
  // 0..255 all belong to quantiser warps, which meet at barrier 3 before reading the tables
  const float qv = threadIdx.x < 256 ? __ldg(a.qtab + threadIdx.x) : 0.f;
  if (threadIdx.x == 0) {
    for (int i = 0; i < C::STAGES; ++i) {
      ptx::mbar_init(&full[i], 1);
      ptx::mbar_init(&empty[i], kQWarps + (R > 0 ? 1 : 0));
    }
    ptx::mbar_init(&done, 1);
    ptx::mbar_init(&never, 1);   // arrived at by nothing (the failure-detection stall waits on it)
    abort_flag = 0;
    ptx::fence_barrier_init();
  }
  if (R > 0 && warp == kMma) {
    ptx::tmem_alloc(&tmem_slot, C::TMEM_COLS);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  // every role's bounded waits start once the previous grid is done (the producer first
  // requests the constant L1 slices, then waits)
  if (warp != kProducer) ptx::griddep_wait();

  if (warp == kProducer) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      ptx::prefetch_tmap(&xmap);
      // The L1 / 1/lambda slices are pack-time constants: those of the first ring pass are
      // requested before waiting for the previous grid (programmatic dependent launch); X,
      // which that grid may have produced, only after.
      int pre = 0;
      for (int c = c0; c < nchunks && pre < C::STAGES; c += nsplit, ++pre) {
        unsigned char* st = ring + pre * C::STAGE_BYTES;
        ptx::mbar_arrive_expect_tx(&full[pre], C::X_BYTES + C::LI_BYTES);
        li_loads<R>(st, a.LI, c, &full[pre]);
      }
      ptx::griddep_wait();
      int stage = 0, issued = 0;
      uint32_t phase = 0;
      for (int c = c0; c < nchunks; c += nsplit, ++issued) {
        unsigned char* st = ring + stage * C::STAGE_BYTES;
        if (issued >= pre) {
          if (!k1_wait(&empty[stage], phase ^ 1u, &abort_flag, a.err, a.wait_ns)) break;
          // the quantiser warps read this stage with ordinary loads before releasing it; the
          // proxy fence orders those reads before the tensor copies that overwrite it
          ptx::fence_proxy_async_smem();
          ptx::mbar_arrive_expect_tx(&full[stage], C::X_BYTES + C::LI_BYTES);
          li_loads<R>(st, a.LI, c, &full[stage]);
        }
        ptx::tma_load_2d(st, &xmap, &full[stage], 64 * c, int(row0));
        if (++stage == C::STAGES) { stage = 0; phase ^= 1u; }
      }
      // every copy issued has landed before shared memory is reused or released
      for (int i = 0; i < C::STAGES; ++i) {
        const int used = issued - i;
        if (used <= 0) continue;
        const uint32_t last_parity = uint32_t(((used - 1) / C::STAGES) & 1);
        const uint64_t t0 = ptx::globaltimer();
        while (!ptx::mbar_try_wait(&full[i], last_parity))
          if (ptx::globaltimer() - t0 > kTimeoutNs) break;
      }
    }
  } else if (warp == kMma) {
    // ------------------------------------------------------------ MMA issuer (down-projection)
    if (R > 0 && lane == 0) {
      const uint32_t tmem = tmem_slot;
      int stage = 0;
      uint32_t phase = 0;
      uint32_t accumulate = 0;
      const bool stalled = a.stall && !k1_wait(&never, 0, &abort_flag, a.err, a.wait_ns);
      for (int c = c0; c < nchunks && !stalled; c += nsplit) {
        if (!k1_wait(&full[stage], phase, &abort_flag, a.err, a.wait_ns)) break;
        ptx::tc_fence_after();
        const uint32_t xs = ptx::smem_u32(ring + stage * C::STAGE_BYTES);
        const uint32_t ls = xs + C::X_BYTES;
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
          ptx::mma_bf16(tmem, ptx::desc_sw128(xs + 32 * kk), ptx::desc_sw128(ls + 32 * kk), C::IDESC, accumulate);
          accumulate = 1;
        }
        ptx::tc_commit(&empty[stage]);
        if (++stage == C::STAGES) { stage = 0; phase ^= 1u; }
      }
      ptx::tc_commit(&done);
    }
  } else {
    // ------------------------------------------------------------ quantiser warps
    if (threadIdx.x < 256) (threadIdx.x < 128 ? s_thr[threadIdx.x] : s_rcp[threadIdx.x - 128]) = qv;
    ptx::bar_sync(3, 32 * kQWarps);
    int stage = 0;
    uint32_t phase = 0;
    for (int c = c0; c < nchunks; c += nsplit) {
      if (!k1_wait(&full[stage], phase, &abort_flag, a.err, a.wait_ns)) break;
      const unsigned char* st = ring + stage * C::STAGE_BYTES;
      // raw bf16 of rows g (w[0]) and g + 8 (w[1]) of this warp, columns 16t .. 16t + 15
      uint32_t w[2][8];
      float il[16];
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int lr = 16 * warp + g + 8 * h;
        const unsigned char* rowp = st + lr * 128;
        const uint4 u0 = *reinterpret_cast<const uint4*>(rowp + (((2 * t) ^ (lr & 7)) << 4));
        const uint4 u1 = *reinterpret_cast<const uint4*>(rowp + (((2 * t + 1) ^ (lr & 7)) << 4));
        w[h][0] = u0.x; w[h][1] = u0.y; w[h][2] = u0.z; w[h][3] = u0.w;
        w[h][4] = u1.x; w[h][5] = u1.y; w[h][6] = u1.z; w[h][7] = u1.w;
      }
      {
        const float4* p = reinterpret_cast<const float4*>(st + C::X_BYTES + C::L_BYTES) + 4 * t;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const float4 v = p[k ^ (t >> 1)];   // bank-spread layout of the 1/lambda part
          il[4 * k] = v.x; il[4 * k + 1] = v.y; il[4 * k + 2] = v.z; il[4 * k + 3] = v.w;
        }
      }
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(&empty[stage]);
      if (++stage == C::STAGES) { stage = 0; phase ^= 1u; }

      const int64_t col = int64_t(c) * 64 + 16 * t;
      // both blocks first (independent chains), then the shuffles, then the stores
      uint32_t s8[2], code0[2], code1[2], word[2];
#pragma unroll
      for (int h = 0; h < 2; ++h) s8[h] = quant_block(w[h], il, a.inv_six, s_thr, s_rcp, &code0[h], &code1[h]);
      // the quad's four scale bytes of a row form one 32-bit word of the tiled layout
#pragma unroll
      for (int h = 0; h < 2; ++h) word[h] = s8[h] << (8 * t);
#pragma unroll
      for (int h = 0; h < 2; ++h) word[h] |= __shfl_xor_sync(kFull, word[h], 1);
#pragma unroll
      for (int h = 0; h < 2; ++h) word[h] |= __shfl_xor_sync(kFull, word[h], 2);
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int64_t row = row0 + 16 * warp + g + 8 * h;
        if (row < M) {
          uint2* dst = reinterpret_cast<uint2*>(a.x_codes + row * (K / 2) + col / 2);
          *dst = make_uint2(code0[h], code1[h]);
        }
        if (t == h) *reinterpret_cast<uint32_t*>(a.x_scales + scale_word_offset(row, c, KG)) = word[h];
      }
    }
    // scale groups past K (K not a multiple of 256) read as zero scales by the GEMM
    if (split == nsplit - 1) {
      for (int c = nchunks; c < KG; ++c) {
        const int64_t row = row0 + 16 * warp + g + 8 * t;
        if (t < 2) *reinterpret_cast<uint32_t*>(a.x_scales + scale_word_offset(row, c, KG)) = 0u;
      }
    }
  }

  // ---- partial down-projection out; the last CTA of the row tile reduces and stores T
  if constexpr (R > 0) {
    __shared__ int s_last;
    float* part = a.partial + (int64_t(blockIdx.x) * kK1MaxSplit + split) * (R * kRows);
    if (warp < 4) {
      // TMEM lane quarter = warp: rows 32 warp + lane; column-major partial, so each store of
      // one column by the warp is 128 contiguous bytes
      // a CTA whose K range is empty (more splits than chunks) contributes zeros
      // the MMAs have completed before TMEM is read (or freed), also after an abort
      k1_drain(&done, 0, a.err);
      const bool ok = !abort_flag && c0 < nchunks;
      ptx::tc_fence_after();
      const uint32_t tbase = tmem_slot + (uint32_t(32 * warp) << 16);
#pragma unroll
      for (int cb = 0; cb < R; cb += 32) {
        uint32_t v[32];
        ptx::tmem_ld_32x32b_x32(tbase + cb, v);
        ptx::tmem_wait_ld();
#pragma unroll
        for (int j = 0; j < 32; ++j)
          if (cb + j < R) part[(cb + j) * kRows + 32 * warp + lane] = ok ? __uint_as_float(v[j]) : 0.f;
      }
      __threadfence();
    }
    ptx::tc_fence_before();
    __syncthreads();
    if (threadIdx.x == 0) {
      unsigned long long* word = a.arrivals + blockIdx.x;
      const unsigned long long tag = a.epoch << 8;
      unsigned long long v = atomicAdd(word, 0ull), nv = 0ull;
      bool swapped = false;
      for (int it = 0; it < 4096 && !swapped; ++it) {
        nv = (v >> 8) == a.epoch ? v + 1 : (tag | 1ull);
        const unsigned long long old = atomicCAS(word, v, nv);
        swapped = old == v;
        v = old;
      }
      if (!swapped) atomicOr(a.err, 8);
      const bool last = swapped && nv == (tag | unsigned(nsplit));
      if (last) atomicExch(word, 0ull);
      s_last = last ? 1 : 0;
      __threadfence();
    }
    __syncthreads();
    if (s_last) {
      // one item = 4 rows x 2 columns; every split's float4 of both columns is loaded before
      // any is added (the adds then run in split order)
      const float* pt = a.partial + int64_t(blockIdx.x) * kK1MaxSplit * (R * kRows);
      const int r_pad = a.r_pad;
      for (int e = threadIdx.x; e < (kRows / 4) * (r_pad / 2); e += blockDim.x) {
        const int rq = e % (kRows / 4), cp = e / (kRows / 4);
        uint32_t v[4] = {0u, 0u, 0u, 0u};
        if (2 * cp < R) {
          float4 p0[kK1MaxSplit], p1[kK1MaxSplit];
#pragma unroll
          for (int q = 0; q < kK1MaxSplit; ++q) {
            if (q < nsplit) {
              const float4* pq = reinterpret_cast<const float4*>(pt + q * (R * kRows) + (2 * cp) * kRows) + rq;
              p0[q] = __ldcg(pq);
              p1[q] = __ldcg(pq + kRows / 4);
            }
          }
          float4 s0 = p0[0], s1 = p1[0];
#pragma unroll
          for (int q = 1; q < kK1MaxSplit; ++q) {
            if (q < nsplit) {
              s0.x += p0[q].x; s0.y += p0[q].y; s0.z += p0[q].z; s0.w += p0[q].w;
              s1.x += p1[q].x; s1.y += p1[q].y; s1.z += p1[q].z; s1.w += p1[q].w;
            }
          }
          const float ia = a.inv_alpha;
          v[0] = ptx::pack_bf16x2(s0.x * ia, s1.x * ia);
          v[1] = ptx::pack_bf16x2(s0.y * ia, s1.y * ia);
          v[2] = ptx::pack_bf16x2(s0.z * ia, s1.z * ia);
          v[3] = ptx::pack_bf16x2(s0.w * ia, s1.w * ia);
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int64_t row = row0 + 4 * rq + i;
          if (row < M) reinterpret_cast<uint32_t*>(a.T + row * r_pad)[cp] = v[i];
        }
      }
    }
    if (warp == kMma) {
      ptx::tc_fence_after();
      ptx::tmem_dealloc(tmem_slot, C::TMEM_COLS);
    }
  }
}

// ------------------------------------------------------------------ tall kernel
// For M large enough to fill the GPU with 32-row tiles, a CTA takes 32 rows and the whole of
// K, so the down-projection needs no split and no cross-CTA reduction.  A stage is CH
// consecutive 64-column chunks (CH x 128 contiguous bytes of every row, so DRAM pages are
// read in long runs): CH 32 x 64 X tiles (TMA) and the chunks' L1 slices and 1/lambda parts
// (bulk copies).
//
// Down-projection for r <= 64 (four chunks a stage): the stage's four 32-row X tiles lie back
// to back, so together they are one 128-row A operand, and the four L1 slices are one
// (4 r)-row B operand.  One tcgen05.mma with M = 128, N = 4 r per 16-wide k-step multiplies
// them; block (q, q) of the product (TMEM lanes 32 q .. 32 q + 31, columns q r .. q r + r - 1)
// is chunk q's contribution to T, the off-diagonal blocks are never read, and T is the sum of
// the four diagonal blocks at the end.  Against one M = 128, N = r product per chunk (whose
// rows 32..127 would be wasted) this reads 2.5x fewer operand bytes from shared memory and
// issues 4x fewer instructions.  For r > 64 each chunk is its own M = 128, N = r product; its A
// rows 32..127 run into the following shared memory and only produce TMEM lanes 32..127,
// which nothing reads (a pad after the ring keeps those reads inside the CTA's shared memory).
//
// The quantiser warps, not the stream, set the pace of this kernel: a warp's blocks are short
// dependency chains, so there are as many warps as the register budget allows (16 with four
// chunks a stage, one 8-row x 64-column piece each).
constexpr int kTallRows = 32;

template <int R>
struct TallCfg {
  static constexpr int CH = R <= 96 ? 4 : 2;                    // chunks per stage
  static constexpr int QW = 4 * CH;                            // quantiser warps: 8 rows of a chunk each
  static constexpr int PRODUCER = QW, MMA = QW + 1, THREADS = 32 * (QW + 2);
  static constexpr int X_TILE = kTallRows * 128;               // 32 rows x 64 bf16
  static constexpr int X_BYTES = CH * X_TILE;
  static constexpr int L_BYTES = R * 128;
  static constexpr int LI_BYTES = CH * (L_BYTES + 256);
  static constexpr int STAGE_BYTES = ((X_BYTES + LI_BYTES + 1023) / 1024) * 1024;
  static constexpr int STAGES = (204 * 1024) / STAGE_BYTES > 8 ? 8 : (204 * 1024) / STAGE_BYTES;
  static constexpr bool STACK = R > 0 && R <= 64;              // one M = 128 product over the four chunks
  static constexpr int N_MMA = STACK ? CH * R : R;
  static constexpr int SPAN = STACK ? X_BYTES : (CH - 1) * X_TILE + 128 * 128;   // farthest A byte read
  static constexpr int PAD = SPAN > STAGE_BYTES ? SPAN - STAGE_BYTES : 0;
  static constexpr int SMEM = STAGES * STAGE_BYTES + PAD + 1024;
  static constexpr int WPC = QW / CH;                          // quantiser warps per chunk
  static constexpr int RPT = kTallRows / WPC / 8;              // rows per thread
  // STACK: every warp quarter q loads 32-column pieces from column q r on
  static constexpr uint32_t TMEM_COLS = STACK ? (R <= 32 ? 128 : 256) : (R <= 32 ? 32 : (R <= 64 ? 64 : 128));
  static constexpr uint32_t IDESC =
      (1u << 4) | (1u << 7) | (1u << 10) | (uint32_t(N_MMA >> 3) << 17) | (uint32_t(128 >> 4) << 24);
  static_assert(!STACK || 3 * R + ((R + 31) / 32) * 32 <= int(TMEM_COLS), "TMEM columns");
  static_assert(!STACK || N_MMA <= 256, "MMA N");
  static_assert(!STACK || 3 * 32 * R * 4 <= STAGE_BYTES, "reduction buffer fits in one stage");
  // K split: this CTA's share [R][32] after the reduction buffer, then rank 0's receiving slots
  static constexpr int PART_OFF = STACK ? 3 * 32 * R : 0;          // floats from the ring's start
  static constexpr int RECV_OFF = PART_OFF + 32 * R;
  static_assert((RECV_OFF + kK1TallMaxSplit * 32 * R) * 4 <= STAGES * STAGE_BYTES, "split shares fit in the ring");
  static_assert(STAGES >= 3, "stages");
  static_assert(RPT == 1, "one row per thread");
  static_assert(QW >= 8, "threads 0..255 (the quantiser-table loads) are quantiser threads");
};

// Stage j's L1 slices and 1/lambda parts: [CH slices][CH 1/lambda parts].
template <int R>
__device__ __forceinline__ void tall_li_loads(unsigned char* dst, const unsigned char* LI, int j, uint64_t* bar) {
  using C = TallCfg<R>;
  const int c0 = C::CH * j;
  const unsigned char* g = LI + int64_t(c0 / kLIGroup) * li_group_bytes(R);
  const int i = c0 % kLIGroup;
  if (C::CH == kLIGroup) {
    ptx::bulk_load(dst, g, C::LI_BYTES, bar);
  } else {
    if (R > 0) ptx::bulk_load(dst, g + i * C::L_BYTES, C::CH * C::L_BYTES, bar);
    ptx::bulk_load(dst + C::CH * C::L_BYTES, g + kLIGroup * C::L_BYTES + i * 256, C::CH * 256, bar);
  }
}

template <int R>
__global__ void __launch_bounds__(TallCfg<R>::THREADS, 1)
    k1_tall_kernel(const __grid_constant__ XMap xmap, K1Args a) {
  using C = TallCfg<R>;
  constexpr int kProducer = C::PRODUCER, kMma = C::MMA, kQWarps = C::QW;
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* ring = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  __shared__ uint64_t full[C::STAGES], empty[C::STAGES], done, never;
  __shared__ volatile int abort_flag;
  __shared__ uint32_t tmem_slot;
  __shared__ float s_thr[128], s_rcp[128];

  ptx::griddep_launch_dependents();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, t = lane & 3;
  const int64_t M = a.M, K = a.K;
  const int64_t KG = scale_groups(K);
  const int nchunks = int(K / 64);
  const int nsteps_all = (nchunks + C::CH - 1) / C::CH;
  // this CTA's 32-row tile and its stages [s_begin, s_begin + nsteps) of K (a.tsplit CTAs per
  // tile at small M, one otherwise)
  const int tsplit = a.tsplit, sp = int(blockIdx.x) % tsplit, rtile = int(blockIdx.x) / tsplit;
  const int s_begin = tsplit > 1 ? sp * a.tsteps : 0;
  const int s_end = tsplit > 1 ? min(nsteps_all, s_begin + a.tsteps) : nsteps_all;
  const int nsteps = s_end > s_begin ? s_end - s_begin : 0;
  const int64_t row0 = int64_t(rtile) * kTallRows;

  // the quantiser tables (pack-time constants) are loaded into registers here and stored after
  // the block barrier, so that no role waits for this load before its first step: threads
  // 0..255 all belong to quantiser warps, which meet at barrier 3 before reading the tables
  const float qv = threadIdx.x < 256 ? __ldg(a.qtab + threadIdx.x) : 0.f;
  if (threadIdx.x == 0) {
    for (int i = 0; i < C::STAGES; ++i) {
      ptx::mbar_init(&full[i], 1);
      ptx::mbar_init(&empty[i], kQWarps + (R > 0 ? 1 : 0));
    }
    ptx::mbar_init(&done, 1);
    ptx::mbar_init(&never, 1);   // arrived at by nothing (the failure-detection stall waits on it)
    abort_flag = 0;
    ptx::fence_barrier_init();
  }
  if (R > 0 && warp == kMma) {
    ptx::tmem_alloc(&tmem_slot, C::TMEM_COLS);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  if (warp != kProducer) ptx::griddep_wait();

  if (warp == kProducer) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      ptx::prefetch_tmap(&xmap);
      // the L1 / 1/lambda parts of the first ring pass are constants: requested before the
      // grid wait
      const int pre = nsteps < C::STAGES ? nsteps : C::STAGES;
      for (int st_i = 0; st_i < pre; ++st_i) {
        unsigned char* st = ring + st_i * C::STAGE_BYTES;
        ptx::mbar_arrive_expect_tx(&full[st_i], C::X_BYTES + C::LI_BYTES);
        tall_li_loads<R>(st + C::X_BYTES, a.LI, s_begin + st_i, &full[st_i]);
      }
      ptx::griddep_wait();
      int stage = 0, issued = 0;
      uint32_t phase = 0;
      for (int j = 0; j < nsteps; ++j, ++issued) {
        unsigned char* st = ring + stage * C::STAGE_BYTES;
        if (j >= pre) {
          if (!k1_wait(&empty[stage], phase ^ 1u, &abort_flag, a.err, a.wait_ns)) break;
          ptx::fence_proxy_async_smem();   // ordinary-load reads of the stage before the refill
          ptx::mbar_arrive_expect_tx(&full[stage], C::X_BYTES + C::LI_BYTES);
          tall_li_loads<R>(st + C::X_BYTES, a.LI, s_begin + j, &full[stage]);
        }
        // a chunk index past K reads as zeros (out-of-range box) and still delivers its bytes
#pragma unroll
        for (int cc = 0; cc < C::CH; ++cc)
          ptx::tma_load_2d(st + cc * C::X_TILE, &xmap, &full[stage], 64 * (C::CH * (s_begin + j) + cc), int(row0));
        if (++stage == C::STAGES) { stage = 0; phase ^= 1u; }
      }
      for (int i = 0; i < C::STAGES; ++i) {       // every copy issued has landed
        const int used = issued - i;
        if (used <= 0) continue;
        const uint32_t last_parity = uint32_t(((used - 1) / C::STAGES) & 1);
        const uint64_t t0 = ptx::globaltimer();
        while (!ptx::mbar_try_wait(&full[i], last_parity))
          if (ptx::globaltimer() - t0 > kTimeoutNs) break;
      }
    }
  } else if (warp == kMma) {
    // ------------------------------------------------------------ MMA issuer (down-projection)
    if (R > 0 && lane == 0) {
      const uint32_t tmem = tmem_slot;
      int stage = 0;
      uint32_t phase = 0;
      uint32_t accumulate = 0;
      const bool stalled = a.stall && !k1_wait(&never, 0, &abort_flag, a.err, a.wait_ns);
      for (int j = 0; j < nsteps && !stalled; ++j) {
        if (!k1_wait(&full[stage], phase, &abort_flag, a.err, a.wait_ns)) break;
        ptx::tc_fence_after();
        const uint32_t xs = ptx::smem_u32(ring + stage * C::STAGE_BYTES);
        const uint32_t ls = xs + C::X_BYTES;
        if constexpr (C::STACK) {
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            ptx::mma_bf16(tmem, ptx::desc_sw128(xs + 32 * kk), ptx::desc_sw128(ls + 32 * kk), C::IDESC, accumulate);
            accumulate = 1;
          }
        } else {
#pragma unroll
          for (int cc = 0; cc < C::CH; ++cc)
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
              ptx::mma_bf16(tmem, ptx::desc_sw128(xs + cc * C::X_TILE + 32 * kk),
                            ptx::desc_sw128(ls + cc * C::L_BYTES + 32 * kk), C::IDESC, accumulate);
              accumulate = 1;
            }
        }
        ptx::tc_commit(&empty[stage]);
        if (++stage == C::STAGES) { stage = 0; phase ^= 1u; }
      }
      ptx::tc_commit(&done);
    }
  } else {
    // ------------------------------------------------------------ quantiser warps
    if (threadIdx.x < 256) (threadIdx.x < 128 ? s_thr[threadIdx.x] : s_rcp[threadIdx.x - 128]) = qv;
    ptx::bar_sync(3, 32 * kQWarps);
    // warp w takes chunk w / 4 of the stage and rows 8 (w % 4) .. 8 (w % 4) + 7; thread (g, t)
    // takes the 16-element block at columns 16 t .. 16 t + 15 of row 8 (w % 4) + g.  Its
    // addresses are computed once and advance by CH chunks a stage.
    const int cc = warp / C::WPC;
    const int r = (warp % C::WPC) * 8 + g;                      // r % 8 == g: the swizzle row
    const int64_t row = row0 + r;
    const bool live = row < M;
    unsigned char* code_p = a.x_codes + row * (K / 2) + (C::CH * s_begin + cc) * 32 + 8 * t;
    unsigned char* scale_p = a.x_scales + scale_word_offset(row, C::CH * s_begin + cc, KG);
    const int xoff = cc * C::X_TILE + r * 128;
    const int u0off = xoff + (((2 * t) ^ g) << 4), u1off = xoff + (((2 * t + 1) ^ g) << 4);
    const int iloff = C::X_BYTES + C::CH * C::L_BYTES + cc * 256 + 64 * t;
    const int kx = t >> 1;                                      // bank-spread layout of 1/lambda
    int stage = 0;
    uint32_t phase = 0;
    for (int j = 0; j < nsteps; ++j, code_p += C::CH * 32, scale_p += C::CH * 512) {
      if (!k1_wait(&full[stage], phase, &abort_flag, a.err, a.wait_ns)) break;
      const unsigned char* st = ring + stage * C::STAGE_BYTES;
      uint32_t w[8];
      float il[16];
      {
        const uint4 u0 = *reinterpret_cast<const uint4*>(st + u0off);
        const uint4 u1 = *reinterpret_cast<const uint4*>(st + u1off);
        w[0] = u0.x; w[1] = u0.y; w[2] = u0.z; w[3] = u0.w;
        w[4] = u1.x; w[5] = u1.y; w[6] = u1.z; w[7] = u1.w;
        const float4* p = reinterpret_cast<const float4*>(st + iloff);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const float4 v = p[k ^ kx];
          il[4 * k] = v.x; il[4 * k + 1] = v.y; il[4 * k + 2] = v.z; il[4 * k + 3] = v.w;
        }
      }
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(&empty[stage]);
      if (++stage == C::STAGES) { stage = 0; phase ^= 1u; }

      if (C::CH * (s_begin + j) + cc >= nchunks) continue;
      uint32_t code0, code1;
      const uint32_t s8 = quant_block(w, il, a.inv_six, s_thr, s_rcp, &code0, &code1);
      // the quad's four scale bytes of this row form one 32-bit word of the tiled layout
      uint32_t word = s8 << (8 * t);
      word |= __shfl_xor_sync(kFull, word, 1);
      word |= __shfl_xor_sync(kFull, word, 2);
      if (live) *reinterpret_cast<uint2*>(code_p) = make_uint2(code0, code1);
      if (t == 0) *reinterpret_cast<uint32_t*>(scale_p) = word;
    }
    // scale groups past K (K not a multiple of 256) read as zero scales by the GEMM (written by
    // the CTA holding the last stage)
    for (int c = nchunks; c < KG && s_end == nsteps_all; ++c)
      if (c % C::CH == cc && t == 0) *reinterpret_cast<uint32_t*>(a.x_scales + scale_word_offset(row, c, KG)) = 0u;
    // rows after the last 32-row tile, up to the end of its 128-row scale tile, belong to no
    // CTA: the last one writes their scales as zeros
    if (blockIdx.x == gridDim.x - 1) {
      const int64_t r_first = row0 + kTallRows, r_end = (row0 / 128) * 128 + 128;
      const int64_t n = (r_end - r_first) * KG;
      for (int64_t i = threadIdx.x; i < n; i += 32 * kQWarps)
        *reinterpret_cast<uint32_t*>(a.x_scales + scale_word_offset(r_first + i / KG, i % KG, KG)) = 0u;
    }
  }

  // ---- T = (X^ L1) / alpha for the CTA's 32 rows
  if constexpr (R > 0) {
    const int64_t row = row0 + lane;
    uint4* trow = reinterpret_cast<uint4*>(a.T + row * a.r_pad);
    // with a K split, the tile's CTAs form a cluster: each keeps its float32 share [R][32 rows]
    // in shared memory (after the ring's reduction buffer), stores it into its slot of cluster
    // rank 0's shared memory, and rank 0 adds the slots in split order
    const bool split = tsplit > 1;
    float* part = reinterpret_cast<float*>(ring) + C::PART_OFF;
    // 32 columns of T from TMEM (plus the other warps' blocks in `red`), scaled, to bf16
    auto emit = [&](int cb, const uint32_t* v, const float* red, bool ok) {
#pragma unroll
      for (int j = 0; j < 32; j += 8) {
        if (cb + j < R) {
          uint32_t o[4];
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            float y[2];
#pragma unroll
            for (int e = 0; e < 2; ++e) {
              const int col = cb + j + 2 * u + e;
              y[e] = __uint_as_float(v[j + 2 * u + e]);
              if (red)
                y[e] = ((y[e] + red[col * 32 + lane]) + red[(R + col) * 32 + lane]) + red[(2 * R + col) * 32 + lane];
              if (split) part[col * 32 + lane] = ok ? y[e] : 0.f;   // this split's share, float32
            }
            o[u] = ok ? ptx::pack_bf16x2(y[0] * a.inv_alpha, y[1] * a.inv_alpha) : 0u;
          }
          if (!split && row < M) trow[(cb + j) / 8] = make_uint4(o[0], o[1], o[2], o[3]);
        }
      }
    };
    if constexpr (C::STACK) {
      // chunk position q's block lies in TMEM lanes 32 q .. 32 q + 31 from column q r on, so
      // warp q reads it; warps 1..3 pass theirs to warp 0 through the ring, free once every
      // quantiser warp is past its last stage (all the ring's copies have landed by then)
      float* red = reinterpret_cast<float*>(ring);   // [3][r][32 lanes]
      if (warp < kQWarps) ptx::bar_sync(1, 32 * kQWarps);
      if (warp < 4) {
        // the MMAs have completed before TMEM is read (or freed), also after an abort
        k1_drain(&done, 0, a.err);
        const bool ok = !abort_flag && nsteps > 0;   // (an empty split contributes zeros)
        ptx::tc_fence_after();
        if (warp > 0) {
#pragma unroll
          for (int cb = 0; cb < R; cb += 32) {
            uint32_t v[32];
            ptx::tmem_ld_32x32b_x32(tmem_slot + (uint32_t(32 * warp) << 16) + uint32_t(warp * R + cb), v);
            ptx::tmem_wait_ld();
#pragma unroll
            for (int j = 0; j < 32; ++j)
              if (cb + j < R) red[((warp - 1) * R + cb + j) * 32 + lane] = __uint_as_float(v[j]);
          }
        }
        ptx::bar_sync(2, 128);
        if (warp == 0) {
#pragma unroll
          for (int cb = 0; cb < R; cb += 32) {
            uint32_t v[32];
            ptx::tmem_ld_32x32b_x32(tmem_slot + uint32_t(cb), v);
            ptx::tmem_wait_ld();
            emit(cb, v, red, ok);
          }
        }
      }
    } else {
      // with a K split the share goes into the ring: every quantiser warp is past its last stage
      if (split && warp < kQWarps) ptx::bar_sync(1, 32 * kQWarps);
    }
    if (!C::STACK && warp == 0) {
      // one product per chunk: T is TMEM lanes 0..31 (read once the MMAs have completed, also
      // after an abort)
      k1_drain(&done, 0, a.err);
      const bool ok = !abort_flag && nsteps > 0;
      ptx::tc_fence_after();
#pragma unroll
      for (int cb = 0; cb < R; cb += 32) {
        uint32_t v[32];
        ptx::tmem_ld_32x32b_x32(tmem_slot + uint32_t(cb), v);
        ptx::tmem_wait_ld();
        emit(cb, v, nullptr, ok);
      }
    }
    if (!split && warp == 0 && row < M)
      for (int j = R; j < a.r_pad; j += 8) trow[j / 8] = make_uint4(0, 0, 0, 0);
    ptx::tc_fence_before();
    __syncthreads();
    if (warp == kMma) {
      ptx::tc_fence_after();
      ptx::tmem_dealloc(tmem_slot, C::TMEM_COLS);
    }
    if (split) {
      // every CTA of the cluster is past its mainloop (rank 0's ring is free to receive), and
      // every share is in its CTA's shared memory
      ptx::cluster_sync();
      // this split's share into slot sp of rank 0's shared memory: remote stores, made visible
      // to rank 0 by the next barrier's release and acquire
      float* recv = reinterpret_cast<float*>(ring) + C::RECV_OFF;
      const uint32_t dst = ptx::mapa(ptx::smem_u32(recv + sp * 32 * R), 0u);
      for (int e = threadIdx.x; e < 8 * R; e += blockDim.x)
        ptx::st_cluster_v4(dst + uint32_t(e) * 16u, reinterpret_cast<const float4*>(part)[e]);
      ptx::cluster_sync();
      if (sp == 0) {
        // T = (sum of the shares in split order) / alpha, 32 rows x r_pad columns (zeros past R)
        for (int e = threadIdx.x; e < 32 * (a.r_pad / 2); e += blockDim.x) {
          const int rr = e % 32, cp = e / 32;
          uint32_t o = 0u;
          if (2 * cp < R) {
            const float* s = recv + (2 * cp) * 32 + rr;
            float s0 = s[0], s1 = s[32];
            for (int q = 1; q < tsplit; ++q) {
              s0 += s[q * 32 * R];
              s1 += s[q * 32 * R + 32];
            }
            o = ptx::pack_bf16x2(s0 * a.inv_alpha, s1 * a.inv_alpha);
          }
          if (row0 + rr < M) reinterpret_cast<uint32_t*>(a.T + (row0 + rr) * a.r_pad)[cp] = o;
        }
      }
    }
  }
}

template <int R>
int launch_tall(const XMap& map, const K1Args& a, const K1Plan& p, cudaStream_t s) {
  using C = TallCfg<R>;
  static int attr_done[64] = {0};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 64 && !attr_done[dev]) {
    cudaError_t e = cudaFuncSetAttribute(k1_tall_kernel<R>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
    if (e != cudaSuccess) return int(e);
    attr_done[dev] = 1;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(unsigned(p.row_tiles * p.nsplit), 1, 1);
  cfg.blockDim = dim3(C::THREADS, 1, 1);
  cfg.dynamicSmemBytes = C::SMEM;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaLaunchAttribute attr2[2] = {attr[0], {}};
  if (p.nsplit > 1) {                             // a tile's split CTAs form one cluster
    attr2[1].id = cudaLaunchAttributeClusterDimension;
    attr2[1].val.clusterDim.x = unsigned(p.nsplit);
    attr2[1].val.clusterDim.y = 1;
    attr2[1].val.clusterDim.z = 1;
    cfg.attrs = attr2;
    cfg.numAttrs = 2;
  }
  K1Args b = a;
  b.tsplit = p.nsplit;
  b.tsteps = p.chunks_per_split / C::CH;
  return int(cudaLaunchKernelEx(&cfg, k1_tall_kernel<R>, map, b));
}

template <int R>
int launch_t(const XMap& map, const K1Args& a, const K1Plan& p, cudaStream_t s) {
  using C = Cfg<R>;
  static int attr_done[64] = {0};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 64 && !attr_done[dev]) {
    cudaError_t e = cudaFuncSetAttribute(k1_kernel<R>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
    if (e != cudaSuccess) return int(e);
    attr_done[dev] = 1;
  }
  // programmatic dependent of the previous kernel in the stream: barrier set-up, TMEM
  // allocation, the tables and the first L1 slices overlap that kernel's drain
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.row_tiles, p.nsplit, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = C::SMEM;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return int(cudaLaunchKernelEx(&cfg, k1_kernel<R>, map, a));
}

}  // namespace

K1Plan k1_plan(int64_t M, int64_t K, int rank, int sm_count) {
  K1Plan p;
  const int nchunks = int(K / 64);
  // enough 32-row tiles to give every other SM one: whole-K CTAs, no split
  // or K short enough that a whole-K CTA beats a split with its cross-CTA reduction (measured:
  // at K = 3072 the 32-row path wins from M = 64 up, at K = 12288 the split wins below ~2400 rows)
  if (ceil_div(M, kTallRows) * 2 >= sm_count || nchunks <= 96) {
    p.tall = true;
    p.row_tiles = int(ceil_div(M, kTallRows));
    // with fewer tiles than half the SMs, every CTA would stream the whole of K for its 32 rows
    // (the kernel's time would not fall with M): split K over up to kK1TallMaxSplit CTAs a tile
    // (one thread-block cluster), in whole stages, so that the tiles' CTAs fill the SMs once
    const int ch = rank <= 96 ? 4 : 2;
    const int nsteps = int(ceil_div(nchunks, ch));
    int ns = 1;
    if (p.row_tiles * 2 < sm_count && p.row_tiles > 0) {
      ns = sm_count / p.row_tiles;
      ns = ns > kK1TallMaxSplit ? kK1TallMaxSplit : ns;
      ns = ns > nsteps ? nsteps : ns;
      ns = ns < 1 ? 1 : ns;
    }
    const int steps = int(ceil_div(nsteps, ns));
    p.nsplit = int(ceil_div(nsteps, steps));       // no empty split
    p.chunks_per_split = steps * ch;
    return p;
  }
  p.row_tiles = int(ceil_div(M, kRows));
  // K splits per 128-row tile: fill one wave of resident CTAs (two per SM), at most kK1MaxSplit,
  // at most the chunk count
  const int slots = 2 * sm_count;
  int ns = p.row_tiles > 0 ? slots / p.row_tiles : 1;
  ns = ns < 1 ? 1 : (ns > kK1MaxSplit ? kK1MaxSplit : ns);
  ns = ns > nchunks ? nchunks : ns;
  p.nsplit = ns;
  p.chunks_per_split = int(ceil_div(nchunks, ns));
  return p;
}

size_t k1_partial_bytes(int64_t M, int rank) {
  return size_t(ceil_div(M, kRows)) * kK1MaxSplit * kRows * size_t(rank) * sizeof(float);
}
size_t k1_arrival_bytes(int64_t M) { return size_t(ceil_div(M, kRows)) * sizeof(unsigned long long); }

int k1_launch(const K1Args& a, const K1Plan& p, void* stream, std::string* err) {
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  XMap map;
  const uint32_t box_rows = p.tall ? uint32_t(kTallRows) : uint32_t(kRows);
  if (!encode_map_2d(map.m, 2, a.X, uint64_t(a.K), uint64_t(a.M), uint64_t(a.K) * 2, 64, box_rows, 1, err))
    return -1;
#define SVDQ_K1_CASE(R) \
  case R: return p.tall ? launch_tall<R>(map, a, p, s) : launch_t<R>(map, a, p, s);
  switch (a.rank) {
    SVDQ_K1_CASE(0)
    SVDQ_K1_CASE(16)
    SVDQ_K1_CASE(32)
    SVDQ_K1_CASE(48)
    SVDQ_K1_CASE(64)
    SVDQ_K1_CASE(80)
    SVDQ_K1_CASE(96)
    SVDQ_K1_CASE(112)
    SVDQ_K1_CASE(128)
    default: return int(cudaErrorInvalidValue);
  }
#undef SVDQ_K1_CASE
}

}  // namespace svdq
