// Internal declarations shared by the host pack, the C-ABI layer and the kernel launchers.
#pragma once

#include <cstddef>
#include <cstdint>
#include <string>
#include <vector>

#include "../../include/svdq.h"

#ifdef __CUDACC__
#define SVDQ_HD __host__ __device__
#else
#define SVDQ_HD
#endif

namespace svdq {

// ------------------------------------------------------------------ host pack (pack_host.cpp)
struct HostPack {
  int64_t N = 0, K = 0, rank = 0;
  std::vector<float> lambda, inv_lambda;   // K
  std::vector<uint16_t> L1;                // K x rank (bf16 bits)
  std::vector<uint16_t> L2;                // rank x N (bf16 bits)
  std::vector<uint8_t> R_codes;            // N x K/2
  std::vector<uint8_t> R_scales;           // N x K/16 (row-major, not tiled)
  std::vector<uint16_t> bias;              // N
  float s_gW = 1.f, s_gX = 1.f, alpha = 1.f;
};

// Validates p and runs smoothing, SVD, residual and NVFP4 quantisation on the CPU.
// R_keep, when non-null, receives the float32 residual R (N x K) that was quantised.
svdq_status_t pack_on_host(const svdq_pack_params_t* p, HostPack* out, std::string* err,
                           std::vector<float>* R_keep = nullptr);

// AWQ-style W4A16 layer: host pack (awq_host.cpp) and GEMV (awq_gemv.cu).
struct AwqHostPack {
  int64_t N = 0, K = 0;
  float alpha = -1.f;
  std::vector<float> s, inv_s;        // K
  std::vector<uint8_t> codes;         // N x K/2
  std::vector<float> scales;          // N x K/64
  std::vector<uint8_t> zeros;         // N x K/64
  std::vector<uint16_t> bias;         // N
};
svdq_status_t awq_pack_host(const svdq_awq_params_t* p, AwqHostPack* out, std::string* err);
struct AwqArgs {
  const uint16_t* X;                  // M x K bf16
  const float* inv_s;                 // K
  const uint8_t* codes;               // N x K/2
  const float* sz;                    // N x K/64 pairs (scale, zero point as float), 16 bytes of padding
  const uint16_t* bias;               // N
  uint16_t* Y;                        // M x N bf16
  int* err;                           // device error word (bounded waits)
  int64_t M, N, K;
};
int awq_launch(const AwqArgs& a, int sm_count, void* stream);

// Activation-quantiser tables for a global scale s_g (host side):
//   thr[c]  smallest float32 amax >= 0 whose block scale E4M3(fl32(amax / fl32(6 s_g))) >= c
//           (c = 0..126; thr[127] = +inf), so the scale code of a block is the number of
//           thresholds <= amax;
//   rcp[c]  fl32(1 / fl32(E4M3value(c) * s_g)) (rcp[0] = 0, unused).
void act_quant_tables(float s_g, float* thr128, float* rcp128);

// Format helpers (host side).
float bf16_to_f32(uint16_t b);
uint16_t f64_to_bf16(double a);
uint8_t e4m3_encode_nonneg(float s);
float e4m3_decode(uint8_t b);
uint8_t e2m1_encode(float v);

// ------------------------------------------------------------------ device layouts
SVDQ_HD inline int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }
SVDQ_HD inline int64_t round_up(int64_t a, int64_t b) { return ceil_div(a, b) * b; }
// 64-column groups per 128-row block of a tiled scale buffer (padded to whole 256-column stages).
SVDQ_HD inline int64_t scale_groups(int64_t K) { return 4 * ceil_div(K, 256); }
SVDQ_HD inline int64_t rank_pad(int64_t r) { return r == 0 ? 0 : round_up(r, 64); }

// ------------------------------------------------------------------ kernel 1 (k1_actquant.cu)
struct K1Args {
  const uint16_t* X;          // M x K bf16 (read through the tensor map passed beside these args)
  const unsigned char* LI;    // per group of four 64-column chunks: four swizzled L1' slices (rank x 128 B), four 1/lambda parts
  uint8_t* x_codes;           // M x K/2
  uint8_t* x_scales;          // tiled
  uint16_t* T;                // M x r_pad bf16 (null if rank == 0)
  float* partial;             // split-K partial sums [row tile][split][rank][128] (rank > 0)
  unsigned long long* arrivals;   // one word per row tile: (epoch << 8) | CTAs arrived
  unsigned long long epoch;   // unique per launch, < 2^56
  int64_t M, K;
  int rank, r_pad;
  float s_gX, inv_six, inv_alpha;
  const float* qtab;          // 256 floats: E4M3 scale thresholds [0,128), reciprocals [128,256)
  int* err;                   // device error word (bounded waits)
  uint64_t wait_ns;           // limit of every bounded wait (nanoseconds)
  int stall;                  // failure-detection tests: the MMA warp waits on a barrier nothing completes
  int tsplit = 1;             // whole-K path: CTAs per 32-row tile, each over tsteps stages of K
  int tsteps = 0;
};
struct K1Plan {
  bool tall = false;          // 32-row tiles over the whole of K (no split) instead of 128-row split tiles
  int row_tiles = 0, nsplit = 1, chunks_per_split = 1;
};
K1Plan k1_plan(int64_t M, int64_t K, int rank, int sm_count);
constexpr int kK1MaxSplit = 8;   // K splits per 128-row tile
constexpr int kK1TallMaxSplit = 8;    // K splits per 32-row tile (one portable cluster; small M)
// Workspace bytes of the split-K partial sums and the arrival words for M rows.
size_t k1_partial_bytes(int64_t M, int rank);
size_t k1_arrival_bytes(int64_t M);
// Encodes the tensor map of X and launches; returns a cudaError_t (or -1 if the map failed).
int k1_launch(const K1Args& a, const K1Plan& plan, void* stream, std::string* err);

// ------------------------------------------------------------------ kernel 2 (k2_fp4gemm.cu)
struct K2Maps {
  alignas(64) unsigned char A[128];    // CUtensorMap: x codes      (u8, K/2 x M, box 128 x 128, swizzle 128)
  alignas(64) unsigned char SFA[128];  // CUtensorMap: x scales     (u8, 256-byte rows of the tiled buffer, box 256 x 8)
  alignas(64) unsigned char T[128];    // CUtensorMap: T            (bf16, r_pad x M, box 64 x 128, swizzle 128)
  alignas(64) unsigned char L2[128];   // CUtensorMap: L2^T         (bf16, r_pad x N, box 64 x 128, swizzle 128)
  alignas(64) unsigned char Y[128];    // CUtensorMap: Y            (bf16, N x M, box 64 x 32, swizzle 128)
};
// Fused MLP epilogue: the layer's output y feeds the next layer of an MLP pair through GELU, so
// kernel 2 writes that layer's kernel-1 outputs for G = bf16(GELU(y)) instead of Y.
struct K2Fuse {
  const float* inv_lambda;    // N: the next layer's 1/lambda
  const float* qtab;          // the next layer's quantiser tables (as K1Args::qtab)
  float inv_six;              // the next layer's fl32(1 / (6 s_gX))
  uint8_t* x_codes;           // M x N/2: the next layer's activation codes
  uint8_t* x_scales;          // tiled, scale_groups(N) groups: its activation scales
  const void* l1f;            // its L1' = diag(1/lambda) L1 in warp-MMA B-fragment order (k2_l1_fragments)
  float* part;                // [2 S][M][rd]: partial G L1' of each unit and column half
  int rd;                     // its kernel rank (0 or a multiple of 16, <= 64)
};
// Weight blocks of kernel 2, one per 256-row pair tile, 256-wide K step and 128-row half, in
// that order (K steps of a tile, then halves, innermost), kK2WeightBlock bytes each: the half's
// 128 rows x 128 bytes of codes as a 128-byte-swizzled TMA tile would leave them in shared
// memory (16-byte chunk c of row r at r * 128 + 16 (c ^ (r % 8))), then the pair tile's 4 KB
// scale block of the step (both halves; see the layer's pack).
constexpr int kK2WeightBlock = 128 * 128 + 4096;
struct K2Args {
  const uint16_t* bias;       // N bf16
  const uint8_t* wt;          // weight blocks (rows padded to 256, K to 256; zero padding)
  int* err;                   // device error word
  int64_t M, N, K;
  int rank;
  float alpha;
  uint64_t wait_ns;           // limit of every bounded wait (nanoseconds)
  int stall;                  // failure-detection tests: the MMA thread waits on a barrier nothing completes
  int unit_len = 1;           // tiles are taken in units of unit_len consecutive column tiles of one row block
  K2Fuse fuse{};              // fused MLP epilogue (k2_fused_launch only)
};
// Default limit of the kernels' bounded waits: two seconds.
constexpr uint64_t kDefaultWaitNs = 2000000000ull;
int k2_launch(const K2Maps& maps, const K2Args& a, int sm_count, void* stream);
size_t k2_smem_bytes();
// Fused MLP epilogue (kernel 2 of the up layer of a pair): maps.Y unused, a.fuse filled,
// a.unit_len from k2_fused_unit_len; then k2_t_reduce_launch sums the partials into T.
constexpr int kFuseMaxRank = 64;
int k2_fused_unit_len(int64_t M, int64_t N, int pairs);
int k2_fused_pairs(int sm_count);   // CTA pairs the fused kernel runs with on this device
int64_t k2_fused_partials(int64_t M, int64_t N, int unit_len);   // partial sums per row (2 S)
int k2_fused_launch(const K2Maps& maps, const K2Args& a, int sm_count, void* stream);
// T[m][j] = bf16(fl32(sum over p of part[p][m][j]) * inv_alpha) for j < rd, 0 for rd <= j < r_pad
int k2_t_reduce_launch(const float* part, int64_t P, int64_t M, int rd, int r_pad, float inv_alpha, uint16_t* T,
                       void* stream);
// Next-layer L1' (K x rd bf16 bits, row-major) -> warp-MMA B fragments: for 16-row step s and
// pair np of 8-column groups, lane l's 16 bytes are {b0, b1} of group 2 np then of 2 np + 1,
// b0 = rows 16 s + 2 (l % 4) + {0, 1} and b1 = rows + 8, column 16 np + 8 g + l / 4.
void k2_l1_fragments(const uint16_t* L1p, int64_t K, int rd, uint16_t* out);
// Elementwise bf16(GELU(y)) with the fused epilogue's arithmetic.
int gelu_launch(const uint16_t* Y, uint16_t* G, int64_t n, int sm_count, void* stream);

// ------------------------------------------------------------------ INT4 variant (int4_path.cu)
// Symmetric INT4 groups: nibble q + 8, q in [-7, 7], one float32 scale per 64 elements along K.
// Activation and weight group scales are stored group-major, [K / 64][rows padded to 128].
void int4_quantize_row(const float* v, int64_t K, uint8_t* codes, float* scales);   // host (pack_host.cpp)
struct alignas(64) Int4K1Maps {
  unsigned char X[128];     // CUtensorMap: X        (bf16, K x M, box 64 x 32, swizzle 128)
  unsigned char L1t[128];   // CUtensorMap: L1'^T    (bf16, K x r_pad, box 64 x r_pad, swizzle 128)
};
struct Int4K1Args {
  const float* inv_lambda;  // K
  uint8_t* codes;           // M x K/2
  float* scales;            // [K/64][scale_ld]
  uint16_t* T;              // M x r_pad bf16, T = X^ L1 (unscaled)
  int64_t M, K, scale_ld;
  int r_pad;
  int* err;                 // device error word
  uint64_t wait_ns;
};
struct alignas(64) Int4K2Maps {
  unsigned char A[128];     // CUtensorMap: x codes  (u8, K/2 x M, box 32 x 128)
  unsigned char B[128];     // CUtensorMap: R codes  (u8, K/2 x N, box 32 x 128)
  unsigned char SA[128];    // CUtensorMap: x scales (f32, M_pad x K/64, box 128 x 1)
  unsigned char SB[128];    // CUtensorMap: R scales (f32, N_pad x K/64, box 128 x 1)
  unsigned char T[128];     // CUtensorMap: T        (bf16, r_pad x M, box 64 x 128, swizzle 128)
  unsigned char L2[128];    // CUtensorMap: L2^T     (bf16, r_pad x N, box 64 x 128, swizzle 128)
};
struct Int4K2Args {
  const uint16_t* bias;     // N bf16
  uint16_t* Y;              // M x N bf16
  int64_t M, N, K;
  int r_pad;
  int* err;
  uint64_t wait_ns;
};
int int4_k1_launch(const Int4K1Maps& maps, const Int4K1Args& a, void* stream);
int int4_k2_launch(const Int4K2Maps& maps, const Int4K2Args& a, void* stream);

// Tensor-map encoding through the driver entry point (api.cu).
// dtype_bytes: 1 (u8), 2 (bf16) or 4 (f32)
bool encode_map_2d(void* map, int dtype_bytes, const void* base, uint64_t inner, uint64_t outer,
                   uint64_t row_stride_bytes, uint32_t box_inner, uint32_t box_outer, int swizzle128,
                   std::string* err);

}  // namespace svdq
