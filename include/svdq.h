/*
 * svdq.h -- C ABI of the SVDQuant W4A4 (NVFP4 / E2M1) linear layer for B300 (sm_103a).
 *
 * The layer (SVDQuant, as the Nunchaku engine runs it; "What SVDQuant actually
 * does" and "How Nunchaku four bit quantization actually works" sections of the
 * aiflownews article on Nunchaku in Diffusers):
 *
 *     Y = alpha * Q4(X diag(lambda)^-1) Q4(R)^T  +  ((X diag(lambda)^-1) L1) L2  +  b
 *
 *   lambda  per-channel smoothing factors that move activation outliers into
 *           the weights (stage one of the method),
 *   L1 L2   the rank-r 16-bit (bfloat16) SVD branch of the smoothed weight
 *           (stage two),
 *   R       the 4-bit residual W diag(lambda) - (L1 L2)^T (stage three),
 *   Q4      NVFP4: E2M1 codes, one E4M3 scale per 16 elements along K,
 *           rounding to nearest even, saturating,
 *   alpha   s_gX * s_gW, the two float32 per-tensor global scales.
 *
 * Conventions (every call):
 *   - Matrices are row-major.  X is M x K, W is N x K (a linear layer's weight),
 *     Y is M x N.  bfloat16 values are passed as their uint16 bit patterns.
 *   - "host" pointers are ordinary CPU memory; "device" pointers are CUDA
 *     global memory on the handle's device.  The caller owns every buffer it
 *     passes; the library never frees caller memory and keeps no pointer to it
 *     after the call returns (except set_workspace, which borrows until reset).
 *   - Every call returns svdq_status_t; no C++ exception crosses the ABI.
 *     svdq_last_error() gives a message for the calling thread's last failure.
 *   - Calls taking a stream are asynchronous on that stream (cudaStream_t
 *     passed as void*, NULL = legacy default stream).  They do not allocate
 *     and do not synchronise.  Kernel launch errors are reported as
 *     SVDQ_ERR_CUDA; a kernel that gave up on a bounded wait records
 *     SVDQ_ERR_TIMEOUT in the handle's device error word (svdq_check_error).
 *   - Shape rules for the CUDA path: K % 64 == 0, N % 16 == 0, 0 <= rank <= 128,
 *     rank % 16 == 0, rank <= min(N, K), M >= 0 (any M; M = 0 is a no-op).
 *   - The device must be compute capability 10.3 (B300); anything else gives
 *     SVDQ_ERR_ARCH before any launch.
 *
 * Device layouts (what svdq_quantize_act writes; documented so that callers
 * and tests can read it):
 *   x_codes   M x K/2 bytes, row-major; element k of a row sits in byte k/2,
 *             low nibble for even k, high nibble for odd k; nibble = E2M1 code
 *             (bit 3 sign, bits 0..2 magnitude index into {0,.5,1,1.5,2,3,4,6}).
 *   x_scales  E4M3 bytes in 128 x 4 tiles, the tensor-core scale layout: with
 *             KG = 4 * ceil(K / 256) groups of 64 columns per row block,
 *             the scale of row m, 16-column block j lives at byte
 *               ((m / 128) * KG + j / 4) * 512 + (m % 32) * 16 + ((m % 128) / 32) * 4 + (j % 4).
 *             Rows are padded to a multiple of 128 (padding rows hold 0).
 *             Size: svdq_scales_bytes(M, K).
 *   T         M x r_pad bfloat16, r_pad = 64 * ceil(rank / 64) (0 if rank == 0),
 *             T[m][j] = round_bf16( (X^ L1)[m][j] / alpha ) for j < rank, 0 beyond.
 *             The 1/alpha folding lets the tensor-core epilogue add the
 *             low-rank product into the same accumulator as the 4-bit product.
 */
#ifndef SVDQ_H_
#define SVDQ_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct svdq_layer* svdq_handle_t; /* opaque; owns all device copies of the packed layer */

typedef enum {
  SVDQ_OK = 0,
  SVDQ_ERR_INVALID_ARG = 1,      /* null pointer, negative size, bad flag      */
  SVDQ_ERR_UNSUPPORTED_SHAPE = 2,/* violates the shape rules above             */
  SVDQ_ERR_ARCH = 3,             /* device is not compute capability 10.3      */
  SVDQ_ERR_OOM = 4,              /* host or device allocation failed           */
  SVDQ_ERR_CUDA = 5,             /* a CUDA runtime call or launch failed       */
  SVDQ_ERR_TIMEOUT = 6,          /* a kernel gave up a bounded wait            */
  SVDQ_ERR_WORKSPACE = 7         /* no workspace, or too small for this M      */
} svdq_status_t;

#define SVDQ_NO_SMOOTH 1u /* lambda = 1: skip smoothing                         */

/* Parameters of the offline packing step. */
typedef struct {
  int64_t N, K, rank;
  const uint16_t* W_bf16;     /* host, N x K, required                                    */
  const uint16_t* bias_bf16;  /* host, N, NULL = zero bias                                */
  const uint16_t* Xcal_bf16;  /* host, Mcal x K calibration activations, NULL = none      */
  int64_t Mcal;
  const float* lambda;        /* host, K; overrides Xcal for lambda when non-NULL         */
  float s_gX;                 /* activation global scale when Xcal is NULL (0 -> 1.0)     */
  const uint16_t* L1_bf16;    /* host, K x rank; with L2 replaces the SVD (NULL = SVD)    */
  const uint16_t* L2_bf16;    /* host, rank x N                                           */
  uint32_t flags;             /* SVDQ_NO_SMOOTH                                           */
  int32_t svd_power_iters;    /* randomized SVD subspace iterations (<= 0 -> 6)           */
  int32_t svd_oversample;     /* extra sketch columns (<= 0 -> 16)                        */
  uint64_t svd_seed;          /* sketch seed                                              */
  int64_t M_max;              /* reserve a library-owned workspace for M <= M_max (0 = none) */
  int32_t device;             /* CUDA device ordinal for the packed layer                */
  void* stream;               /* cudaStream_t used for the upload                         */
} svdq_pack_params_t;

/* The packed layer in canonical host layouts (caller-allocated buffers). */
typedef struct {
  float* lambda;        /* K                                                   */
  float* inv_lambda;    /* K, fl32(1 / lambda)                                 */
  uint16_t* L1_bf16;    /* K x rank                                            */
  uint16_t* L2_bf16;    /* rank x N                                            */
  uint8_t* R_codes;     /* N x K/2, same nibble order as x_codes               */
  uint8_t* R_scales;    /* N x K/16 E4M3, row-major (not tiled)                */
  uint16_t* bias_bf16;  /* N                                                   */
  float s_gW, s_gX, alpha;
} svdq_packed_host_t;

typedef struct {
  int64_t N, K, rank, lora_rank, r_pad, M_max;   /* r_pad: T width, 64 * ceil((rank + lora_rank) / 64) */
  float s_gW, s_gX, alpha;
  int32_t device, sm_count;
} svdq_info_t;

/*
 * svdq_pack_host -- the offline step alone, on the CPU (no CUDA call).
 * Smoothing lambda_c = sqrt(max|X_c| / max|W_c|) (stage one), top-rank SVD of
 * (W diag(lambda))^T by randomized subspace iteration with Sigma on L2 (stage
 * two), R = W diag(lambda) - (L1 L2)^T against the bf16 factors, NVFP4
 * quantisation of R with s_gW = amax|R| / 2688 (stage three).  All outputs go
 * to caller buffers in `out`.  Errors: INVALID_ARG, UNSUPPORTED_SHAPE, OOM.
 */
svdq_status_t svdq_pack_host(const svdq_pack_params_t* p, svdq_packed_host_t* out);

/*
 * svdq_pack_weights -- svdq_pack_host, then the device layouts, uploaded to
 * handle-owned device memory on p->device (cudaMalloc + cudaMemcpyAsync on
 * p->stream, synchronised before return).  *out receives the handle; destroy
 * it with svdq_destroy.  With p->M_max > 0 a workspace for M <= M_max is
 * reserved as by svdq_reserve.
 */
svdq_status_t svdq_pack_weights(const svdq_pack_params_t* p, svdq_handle_t* out);

/* Frees every device and host allocation the handle owns.  NULL is a no-op. */
svdq_status_t svdq_destroy(svdq_handle_t h);

svdq_status_t svdq_get_info(svdq_handle_t h, svdq_info_t* info);

/* Copy of the packed layer in canonical host layouts (see svdq_packed_host_t). */
svdq_status_t svdq_export(svdq_handle_t h, svdq_packed_host_t* out);

/*
 * svdq_attach_lora -- appends a LoRA adapter to the 16-bit low-rank branch without touching
 * the quantised residual: the forward becomes Y = (SVDQuant layer) + scale * (X A) B.  The
 * pages note that SVDQuant works with existing LoRA adapters without re-quantisation
 * (aiflownews article on Nunchaku, "What SVDQuant actually does"); here the adapter's factors
 * are concatenated onto L1 and L2, so the kernels run with rank + r_lora and the up- and
 * down-projections of both share the same passes.
 *   A_bf16  host, K x r_lora row-major (bf16 bits); the library keeps bf16(scale * A)
 *   B_bf16  host, r_lora x N row-major (bf16 bits)
 *   r_lora  multiple of 16 with rank + r_lora <= 128; 0 removes the adapter (A, B may be NULL)
 * Synchronises the handle's device, then replaces the handle's low-rank buffers; the layer's
 * own workspace grows if needed, a lent one must already be large enough (else
 * SVDQ_ERR_WORKSPACE and the layer is unchanged).  Errors: INVALID_ARG, UNSUPPORTED_SHAPE,
 * WORKSPACE, OOM, CUDA.  svdq_export keeps returning the SVD factors alone.
 */
svdq_status_t svdq_attach_lora(svdq_handle_t h, const uint16_t* A_bf16, const uint16_t* B_bf16, int64_t r_lora,
                               float scale, void* stream);

/* Bytes of the activation-scale buffer for M rows (tiled layout above). */
int64_t svdq_scales_bytes(int64_t M, int64_t K);

/*
 * Workspace: the forward keeps the quantised activations, T and the split-K
 * partial sums of the down-projection in a device workspace (no part of it
 * needs clearing by the caller).
 * svdq_workspace_size gives the bytes needed for M rows; svdq_reserve makes the
 * handle allocate (cudaMalloc) and own one for M <= M_max; svdq_set_workspace
 * lends caller memory instead (256-byte aligned, NULL to drop it).
 * host_staging is the number of device staging slots for host X and Y: 0 none,
 * 1 for svdq_linear_forward_host, 2 (or more, taken as 2) also for
 * svdq_linear_forward_host_batch; each slot adds M*K*2 + M*N*2 bytes.
 * Concurrent calls on one handle share the workspace and must be ordered on one
 * stream.
 */
svdq_status_t svdq_workspace_size(svdq_handle_t h, int64_t M, int32_t host_staging, size_t* bytes);
svdq_status_t svdq_reserve(svdq_handle_t h, int64_t M_max, int32_t host_staging);
svdq_status_t svdq_set_workspace(svdq_handle_t h, void* dev_ptr, size_t bytes, int64_t M_max,
                                 int32_t host_staging);

/*
 * svdq_quantize_act -- kernel 1 alone: x^ = fl32(x * inv_lambda), NVFP4 codes
 * and E4M3 block scales of x^ (block quantiser with s_gX, bit-exact with the
 * format rules above) and T = X^ L1 / alpha (low-rank down-projection of stage
 * two, float32 accumulation, bfloat16 out).  X: device M x K bf16.  x_codes,
 * x_scales, T: device buffers in the layouts above (T may be NULL when
 * rank == 0).  Uses the handle's workspace for the split-K partial sums.
 * Scale bytes of the groups past K (K not a multiple of 256) are written as zero.
 */
svdq_status_t svdq_quantize_act(svdq_handle_t h, const void* X_bf16, int64_t M, void* x_codes,
                                void* x_scales, void* T_bf16, void* stream);

/*
 * svdq_gemm_quantized -- kernel 2 alone on already-quantised activations:
 * Y = alpha * (acc_fp4 + T L2) + b with the block-scaled FP4 tensor-core GEMM
 * (the 4-bit branch) and the low-rank up-projection added into the same
 * accumulator.  Inputs in the layouts above; Y: device M x N bf16, fully
 * overwritten, written once.
 */
svdq_status_t svdq_gemm_quantized(svdq_handle_t h, const void* x_codes, const void* x_scales,
                                  const void* T_bf16, void* Y_bf16, int64_t M, void* stream);

/*
 * svdq_linear_forward -- the layer: kernel 1 then kernel 2 on `stream`.
 * X: device M x K bf16 (read once).  Y: device M x N bf16 (written once).  Needs a
 * workspace for M (svdq_reserve / svdq_set_workspace).  X and Y must not overlap each other
 * or the workspace's kernel scratch: SVDQ_ERR_INVALID_ARG otherwise.
 */
svdq_status_t svdq_linear_forward(svdq_handle_t h, const void* X_bf16, void* Y_bf16, int64_t M,
                                  void* stream);

/*
 * svdq_linear_forward_host -- the layer on HOST buffers: copies X (host, ideally
 * pinned) to the workspace's device staging, runs svdq_linear_forward, copies Y
 * back to host and synchronises the stream.  Needs a workspace reserved with
 * host_staging != 0.
 */
svdq_status_t svdq_linear_forward_host(svdq_handle_t h, const uint16_t* X_host, uint16_t* Y_host,
                                       int64_t M, void* stream);

/*
 * svdq_linear_forward_host_batch -- B layer calls on HOST buffers, pipelined: step b reads
 * X_host[b] (M x K bf16) and writes Y_host[b] (M x N bf16), b < B.  The kernels run on `stream`;
 * the uploads and downloads run on two copy streams the handle creates on first use.  Steps
 * alternate between two device staging slots, so step b+1's upload and step b-1's download
 * overlap step b's kernels and each other.  Returns after every Y_host[b] holds its result.
 *   X_host, Y_host: arrays of B host pointers (caller-owned; pinned memory lets the copies run
 *   asynchronously, pageable memory works but serialises them).  Y_host[b] must not overlap any
 *   X_host[c] or another Y_host[c].
 *   Work already queued on `stream` completes before the first upload starts.
 *   Errors: SVDQ_ERR_INVALID_ARG (null handle or pointers, negative M or B),
 *   SVDQ_ERR_WORKSPACE (no workspace with two staging slots for M), SVDQ_ERR_CUDA.  B == 0
 *   or M == 0 does nothing.
 */
svdq_status_t svdq_linear_forward_host_batch(svdq_handle_t h, const uint16_t* const* X_host,
                                             uint16_t* const* Y_host, int32_t B, int64_t M,
                                             void* stream);

/*
 * svdq_linear_forward_noalloc -- the same layer as svdq_linear_forward for callers that must
 * not allocate device memory when they run it: code inside a framework's memory pool or budget
 * (a library-owned cudaMalloc would bypass the pool and may not fit), and latency-critical
 * loops that cannot take cudaMalloc's implicit synchronisation.  Instead of the handle's
 * workspace it uses a statically sized scratch array that the library holds on every device it
 * is loaded on (32 MiB per device, kept until the process exits), so the call makes no
 * allocation of any kind.  The SVDQuant/Nunchaku pages have no counterpart; it is an interface
 * convenience of this library.
 *   X: device M x K bf16, Y: device M x N bf16 (as svdq_linear_forward); neither may overlap
 *   the other or the static scratch (SVDQ_ERR_INVALID_ARG).
 *   The scratch array's device address is looked up with cudaGetSymbolAddress, with the
 *   handle's device current, on every call made outside stream capture, so a device reset
 *   between calls does no harm.  A call on a stream that is capturing uses the address found by
 *   the last call outside capture on that device, and fails with SVDQ_ERR_INVALID_ARG if there
 *   was none: make the first call on a device before any stream capture.
 *   Every call shares the one scratch array, which keeps the last call's contents (nothing in it
 *   needs clearing: kernel 2 reads only what kernel 1 wrote in the same call, and the split-K
 *   arrival words carry a per-launch epoch).  Calls that overlap on the GPU (different streams,
 *   or different handles on the same device without ordering) race on it.  Order them on one
 *   stream.
 *   Errors: SVDQ_ERR_WORKSPACE when M needs more scratch than 32 MiB (svdq_workspace_size with
 *   host_staging = 0 gives the requirement), plus the errors of svdq_linear_forward.
 */
svdq_status_t svdq_linear_forward_noalloc(svdq_handle_t h, const void* X_bf16, void* Y_bf16, int64_t M,
                                          void* stream);

/*
 * svdq_set_wait_limit -- failure detection.  Every wait inside the kernels (on a barrier that
 * another warp, the other CTA of a pair or a copy engine completes) gives up after a limit,
 * records SVDQ_ERR_TIMEOUT in the handle's device error word, finishes or waits out the work it
 * started and returns, so a lost signal never hangs the GPU.  This call sets that limit for the
 * handle's later launches (wait_ns nanoseconds; 0 restores the default of two seconds).
 * stall_kernel = 1 or 2 makes the MMA warp of kernel 1 or kernel 2 wait on a barrier that nothing
 * completes, so that its wait runs out: the way tests exercise the path without faulting a GPU.
 * 0 turns it off.  The SVDQuant pages have no counterpart; it is a diagnostics hook.
 *   Errors: SVDQ_ERR_INVALID_ARG (null handle, stall_kernel outside 0..2).
 */
svdq_status_t svdq_set_wait_limit(svdq_handle_t h, uint64_t wait_ns, int32_t stall_kernel);

/*
 * svdq_check_error -- synchronises the handle's device, reads and clears the
 * device error word that the kernels set when a bounded wait gives up.
 * Returns SVDQ_OK or SVDQ_ERR_TIMEOUT (or SVDQ_ERR_CUDA for a sticky CUDA error).
 */
svdq_status_t svdq_check_error(svdq_handle_t h);

const char* svdq_status_string(svdq_status_t s);
const char* svdq_last_error(void);

/* ==================================================================================
 * MLP pair: two SVDQuant layers with GELU between them, the up layer's output feeding the down
 * layer (the FLUX transformer block's feed-forward: K -> N_up -> N).
 *
 * The pages' Nunchaku section says the low-rank and 4-bit branches run as one fused operation
 * that shares inputs and outputs so that memory-bound diffusion transformers avoid redundant
 * memory traffic (aiflownews article on Nunchaku in Diffusers, "Nunchaku: the inference engine
 * that makes SVDQuant practical").  The pair carries that sharing across the activation: the up
 * layer's kernel 2 applies GELU to its bf16 output tile and writes the down layer's kernel-1
 * outputs for it (NVFP4 codes, E4M3 block scales and the low-rank down-projection T), so the
 * up layer's output is never written to memory and the down layer's kernel 1 never runs.
 *
 * Arithmetic (identical to running the layers apart with svdq_gelu_bf16 between them, except
 * for the float32 summation order of T):
 *   Y_up = bf16(alpha_up * acc + b_up)              the up layer's output, bit for bit
 *   G    = bf16(GELU(Y_up)),  GELU(y) = y * Phi(y), Phi the standard normal CDF (the pages
 *          name no activation formula: this is GELU's definition, not the tanh approximation),
 *          evaluated in float32 as y Q(|y|) (y <= 0) or y (1 - Q(y)) with the normal tail
 *          Q(u) = erfc(u / sqrt(2)) / 2 from the Chebyshev fit of erfc in Numerical Recipes
 *          (section 6.2, erfcc); relative error below 2^-19 (y >= 0), 2^-19 + y^2 2^-22 (y < 0)
 *   codes, scales of G: the down layer's smoothing and NVFP4 quantiser (as svdq_quantize_act)
 *   T    = bf16(fl32(sum of partial G L1') * fl32(1 / alpha_down)), L1' = diag(1/lambda) L1 in
 *          bf16 as kernel 1 uses it; the partial sums (float32, one per run of column tiles and
 *          half tile) are added in a fixed order, so T is reproducible from run to run.
 * Limits: the up layer's N equals the down layer's K; the down layer's kernel rank (SVD rank
 * plus any LoRA rank) is at most 64.  The pair keeps the down layer's L1' in the order the
 * epilogue reads it; attaching LoRA factors to the down layer afterwards invalidates the pair
 * (its calls then return SVDQ_ERR_INVALID_ARG).  Both handles must outlive the pair.
 * Errors: the fused kernel reports bounded-wait expiry on the up handle's error word, the down
 * layer's kernel 2 on the down handle's; svdq_mlp_check_error reads both.
 * ================================================================================== */
typedef struct svdq_mlp* svdq_mlp_t;

/* svdq_mlp_create -- binds two packed layers (up: N_up x K, down: N x N_up) on one device and
 * allocates the pair's buffers for up to M_max rows: the down layer's L1' in fragment order
 * (N_up x rank bf16) and the partial sums of T (at most about 2 * N_up/256 * M_max * rank * 4
 * bytes, far less at large M).  Errors: SVDQ_ERR_INVALID_ARG (null, same handle twice, other
 * devices, N_up != K_down), SVDQ_ERR_UNSUPPORTED_SHAPE (down rank > 64), SVDQ_ERR_OOM. */
svdq_status_t svdq_mlp_create(svdq_handle_t up, svdq_handle_t down, int64_t M_max, svdq_mlp_t* out);
svdq_status_t svdq_mlp_destroy(svdq_mlp_t p);

/* svdq_mlp_up_quantize -- the up layer's kernel 1 on X (device M x K bf16), then its kernel 2
 * with the fused epilogue and the reduction of T: writes the down layer's kernel-1 outputs for
 * G = bf16(GELU(Y_up)) into x_codes (M x N_up/2), x_scales (tiled, svdq_scales_bytes(M, N_up))
 * and T (M x r_pad_down bf16; may be NULL when the down rank is 0), exactly the buffers
 * svdq_gemm_quantized of the down layer consumes.  Uses the up layer's workspace
 * (svdq_reserve(up, >= M)).  M <= M_max.  Outputs must not overlap X or each other. */
svdq_status_t svdq_mlp_up_quantize(svdq_mlp_t p, const void* X_bf16, int64_t M, void* x_codes,
                                   void* x_scales, void* T_bf16, void* stream);

/* svdq_mlp_forward -- the whole pair on `stream`: svdq_mlp_up_quantize into the down layer's
 * workspace, then the down layer's kernel 2.  X: device M x K bf16; Y: device M x N bf16
 * (written once).  Needs both layers' workspaces for M (svdq_reserve) and M <= M_max.  X and Y
 * must not overlap each other or either workspace's kernel scratch. */
svdq_status_t svdq_mlp_forward(svdq_mlp_t p, const void* X_bf16, void* Y_bf16, int64_t M, void* stream);

/* svdq_mlp_check_error -- svdq_check_error of the up layer, then of the down layer (both are
 * read and cleared); returns the first failure. */
svdq_status_t svdq_mlp_check_error(svdq_mlp_t p);

/* svdq_gelu_bf16 -- G[i] = bf16(GELU(Y[i])) for n bf16 values (n % 8 == 0, 16-byte aligned
 * device buffers, G == Y allowed), with the fused epilogue's arithmetic: the unfused pair is
 * svdq_linear_forward(up), this, svdq_linear_forward(down).  Runs on the current device. */
svdq_status_t svdq_gelu_bf16(const void* Y_bf16, void* G_bf16, int64_t n, void* stream);

/* ==================================================================================
 * INT4 variant of the SVDQuant layer
 *
 * The pages say SVDQuant supports both INT4 and FP4 and that Nunchaku runs INT4 kernels on
 * hardware older than Blackwell (aiflownews article on Nunchaku, "What SVDQuant actually does",
 * "How Nunchaku four bit quantization actually works"); they give no INT4 group size or scale
 * format.  Reading used here: the same smoothing, low-rank branch and residual as the NVFP4
 * layer, with the residual and the smoothed activations quantised to symmetric INT4 groups:
 *   q = clamp(rint(fl32(v * fl32(1 / s))), -7, 7), ties to even, s = fl32(amax / 7) per 64
 *   consecutive elements along K (s = 0 and q = 0 for an all-zero group),
 *   Y = sum_g sX[m, g] sW[n, g] (sum_{k in g} qx qw) + (X^ L1) L2 + b,   bf16 out.
 * This part's tensor cores have no integer MMA of the tcgen05 family, and the per-group scales
 * sit inside the K sum, so the GEMM unpacks the codes to bf16 and runs warp-level MMAs, finishing
 * each group's exact integer sum in float32 registers before scaling it.
 * Layouts:
 *   codes    rows x K/2 bytes, element k in byte k/2 (low nibble for even k), nibble = q + 8.
 *   scales   device: group-major float32, [K/64][svdq_int4_scale_ld(rows)] (scale of row m, group
 *            g at g * ld + m; rows past the last are padding); host export: rows x K/64 row-major.
 *   T        rows x r_pad bf16, T = X^ L1 (not divided by anything), r_pad = 64 * ceil(rank / 64).
 * Shape rules: K % 64 == 0, N % 16 == 0, rank % 16 == 0, 0 <= rank <= min(128, N, K).
 * ================================================================================== */
typedef struct svdq_int4_layer* svdq_int4_handle_t;

/* The packed INT4 layer in canonical host layouts (caller-allocated buffers, NULL = skip). */
typedef struct {
  float* lambda;        /* K                                                   */
  float* inv_lambda;    /* K                                                   */
  uint16_t* L1_bf16;    /* K x rank                                            */
  uint16_t* L2_bf16;    /* rank x N                                            */
  uint8_t* R_codes;     /* N x K/2                                             */
  float* R_scales;      /* N x K/64, row-major                                 */
  uint16_t* bias_bf16;  /* N                                                   */
} svdq_int4_host_t;

/* Rows of a group-major scale buffer for `rows` rows: 128 * ceil(rows / 128). */
int64_t svdq_int4_scale_ld(int64_t rows);

/*
 * svdq_int4_pack_host -- the INT4 offline step on the CPU (no CUDA call): smoothing, the
 * randomized top-rank SVD, the residual against the bf16 factors, INT4 groups.  Uses the fields
 * of svdq_pack_params_t as svdq_pack_host does (s_gX is ignored: the INT4 groups need no global
 * scale).  Errors: INVALID_ARG, UNSUPPORTED_SHAPE, OOM.
 */
svdq_status_t svdq_int4_pack_host(const svdq_pack_params_t* p, svdq_int4_host_t* out);

/*
 * svdq_int4_pack -- svdq_int4_pack_host, then the device layouts uploaded to p->device
 * (synchronised before return); reserves a workspace for M <= p->M_max when M_max > 0.
 * Errors: those of svdq_int4_pack_host, ARCH, OOM, CUDA.
 */
svdq_status_t svdq_int4_pack(const svdq_pack_params_t* p, svdq_int4_handle_t* out);
svdq_status_t svdq_int4_export(svdq_int4_handle_t h, svdq_int4_host_t* out);

/* Library-owned workspace for svdq_int4_forward with M <= M_max (replaces any earlier one). */
svdq_status_t svdq_int4_reserve(svdq_int4_handle_t h, int64_t M_max);

/*
 * svdq_int4_quantize_act -- kernel int4_k1 alone: x^ = fl32(x * inv_lambda), INT4 groups of x^
 * (bit-exact with the quantiser above) and T = X^ L1 (float32 accumulation, bf16 out).
 * X: device M x K bf16; x_codes: device M x K/2; x_scales: device float32 group-major with
 * ld = svdq_int4_scale_ld(M); T: device M x r_pad bf16 (NULL when rank == 0).  16-byte aligned.
 */
svdq_status_t svdq_int4_quantize_act(svdq_int4_handle_t h, const void* X_bf16, int64_t M, void* x_codes,
                                     float* x_scales, void* T_bf16, void* stream);

/*
 * svdq_int4_forward -- the INT4 layer: kernel int4_k1 then kernel int4_k2 on `stream`.
 * X: device M x K bf16; Y: device M x N bf16, fully overwritten.  X, Y and the workspace must
 * not overlap.  Errors: INVALID_ARG, WORKSPACE (no workspace for M), CUDA.
 */
svdq_status_t svdq_int4_forward(svdq_int4_handle_t h, const void* X_bf16, void* Y_bf16, int64_t M, void* stream);

/* Synchronises, reads and clears the device error word (SVDQ_ERR_TIMEOUT if a wait gave up). */
svdq_status_t svdq_int4_check_error(svdq_int4_handle_t h);
svdq_status_t svdq_int4_destroy(svdq_int4_handle_t h);

/* ==================================================================================
 * AWQ-style W4A16 linear layer (the modulation / adaptive-normalisation layers)
 *
 * The pages keep 16-bit activations and quantise only the weights to four bits, AWQ style,
 * for the layers where 4-bit activations cost too much accuracy (aiflownews article on
 * Nunchaku, "How Nunchaku four bit quantization actually works").  Readings (the pages give none):
 *   - weights W diag(s) in groups of 64 consecutive input channels of an output row:
 *     asymmetric 4-bit codes q in [0, 15], float32 scale sc and zero point z in [0, 15]:
 *       sc = fl32(max(w_max - w_min, 1e-5) / 15), z = clamp(rint(-w_min / sc), 0, 15),
 *       q = clamp(rint(w / sc) + z, 0, 15)
 *   - activation-aware per-channel scales s_c = a_c^alpha / sqrt(max s * min s),
 *     a_c = mean_m |Xcal_mc|, alpha in {0, 0.05, ..., 0.95} picked by the smallest
 *     calibration output error (all ones without calibration data)
 *   - forward: x' = fl32(x * fl32(1 / s_c)), Y = x' ((q - z) sc)^T + b, bf16 out; the kernel
 *     multiplies in fp16 (x' rounded to fp16) and sums four products in fp16 before float32.
 *     A row of x' whose largest magnitude exceeds 512 is scaled by an exact power of two for
 *     the fp16 part and its sums scaled back, so no input magnitude overflows the fp16 sums.
 *     Built for the small-M (GEMV-like) modulation shapes: the weights are streamed from HBM
 *     once per 8 rows of X.
 * ================================================================================== */
typedef struct svdq_awq_layer* svdq_awq_handle_t;

typedef struct {
  int64_t N, K;                /* K % 64 == 0                                                 */
  const uint16_t* W_bf16;      /* host, N x K row-major                                       */
  const uint16_t* bias_bf16;   /* host, N, NULL = zero bias                                   */
  const uint16_t* Xcal_bf16;   /* host, Mcal x K calibration activations, NULL = no search    */
  int64_t Mcal;
  const float* s;              /* host, K: per-channel scales to use instead of the search    */
  int32_t device;
  void* stream;                /* cudaStream_t for the upload                                 */
} svdq_awq_params_t;

typedef struct {
  float* s;                    /* K                                                           */
  float* inv_s;                /* K, fl32(1 / s)                                              */
  uint8_t* codes;              /* N x K/2, element 2j in the low nibble of byte j             */
  float* scales;               /* N x K/64                                                    */
  uint8_t* zeros;              /* N x K/64                                                    */
  uint16_t* bias_bf16;         /* N                                                           */
  float alpha;                 /* searched exponent, -1 if none                               */
} svdq_awq_host_t;

/* Host quantisation alone (no CUDA call); all outputs in caller buffers.
 * Errors: INVALID_ARG, UNSUPPORTED_SHAPE. */
svdq_status_t svdq_awq_pack_host(const svdq_awq_params_t* p, svdq_awq_host_t* out);
/* svdq_awq_pack_host, then the packed weights uploaded to handle-owned device memory.
 * Errors: as svdq_awq_pack_host, plus ARCH, OOM, CUDA. */
svdq_status_t svdq_awq_pack(const svdq_awq_params_t* p, svdq_awq_handle_t* out);
svdq_status_t svdq_awq_destroy(svdq_awq_handle_t h);
/* Copy of the packed layer (buffers as in svdq_awq_host_t, caller-owned). */
svdq_status_t svdq_awq_export(svdq_awq_handle_t h, svdq_awq_host_t* out);
/* Y (device, M x N bf16) = x' W'^T + b for X (device, M x K bf16); asynchronous on stream,
 * allocates nothing; X and Y 16-byte aligned, not aliased; M = 0 is a no-op.
 * Errors: INVALID_ARG, CUDA. */
svdq_status_t svdq_awq_forward(svdq_awq_handle_t h, const void* X_bf16, void* Y_bf16, int64_t M, void* stream);
/* Synchronises the layer's device, reads and clears its device error word: TIMEOUT if a
 * kernel gave up a bounded wait since the last check. */
svdq_status_t svdq_awq_check_error(svdq_awq_handle_t h);

#ifdef __cplusplus
}
#endif

#endif /* SVDQ_H_ */
