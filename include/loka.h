/*
 * loka.h -- C ABI of the GB300 (sm_103a) FP8 linear + normalization library.
 *
 * The operation is the FP8 linear layer of a large recommendation model: a
 * small GEMM followed immediately by a normalization, whose quantization
 * overhead can cancel the FP8 gain ("LoKA: Low-precision Kernel Applications
 * for Recommendation Models at Scale", section I and section II-C "Key
 * findings").  The library computes, on one GPU:
 *
 *   amax -> scale -> E4M3 cast of activations X[M,K] and weights W[N,K]
 *   -> FP8 GEMM with fp32 accumulation (tcgen05 tensor cores, TMEM)
 *   -> epilogue: dequantize, add bias, LayerNorm, RMSNorm or BlockNorm,
 *      optional Hard Swish, bf16 store and/or E4M3 codes for the next layer
 *
 * plus square 32x32-block quantization with a transposed copy (GEM Training
 * page), a per-layer quantization-error probe (LoKA section III-A, MERE of
 * FP8(Wx+b) against a high-precision Wx+b) with the probe's online input
 * statistics, Cholesky factor and sampler (section III-A 1), and a variant
 * selector (LoKA section III-C, Dispatch).
 *
 * Conventions for every call:
 *   - Pointers named as device pointers must be device memory of the current
 *     CUDA device; the caller owns all memory.  No call allocates device
 *     memory; calls that need temporary space take a caller-provided
 *     workspace, whose size the matching *_workspace_size() call returns.
 *   - Work is enqueued on `stream` (a cudaStream_t, NULL = legacy default
 *     stream) and is asynchronous, except where a call says it synchronizes.
 *   - Argument errors are found on the host before anything is launched; the
 *     call then returns a non-zero loka_status and loka_last_error() gives a
 *     message.  Launch failures return LOKA_ERR_CUDA.
 *   - Kernels never spin forever: every wait inside a kernel has a time
 *     limit; a kernel that gives up sets a device status flag and returns.
 *     loka_device_status() (or the next synchronizing call) reports it as
 *     LOKA_ERR_TIMEOUT.
 *   - Tensors are row-major.  X is [M,K] (K contiguous), W is [N,K] (the
 *     nn.Linear layout; the GEMM is Y = X W^T), Y is [M,N].
 *   - Not thread-safe per stream; calls on different streams may overlap.
 */
#ifndef LOKA_H_
#define LOKA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef int32_t loka_status;
#define LOKA_OK 0
#define LOKA_ERR_INVALID_ARG 1   /* bad pointer, size, alignment or enum   */
#define LOKA_ERR_UNSUPPORTED 2   /* valid but not implemented (e.g. N)    */
#define LOKA_ERR_WORKSPACE 3     /* workspace missing or too small         */
#define LOKA_ERR_TIMEOUT 4       /* a kernel wait ran out of time          */
#define LOKA_ERR_CUDA 5          /* a CUDA runtime/driver call failed      */
#define LOKA_ERR_NUMERIC 6       /* a numerical precondition failed (e.g. a
                                    covariance not positive definite)     */

/* Scaling granularity of the E4M3 cast (LoKA section II-C / Table VI name
 * tensorwise, rowwise and blockwise recipes; the GEM Training page, "Low
 * Precision Flash Attention", places MXFP8 scale factors along K). */
#define LOKA_SCALE_TENSOR 0      /* one fp32 scale for the whole tensor    */
#define LOKA_SCALE_ROW 1         /* one fp32 scale per row                 */
#define LOKA_SCALE_MX32 2        /* one E8M0 scale per 1x32 block along K  */
#define LOKA_BF16 3              /* no quantization: bf16 GEMM (fallback)  */
#define LOKA_SCALE_BLOCK32 4     /* one E8M0 scale per 32x32 block          */

/* Normalization applied to each output row (LoKA section III-B). */
#define LOKA_NORM_NONE 0
#define LOKA_NORM_LAYER 1        /* (v-mean)/sqrt(var+eps)*gamma+beta      */
#define LOKA_NORM_RMS 2          /* v/sqrt(mean(v^2)+eps)*gamma            */
#define LOKA_NORM_BLOCK_RMS 3    /* RMSNorm over each norm_block columns    */
#define LOKA_ACT_NONE 0
#define LOKA_ACT_HARDSWISH 1     /* y*min(max(y+3,0),6)/6 after the norm     */

/* Library version, (major << 16) | minor. */
int32_t loka_version(void);

/* Message for the last non-OK status returned on this host thread. */
const char* loka_last_error(void);

/* Synchronizes `stream`, then reads and clears the device status flag that
 * kernels set when a wait runs out of time.  Returns LOKA_OK,
 * LOKA_ERR_TIMEOUT or LOKA_ERR_CUDA. */
loka_status loka_device_status(void* stream);

/* Diagnostic: launches one kernel whose only wait can never complete (an
 * mbarrier that nothing arrives at).  Its bounded wait gives up after
 * limit_ns nanoseconds (0 < limit_ns <= 1e10), sets the device status flag
 * and returns, so the next loka_device_status() reports LOKA_ERR_TIMEOUT and
 * the GPU context stays usable.  Exists to test the timeout path without
 * ever hanging or faulting a GPU.  Asynchronous. */
loka_status loka_selftest_watchdog(uint64_t limit_ns, void* stream);

/* Diagnostic: the dense tensor-core peak of this GPU, for the tensor-pipe
 * share of the FP8 contraction (LoKA page, Table I lists the GB300's dense
 * FP8 rate; the pages rate FP8 GEMMs by their fraction of it).  Launches one
 * CTA per SM; each issues `mmas_per_sm` tcgen05 MMAs of M = 128, N = 256 and
 * one 32-byte K step (kind 0: E4M3 x E4M3, K = 32; kind 1: bf16 x bf16,
 * K = 16; fp32 accumulation in tensor memory) on zero-filled shared-memory
 * tiles, with no memory traffic.  The caller times the launch with events
 * on `stream`: FLOPs = SMs * mmas_per_sm * 2 * 128 * 256 * K.  1 <=
 * mmas_per_sm <= 2^32.  Asynchronous; LOKA_ERR_INVALID_ARG for another kind
 * or count. */
loka_status loka_selftest_mma_peak(int32_t kind, int64_t mmas_per_sm, void* stream);

/* ------------------------------------------------------------------------
 * loka_quantize_fp8 -- amax, scale selection and E4M3 cast of one tensor.
 *
 * Defined by LoKA section II-C (FP8 recipes: tensorwise, rowwise, blockwise)
 * and the MX block scaling the GEM Training page uses (scale factors along
 * K).  For x of shape [rows, cols] (bf16, device, 16-byte aligned,
 * cols % 32 == 0) whose rows start ld elements apart (ld >= cols,
 * ld % 8 == 0; ld == cols for a dense tensor, larger for a column slice of
 * a wider one):
 *   LOKA_SCALE_TENSOR: amax = max|x|;  inv = fl32(448/amax); q = E4M3(fl32(x*inv));
 *                      scales[0] = fl32(amax/448)  (fp32, 1 element)
 *   LOKA_SCALE_ROW:    the same per row; scales is fp32 [rows]
 *   LOKA_SCALE_MX32:   per block of 32 along cols: e = clamp(floor(log2 amax)-8,
 *                      -127, 127); q = E4M3(x * 2^-e); scales is uint8 E8M0
 *                      [rows, cols/32] holding e + 127
 * amax == 0 gives scale 1 (tensor/row) or E8M0 code 0 (MX).  E4M3 rounding
 * is to nearest, ties to even, saturating at +-448; NaN stays NaN.
 * q: uint8 [rows, cols] device, dense (16-byte aligned).  workspace: device, at
 * least loka_quantize_fp8_workspace_size() bytes (0 for ROW and MX32; NULL
 * allowed then).  Asynchronous.
 * ---------------------------------------------------------------------- */
size_t loka_quantize_fp8_workspace_size(int64_t rows, int64_t cols, int32_t mode);
/* LOKA_SCALE_BLOCK32 (also taken by loka_quantize_fp8): square 32 x 32
 * blocks, the [32, 32] block quantization of the GEM Training page ("Low
 * Precision Flash Attention": one scale per 32x32 block makes quantization
 * transpose-invariant, so a tensor is quantized once for the GEMMs that take
 * it and its transpose).  Per block of rows 32i..32i+31 and cols
 * 32j..32j+31: e = clamp(floor(log2 amax) - 8, -127, 127) (the MX rule),
 * q = E4M3(x * 2^-e); scales is uint8 E8M0 [ceil(rows/32), cols/32] holding
 * e + 127 (a ragged last block row covers the rows that exist).  The
 * quantization of the transpose is the transpose of the codes and scales. */
loka_status loka_quantize_fp8(const void* x, int64_t rows, int64_t cols, int64_t ld, int32_t mode,
                              void* q, void* scales, void* workspace, size_t workspace_bytes,
                              void* stream);

/* loka_quantize_fp8_block32 -- LOKA_SCALE_BLOCK32 codes and scales, and in
 * the same pass, when q_t is not NULL, the codes of x transposed: q_t uint8
 * [cols, rows] (device, 16-byte aligned; rows % 32 == 0), equal to the codes
 * of quantizing x^T, whose scales are the transpose of scales.  ld is x's
 * row stride in elements, as for loka_quantize_fp8.
 * Asynchronous; no workspace. */
loka_status loka_quantize_fp8_block32(const void* x, int64_t rows, int64_t cols, int64_t ld, void* q, void* q_t,
                                      void* scales, void* stream);

/* ------------------------------------------------------------------------
 * loka_fp8_linear_norm -- Y = Norm(dequant(E4M3(X) E4M3(W)^T) + b), bf16.
 *
 * Defined by LoKA section II-C (the FP8 linear y = Wx + b), section III-B
 * "Block-wise Normalization" (the normalization fused into the GEMM
 * epilogue while the output row is still on chip; case 1, a whole output row
 * per thread block) and section I (wide ensembles of small GEMMs: a grouped
 * call runs several independent layers in one launch).
 *
 * One descriptor per independent layer (group).  All groups of one call must
 * share N, K, mode, norm, norm_block, eps, act and the *_is_fp8 flags; M
 * may differ.
 *   M >= 0; K >= 32 and a multiple of 32; N a multiple of 32 from 32 to
 *   2048 (the pages' production shapes, LoKA section II-C, include widths
 *   such as 768); anything else is LOKA_ERR_UNSUPPORTED.  A K that is not a
 *   multiple of 128 is read as zero-padded to the next one (no effect on
 *   the result).  Rows of up to 256 columns run on one CTA of 64, 128, 192
 *   or 256 columns (the columns past N hold nothing); rows wider than 256
 *   are split into 256-column slices, the last one partial: with LayerNorm
 *   or RMSNorm over a thread-block cluster of 2, 4 or 8 CTAs that merge
 *   their row statistics (weighted by the columns each holds) through
 *   distributed shared memory; with no norm or BlockNorm over
 *   ceil(N/256) independent CTAs (no statistic spans the row).
 *   x: bf16 [M,K] (x_is_fp8 = 0) or E4M3 [M,K] with x_scales as produced by
 *      loka_quantize_fp8 (x_is_fp8 = 1).  Same for w / w_scales / w_is_fp8.
 *   mode: LOKA_SCALE_* (LOKA_BF16 runs the bf16 GEMM; *_is_fp8 must be 0).
 *   LOKA_SCALE_BLOCK32 runs the block-scaled MMA of MX with each row taking
 *   its 32-row block's scales (caller-quantized operands: the scales of
 *   loka_quantize_fp8 with that mode).
 *   bias, gamma, beta: bf16 [N] or NULL (0, 1, 0).  y: bf16 [M,N] (see y_q).
 *   eps: added to the variance (LayerNorm) or mean square (RMSNorm).
 * Accumulation is fp32 in tensor memory; the epilogue works in fp32.
 * BlockNorm (LoKA section III-B 2 "Block-wise Normalization": RMSNorm
 * applied to (Wx + b).view(-1, BlockN), an unparameterized grouped RMSNorm
 * that needs no statistics across thread blocks): norm LOKA_NORM_BLOCK_RMS
 * normalizes every norm_block consecutive columns of a row by their own
 * root mean square (+ eps), then multiplies by gamma when given.
 * norm_block is 32, 64, 128 or 256 and divides N; rows wider than 256 need
 * no cluster exchange then.  Hard Swish (LoKA section III-B 3):
 * act LOKA_ACT_HARDSWISH applies y * min(max(y + 3, 0), 6) / 6 to the
 * normalized (and gamma/beta-scaled) output, before the bf16 rounding and
 * the quantized output.  Every group shares norm, norm_block and act.
 * Quantized output (PreNorm fusion, the GEM Training page, "Handling
 * Quantization Overhead": the next layer's activation quantization fused
 * into this layer's normalization): when y_q is set, the epilogue also
 * writes y_q and y_q_scales, equal byte for byte to what
 * loka_quantize_fp8(Y, M, N, y_q_mode) writes for the bf16 output Y of the
 * same call, so they feed the next layer as x / x_scales with x_is_fp8 = 1.
 * y may then be NULL (no bf16 copy).  y_q_mode LOKA_SCALE_ROW needs
 * N <= 256 (one CTA holds the row; LOKA_ERR_UNSUPPORTED otherwise);
 * LOKA_SCALE_MX32 takes every N (a block is 32 columns of one CTA);
 * LOKA_SCALE_TENSOR is LOKA_ERR_UNSUPPORTED (its amax needs every row before
 * the first code).  y_q is 16-byte aligned, y_q_scales 4-byte aligned for
 * ROW; every group sets y_q, or none does.  Not with mode LOKA_BF16.
 * workspace: device, loka_fp8_linear_norm_workspace_size() bytes (holds the
 * quantized operands and scales of bf16 inputs).  Asynchronous.
 * num_groups in [1, 16].  `descs` is a host array.
 * ---------------------------------------------------------------------- */
typedef struct loka_linear_desc {
  int64_t M, N, K;
  int32_t mode;          /* LOKA_SCALE_* or LOKA_BF16 */
  int32_t norm;          /* LOKA_NORM_* */
  float eps;
  int32_t x_is_fp8;
  int32_t w_is_fp8;
  int32_t y_q_mode;      /* scaling of y_q: LOKA_SCALE_ROW or LOKA_SCALE_MX32 (read when y_q is set) */
  const void* x;         /* device */
  const void* x_scales;  /* device, used when x_is_fp8 */
  const void* w;         /* device */
  const void* w_scales;  /* device, used when w_is_fp8 */
  const void* bias;      /* device bf16 [N] or NULL */
  const void* gamma;     /* device bf16 [N] or NULL */
  const void* beta;      /* device bf16 [N] or NULL */
  void* y;               /* device bf16 [M,N]; may be NULL when y_q is set */
  void* y_q;             /* device E4M3 [M,N] of the bf16 output for the next layer, or NULL */
  void* y_q_scales;      /* device fp32 [M] (LOKA_SCALE_ROW) or uint8 E8M0 [M,N/32] (LOKA_SCALE_MX32) */
  int32_t norm_block;    /* LOKA_NORM_BLOCK_RMS: columns per block (32, 64, 128 or 256) */
  int32_t act;           /* LOKA_ACT_NONE or LOKA_ACT_HARDSWISH */
} loka_linear_desc;

size_t loka_fp8_linear_norm_workspace_size(const loka_linear_desc* descs, int32_t num_groups);
loka_status loka_fp8_linear_norm(const loka_linear_desc* descs, int32_t num_groups,
                                 void* workspace, size_t workspace_bytes, void* stream);

/* ------------------------------------------------------------------------
 * loka_fp8_linear_norm_static -- loka_fp8_linear_norm without any allocation.
 *
 * The pages have no counterpart to this call; it exists for callers that
 * cannot allocate device memory: code running where no allocator is reachable
 * (a plugin handed only input and output buffers by its host framework, or a
 * runtime that forbids cudaMalloc on its path) and so cannot supply the
 * workspace that loka_fp8_linear_norm needs for the quantized operands.
 *
 * Same arguments, semantics and results as loka_fp8_linear_norm, minus the
 * workspace: the scratch is a built-in 4 MiB device array owned by the
 * library (every GPU that loads the library holds it until the process
 * exits).  Calls whose quantized operands and scales need more than 4 MiB
 * (loka_fp8_linear_norm_workspace_size() > 4194304) fail with
 * LOKA_ERR_WORKSPACE before anything is launched.  The call allocates
 * nothing itself (no cudaMalloc, cudaFree or allocating library routine).
 * The first call on a device looks up the array's device address (a host
 * runtime query, done once per device); make that first call before any
 * stream capture.  Every call shares the one array and leaves its contents
 * behind; the call clears what must start at zero.  Calls that overlap on
 * the GPU (different streams, or different host threads) race on the array:
 * serialize them.
 * ---------------------------------------------------------------------- */
loka_status loka_fp8_linear_norm_static(const loka_linear_desc* descs, int32_t num_groups, void* stream);

/* ------------------------------------------------------------------------
 * loka_quant_error -- quantization-error probe of one layer.
 *
 * Defined by LoKA section II-C "Error Analysis" (MERE: the mean element-wise
 * relative error |out-ref|/|ref| of a low-precision output against a
 * high-precision one) and section III-A "Offline Error Quantification"
 * (loss = MERE(FP8(Wx+b), high-precision(Wx+b)) per layer, Fig. 5).
 * out = the FP8 linear output before normalization in fp32 (desc->mode);
 * ref = the bf16-input linear with fp32 accumulation.  desc->y is ignored.
 * Reports, over all M*N elements:
 *   mere        mean of |out-ref|/|ref| over elements with ref != 0
 *   rel_err_fro ||out-ref||_F / ||ref||_F
 *   max_abs     max |out-ref|
 *   max_abs_post_norm  max |Norm(out) - Norm(ref)| with the layer's norm,
 *               norm_block, eps, gamma, beta and act (fp32 outputs before
 *               the bf16 rounding); equals max_abs when the layer has
 *               neither a norm nor an activation
 *   zero_ref_count, count
 * workspace: loka_quant_error_workspace_size() bytes.  SYNCHRONIZES the
 * stream; `stats` is a host pointer.
 * ---------------------------------------------------------------------- */
typedef struct loka_error_stats {
  double mere;
  double rel_err_fro;
  double max_abs;
  double max_abs_post_norm;
  int64_t zero_ref_count;
  int64_t count;
} loka_error_stats;

size_t loka_quant_error_workspace_size(const loka_linear_desc* desc);
loka_status loka_quant_error(const loka_linear_desc* desc, void* workspace, size_t workspace_bytes,
                             loka_error_stats* stats, void* stream);

/* ------------------------------------------------------------------------
 * loka_dispatch_select -- choose a variant for one layer (host only).
 *
 * Defined by LoKA section III-C "Library and Recipe Selection": filter the
 * candidates by expected error (MERE below a threshold, typically 0.2) and by
 * speedup over the high-precision path (typically > 1.05x), then take the one
 * with the highest measured throughput; section VI "Limitations": a layer
 * with no qualifying candidate runs in high precision (LOKA_BF16).
 * table: host array of n measured rows.  A query matches rows with equal N,
 * K and norm; among them the rows nearest in log2(M) (ties: larger M) and in
 * outlier fraction (ties: larger) are the candidates.  Filters: rel_err <=
 * max_rel_err; mere < max_mere when max_mere >= 0; t_bf16/t > min_speedup
 * when min_speedup >= 0 (needs a LOKA_BF16 row).  Smallest time wins; ties
 * go to smaller rel_err, then the smaller variant id.  *choice (host) gets a
 * LOKA_SCALE_* / LOKA_BF16 value.  Pure host code, no GPU work.
 * ---------------------------------------------------------------------- */
typedef struct loka_problem {
  int64_t M, N, K;
  int32_t norm;
  int32_t reserved;
  double outlier_frac;
} loka_problem;

typedef struct loka_dispatch_entry {
  loka_problem p;
  int32_t variant;
  int32_t reserved;
  double time_us;
  double rel_err;
  double mere;
} loka_dispatch_entry;

typedef struct loka_policy {
  double max_rel_err;   /* e.g. 1e-2 */
  double max_mere;      /* e.g. 0.2; < 0 disables */
  double min_speedup;   /* e.g. 1.05; < 0 disables */
} loka_policy;

loka_status loka_dispatch_select(const loka_dispatch_entry* table, int64_t n, const loka_problem* p,
                                 const loka_policy* policy, int32_t* choice);

/* ------------------------------------------------------------------------
 * LoKA Probe: online learning of a layer's input distribution, and sampling.
 *
 * Defined by LoKA section III-A 1 "Online Distribution Learning": the batch
 * dimension is independent, so a layer's inputs are modeled per feature by
 * a mean and a covariance, tracked with a batched Welford / Chan update in
 * higher precision; synthetic inputs are T' = 1 mu^T + Z L^T with
 * Z ~ N(0, I) and L L^T = Sigma + eps I.
 *
 * loka_probe_stats_update merges a batch x (bf16 [B, K], device, 16-byte
 * aligned) into *stats: with the batch mean mu_b and scatter
 * S_b = (x - mu_b)^T (x - mu_b), n += B, mu += (B / n_new)(mu_b - mu),
 * scatter += S_b + (n_old B / n_new) d d^T, d = mu_b - mu_old.  mu (fp64 [K])
 * and scatter (fp64 [K, K], the unnormalized scatter matrix; the unbiased
 * covariance is scatter / (n - 1)) are caller-owned device arrays; n is
 * advanced on the host when the call is queued.  x^T x runs on the tensor
 * cores in fp32 over split-K groups of up to 4096 rows, summed and centred
 * in fp64 (raw moments: exact enough when |mean| is not far above the
 * standard deviation, as for normalized activations).  K is 128, 256, 512,
 * 1024 or 2048; B <= 2^24.  workspace: loka_probe_stats_workspace_size()
 * bytes, 256-byte aligned.  Asynchronous.
 *
 * loka_probe_sample_inputs writes out (bf16 [B, K]) = Z L^T + mu, Z the
 * counter-based normals of `seed` (SplitMix64 random number i from state
 * seed + (i + 1) * 0x9E3779B97F4A7C15; Box-Muller on 24-bit uniforms in
 * fp32; Z[b, k] is normal b K + k), mu bf16 [K], chol = L bf16 [K, K]
 * row-major (the caller's Cholesky factor of the regularized covariance).
 * workspace: loka_probe_sample_workspace_size() bytes.  Asynchronous.
 * ---------------------------------------------------------------------- */
typedef struct loka_input_stats {
  int64_t n;             /* rows merged so far (host) */
  int64_t K;             /* features */
  double* mu;            /* device fp64 [K] */
  double* scatter;       /* device fp64 [K, K] */
} loka_input_stats;

size_t loka_probe_stats_workspace_size(int64_t B, int64_t K);
/* loka_probe_covariance: cov (fp64 [K, K], device, caller-owned) =
 * scatter / (n - 1), the unbiased covariance of the rows merged so far
 * (section III-A 1: the covariance the sampler draws from).  n >= 2.
 * Asynchronous. */
loka_status loka_probe_covariance(const loka_input_stats* stats, double* cov, void* stream);
loka_status loka_probe_stats_update(loka_input_stats* stats, const void* x, int64_t B, void* workspace,
                                    size_t workspace_bytes, void* stream);
/* loka_probe_cholesky: L (bf16 [K, K] row-major, lower, zero above the
 * diagonal) with L L^T = Sigma + eps I, Sigma = scatter / (n - 1) and
 * eps = eps_rel * trace(Sigma) / K (the page suggests about 1e-6), and mu as
 * bf16 [K]: the inputs of loka_probe_sample_inputs.  fp32 left-looking
 * factorization on one thread block (a once-per-snapshot K x K step).
 * n >= 2.  LOKA_ERR_NUMERIC when a pivot is not positive.  Synchronizes
 * the stream.  workspace: loka_probe_cholesky_workspace_size() bytes. */
size_t loka_probe_cholesky_workspace_size(int64_t K);
loka_status loka_probe_cholesky(const loka_input_stats* stats, double eps_rel, void* chol, void* mu_out,
                                void* workspace, size_t workspace_bytes, void* stream);
size_t loka_probe_sample_workspace_size(int64_t B, int64_t K);
loka_status loka_probe_sample_inputs(const void* mu, const void* chol, int64_t B, int64_t K, uint64_t seed,
                                     void* out, void* workspace, size_t workspace_bytes, void* stream);

/* ------------------------------------------------------------------------
 * LoKA Probe: the weight model.
 *
 * Defined by LoKA section III-A 1, "Optimized Weight Distribution Modeling"
 * and "Sampling learned distributions" (b): a weight W [R, C] is modeled as
 * matrix-normal, W ~ MN(M, U, V), vec(W) ~ N(vec(M), V (x) U), with the row
 * covariance U [R, R] and column covariance V [C, C] tracked by a
 * Kronecker-factor (flip-flop) update smoothed by an exponential moving
 * average, through linear solves against regularized Cholesky factors.
 *
 * loka_probe_weight_update merges one weight w (bf16 [R, C], device) into
 * *stats.  The first call (n == 0) starts the model: M = W, U = I, V = I.
 * Every later call, with eps_A = eps_rel * trace(A) / dim(A) on the matrix A
 * it regularizes (the page suggests eps_rel about 1e-6):
 *   Wc = W - M;  L_V L_V^T = V + eps_V I,  U' = (Wc L_V^-T)(Wc L_V^-T)^T / C;
 *   L_U L_U^T = U + eps_U I,  V' = (L_U^-1 Wc)^T (L_U^-1 Wc) / R
 *   (both with the U, V held before the call);
 *   U'' = m U + (1-m) U',  V'' = m V + (1-m) V'  (m = momentum, in [0, 1));
 *   U = (U'' + U''^T)/2 + eps_U I,  V = (V'' + V''^T)/2 + eps_V I;
 *   s = trace(U)/R,  U /= s,  V *= s  (V (x) U unchanged);  M = m M + (1-m) W.
 * mean (fp32 [R, C]), U (fp32 [R, R]) and V (fp32 [C, C], all row-major)
 * are caller-owned device arrays; n is advanced on the host.  fp32 SIMT
 * kernels (a once-per-probe-interval step off the data-parallel path).
 * 2 <= R, C <= 2048, C even.  LOKA_ERR_NUMERIC when a factor's pivot is not
 * positive.  Synchronizes the stream (except for the first call).
 *
 * loka_probe_sample_weights writes out (bf16 [R, C]) = M + L_U Z L_V^T with
 * L_U L_U^T = U + eps_U I, L_V L_V^T = V + eps_V I and Z the counter-based
 * normals of `seed` (Z[r, c] is normal r C + c, the stream of
 * loka_probe_sample_inputs, in fp32).  Synchronizes the stream.
 * workspace: loka_probe_weight_workspace_size(R, C) bytes, 256-byte aligned,
 * for both calls.
 * ---------------------------------------------------------------------- */
typedef struct loka_weight_stats {
  int64_t n;             /* updates merged so far (host) */
  int64_t R;             /* weight rows */
  int64_t C;             /* weight columns */
  float* mean;           /* device fp32 [R, C] */
  float* U;              /* device fp32 [R, R] */
  float* V;              /* device fp32 [C, C] */
} loka_weight_stats;

size_t loka_probe_weight_workspace_size(int64_t R, int64_t C);
loka_status loka_probe_weight_update(loka_weight_stats* stats, const void* w, double momentum, double eps_rel,
                                     void* workspace, size_t workspace_bytes, void* stream);
loka_status loka_probe_sample_weights(const loka_weight_stats* stats, double eps_rel, uint64_t seed, void* out,
                                      void* workspace, size_t workspace_bytes, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* LOKA_H_ */
