// Internal declarations shared by the library's translation units (not part
// of the C ABI; see include/loka.h for that).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace loka {

constexpr int kScaleTensor = 0;
constexpr int kScaleRow = 1;
constexpr int kScaleMx32 = 2;
constexpr int kBf16 = 3;
constexpr int kScaleBlock32 = 4;   // square 32 x 32 blocks, E8M0 scales

constexpr int kNormNone = 0;
constexpr int kNormLayer = 1;
constexpr int kNormRms = 2;
constexpr int kNormBlockRms = 3;   // RMSNorm over fixed blocks of the output row (BlockNorm)
constexpr int kActNone = 0;
constexpr int kActHardSwish = 1;

constexpr int kMaxGroups = 16;
constexpr int kMaxQuantJobs = 2 * kMaxGroups;

// One tensor to quantize: x bf16 [rows, cols] -> q E4M3 [rows, cols] +
// scales (fp32 [1] / fp32 [rows] / E8M0 [rows, cols/32]).
struct QuantJob {
  const void* x;
  uint8_t* q;
  void* scales;
  unsigned* amax_slot;   // tensorwise only: 4-byte accumulator, zeroed by the launcher
  uint8_t* sf_tc;        // MX / 32x32 blocks, optional: E8M0 codes again in the tensor-memory copy
                         // layout (32x32 blocks: every row of a block row repeats its codes)
  uint8_t* q_t;          // 32x32 blocks only, optional: the codes transposed, [cols, rows]
  int64_t rows;
  int64_t cols;
  int64_t ld;            // elements between the starts of consecutive rows of x (>= cols, % 8 == 0)
  int64_t row_begin;     // first row of this job in the launch's joint row space (32x32 blocks:
                         // first unit of 32 rows x 256 columns, set by launch_quantize)
};

struct QuantJobs {
  QuantJob j[kMaxQuantJobs];
  int n;
  int64_t total_rows;
};

cudaError_t launch_quantize(const QuantJobs& jobs, int mode, int sms, cudaStream_t stream);

// MX scale factors in the tensor-memory copy layout: for row block rb (128
// rows) and K block kb (128 elements = 4 codes per row), a 512-byte block at
// (rb * ceil(K/128) + kb) * 512; inside it row m, code kk sits at byte
// (m % 32) * 16 + ((m % 128) / 32) * 4 + kk.  tcgen05.cp.32x128b.warpx4 of
// such a block puts the codes of row m in TMEM lane m, column (m % 128) / 32,
// byte kk.
__host__ __device__ inline int64_t sf_tc_offset(int64_t m, int64_t blk32, int64_t kb128_count) {
  const int64_t rb = m >> 7, kb = blk32 >> 2, kk = blk32 & 3;
  return (rb * kb128_count + kb) * 512 + (m & 31) * 16 + ((m & 127) >> 5) * 4 + kk;
}
__host__ __device__ inline int64_t sf_tc_bytes(int64_t rows, int64_t cols) {
  return ((rows + 127) / 128) * ((cols + 127) / 128) * 512;
}

// Rewrites logical E8M0 codes into the tensor-memory copy layout: [rows,
// cols/32] (row_div 1, MX) or [ceil(rows/32), cols/32] (row_div 32, square
// blocks: each row takes its block row's codes).
cudaError_t launch_sf_permute(const uint8_t* logical, uint8_t* tc, int64_t rows, int64_t cols, int row_div, int sms,
                              cudaStream_t stream);

// ------------------------------------------------------------------ GEMM
// Per-group arguments of the fused GEMM + normalization kernel.
struct GemmGroup {
  CUtensorMap tm_a;      // A [M,K] (E4M3 or bf16), box {128 bytes of K, 128 rows}
  CUtensorMap tm_b;      // B [N,K], box {128 bytes of K, min(N,256) rows}
  const float* sx;       // per-row [M] / per-tensor [1] activation scale, or null (=1)
  const float* sw;       // per-row [N] / per-tensor [1] weight scale, or null (=1)
  const uint8_t* sfa_tc; // MX: A scale codes in the tensor-memory copy layout
  const uint8_t* sfb_tc; // MX: B scale codes in the tensor-memory copy layout
  const uint16_t* bias;  // bf16 [N] or null
  const uint16_t* gamma; // bf16 [N] or null
  const uint16_t* beta;  // bf16 [N] or null
  void* y;               // output (the fp32 output is stored directly); the quantized
                         // output kind may leave it null (no bf16 copy)
  const uint16_t* xbf;   // in-kernel activation quantization: bf16 X [M, K] (dense rows)
  uint8_t* yq;           // quantized output kind: E4M3 codes [M, N] of the bf16 output
  void* yq_scales;       // and their scales: fp32 [M] (per row) or E8M0 [M, N/32] (MX)
  int64_t M;
  int32_t tile_begin;    // first tile of this group in the launch's tile space
  int32_t sx_per_row;    // 1: sx has M entries, 0: one entry
  int32_t sw_per_row;
  int32_t b_box_rows;    // rows of tm_b's box: the columns one CTA owns (checked before a launch)
};

struct GemmParams {
  GemmGroup g[kMaxGroups];
  int32_t num_groups;
  int32_t total_tiles;
  int32_t K;
  int32_t norm;
  float eps;
  int32_t stages;        // shared-memory ring depth (set by the launcher)
  int32_t w_ready;       // 1: W and its scales were complete before the launch that precedes
                         // this GEMM, so resident W may load before waiting for that launch
  int32_t x_ready;       // 1: the bf16 X was complete before the launch that precedes this GEMM
                         // (in-kernel quantization reads it before waiting for that launch)
  int32_t a_bufs;        // in-kernel quantization: quantized A tiles in shared memory (1 or 2)
  int32_t yq_mode;       // quantized output kind: kScaleRow or kScaleMx32
  int32_t norm_block;    // BlockNorm block (32, 64, 128 or 256 columns)
  int32_t act;           // kActNone or kActHardSwish, after the normalization
  int32_t slices;        // CL == 1 launches: independent column slices per row (1 = none)
  int32_t n_cols;        // columns of an output row (the layer's N; set by the launcher)
  float inv_n_cols;      // 1 / n_cols
  // cluster merge of row statistics (Chan), CTA j of a cluster holding the
  // row's columns from j * 256 on: chan_w[j] = n_b / (n_a + n_b) and
  // chan_c[j] = n_a n_b / (n_a + n_b) with n_a = 256 j and n_b its columns
  // (0 for a CTA past the row's end); set by the launcher
  float chan_w[8];
  float chan_c[8];
  unsigned* status;      // device status word
  uint64_t wait_limit_ns;
};

// kE4M3Qx: A is the caller's bf16 X, quantized per row inside the GEMM (the
// codes go straight into the shared-memory A tile); B is E4M3 W with per-row
// scales.
enum class OperandKind : int { kE4M3 = 0, kBf16 = 1, kMxE4M3 = 2, kE4M3Qx = 3 };
// kQuant: E4M3 codes and scales of the bf16 output (plus the bf16 output when
// its pointer is set)
enum class OutKind : int { kBf16 = 0, kF32 = 1, kQuant = 2 };

// How an output row of N columns is split: `local` columns per CTA; `cl`
// CTAs of a thread-block cluster per tile (row statistics exchanged), or
// `slices` independent CTAs per tile (no statistic spans the row).
struct GemmRoute {
  int local, cl, slices;
};
GemmRoute gemm_route(int N, int norm);
// (columns per CTA, cluster size) of a row of N columns whose statistics
// span it; false when N is not a multiple of 32 in [32, 2048].
bool split_n_host(int N, int* local, int* cl);

// Launches the persistent GEMM + epilogue kernel for N columns (fills in
// p.stages and p.slices; tm_b must have been encoded with a box of
// gemm_route(...).local rows, recorded in b_box_rows).
cudaError_t launch_gemm_norm(GemmParams& p, int N, OperandKind op, OutKind out, int sms, cudaStream_t stream);

// Whether the kernel has a shared-memory plan for this N, K and operand type.
bool gemm_supported(int N, int K, OperandKind op);
// Whether the GEMM quantizes bf16 X per row itself (kE4M3Qx) for this row
// width, K and output kind: where it has a plan that keeps W resident beside
// two A tiles.
bool gemm_qx_supported(int N, int K, int norm, OutKind out);

// Probe reduction: accumulates MERE / Frobenius / max statistics of out vs ref.
cudaError_t launch_error_reduce(const float* out, const float* ref, int64_t n, double* acc, int sms, cudaStream_t stream);

// Probe statistics (probe_stats.cu): X [B,K] -> X^T as G groups [K, Bg]
// (zero-padded) plus per-128-row-tile column sums; then the ordered merge of
// the GEMM partials (fp32 [G][K][K]) into mu and S (fp64, Chan update); and
// the counter-based normals of the sampler (bf16).
cudaError_t launch_stats_transpose(const void* x, int64_t B, int64_t K, int64_t Bg, int G, void* xt, float* colpart,
                                   cudaStream_t stream);
cudaError_t launch_stats_merge(const float* colpart, int64_t tiles, const float* partials, int G, int64_t K,
                               double* colwork /* 35 K fp64 */, double* mu, double* S, int64_t n_old, int64_t nb,
                               int sms, cudaStream_t stream);
cudaError_t launch_normals(uint64_t seed, int64_t count, void* z, int sms, cudaStream_t stream);
cudaError_t launch_normals_f32(uint64_t seed, int64_t count, float* z, int sms, cudaStream_t stream);

// Probe weight model (probe_weights.cu): the matrix-normal W ~ MN(M, U, V)
// of a weight [R, C].  Workspace (fp32 unless noted): Wc, W_V, W_U [R, C];
// L_U, U' [R, R]; L_V, V' [C, C]; 2 fp64 traces and a status word.
struct WeightWork {
  float *wc, *wv, *wu, *lu, *u1, *lv, *v1;
  double* trace;   // [2]
  int* status;     // [2]: a non-positive pivot in the factor of U (0) or V (1)
};
// First update: M = W, U = I, V = I.
cudaError_t launch_weight_init(const void* w, int64_t R, int64_t C, float* M, float* U, float* V, int sms,
                               cudaStream_t stream);
// One flip-flop update of (M, U, V) with W (bf16 [R, C]), momentum m.
cudaError_t launch_weight_update(const void* w, int64_t R, int64_t C, double m, double eps_rel, float* M, float* U,
                                 float* V, const WeightWork& ws, int sms, cudaStream_t stream);
// W' = M + L_U Z L_V^T (bf16 [R, C]); Z: the seed's counter-based normals.
cudaError_t launch_weight_sample(const float* M, const float* U, const float* V, int64_t R, int64_t C, double eps_rel,
                                 uint64_t seed, void* out, const WeightWork& ws, int sms, cudaStream_t stream);
// cov (fp64 [K, K]) = S / (n - 1)
cudaError_t launch_covariance(const double* S, int64_t K, int64_t n, double* cov, int sms, cudaStream_t stream);
// Cholesky factor of S / (n - 1) + eps I (one block, fp32; A: K x K fp32
// scratch); L and mu_out bf16; *status = 1 if not positive definite.
cudaError_t launch_cholesky(const double* S, const double* mu, int64_t K, int64_t n, double eps_rel, float* A,
                            void* L, void* mu_out, int* status, cudaStream_t stream);

// Watchdog self-test: waits on a barrier that nothing completes.
cudaError_t launch_watchdog_selftest(unsigned* status, uint64_t limit_ns, cudaStream_t stream);
// Tensor-core peak: one CTA per SM issuing `mmas` back-to-back MMAs (kind 0
// E4M3, 1 bf16) on shared-memory tiles (mma_peak.cu).
cudaError_t launch_mma_peak(int kind, int64_t mmas, int sms, unsigned* status, uint64_t limit_ns, cudaStream_t stream);

}  // namespace loka
