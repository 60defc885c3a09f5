// LoKA Probe: online learning of a layer's input distribution (running mean
// and scatter matrix, merged batch by batch) and sampling of synthetic
// inputs from it.
//
// Defined by "LoKA: Low-precision Kernel Applications for Recommendation
// Models at Scale", section III-A 1 "Online Distribution Learning": the batch
// dimension is independent, so a layer's activations are modeled per feature
// by their mean and covariance, tracked with a batched Welford / Chan update
// (accumulated in higher precision); synthetic inputs are
// T' = 1 mu^T + Z L^T with Z ~ N(0, I) and L the Cholesky factor of the
// regularized covariance.
//
// The batch scatter X^T X is a dense contraction over the batch and runs on
// the tensor cores through the fused GEMM (bf16 operands, fp32 output, no
// norm), split over the batch: the transpose kernel below writes X^T as G
// groups [K, Bg] (batch rows zero-padded to a multiple of 128, which adds
// nothing to the sums), the grouped GEMM makes one fp32 [K, K] partial per
// group, and the merge kernel adds the partials in group order in fp64,
// centres them with the column sums and applies the Chan update.
#include "loka_internal.h"
#include "ptx.cuh"

namespace loka {

namespace {

constexpr int kTRows = 128;   // batch rows per transpose tile
constexpr int kTCols = 64;    // features per transpose tile

// X [B, K] bf16 -> Xt [G][K][Bg] bf16 (rows b >= B are zero) and per-tile
// column sums colpart[tile][K] (fp32, the tile's 128 rows).  One 256-thread
// block per (128-row tile, 64-feature tile).
__global__ void __launch_bounds__(256) stats_transpose_kernel(const uint16_t* __restrict__ x, int64_t B, int64_t K,
                                                              int64_t Bg, uint16_t* __restrict__ xt,
                                                              float* __restrict__ colpart) {
  __shared__ uint16_t tile[kTRows][kTCols + 2];
  __shared__ float part[4][kTCols];
  const int64_t rt = blockIdx.x, ct = blockIdx.y;
  const int64_t b0 = rt * kTRows, c0 = ct * kTCols;
  const int t = threadIdx.x;
  // coalesced load: 8 threads per row (16 bytes each), 32 rows per pass
  for (int pass = 0; pass < kTRows / 32; ++pass) {
    const int r = pass * 32 + (t >> 3), q = t & 7;
    const int64_t b = b0 + r;
    uint4 v = make_uint4(0, 0, 0, 0);
    if (b < B) v = *reinterpret_cast<const uint4*>(x + b * K + c0 + q * 8);
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      tile[r][q * 8 + 2 * e] = static_cast<uint16_t>(w[e] & 0xFFFFu);
      tile[r][q * 8 + 2 * e + 1] = static_cast<uint16_t>(w[e] >> 16);
    }
  }
  __syncthreads();
  // column sums: feature c = t % 64 over rows 32h .. 32h + 31, then the 4 parts
  {
    const int c = t & 63, h = t >> 6;
    float s = 0.0f;
    for (int r = 0; r < 32; ++r) s += __uint_as_float(static_cast<uint32_t>(tile[h * 32 + r][c]) << 16);
    part[h][c] = s;
  }
  // transposed store: feature row c0 + c of group g gets the tile's 128
  // batch rows, 16 bytes (8 rows) per thread, 16 threads per feature row
  const int64_t g = b0 / Bg, lb0 = b0 - g * Bg;
  for (int pass = 0; pass < kTCols / 16; ++pass) {
    const int c = pass * 16 + (t >> 4), r8 = t & 15;
    uint32_t w[4];
#pragma unroll
    for (int e = 0; e < 4; ++e)
      w[e] = static_cast<uint32_t>(tile[r8 * 8 + 2 * e][c]) | (static_cast<uint32_t>(tile[r8 * 8 + 2 * e + 1][c]) << 16);
    *reinterpret_cast<uint4*>(xt + (g * K + c0 + c) * Bg + lb0 + r8 * 8) = make_uint4(w[0], w[1], w[2], w[3]);
  }
  __syncthreads();
  if (t < kTCols) colpart[rt * K + c0 + t] = part[0][t] + part[1][t] + part[2][t] + part[3][t];
}

constexpr int kSumChunks = 32;   // tile chunks of the first column-sum stage

// Column sums, stage 1: part[chunk][k] = sum of colpart[tile][k] over the
// chunk's tiles (fp64, in tile order).  Block (column block of 32, chunk);
// warp w takes tiles w, w + 8, ... of the chunk, then the 8 warp sums are
// added in warp order.
__global__ void __launch_bounds__(256) stats_colsum_kernel(const float* __restrict__ colpart, int64_t tiles, int64_t K,
                                                           double* __restrict__ part) {
  __shared__ double wsum[8][32];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t k = static_cast<int64_t>(blockIdx.x) * 32 + lane;
  const int64_t per = (tiles + kSumChunks - 1) / kSumChunks;
  const int64_t t0 = static_cast<int64_t>(blockIdx.y) * per;
  const int64_t t1 = t0 + per < tiles ? t0 + per : tiles;
  double s = 0.0;
  for (int64_t t = t0 + warp; t < t1; t += 8) s += static_cast<double>(colpart[t * K + k]);
  wsum[warp][lane] = s;
  __syncthreads();
  if (warp == 0) {
    double a = wsum[0][lane];
#pragma unroll
    for (int w = 1; w < 8; ++w) a += wsum[w][lane];
    part[blockIdx.y * K + k] = a;
  }
}

// Column sums, stage 2, and the per-column terms of the update: s = sum of
// the chunks in order, m = s / B (the batch mean), d = m - mu_old.
__global__ void __launch_bounds__(256) stats_colprep_kernel(const double* __restrict__ part, int64_t K,
                                                            const double* __restrict__ mu, double nb,
                                                            double* __restrict__ col) {
  const int64_t k = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (k >= K) return;
  double s = 0.0;
  for (int c = 0; c < kSumChunks; ++c) s += part[c * K + k];
  const double m = s / nb;
  col[k] = s;
  col[K + k] = m;
  col[2 * K + k] = m - mu[k];
}

// Chan update of the scatter matrix: S += S_b + (n_old B / n_new) d d^T with
// S_b = sum_g Y_g - s m^T (raw moments centred; s = column sums, m = s / B).
__global__ void __launch_bounds__(256) stats_merge_kernel(const float* __restrict__ partials, int G, int64_t K,
                                                          const double* __restrict__ col, double* __restrict__ S,
                                                          double w) {
  const int64_t kk = K * K;
  const double* s = col;
  const double* m = col + K;
  const double* d = col + 2 * K;
  for (int64_t e = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; e < kk;
       e += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t i = e / K, j = e - i * K;
    // the G (<= 16) partials, loaded together, added in group order
    float v[kMaxGroups];
#pragma unroll
    for (int g = 0; g < kMaxGroups; ++g) v[g] = g < G ? partials[g * kk + e] : 0.0f;
    double raw = 0.0;
#pragma unroll
    for (int g = 0; g < kMaxGroups; ++g) raw += static_cast<double>(v[g]);
    S[e] += (raw - s[i] * m[j]) + w * d[i] * d[j];
  }
}

// mu += (B / n_new) d
__global__ void __launch_bounds__(256) stats_mean_kernel(const double* __restrict__ col, double* __restrict__ mu,
                                                         int64_t K, double f) {
  const int64_t k = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (k >= K) return;
  mu[k] += f * col[2 * K + k];
}

// SplitMix64 output for state `s` (the output function of SplittableRandom).
__device__ __forceinline__ uint64_t splitmix64(uint64_t s) {
  uint64_t z = s;
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

// Z [count] bf16: normal pair j from random numbers 2j and 2j + 1 of the
// seed's counter-based stream (state seed + (i + 1) * golden gamma), by
// Box-Muller on 24-bit uniforms, in fp32.
// Normal pair j as bf16 (packed, F32 = false) or fp32 (F32 = true).
template <bool F32>
__global__ void __launch_bounds__(256) normals_kernel(uint64_t seed, int64_t pairs, void* __restrict__ z) {
  constexpr uint64_t kGamma = 0x9E3779B97F4A7C15ull;
  for (int64_t j = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; j < pairs;
       j += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const uint64_t i0 = static_cast<uint64_t>(2 * j);
    const uint64_t r1 = splitmix64(seed + (i0 + 1) * kGamma);
    const uint64_t r2 = splitmix64(seed + (i0 + 2) * kGamma);
    const float u1 = static_cast<float>((r1 >> 40) + 1) * 0x1p-24f;   // (0, 1], exact
    const float u2 = static_cast<float>(r2 >> 40) * 0x1p-24f;         // [0, 1), exact
    const float rad = sqrtf(-2.0f * logf(u1));
    float s, c;
    sincospif(2.0f * u2, &s, &c);
    if (F32)
      static_cast<float2*>(z)[j] = make_float2(rad * c, rad * s);
    else
      static_cast<uint32_t*>(z)[j] = pack_bf16x2(rad * c, rad * s);
  }
}

// The regularized covariance and its Cholesky factor, on one block:
// A = S / (n - 1) + eps I with eps = eps_rel * trace(S / (n - 1)) / K (fp32,
// from the fp64 scatter), factored in place column by column (left-looking:
// L_jj = sqrt(A_jj - sum_k L_jk^2), L_ij = (A_ij - sum_k L_ik L_jk) / L_jj,
// k < j), row j's finished entries staged in shared memory.  Writes L (bf16,
// zero above the diagonal) and mu (bf16); *status = 1 when a pivot is not
// positive (A not positive definite).
__global__ void __launch_bounds__(1024) cholesky_kernel(const double* __restrict__ S, const double* __restrict__ mu,
                                                        int64_t K, double inv_n1, double eps_rel, float* __restrict__ A,
                                                        uint16_t* __restrict__ L, uint16_t* __restrict__ mu_out,
                                                        int* __restrict__ status) {
  extern __shared__ float rowj[];            // K floats
  __shared__ double red[32];
  __shared__ float pivot;
  __shared__ int bad;
  const int t = threadIdx.x, nt = blockDim.x;
  const int lane = t & 31, warp = t >> 5;
  // trace of S / (n - 1)
  double tr = 0.0;
  for (int64_t i = t; i < K; i += nt) tr += S[i * K + i] * inv_n1;
  for (int o = 16; o > 0; o >>= 1) tr += __shfl_xor_sync(0xffffffffu, tr, o);
  if (lane == 0) red[warp] = tr;
  if (t == 0) bad = 0;
  __syncthreads();
  if (t == 0) {
    double a = 0.0;
    for (int w = 0; w < nt / 32; ++w) a += red[w];
    red[0] = a;
  }
  __syncthreads();
  const double eps = eps_rel * red[0] / static_cast<double>(K);
  for (int64_t e = t; e < K * K; e += nt) {
    const int64_t i = e / K, j = e - i * K;
    A[e] = static_cast<float>(S[e] * inv_n1 + (i == j ? eps : 0.0));
  }
  __syncthreads();
  for (int64_t j = 0; j < K; ++j) {
    for (int64_t k = t; k < j; k += nt) rowj[k] = A[j * K + k];
    __syncthreads();
    // diagonal
    float s = 0.0f;
    for (int64_t k = t; k < j; k += nt) s = fmaf(rowj[k], rowj[k], s);
    for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
    if (lane == 0) red[warp] = s;
    __syncthreads();
    if (t == 0) {
      float a = 0.0f;
      for (int w = 0; w < nt / 32; ++w) a += static_cast<float>(red[w]);
      const float d = A[j * K + j] - a;
      if (!(d > 0.0f)) bad = 1;
      pivot = d > 0.0f ? sqrtf(d) : 1.0f;
      A[j * K + j] = pivot;
    }
    __syncthreads();
    if (bad) break;
    const float inv = 1.0f / pivot;
    for (int64_t i = j + 1 + t; i < K; i += nt) {
      float dot = 0.0f;
      const float* ri = A + i * K;
      for (int64_t k = 0; k < j; ++k) dot = fmaf(ri[k], rowj[k], dot);
      A[i * K + j] = (A[i * K + j] - dot) * inv;
    }
    __syncthreads();
  }
  if (t == 0) *status = bad;
  for (int64_t e = t; e < K * K; e += nt) {
    const int64_t i = e / K, j = e - i * K;
    const float v = j <= i ? A[e] : 0.0f;
    L[e] = static_cast<uint16_t>(pack_bf16x2(v, 0.0f) & 0xFFFFu);
  }
  for (int64_t i = t; i < K; i += nt) mu_out[i] = static_cast<uint16_t>(pack_bf16x2(static_cast<float>(mu[i]), 0.0f) & 0xFFFFu);
}

// cov = S / (n - 1): the unbiased covariance of the merged rows (fp64,
// one IEEE division per entry).
__global__ void __launch_bounds__(256) covariance_kernel(const double* __restrict__ S, int64_t count, double n1,
                                                         double* __restrict__ cov) {
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < count;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x)
    cov[i] = S[i] / n1;
}

int grid_for(int64_t n, int sms) {
  int64_t b = (n + 255) / 256;
  if (b > static_cast<int64_t>(sms) * 8) b = static_cast<int64_t>(sms) * 8;
  return static_cast<int>(b < 1 ? 1 : b);
}

}  // namespace

cudaError_t launch_stats_transpose(const void* x, int64_t B, int64_t K, int64_t Bg, int G, void* xt, float* colpart,
                                   cudaStream_t stream) {
  const int64_t tiles = static_cast<int64_t>(G) * Bg / kTRows;
  const dim3 grid(static_cast<unsigned>(tiles), static_cast<unsigned>(K / kTCols));
  stats_transpose_kernel<<<grid, 256, 0, stream>>>(static_cast<const uint16_t*>(x), B, K, Bg,
                                                    static_cast<uint16_t*>(xt), colpart);
  return cudaGetLastError();
}

cudaError_t launch_stats_merge(const float* colpart, int64_t tiles, const float* partials, int G, int64_t K,
                               double* colwork, double* mu, double* S, int64_t n_old, int64_t nb, int sms,
                               cudaStream_t stream) {
  double* part = colwork;                        // [kSumChunks][K]
  double* col = colwork + kSumChunks * K;        // s, m, d: [3][K]
  const double dn = static_cast<double>(n_old), db = static_cast<double>(nb);
  stats_colsum_kernel<<<dim3(static_cast<unsigned>(K / 32), kSumChunks), 256, 0, stream>>>(colpart, tiles, K, part);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  stats_colprep_kernel<<<static_cast<unsigned>((K + 255) / 256), 256, 0, stream>>>(part, K, mu, db, col);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  stats_merge_kernel<<<grid_for(K * K, sms), 256, 0, stream>>>(partials, G, K, col, S, dn * db / (dn + db));
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  stats_mean_kernel<<<static_cast<unsigned>((K + 255) / 256), 256, 0, stream>>>(col, mu, K, db / (dn + db));
  return cudaGetLastError();
}

cudaError_t launch_cholesky(const double* S, const double* mu, int64_t K, int64_t n, double eps_rel, float* A,
                            void* L, void* mu_out, int* status, cudaStream_t stream) {
  const size_t smem = static_cast<size_t>(K) * sizeof(float);
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(cholesky_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
  }
  cholesky_kernel<<<1, 1024, smem, stream>>>(S, mu, K, 1.0 / static_cast<double>(n - 1), eps_rel, A,
                                             static_cast<uint16_t*>(L), static_cast<uint16_t*>(mu_out), status);
  return cudaGetLastError();
}

cudaError_t launch_covariance(const double* S, int64_t K, int64_t n, double* cov, int sms, cudaStream_t stream) {
  covariance_kernel<<<grid_for(K * K, sms), 256, 0, stream>>>(S, K * K, static_cast<double>(n - 1), cov);
  return cudaGetLastError();
}

cudaError_t launch_normals(uint64_t seed, int64_t count, void* z, int sms, cudaStream_t stream) {
  const int64_t pairs = count / 2;
  normals_kernel<false><<<grid_for(pairs, sms), 256, 0, stream>>>(seed, pairs, z);
  return cudaGetLastError();
}

cudaError_t launch_normals_f32(uint64_t seed, int64_t count, float* z, int sms, cudaStream_t stream) {
  const int64_t pairs = count / 2;
  normals_kernel<true><<<grid_for(pairs, sms), 256, 0, stream>>>(seed, pairs, z);
  return cudaGetLastError();
}

}  // namespace loka
