// LoKA Probe: online learning of a layer's weight distribution, and sampling.
//
// Defined by "LoKA: Low-precision Kernel Applications for Recommendation
// Models at Scale", section III-A 1 "Online Distribution Learning",
// paragraph "Optimized Weight Distribution Modeling", and "Sampling learned
// distributions" (b).  A weight W [R, C] is modeled as matrix-normal,
// W ~ MN(M, U, V) (vec(W) ~ N(vec(M), V (x) U)), with the row covariance U
// [R, R] and the column covariance V [C, C] tracked by a Kronecker-factor
// (flip-flop) update smoothed by an exponential moving average, using linear
// solves against regularized Cholesky factors instead of inverses:
//
//   Wc = W - M
//   L_V L_V^T = V + eps_V I,   W_V = Wc L_V^{-T},   U' = W_V W_V^T / C
//   L_U L_U^T = U + eps_U I,   W_U = L_U^{-1} Wc,   V' = W_U^T W_U / R
//   U'' = m U + (1 - m) U',   V'' = m V + (1 - m) V'
//   U = (U'' + U''^T)/2 + eps_U I,   V = (V'' + V''^T)/2 + eps_V I
//   s = trace(U) / R,   U <- U / s,   V <- s V,   M <- m M + (1 - m) W
//
// with eps_A = eps_rel * trace(A) / dim(A) on the matrix it regularizes.
// Sampling: W' = M + L_U Z L_V^T, Z the seed's counter-based normals.
//
// This runs once per probe interval, off the data-parallel path, on small
// matrices (R, C <= 2048): plain fp32 SIMT kernels.  The factorizations run
// on one thread block per matrix (both in one launch), the triangular solves
// one warp per right-hand side, the products through a shared-memory tiled
// fp32 GEMM.
#include "loka_internal.h"
#include "ptx.cuh"

namespace loka {

namespace {

int grid_of(int64_t n, int sms) {
  int64_t b = (n + 255) / 256;
  if (b > static_cast<int64_t>(sms) * 8) b = static_cast<int64_t>(sms) * 8;
  return static_cast<int>(b < 1 ? 1 : b);
}

__device__ __forceinline__ float bf16f(uint16_t h) { return __uint_as_float(static_cast<uint32_t>(h) << 16); }

__global__ void __launch_bounds__(256) weight_init_kernel(const uint16_t* __restrict__ w, int64_t R, int64_t C,
                                                          float* __restrict__ M, float* __restrict__ U,
                                                          float* __restrict__ V) {
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  const int64_t t0 = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  for (int64_t i = t0; i < R * C; i += stride) M[i] = bf16f(w[i]);
  for (int64_t i = t0; i < R * R; i += stride) U[i] = (i / R == i % R) ? 1.0f : 0.0f;
  for (int64_t i = t0; i < C * C; i += stride) V[i] = (i / C == i % C) ? 1.0f : 0.0f;
}

__global__ void __launch_bounds__(256) weight_center_kernel(const uint16_t* __restrict__ w, const float* __restrict__ M,
                                                            int64_t n, float* __restrict__ wc) {
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x)
    wc[i] = bf16f(w[i]) - M[i];
}

// L L^T = A + eps I (eps = eps_rel * trace(A) / n), block b factors matrix b
// (A0, n0 -> L0 or A1, n1 -> L1), left-looking, in place in L:
//   L_jj = sqrt(A_jj - sum_{k<j} L_jk^2),  L_ij = (A_ij - sum_{k<j} L_ik L_jk) / L_jj.
// Row j's finished entries are staged in shared memory; zeros above the
// diagonal; status[b] = 1 when a pivot is not positive.
__global__ void __launch_bounds__(1024) chol_reg_kernel(const float* __restrict__ A0, int n0, float* __restrict__ L0,
                                                        const float* __restrict__ A1, int n1, float* __restrict__ L1,
                                                        double eps_rel, int* __restrict__ status) {
  extern __shared__ float rowj[];
  __shared__ double red[32];
  __shared__ float pivot;
  __shared__ int bad;
  const float* A = blockIdx.x == 0 ? A0 : A1;
  float* L = blockIdx.x == 0 ? L0 : L1;
  const int n = blockIdx.x == 0 ? n0 : n1;
  const int t = threadIdx.x, nt = blockDim.x, lane = t & 31, warp = t >> 5;
  double tr = 0.0;
  for (int i = t; i < n; i += nt) tr += A[static_cast<int64_t>(i) * n + i];
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
  const float eps = static_cast<float>(eps_rel * red[0] / n);
  for (int64_t e = t; e < static_cast<int64_t>(n) * n; e += nt) {
    const int64_t i = e / n, j = e - i * n;
    L[e] = A[e] + (i == j ? eps : 0.0f);
  }
  __syncthreads();
  for (int j = 0; j < n; ++j) {
    for (int k = t; k < j; k += nt) rowj[k] = L[static_cast<int64_t>(j) * n + k];
    __syncthreads();
    float s = 0.0f;
    for (int k = t; k < j; k += nt) s = fmaf(rowj[k], rowj[k], s);
    for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
    if (lane == 0) red[warp] = s;
    __syncthreads();
    if (t == 0) {
      float a = 0.0f;
      for (int w = 0; w < nt / 32; ++w) a += static_cast<float>(red[w]);
      const float d = L[static_cast<int64_t>(j) * n + j] - a;
      if (!(d > 0.0f)) bad = 1;
      pivot = d > 0.0f ? sqrtf(d) : 1.0f;
      L[static_cast<int64_t>(j) * n + j] = pivot;
    }
    __syncthreads();
    if (bad) break;
    const float inv = 1.0f / pivot;
    for (int i = j + 1 + t; i < n; i += nt) {
      float* ri = L + static_cast<int64_t>(i) * n;
      float dot = 0.0f;
      for (int k = 0; k < j; ++k) dot = fmaf(ri[k], rowj[k], dot);
      ri[j] = (ri[j] - dot) * inv;
    }
    __syncthreads();
  }
  if (t == 0) status[blockIdx.x] = bad;
  for (int64_t e = t; e < static_cast<int64_t>(n) * n; e += nt) {
    const int64_t i = e / n, j = e - i * n;
    if (j > i) L[e] = 0.0f;
  }
}

// Forward substitution, one warp per right-hand side r < rhs: x with
// L x = b, b_j = B[r*bs + j*bj], written to X[r*xs + j*xj] (n unknowns,
// L lower triangular n x n, row-major).  x stays in shared memory (n floats
// per warp) until it is written out.
__global__ void __launch_bounds__(128) trsv_lower_kernel(const float* __restrict__ L, int n, const float* __restrict__ B,
                                                         int64_t bs, int64_t bj, int64_t rhs, float* __restrict__ X,
                                                         int64_t xs, int64_t xj) {
  extern __shared__ float xbuf[];
  const int lane = threadIdx.x & 31, wib = threadIdx.x >> 5;
  float* x = xbuf + static_cast<int64_t>(wib) * n;
  const int64_t r = static_cast<int64_t>(blockIdx.x) * (blockDim.x >> 5) + wib;
  if (r >= rhs) return;
  for (int j = 0; j < n; ++j) {
    const float* lj = L + static_cast<int64_t>(j) * n;
    float s = 0.0f;
    for (int k = lane; k < j; k += 32) s = fmaf(lj[k], x[k], s);
    for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
    if (lane == 0) x[j] = (B[r * bs + j * bj] - s) / lj[j];
    __syncwarp();
  }
  for (int j = lane; j < n; j += 32) X[r * xs + j * xj] = x[j];
}

// C[i, j] = alpha * sum_k A(i, k) B(k, j) (+ D[i, j] when D is set), with
// A(i, k) = A[i*ai + k*ak], B(k, j) = B[k*bk + j*bj]; C row-major (ldc),
// fp32 or bf16 (out_bf16).  16 x 16 output tiles, K in steps of 16 through
// shared memory; fp32 accumulation in k order.
__global__ void __launch_bounds__(256) gemm_f32_kernel(int64_t Mr, int64_t Nc, int64_t K, const float* __restrict__ A,
                                                       int64_t ai, int64_t ak, const float* __restrict__ B, int64_t bk,
                                                       int64_t bj, float alpha, const float* __restrict__ D,
                                                       void* __restrict__ Cout, int64_t ldc, int out_bf16) {
  __shared__ float as[16][17];
  __shared__ float bs[16][17];
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
  const int64_t i = static_cast<int64_t>(blockIdx.y) * 16 + ty;
  const int64_t j = static_cast<int64_t>(blockIdx.x) * 16 + tx;
  float acc = 0.0f;
  for (int64_t k0 = 0; k0 < K; k0 += 16) {
    const int64_t ia = static_cast<int64_t>(blockIdx.y) * 16 + ty, ka = k0 + tx;
    as[ty][tx] = (ia < Mr && ka < K) ? A[ia * ai + ka * ak] : 0.0f;
    const int64_t kb = k0 + ty, jb = static_cast<int64_t>(blockIdx.x) * 16 + tx;
    bs[ty][tx] = (kb < K && jb < Nc) ? B[kb * bk + jb * bj] : 0.0f;
    __syncthreads();
#pragma unroll
    for (int k = 0; k < 16; ++k) acc = fmaf(as[ty][k], bs[k][tx], acc);
    __syncthreads();
  }
  if (i < Mr && j < Nc) {
    float v = alpha * acc;
    if (D != nullptr) v += D[i * ldc + j];
    if (out_bf16)
      static_cast<uint16_t*>(Cout)[i * ldc + j] = static_cast<uint16_t>(pack_bf16x2(v, 0.0f) & 0xFFFFu);
    else
      static_cast<float*>(Cout)[i * ldc + j] = v;
  }
}

// The moving average of both factors, symmetrized: S = ((m X + (1-m) X') +
// (m X + (1-m) X')^T) / 2 for X = U (n = R) and X = V (n = C), into the
// estimate buffers (each element reads its transpose partner only).
__global__ void __launch_bounds__(256) weight_ema_kernel(const float* __restrict__ U, float* __restrict__ U1, int64_t R,
                                                         const float* __restrict__ V, float* __restrict__ V1, int64_t C,
                                                         float m, float* __restrict__ Us, float* __restrict__ Vs) {
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  const int64_t t0 = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  const float m1 = 1.0f - m;
  for (int64_t e = t0; e < R * R; e += stride) {
    const int64_t i = e / R, j = e - i * R;
    const float a = fmaf(m, U[e], m1 * U1[e]), b = fmaf(m, U[j * R + i], m1 * U1[j * R + i]);
    Us[e] = 0.5f * (a + b);
  }
  for (int64_t e = t0; e < C * C; e += stride) {
    const int64_t i = e / C, j = e - i * C;
    const float a = fmaf(m, V[e], m1 * V1[e]), b = fmaf(m, V[j * C + i], m1 * V1[j * C + i]);
    Vs[e] = 0.5f * (a + b);
  }
}

// trace[0] = trace(Us), trace[1] = trace(Vs), fp64 in a fixed order.
__global__ void __launch_bounds__(256) weight_trace_kernel(const float* __restrict__ Us, int64_t R,
                                                           const float* __restrict__ Vs, int64_t C,
                                                           double* __restrict__ trace) {
  __shared__ double red[2][8];
  const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
  double a = 0.0, b = 0.0;
  for (int64_t i = t; i < R; i += blockDim.x) a += Us[i * R + i];
  for (int64_t i = t; i < C; i += blockDim.x) b += Vs[i * C + i];
  for (int o = 16; o > 0; o >>= 1) {
    a += __shfl_xor_sync(0xffffffffu, a, o);
    b += __shfl_xor_sync(0xffffffffu, b, o);
  }
  if (lane == 0) {
    red[0][warp] = a;
    red[1][warp] = b;
  }
  __syncthreads();
  if (t == 0) {
    double sa = 0.0, sb = 0.0;
    for (int w = 0; w < 8; ++w) {
      sa += red[0][w];
      sb += red[1][w];
    }
    trace[0] = sa;
    trace[1] = sb;
  }
}

// U = (Us + eps_U I) / s, V = (Vs + eps_V I) * s with s = trace(U) / R =
// trace(Us) (1 + eps_rel) / R; M <- m M + (1 - m) W.
__global__ void __launch_bounds__(256) weight_final_kernel(const float* __restrict__ Us, const float* __restrict__ Vs,
                                                           const double* __restrict__ trace, int64_t R, int64_t C,
                                                           double eps_rel, float m, const uint16_t* __restrict__ w,
                                                           float* __restrict__ M, float* __restrict__ U,
                                                           float* __restrict__ V) {
  const double eu = eps_rel * trace[0] / static_cast<double>(R);
  const double ev = eps_rel * trace[1] / static_cast<double>(C);
  const double s = (trace[0] + static_cast<double>(R) * eu) / static_cast<double>(R);
  const float inv_s = static_cast<float>(1.0 / s), sf = static_cast<float>(s);
  const float euf = static_cast<float>(eu), evf = static_cast<float>(ev);
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  const int64_t t0 = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  for (int64_t e = t0; e < R * R; e += stride) U[e] = (Us[e] + (e / R == e % R ? euf : 0.0f)) * inv_s;
  for (int64_t e = t0; e < C * C; e += stride) V[e] = (Vs[e] + (e / C == e % C ? evf : 0.0f)) * sf;
  for (int64_t e = t0; e < R * C; e += stride) M[e] = fmaf(m, M[e], (1.0f - m) * bf16f(w[e]));
}

cudaError_t launch_chol2(const float* A0, int n0, float* L0, const float* A1, int n1, float* L1, double eps_rel,
                         int* status, cudaStream_t stream) {
  const int nmax = n0 > n1 ? n0 : n1;
  const size_t smem = static_cast<size_t>(nmax) * sizeof(float);
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(chol_reg_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
  }
  chol_reg_kernel<<<2, 1024, smem, stream>>>(A0, n0, L0, A1, n1, L1, eps_rel, status);
  return cudaGetLastError();
}

cudaError_t launch_trsv(const float* L, int n, const float* B, int64_t bs, int64_t bj, int64_t rhs, float* X, int64_t xs,
                        int64_t xj, cudaStream_t stream) {
  const size_t smem = static_cast<size_t>(4) * n * sizeof(float);   // 4 warps per block
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(trsv_lower_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
  }
  trsv_lower_kernel<<<static_cast<unsigned>((rhs + 3) / 4), 128, smem, stream>>>(L, n, B, bs, bj, rhs, X, xs, xj);
  return cudaGetLastError();
}

cudaError_t launch_gemm_f32(int64_t Mr, int64_t Nc, int64_t K, const float* A, int64_t ai, int64_t ak, const float* B,
                            int64_t bk, int64_t bj, float alpha, const float* D, void* C, int64_t ldc, bool out_bf16,
                            cudaStream_t stream) {
  const dim3 grid(static_cast<unsigned>((Nc + 15) / 16), static_cast<unsigned>((Mr + 15) / 16));
  gemm_f32_kernel<<<grid, 256, 0, stream>>>(Mr, Nc, K, A, ai, ak, B, bk, bj, alpha, D, C, ldc, out_bf16 ? 1 : 0);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_weight_init(const void* w, int64_t R, int64_t C, float* M, float* U, float* V, int sms,
                               cudaStream_t stream) {
  int64_t n = R * C;
  if (R * R > n) n = R * R;
  if (C * C > n) n = C * C;
  weight_init_kernel<<<grid_of(n, sms), 256, 0, stream>>>(static_cast<const uint16_t*>(w), R, C, M, U, V);
  return cudaGetLastError();
}

cudaError_t launch_weight_update(const void* w, int64_t R, int64_t C, double m, double eps_rel, float* M, float* U,
                                 float* V, const WeightWork& ws, int sms, cudaStream_t stream) {
  const uint16_t* wb = static_cast<const uint16_t*>(w);
  weight_center_kernel<<<grid_of(R * C, sms), 256, 0, stream>>>(wb, M, R * C, ws.wc);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  // L_U L_U^T = U + eps_U I and L_V L_V^T = V + eps_V I (one launch)
  if ((e = launch_chol2(U, static_cast<int>(R), ws.lu, V, static_cast<int>(C), ws.lv, eps_rel, ws.status, stream)) !=
      cudaSuccess)
    return e;
  // W_V = Wc L_V^{-T}: row r of W_V solves L_V y = Wc[r, :]^T
  if ((e = launch_trsv(ws.lv, static_cast<int>(C), ws.wc, C, 1, R, ws.wv, C, 1, stream)) != cudaSuccess) return e;
  // W_U = L_U^{-1} Wc: column c of W_U solves L_U z = Wc[:, c]
  if ((e = launch_trsv(ws.lu, static_cast<int>(R), ws.wc, 1, C, C, ws.wu, 1, C, stream)) != cudaSuccess) return e;
  // U' = W_V W_V^T / C [R, R];  V' = W_U^T W_U / R [C, C]
  if ((e = launch_gemm_f32(R, R, C, ws.wv, C, 1, ws.wv, 1, C, 1.0f / static_cast<float>(C), nullptr, ws.u1, R, false,
                           stream)) != cudaSuccess)
    return e;
  if ((e = launch_gemm_f32(C, C, R, ws.wu, 1, C, ws.wu, C, 1, 1.0f / static_cast<float>(R), nullptr, ws.v1, C, false,
                           stream)) != cudaSuccess)
    return e;
  // the moving averages, symmetrized (into the factor buffers, free now)
  int64_t n = R * R > C * C ? R * R : C * C;
  weight_ema_kernel<<<grid_of(n, sms), 256, 0, stream>>>(U, ws.u1, R, V, ws.v1, C, static_cast<float>(m), ws.lu, ws.lv);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  weight_trace_kernel<<<1, 256, 0, stream>>>(ws.lu, R, ws.lv, C, ws.trace);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  if (R * C > n) n = R * C;
  weight_final_kernel<<<grid_of(n, sms), 256, 0, stream>>>(ws.lu, ws.lv, ws.trace, R, C, eps_rel, static_cast<float>(m),
                                                           wb, M, U, V);
  return cudaGetLastError();
}

cudaError_t launch_weight_sample(const float* M, const float* U, const float* V, int64_t R, int64_t C, double eps_rel,
                                 uint64_t seed, void* out, const WeightWork& ws, int sms, cudaStream_t stream) {
  cudaError_t e = launch_chol2(U, static_cast<int>(R), ws.lu, V, static_cast<int>(C), ws.lv, eps_rel, ws.status, stream);
  if (e != cudaSuccess) return e;
  // Z [R, C]: normal r C + c of the seed
  if ((e = launch_normals_f32(seed, R * C, ws.wc, sms, stream)) != cudaSuccess) return e;
  // T = Z L_V^T [R, C], then W' = M + L_U T (bf16)
  if ((e = launch_gemm_f32(R, C, C, ws.wc, C, 1, ws.lv, 1, C, 1.0f, nullptr, ws.wv, C, false, stream)) != cudaSuccess)
    return e;
  return launch_gemm_f32(R, C, R, ws.lu, R, 1, ws.wv, C, 1, 1.0f, M, out, C, true, stream);
}

}  // namespace loka
