// amax -> scale -> E4M3 cast kernels (tensorwise, rowwise, MX 1x32).
//
// Defined by "LoKA: Low-precision Kernel Applications for Recommendation
// Models at Scale", section II-C (FP8 recipes with tensorwise / rowwise /
// blockwise scaling, whose quantization cost is over 30% of GEMM latency) and
// by the MXFP8 block scaling on the GEM Training page ("Low Precision Flash
// Attention": scale factors along each GEMM's K dimension).
//
// These are HBM-bound streaming kernels: every thread moves 16-byte vectors
// (8 bf16 in, 8 E4M3 codes out), a warp covers 512 contiguous input bytes per
// load, and the row amax is a warp-shuffle reduction, so the data are read
// from HBM exactly once.  Several tensors (the X and W of every group of a
// grouped layer) are handled by one launch through a job table.
#include <atomic>

#include "loka_internal.h"
#include "ptx.cuh"
#include "quant_math.cuh"

namespace loka {

namespace {

__device__ __forceinline__ int find_job(const QuantJobs& jobs, int64_t gr) {
  int j = 0;
  while (j + 1 < jobs.n && jobs.j[j + 1].row_begin <= gr) ++j;
  return j;
}

// One warp per row.  V = 16-byte vectors per lane kept in registers
// (cols <= 256 * V).  MODE 1 = rowwise, MODE 2 = MX 1x32.
template <int MODE, int V>
__global__ void __launch_bounds__(256) quant_rows_kernel(const __grid_constant__ QuantJobs jobs) {
  launch_dependents();   // the GEMM that follows may start its prologue
  const int lane = threadIdx.x & 31;
  const int64_t warp0 = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int64_t nwarps = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
  for (int64_t gr = warp0; gr < jobs.total_rows; gr += nwarps) {
    const QuantJob& job = jobs.j[find_job(jobs, gr)];
    const int64_t row = gr - job.row_begin;
    const int nvec = static_cast<int>(job.cols >> 3);
    const uint4* src = reinterpret_cast<const uint4*>(job.x) + row * (job.ld >> 3);
    uint2* dst = reinterpret_cast<uint2*>(job.q + row * job.cols);
    uint4 v[V];
#pragma unroll
    for (int i = 0; i < V; ++i) {
      const int idx = i * 32 + lane;
      v[i] = idx < nvec ? __ldcs(src + idx) : make_uint4(0, 0, 0, 0);
    }
    if (MODE == kScaleRow) {
      float m = 0.0f;
#pragma unroll
      for (int i = 0; i < V; ++i) m = abs_max8(v[i], m);
      m = warp_max(m);
      float inv, scale;
      row_scales(m, inv, scale);
#pragma unroll
      for (int i = 0; i < V; ++i) {
        const int idx = i * 32 + lane;
        if (idx < nvec) dst[idx] = cast8(v[i], inv);
      }
      if (lane == 0) reinterpret_cast<float*>(job.scales)[row] = scale;
    } else {
      uint8_t* sc = reinterpret_cast<uint8_t*>(job.scales) + row * (job.cols >> 5);
#pragma unroll
      for (int i = 0; i < V; ++i) {
        const int idx = i * 32 + lane;
        float m = abs_max8(v[i], 0.0f);
        m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 1));
        m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 2));
        const int e = mx_exponent(m);
        if (idx < nvec) {
          dst[idx] = cast8(v[i], pow2_neg(e));
          if ((lane & 3) == 0) {
            sc[idx >> 2] = static_cast<uint8_t>(e + 127);
            if (job.sf_tc != nullptr) job.sf_tc[sf_tc_offset(row, idx >> 2, (job.cols + 127) >> 7)] = static_cast<uint8_t>(e + 127);
          }
        }
      }
    }
  }
}

// Rows of at most 128 columns: LPR lanes per row (one 16-byte vector each,
// LPR * 8 columns), 32 / LPR rows per warp step, and U steps loaded before
// any is processed, so a warp keeps U * 512 bytes in flight where one row
// per half-warp would keep 128 to 256.  Reductions stay within a row's LPR
// lanes.  Same arithmetic as quant_rows_kernel.
template <int MODE, int LPR>
__global__ void __launch_bounds__(256) quant_rows_narrow_kernel(const __grid_constant__ QuantJobs jobs) {
  launch_dependents();   // the GEMM that follows may start its prologue
  constexpr int RPW = 32 / LPR;   // rows per warp step
  constexpr int U = 4;            // steps in flight
  const int lane = threadIdx.x & 31;
  const int hl = lane % LPR;      // lane within the row = its vector
  const int sub = lane / LPR;     // row within the step
  const int64_t warp0 = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int64_t nwarps = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
  // every lane of a warp runs the loop the same number of times (base is
  // per warp); rows past the last one are dummies that load nothing
  for (int64_t base = warp0 * RPW * U; base < jobs.total_rows; base += nwarps * RPW * U) {
    uint4 v[U];
    const QuantJob* jb[U];
    int64_t row[U];
    bool live[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int64_t gr = base + u * RPW + sub;
      live[u] = gr < jobs.total_rows;
      jb[u] = &jobs.j[find_job(jobs, live[u] ? gr : 0)];
      row[u] = (live[u] ? gr : 0) - jb[u]->row_begin;
      const int nvec = static_cast<int>(jb[u]->cols >> 3);
      const uint4* src = reinterpret_cast<const uint4*>(jb[u]->x) + row[u] * (jb[u]->ld >> 3);
      v[u] = (live[u] && hl < nvec) ? __ldcs(src + hl) : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const QuantJob& job = *jb[u];
      const int nvec = static_cast<int>(job.cols >> 3);
      const bool act = live[u] && hl < nvec;
      uint2* dst = reinterpret_cast<uint2*>(job.q + row[u] * job.cols);
      if (MODE == kScaleRow) {
        float m = abs_max8(v[u], 0.0f);
#pragma unroll
        for (int o = 1; o < LPR; o <<= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
        float inv, scale;
        row_scales(m, inv, scale);
        if (act) dst[hl] = cast8(v[u], inv);
        if (live[u] && hl == 0) reinterpret_cast<float*>(job.scales)[row[u]] = scale;
      } else {
        float m = abs_max8(v[u], 0.0f);
        m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 1));
        m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 2));
        const int e = mx_exponent(m);
        if (act) {
          dst[hl] = cast8(v[u], pow2_neg(e));
          if ((hl & 3) == 0) {
            uint8_t* sc = reinterpret_cast<uint8_t*>(job.scales) + row[u] * (job.cols >> 5);
            sc[hl >> 2] = static_cast<uint8_t>(e + 127);
            if (job.sf_tc != nullptr)
              job.sf_tc[sf_tc_offset(row[u], hl >> 2, (job.cols + 127) >> 7)] = static_cast<uint8_t>(e + 127);
          }
        }
      }
    }
  }
}

// Rows of at most 256 columns: one half-warp per row, two rows per warp.
// Lane l of a half holds vectors l and l + 16 of its row (512 contiguous
// bytes per row per load pair), so a warp keeps two rows' bytes in flight
// where a whole warp per row would keep one; reductions stay within the
// half (shuffle offsets 1..8).  Same arithmetic as quant_rows_kernel.
template <int MODE>
__global__ void __launch_bounds__(256) quant_rows_half_kernel(const __grid_constant__ QuantJobs jobs) {
  launch_dependents();   // the GEMM that follows may start its prologue
  const int lane = threadIdx.x & 31;
  const int hl = lane & 15;                          // lane within the half
  const int64_t half0 = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 4;
  const int64_t nhalves = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 4;
  // both halves of a warp run the loop the same number of times (nhalves is
  // even and the halves' rows differ by 1), so the full-mask shuffles below
  // stay convergent; a half past the last row works on a dummy row
  for (int64_t base = half0 & ~int64_t(1); base < jobs.total_rows; base += nhalves) {
    const int64_t gr = base + (half0 & 1);
    const bool live = gr < jobs.total_rows;
    const QuantJob& job = jobs.j[find_job(jobs, live ? gr : base)];
    const int64_t row = (live ? gr : base) - job.row_begin;
    const int nvec = static_cast<int>(job.cols >> 3);
    const uint4* src = reinterpret_cast<const uint4*>(job.x) + row * (job.ld >> 3);
    uint2* dst = reinterpret_cast<uint2*>(job.q + row * job.cols);
    uint4 v[2];
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const int idx = i * 16 + hl;
      v[i] = (live && idx < nvec) ? __ldcs(src + idx) : make_uint4(0, 0, 0, 0);
    }
    if (MODE == kScaleRow) {
      float m = abs_max8(v[1], abs_max8(v[0], 0.0f));
#pragma unroll
      for (int o = 1; o < 16; o <<= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
      float inv, scale;
      row_scales(m, inv, scale);
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        const int idx = i * 16 + hl;
        if (live && idx < nvec) dst[idx] = cast8(v[i], inv);
      }
      if (live && hl == 0) reinterpret_cast<float*>(job.scales)[row] = scale;
    } else {
      uint8_t* sc = reinterpret_cast<uint8_t*>(job.scales) + row * (job.cols >> 5);
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        const int idx = i * 16 + hl;
        float m = abs_max8(v[i], 0.0f);
        m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 1));
        m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 2));
        const int e = mx_exponent(m);
        if (live && idx < nvec) {
          dst[idx] = cast8(v[i], pow2_neg(e));
          if ((hl & 3) == 0) {
            sc[idx >> 2] = static_cast<uint8_t>(e + 127);
            if (job.sf_tc != nullptr) job.sf_tc[sf_tc_offset(row, idx >> 2, (job.cols + 127) >> 7)] = static_cast<uint8_t>(e + 127);
          }
        }
      }
    }
  }
}

// Rows longer than 2048 elements: amax pass, then a cast pass that re-reads
// the row (it is still in L1/L2).  Same arithmetic as above.
template <int MODE>
__global__ void __launch_bounds__(256) quant_rows_long_kernel(const __grid_constant__ QuantJobs jobs) {
  launch_dependents();   // the GEMM that follows may start its prologue
  const int lane = threadIdx.x & 31;
  const int64_t warp0 = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int64_t nwarps = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
  for (int64_t gr = warp0; gr < jobs.total_rows; gr += nwarps) {
    const QuantJob& job = jobs.j[find_job(jobs, gr)];
    const int64_t row = gr - job.row_begin;
    const int nvec = static_cast<int>(job.cols >> 3);
    const uint4* src = reinterpret_cast<const uint4*>(job.x) + row * (job.ld >> 3);
    uint2* dst = reinterpret_cast<uint2*>(job.q + row * job.cols);
    if (MODE == kScaleRow) {
      float m = 0.0f;
      for (int idx = lane; idx < nvec; idx += 32) m = abs_max8(__ldg(src + idx), m);
      m = warp_max(m);
      float inv, scale;
      row_scales(m, inv, scale);
      for (int idx = lane; idx < nvec; idx += 32) dst[idx] = cast8(__ldg(src + idx), inv);
      if (lane == 0) reinterpret_cast<float*>(job.scales)[row] = scale;
    } else {
      uint8_t* sc = reinterpret_cast<uint8_t*>(job.scales) + row * (job.cols >> 5);
      for (int base = 0; base < nvec; base += 32) {   // nvec % 4 == 0: whole blocks per step
        const int idx = base + lane;
        const uint4 v = idx < nvec ? __ldcs(src + idx) : make_uint4(0, 0, 0, 0);
        float m = abs_max8(v, 0.0f);
        m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 1));
        m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 2));
        const int e = mx_exponent(m);
        if (idx < nvec) {
          dst[idx] = cast8(v, pow2_neg(e));
          if ((lane & 3) == 0) {
            sc[idx >> 2] = static_cast<uint8_t>(e + 127);
            if (job.sf_tc != nullptr) job.sf_tc[sf_tc_offset(row, idx >> 2, (job.cols + 127) >> 7)] = static_cast<uint8_t>(e + 127);
          }
        }
      }
    }
  }
}

// Source vector of dense vector index i (8 elements) of a job whose rows may
// be strided (ld > cols).
__device__ __forceinline__ const uint4* strided_vec(const QuantJob& job, int64_t i) {
  const uint4* src = reinterpret_cast<const uint4*>(job.x);
  if (job.ld == job.cols) return src + i;
  const int64_t cv = job.cols >> 3;
  const int64_t r = i / cv;
  return src + r * (job.ld >> 3) + (i - r * cv);
}

// Tensorwise pass 1: amax of each job into its slot (fp32 bits; the slot must
// be zero beforehand).  blockIdx.y = job.
__global__ void __launch_bounds__(256) amax_tensor_kernel(const __grid_constant__ QuantJobs jobs) {
  const QuantJob& job = jobs.j[blockIdx.y];
  const int64_t nvec = (job.rows * job.cols) >> 3;
  float m = 0.0f;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < nvec;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x)
    m = abs_max8(__ldg(strided_vec(job, i)), m);
  m = warp_max(m);
  __shared__ float red[8];
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = m;
  __syncthreads();
  if (threadIdx.x < 32) {
    m = threadIdx.x < (blockDim.x >> 5) ? red[threadIdx.x] : 0.0f;
    m = warp_max(m);
    // non-negative floats order like their bit patterns
    if (threadIdx.x == 0 && !(m != m)) atomicMax(job.amax_slot, __float_as_uint(m));
  }
}

// Tensorwise pass 2: cast with the tensor's scale; block (0, job) writes it.
__global__ void __launch_bounds__(256) cast_tensor_kernel(const __grid_constant__ QuantJobs jobs) {
  launch_dependents();
  const QuantJob& job = jobs.j[blockIdx.y];
  const float amax = __uint_as_float(*reinterpret_cast<volatile unsigned*>(job.amax_slot));
  float inv, scale;
  row_scales(amax, inv, scale);
  if (blockIdx.x == 0 && threadIdx.x == 0) reinterpret_cast<float*>(job.scales)[0] = scale;
  const int64_t nvec = (job.rows * job.cols) >> 3;
  uint2* dst = reinterpret_cast<uint2*>(job.q);
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < nvec;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x)
    dst[i] = cast8(__ldcs(strided_vec(job, i)), inv);
}

__global__ void __launch_bounds__(256) sf_permute_kernel(const uint8_t* __restrict__ logical, uint8_t* __restrict__ tc,
                                                         int64_t rows, int64_t cols, int row_div) {
  const int64_t nb = cols >> 5;
  const int64_t total = rows * nb;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < total;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t m = i / nb, b = i - m * nb;
    tc[sf_tc_offset(m, b, (cols + 127) >> 7)] = logical[(m / row_div) * nb + b];
  }
}

// Square 32 x 32 blocks (GEM Training page, "Low Precision Flash Attention":
// one scale per [32, 32] block, so the quantization of X^T is the transpose
// of that of X and a tensor is quantized once for both GEMM directions).
// One 256-thread block per unit of 32 rows x 256 columns (8 blocks): warp w
// loads rows 4w..4w+3 of the strip, each lane 8 columns of each row (16-byte
// vectors, 512 contiguous bytes per row per warp).  A block's amax merges the
// 4 lanes of its 32 columns (shuffles), then the 8 warps (shared memory); the
// exponent rule is the MX one.  Codes go out row by row; the optional
// transposed copy is staged in shared memory and transposed 4 x 4 bytes at a
// time (byte permutes), each of 64 threads writing the 32 codes of 4
// transposed rows as whole 32-byte sectors.
__global__ void __launch_bounds__(256) quant_block32_kernel(const __grid_constant__ QuantJobs jobs) {
  launch_dependents();   // the GEMM that follows may start its prologue
  __shared__ float red[8][8];                        // [warp][block] partial amax
  __shared__ int ex[8];                              // the unit's block exponents
  __shared__ __align__(16) uint8_t tile[32][256 + 16];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int64_t u = blockIdx.x; u < jobs.total_rows; u += gridDim.x) {
    const QuantJob& job = jobs.j[find_job(jobs, u)];
    const int64_t lu = u - job.row_begin;
    const int64_t segs = (job.cols + 255) >> 8;
    const int64_t rb = lu / segs, seg = lu - rb * segs;
    const int64_t r0 = rb * 32, c0 = seg * 256;
    const int64_t nvec = job.ld >> 3;   // source row stride in vectors
    const uint4* src = reinterpret_cast<const uint4*>(job.x);
    const bool col_ok = c0 + 8 * lane < job.cols;
    uint4 v[4];
    float m = 0.0f;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int64_t row = r0 + 4 * warp + i;
      v[i] = (col_ok && row < job.rows) ? __ldcs(src + row * nvec + (c0 >> 3) + lane) : make_uint4(0, 0, 0, 0);
      m = abs_max8(v[i], m);
    }
    m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 1));
    m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 2));
    if ((lane & 3) == 0) red[warp][lane >> 2] = m;
    __syncthreads();
    if (warp == 0 && lane < 8) {
      float a = red[0][lane];
#pragma unroll
      for (int w = 1; w < 8; ++w) a = fmaxf(a, red[w][lane]);
      ex[lane] = mx_exponent(a);
    }
    __syncthreads();
    const float mul = pow2_neg(ex[lane >> 2]);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int64_t row = r0 + 4 * warp + i;
      const uint2 c = cast8(v[i], mul);
      if (col_ok && row < job.rows) reinterpret_cast<uint2*>(job.q + row * job.cols + c0)[lane] = c;
      if (job.q_t != nullptr) reinterpret_cast<uint2*>(&tile[4 * warp + i][0])[lane] = c;
    }
    const int64_t nb = job.cols >> 5;
    if (warp == 0 && lane < 8 && c0 + 32 * lane < job.cols)
      reinterpret_cast<uint8_t*>(job.scales)[rb * nb + (c0 >> 5) + lane] = static_cast<uint8_t>(ex[lane] + 127);
    if (job.sf_tc != nullptr) {
      const int64_t row = r0 + (threadIdx.x >> 3);
      const int b = threadIdx.x & 7;
      if (row < job.rows && c0 + 32 * b < job.cols)
        job.sf_tc[sf_tc_offset(row, (c0 >> 5) + b, (job.cols + 127) >> 7)] = static_cast<uint8_t>(ex[b] + 127);
    }
    if (job.q_t != nullptr) {
      __syncthreads();
      // threads 0..63: columns 4g..4g+3 of the unit, all 32 rows of the
      // strip, transposed 4 x 4 bytes at a time; each transposed row then
      // gets its 32 codes as two 16-byte stores (one whole sector)
      const int g = threadIdx.x;
      if (g < 64 && c0 + 4 * g < job.cols) {
        uint32_t col[4][8];
#pragma unroll
        for (int rb = 0; rb < 8; ++rb) {
          uint32_t q4[4];
#pragma unroll
          for (int r = 0; r < 4; ++r) q4[r] = *reinterpret_cast<const uint32_t*>(&tile[4 * rb + r][4 * g]);
          const uint32_t lo01 = __byte_perm(q4[0], q4[1], 0x5140), hi01 = __byte_perm(q4[0], q4[1], 0x7362);
          const uint32_t lo23 = __byte_perm(q4[2], q4[3], 0x5140), hi23 = __byte_perm(q4[2], q4[3], 0x7362);
          col[0][rb] = __byte_perm(lo01, lo23, 0x5410);
          col[1][rb] = __byte_perm(lo01, lo23, 0x7632);
          col[2][rb] = __byte_perm(hi01, hi23, 0x5410);
          col[3][rb] = __byte_perm(hi01, hi23, 0x7632);
        }
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          uint4* out = reinterpret_cast<uint4*>(job.q_t + (c0 + 4 * g + c) * job.rows + r0);
          out[0] = make_uint4(col[c][0], col[c][1], col[c][2], col[c][3]);
          out[1] = make_uint4(col[c][4], col[c][5], col[c][6], col[c][7]);
        }
      }
    }
    __syncthreads();   // the next unit reuses red, ex and tile
  }
}

// One wave of the grid-stride kernel: as many 256-thread blocks as are
// resident at once (the register count decides; asked once per kernel and
// device), never more than one warp per row.  V = 0: the long-row kernel;
// V = -1: half-warp rows (at most 256 columns); V = -4, -8, -16: -V lanes per
// row (at most 32, 64, 128 columns); V > 0: V vectors per lane.
template <int MODE, int V>
constexpr auto rows_kernel() {
  if constexpr (V == 0)
    return quant_rows_long_kernel<MODE>;
  else if constexpr (V == -1)
    return quant_rows_half_kernel<MODE>;
  else if constexpr (V < -1)
    return quant_rows_narrow_kernel<MODE, -V>;
  else
    return quant_rows_kernel<MODE, V>;
}

template <int MODE, int V>
cudaError_t launch_one_wave(const QuantJobs& jobs, int sms, cudaStream_t stream) {
  const int threads = 256;
  auto kern = rows_kernel<MODE, V>();
  static std::atomic<int> per_sm[64];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  int occ = per_sm[dev & 63].load();
  if (occ == 0) {
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kern, threads, 0);
    if (e != cudaSuccess) return e;
    if (occ < 1) occ = 1;
    per_sm[dev & 63].store(occ);
  }
  // rows one block takes per pass: 8 warps x rows per warp (x 4 steps for
  // the narrow kernel)
  constexpr int64_t kRowsPerBlock = V == -1 ? 16 : (V < -1 ? 8 * (32 / -V) * 4 : 8);
  int64_t blocks = (jobs.total_rows + kRowsPerBlock - 1) / kRowsPerBlock;
  const int64_t cap = static_cast<int64_t>(sms) * occ;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  kern<<<static_cast<unsigned>(blocks), threads, 0, stream>>>(jobs);
  return cudaGetLastError();
}

template <int MODE>
cudaError_t launch_rows(const QuantJobs& jobs, int max_cols, int sms, cudaStream_t stream) {
  if (max_cols <= 32) return launch_one_wave<MODE, -4>(jobs, sms, stream);     // 4 lanes per row
  if (max_cols <= 64) return launch_one_wave<MODE, -8>(jobs, sms, stream);     // 8 lanes per row
  if (max_cols <= 128) return launch_one_wave<MODE, -16>(jobs, sms, stream);   // 16 lanes per row
  if (max_cols <= 256) return launch_one_wave<MODE, -1>(jobs, sms, stream);    // half-warp rows
  if (max_cols <= 512) return launch_one_wave<MODE, 2>(jobs, sms, stream);
  if (max_cols <= 1024) return launch_one_wave<MODE, 4>(jobs, sms, stream);
  if (max_cols <= 2048) return launch_one_wave<MODE, 8>(jobs, sms, stream);
  return launch_one_wave<MODE, 0>(jobs, sms, stream);
}

}  // namespace

cudaError_t launch_sf_permute(const uint8_t* logical, uint8_t* tc, int64_t rows, int64_t cols, int row_div, int sms,
                              cudaStream_t stream) {
  const int64_t total = rows * (cols >> 5);
  if (total == 0) return cudaSuccess;
  int64_t blocks = (total + 255) / 256;
  if (blocks > static_cast<int64_t>(sms) * 4) blocks = static_cast<int64_t>(sms) * 4;
  sf_permute_kernel<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(logical, tc, rows, cols, row_div);
  return cudaGetLastError();
}

cudaError_t launch_quantize(const QuantJobs& jobs, int mode, int sms, cudaStream_t stream) {
  if (jobs.n == 0 || jobs.total_rows == 0) return cudaSuccess;
  int max_cols = 0;
  int64_t max_elems = 0;
  for (int i = 0; i < jobs.n; ++i) {
    if (jobs.j[i].cols > max_cols) max_cols = static_cast<int>(jobs.j[i].cols);
    if (jobs.j[i].rows * jobs.j[i].cols > max_elems) max_elems = jobs.j[i].rows * jobs.j[i].cols;
  }
  if (mode == kScaleRow) return launch_rows<kScaleRow>(jobs, max_cols, sms, stream);
  if (mode == kScaleMx32) return launch_rows<kScaleMx32>(jobs, max_cols, sms, stream);
  if (mode == kScaleBlock32) {
    // units of 32 rows x 256 columns, numbered across the jobs
    QuantJobs u = jobs;
    int64_t units = 0;
    for (int i = 0; i < u.n; ++i) {
      u.j[i].row_begin = units;
      units += ((u.j[i].rows + 31) / 32) * ((u.j[i].cols + 255) / 256);
    }
    u.total_rows = units;
    if (units == 0) return cudaSuccess;
    static std::atomic<int> per_sm[64];
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    int occ = per_sm[dev & 63].load();
    if (occ == 0) {
      e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, quant_block32_kernel, 256, 0);
      if (e != cudaSuccess) return e;
      if (occ < 1) occ = 1;
      per_sm[dev & 63].store(occ);
    }
    int64_t blocks = units;
    if (blocks > static_cast<int64_t>(sms) * occ) blocks = static_cast<int64_t>(sms) * occ;
    quant_block32_kernel<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(u);
    return cudaGetLastError();
  }
  if (mode == kScaleTensor) {
    for (int i = 0; i < jobs.n; ++i) {
      cudaError_t e = cudaMemsetAsync(jobs.j[i].amax_slot, 0, sizeof(unsigned), stream);
      if (e != cudaSuccess) return e;
    }
    int64_t per_job = (max_elems / 8 + 255) / 256;
    const int64_t cap = (static_cast<int64_t>(sms) * 8 + jobs.n - 1) / jobs.n;
    if (per_job > cap) per_job = cap;
    if (per_job < 1) per_job = 1;
    const dim3 grid(static_cast<unsigned>(per_job), static_cast<unsigned>(jobs.n));
    amax_tensor_kernel<<<grid, 256, 0, stream>>>(jobs);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    cast_tensor_kernel<<<grid, 256, 0, stream>>>(jobs);
    return cudaGetLastError();
  }
  return cudaErrorInvalidValue;
}

}  // namespace loka
