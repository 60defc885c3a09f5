// Quantization-error probe reduction and the watchdog self-test kernel.
//
// The probe follows "LoKA: Low-precision Kernel Applications for
// Recommendation Models at Scale", section II-C "Error Analysis" (MERE, the
// mean element-wise relative error against a high-precision reference) and
// section III-A "Offline Error Quantification" (the per-layer error of
// FP8(Wx+b) against the high-precision Wx+b).  The reduction reads the two
// fp32 outputs once (HBM-bound) and accumulates, in fp64:
//   acc[0] = sum over ref != 0 of |out-ref|/|ref|
//   acc[1] = number of ref != 0
//   acc[2] = sum (out-ref)^2
//   acc[3] = sum ref^2
//   acc[4] = max |out-ref| (as the bits of a non-negative double)
#include "loka_internal.h"
#include "ptx.cuh"

namespace loka {

namespace {

__device__ __forceinline__ double warp_sum(double v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

__device__ __forceinline__ double warp_maxd(double v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmax(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

__global__ void __launch_bounds__(256) error_reduce_kernel(const float* __restrict__ out, const float* __restrict__ ref,
                                                           int64_t n, double* __restrict__ acc) {
  double rel = 0.0, nz = 0.0, d2 = 0.0, r2 = 0.0, mx = 0.0;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  const int64_t n4 = n >> 2;
  const float4* o4 = reinterpret_cast<const float4*>(out);
  const float4* r4 = reinterpret_cast<const float4*>(ref);
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n4; i += stride) {
    const float4 a = __ldcs(o4 + i);
    const float4 b = __ldcs(r4 + i);
    const float av[4] = {a.x, a.y, a.z, a.w};
    const float bv[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const double d = static_cast<double>(av[e]) - static_cast<double>(bv[e]);
      const double r = bv[e];
      if (r != 0.0) {
        rel += fabs(d) / fabs(r);
        nz += 1.0;
      }
      d2 += d * d;
      r2 += r * r;
      mx = fmax(mx, fabs(d));
    }
  }
  for (int64_t i = (n4 << 2) + static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n; i += stride) {
    const double d = static_cast<double>(out[i]) - static_cast<double>(ref[i]);
    const double r = ref[i];
    if (r != 0.0) {
      rel += fabs(d) / fabs(r);
      nz += 1.0;
    }
    d2 += d * d;
    r2 += r * r;
    mx = fmax(mx, fabs(d));
  }
  rel = warp_sum(rel);
  nz = warp_sum(nz);
  d2 = warp_sum(d2);
  r2 = warp_sum(r2);
  mx = warp_maxd(mx);
  __shared__ double red[5][8];
  const int w = threadIdx.x >> 5;
  if ((threadIdx.x & 31) == 0) {
    red[0][w] = rel;
    red[1][w] = nz;
    red[2][w] = d2;
    red[3][w] = r2;
    red[4][w] = mx;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    double s[5] = {0, 0, 0, 0, 0};
    for (int i = 0; i < static_cast<int>(blockDim.x >> 5); ++i) {
      for (int k = 0; k < 4; ++k) s[k] += red[k][i];
      s[4] = fmax(s[4], red[4][i]);
    }
    for (int k = 0; k < 4; ++k) atomicAdd(acc + k, s[k]);
    atomicMax(reinterpret_cast<unsigned long long*>(acc + 4), static_cast<unsigned long long>(__double_as_longlong(s[4])));
  }
}

// Waits on an mbarrier that nothing ever arrives at; the bounded wait gives
// up after limit_ns, records kErrSelftest and returns.  Used to show that a
// stuck wait becomes an error status rather than a hung GPU.
__global__ void watchdog_selftest_kernel(unsigned* status, uint64_t limit_ns) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    abort_flag = 0;
    mbar_init(smem_u32(&bar), 1);
    fence_barrier_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    const Watchdog wd{&abort_flag, status, limit_ns};
    wait_parity(wd, smem_u32(&bar), 0, kErrSelftest);
  }
  __syncthreads();
}

}  // namespace

cudaError_t launch_error_reduce(const float* out, const float* ref, int64_t n, double* acc, int sms, cudaStream_t stream) {
  cudaError_t e = cudaMemsetAsync(acc, 0, 5 * sizeof(double), stream);
  if (e != cudaSuccess || n == 0) return e;
  int64_t blocks = (n / 4 + 255) / 256;
  const int64_t cap = static_cast<int64_t>(sms) * 4;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  error_reduce_kernel<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(out, ref, n, acc);
  return cudaGetLastError();
}

cudaError_t launch_watchdog_selftest(unsigned* status, uint64_t limit_ns, cudaStream_t stream) {
  watchdog_selftest_kernel<<<1, 32, 0, stream>>>(status, limit_ns);
  return cudaGetLastError();
}

}  // namespace loka
