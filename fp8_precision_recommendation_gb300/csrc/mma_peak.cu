// Dense tensor-core throughput of this GPU, measured with the same tcgen05
// instructions the GEMM issues: the FP8 peak (kind::f8f6f4, E4M3 x E4M3 ->
// fp32) against which the contraction's tensor-pipe share is measured, and
// the bf16 peak (kind::f16) for a check against the library GEMM's number.
//
// One CTA per SM (its shared memory keeps a second one off the SM).  Thread
// 0 issues `mmas` MMAs of M = 128, N = 256 and one 32-byte K step (K = 32
// E4M3 or 16 bf16 values) from two zero-filled shared-memory tiles into one
// tensor-memory accumulator, cycling over the four K steps of a 128-byte
// row; the tensor pipe queues them back to back.  Nothing is loaded from
// memory, so the launch time is the pipe's alone.  The final commit is
// awaited with a time limit.
#include "loka_internal.h"
#include "ptx.cuh"

namespace loka {
namespace {

constexpr int kPeakM = 128;
constexpr int kPeakN = 256;
constexpr uint32_t kPeakSmem = 128 * 1024;   // > half of the SM's shared memory: one CTA per SM

__global__ void __launch_bounds__(128, 1) mma_peak_kernel(int kind, int64_t mmas, unsigned* status, uint64_t limit_ns) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  __shared__ uint64_t done_bar;
  __shared__ uint32_t tmem_base;
  __shared__ int abort_flag;
  // 1024-byte aligned operand tiles: A 128 rows x 128 bytes, B 256 x 128
  const uint32_t base = (smem_u32(smem_raw) + 1023u) & ~1023u;
  const uint32_t a_addr = base, b_addr = base + kPeakM * 128;
  uint8_t* gen = smem_raw + (base - smem_u32(smem_raw));
  for (int i = threadIdx.x; i < (kPeakM + kPeakN) * 128 / 16; i += blockDim.x)
    reinterpret_cast<uint4*>(gen)[i] = make_uint4(0u, 0u, 0u, 0u);
  const int warp = threadIdx.x >> 5;
  if (threadIdx.x == 0) {
    abort_flag = 0;
    mbar_init(smem_u32(&done_bar), 1);
    fence_barrier_init();
  }
  if (warp == 0) {
    tmem_alloc(smem_u32(&tmem_base), kPeakN);
    tmem_relinquish();
  }
  fence_proxy_async_smem();   // the zeros are read by the tensor core
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (threadIdx.x == 0) {
    const uint32_t d = tmem_base;
    const uint32_t idesc = kind == 0 ? idesc_dense(0, 0, kPeakM, kPeakN) : idesc_dense(1, 1, kPeakM, kPeakN);
    for (int64_t i = 0; i < mmas; ++i) {
      const uint32_t k = static_cast<uint32_t>(i & 3) * 32u;
      const uint64_t adesc = sdesc_k128_sw128(a_addr + k), bdesc = sdesc_k128_sw128(b_addr + k);
      if (kind == 0)
        mma_f8f6f4(d, adesc, bdesc, idesc, i != 0);
      else
        mma_f16(d, adesc, bdesc, idesc, i != 0);
    }
    mma_commit(smem_u32(&done_bar));
    const Watchdog wd{&abort_flag, status, limit_ns};
    if (!wait_parity(wd, smem_u32(&done_bar), 0, kErrSelftest)) wait_parity_drain(wd, smem_u32(&done_bar), 0);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0) tmem_dealloc(tmem_base, kPeakN);
}

}  // namespace

cudaError_t launch_mma_peak(int kind, int64_t mmas, int sms, unsigned* status, uint64_t limit_ns, cudaStream_t stream) {
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(mma_peak_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kPeakSmem);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  mma_peak_kernel<<<sms, 128, kPeakSmem, stream>>>(kind, mmas, status, limit_ns);
  return cudaGetLastError();
}

}  // namespace loka
