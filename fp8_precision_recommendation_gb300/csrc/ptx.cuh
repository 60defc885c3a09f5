// Inline-PTX wrappers for sm_103a: mbarriers, TMA (cp.async.bulk.tensor),
// tcgen05 (TMEM alloc, MMA, commit, ld), E4M3 conversion, and bounded waits.
//
// Every wait in this library goes through wait_parity(), which gives up after
// a time limit, records a code in the device status word and tells the
// caller to abandon its loop, so no kernel can spin forever.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace loka {

// Status bits a kernel may OR into the device status word.
enum : unsigned {
  kErrProducerWait = 1u,
  kErrMmaWait = 2u,
  kErrEpilogueWait = 4u,
  kErrDrainWait = 8u,
  kErrSelftest = 16u,
  kErrMisaligned = 32u,
  kErrClusterWait = 64u,
  // in-kernel quantization: which hand-off gave up
  kErrQuantWait = 128u,      // a quantizer warp (staging slot, A tile or row-scale buffer)
  kErrTeamWait = 256u,       // an epilogue team's shared-vector barrier
  kErrRowScaleWait = 512u,   // the epilogue waiting for a tile's row scales
  kErrTeardownWait = 1024u,  // the MMA warp waiting for the epilogue before freeing tensor memory
};

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// ----------------------------------------------------------------- mbarrier
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}

// Suspending wait: the thread sleeps in hardware until the phase completes
// or about kSuspendHintNs pass, so a waiting warp takes no issue slots from
// the warps that are working.
constexpr uint32_t kSuspendHintNs = 1000000;

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity), "r"(kSuspendHintNs)
      : "memory");
  return ok != 0;
}

// Shared abort word: once any thread of the CTA gives up, every later wait
// returns false at once instead of running its own full time limit.
struct Watchdog {
  volatile int* abort_flag;   // shared memory
  unsigned* status;           // device status word (global)
  uint64_t limit_ns;
};

__device__ __forceinline__ bool wait_parity(const Watchdog& wd, uint32_t bar, uint32_t parity, unsigned code) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if (*wd.abort_flag) return false;
    if (global_timer_ns() - t0 > wd.limit_ns) {
      *wd.abort_flag = 1;
      atomicOr(wd.status, code);
      return false;
    }
  }
}

// Bounded wait used only while draining after an abort: it ignores the abort
// flag (the point is to let copies already in flight land) but keeps a limit.
__device__ __forceinline__ bool wait_parity_drain(const Watchdog& wd, uint32_t bar, uint32_t parity) {
  const uint64_t t0 = global_timer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (global_timer_ns() - t0 > wd.limit_ns) {
      atomicOr(wd.status, kErrDrainWait);
      return false;
    }
  }
  return true;
}

__device__ __forceinline__ void named_bar_sync(uint32_t id, uint32_t threads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

// bar.sync that also ORs `pred` over the participating threads: every thread
// gets the same answer, so a decision taken on it is uniform.
__device__ __forceinline__ bool named_bar_or(uint32_t id, uint32_t threads, bool pred) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.u32 p, %1, 0;\n\tbar.red.or.pred p, %2, %3, p;\n\tselp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(r)
      : "r"(pred ? 1u : 0u), "r"(id), "r"(threads)
      : "memory");
  return r != 0;
}

// Programmatic dependent launch: a kernel launched after this one with
// programmatic stream serialization may start (its prologue) once every CTA
// of this grid has executed launch_dependents; it must call
// wait_prerequisite_grids before touching memory this grid writes, which
// returns once this grid has completed and its writes are visible.
__device__ __forceinline__ void launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void wait_prerequisite_grids() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// ------------------------------------------------------------------ clusters
__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

// Address of the same shared-memory location in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t mapa_shared(uint32_t addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
  return r;
}

// Asynchronous store of two floats into shared memory of a CTA of the
// cluster; the destination CTA's mbarrier `cluster_bar` counts the 8 bytes
// (complete_tx) once they have landed, so the receiver needs no release from
// the sender.
__device__ __forceinline__ void st_async_f32x2(uint32_t cluster_addr, float a, float b, uint32_t cluster_bar) {
  asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.v2.f32 [%0], {%1, %2}, [%3];" ::"r"(cluster_addr),
               "f"(a), "f"(b), "r"(cluster_bar)
               : "memory");
}

// Arrive (no memory ordering) on an mbarrier of (possibly) another CTA.
__device__ __forceinline__ void mbar_arrive_cluster_relaxed(uint32_t cluster_bar) {
  asm volatile("mbarrier.arrive.relaxed.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_bar) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait_acq_cluster(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity), "r"(kSuspendHintNs)
      : "memory");
  return ok != 0;
}

// Bounded wait for arrivals from the CTAs of the cluster (acquire scope).
__device__ __forceinline__ bool wait_parity_cluster(const Watchdog& wd, uint32_t bar, uint32_t parity, unsigned code) {
  if (mbar_try_wait_acq_cluster(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  while (true) {
    if (mbar_try_wait_acq_cluster(bar, parity)) return true;
    if (*wd.abort_flag) return false;
    if (global_timer_ns() - t0 > wd.limit_ns) {
      *wd.abort_flag = 1;
      atomicOr(wd.status, code);
      return false;
    }
  }
}

// Whole-cluster barrier (every thread of every CTA of the cluster).
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// ---------------------------------------------------------------------- TMA
__device__ __forceinline__ void tma_prefetch_desc(const void* tmap) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(tmap)) : "memory");
}

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const void* tmap, uint32_t bar, int32_t x, int32_t y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4}], [%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(tmap)), "r"(bar), "r"(x), "r"(y)
      : "memory");
}

// 1-D bulk copy global -> shared, completing on an mbarrier (16-byte aligned
// addresses, size a multiple of 16).
__device__ __forceinline__ void bulk_load_1d(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
               "l"(src), "r"(bytes), "r"(bar)
               : "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Warpgroup register reallocation: every thread of the 4 warps of a
// warpgroup executes the same call.  dec returns registers to the CTA's pool;
// inc waits until the pool can give the warpgroup R registers per thread.
// The per-warpgroup counts must add up to no more than the registers the
// CTA was launched with.
template <int R>
__device__ __forceinline__ void regs_dec() {
  asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(R));
}
template <int R>
__device__ __forceinline__ void regs_inc() {
  asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(R));
}

// 16-byte asynchronous copy global -> shared through the load/store path
// (bypassing L1); src_bytes < 16 fills the rest with zeros (0: all zeros,
// nothing read).  Completion is tracked per thread by commit groups.
__device__ __forceinline__ void cp_async_16(uint32_t dst, const void* src, uint32_t src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(src_bytes) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
// Waits until at most N of this thread's most recent commit groups are pending.
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// 16 bytes from shared memory.
__device__ __forceinline__ uint4 ld_shared_v4(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr) : "memory");
  return v;
}

// 8 bytes into shared memory.
__device__ __forceinline__ void st_shared_v2(uint32_t addr, uint2 v) {
  asm volatile("st.shared.v2.b32 [%0], {%1, %2};" ::"r"(addr), "r"(v.x), "r"(v.y) : "memory");
}

// ------------------------------------------------------------------ tcgen05
__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem), "r"(ncols) : "memory");
}

__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// D[tmem] (+)= A[smem] * B[smem]^T, both K-major, one CTA.
__device__ __forceinline__ void mma_f8f6f4(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

__device__ __forceinline__ void mma_f16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Block-scaled MXFP8: one E8M0 scale per 32 K-elements for each row of A
// and each row of B, read from tensor memory.
__device__ __forceinline__ void mma_mxf8f6f4(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                             uint32_t sfa_tmem, uint32_t sfb_tmem, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %6, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], %1, %2, %3, [%4], [%5], p;\n\t}" ::"r"(
          d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
      : "memory");
}

// Copies a 32-row x 16-byte shared-memory block into tensor memory, lanes
// 0-31 of every lane quadrant (the same 16 bytes replicated 4 times),
// columns [col, col + 4).
__device__ __forceinline__ void tmem_cp_32x128b_warpx4(uint32_t taddr, uint64_t sdesc) {
  asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(sdesc) : "memory");
}

__device__ __forceinline__ void mma_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar) : "memory");
}

// 16 lanes x 256 bits, repeated 4 times along columns (32 columns in all).
// Thread t of the warp gets, for repetition i = 0..3 (columns 8i..8i+7):
//   r[4i+0], r[4i+1] = lane (base + t/4),     columns 8i + 2(t%4) + {0, 1}
//   r[4i+2], r[4i+3] = lane (base + 8 + t/4), columns 8i + 2(t%4) + {0, 1}
__device__ __forceinline__ void tmem_ld_16x256b_x4(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.16x256b.x4.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
        "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr)
      : "memory");
}

__device__ __forceinline__ void tmem_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// The inverse of tmem_ld_16x256b_x4: thread t writes r[] to the lanes and
// columns it would read them from.
__device__ __forceinline__ void tmem_st_16x256b_x4(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.16x256b.x4.b32 [%0], "
      "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]),
      "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
      : "memory");
}

// This thread's tensor-memory stores are complete (before it reads them back).
__device__ __forceinline__ void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// Makes every register of a tcgen05.ld destination appear redefined after
// tcgen05.wait::ld, so no use of it can be scheduled before the wait.
template <int NR>
__device__ __forceinline__ void reg_fence(uint32_t (&r)[NR]) {
#pragma unroll
  for (int i = 0; i < NR; ++i) asm volatile("" : "+r"(r[i])::"memory");
}

// Shared-memory matrix descriptor for a K-major operand tile whose rows are
// 128 bytes, stored with the 128-byte swizzle (8-row atoms of 1024 bytes, as
// TMA writes them with CU_TENSOR_MAP_SWIZZLE_128B).  Fields: start address
// >> 4 (bits 0-13), leading byte offset >> 4 (16-29, unused for this layout),
// stride byte offset >> 4 (32-45: 1024 between 8-row groups), descriptor
// version 1 (46-47), base offset 0 (49-51), swizzle mode 2 = 128B (61-63).
__device__ __forceinline__ uint64_t sdesc_k128_sw128(uint32_t smem_addr) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((smem_addr & 0x3FFFF) >> 4);
  d |= static_cast<uint64_t>(1) << 16;
  d |= static_cast<uint64_t>(1024 >> 4) << 32;
  d |= static_cast<uint64_t>(1) << 46;
  d |= static_cast<uint64_t>(2) << 61;
  return d;
}

// Shared-memory descriptor of an unswizzled block of 16-byte rows stored
// contiguously (core matrices of 8 rows x 16 bytes, 128 bytes apart), as the
// source of tcgen05.cp: stride byte offset 128, swizzle mode 0.
__device__ __forceinline__ uint64_t sdesc_rows16(uint32_t smem_addr) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((smem_addr & 0x3FFFF) >> 4);
  d |= static_cast<uint64_t>(128 >> 4) << 32;
  d |= static_cast<uint64_t>(1) << 46;
  return d;
}

// Instruction descriptor for kind::mxf8f6f4 block scaling (E4M3 A and B,
// fp32 D): B scale-factor byte id (bits 4-5), A/B formats 0 = E4M3, N >> 3
// (17-22), scale type 1 = UE8M0 (23), M >> 4 (24-28), A scale-factor byte id
// (29-30).  The byte id picks which of the four E8M0 codes packed in each
// 32-bit tensor-memory word applies to this K-step of 32.
__host__ __device__ constexpr uint32_t idesc_mx(uint32_t m, uint32_t n, uint32_t sf_id) {
  return (sf_id << 4) | ((n >> 3) << 17) | (1u << 23) | ((m >> 4) << 24) | (sf_id << 29);
}

// Instruction descriptor for kind::f16 / kind::f8f6f4: D fp32 (bits 4-5 = 1),
// A/B formats (7-9, 10-12), K-major A and B (15, 16 = 0), N >> 3 (17-22),
// M >> 4 (24-28).
__host__ __device__ constexpr uint32_t idesc_dense(uint32_t a_fmt, uint32_t b_fmt, uint32_t m, uint32_t n) {
  return (1u << 4) | (a_fmt << 7) | (b_fmt << 10) | ((n >> 3) << 17) | ((m >> 4) << 24);
}

// Predicated global stores (no branch around them).
__device__ __forceinline__ void st_global_pred_v2f32(void* ptr, float2 v, uint32_t pred) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %3, 0;\n\t@p st.global.v2.f32 [%0], {%1, %2};\n\t}" ::"l"(ptr), "f"(v.x),
      "f"(v.y), "r"(pred)
      : "memory");
}

__device__ __forceinline__ void st_global_pred_v2b32(void* ptr, uint32_t a, uint32_t b, uint32_t pred) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %3, 0;\n\t@p st.global.v2.b32 [%0], {%1, %2};\n\t}" ::"l"(ptr), "r"(a),
      "r"(b), "r"(pred)
      : "memory");
}

__device__ __forceinline__ void st_global_pred_v4b32(void* ptr, const uint32_t (&v)[4], uint32_t pred) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %5, 0;\n\t@p st.global.v4.b32 [%0], {%1, %2, %3, %4};\n\t}" ::"l"(ptr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(pred)
      : "memory");
}

// Transposes a 4 x 4 block of 32-bit values held by the 4 lanes of a group
// (lane bits 0-1 = q): on return, element j of lane q is what element q of
// lane j was.  Two butterfly stages, each swapping one bit of the lane index
// with the same bit of the element index.
__device__ __forceinline__ void transpose4_lanes(uint32_t (&x)[4], int q) {
  const bool b0 = (q & 1) != 0;
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const uint32_t send = b0 ? x[2 * h] : x[2 * h + 1];
    const uint32_t recv = __shfl_xor_sync(0xffffffffu, send, 1);
    if (b0) x[2 * h] = recv;
    else x[2 * h + 1] = recv;
  }
  const bool b1 = (q & 2) != 0;
#pragma unroll
  for (int l = 0; l < 2; ++l) {
    const uint32_t send = b1 ? x[l] : x[l + 2];
    const uint32_t recv = __shfl_xor_sync(0xffffffffu, send, 2);
    if (b1) x[l] = recv;
    else x[l + 2] = recv;
  }
}

// -------------------------------------------------------------- conversions
// Two fp32 -> two E4M3 codes, round to nearest even, saturating to +-448
// (NaN stays NaN).  `lo` lands in the low byte.
__device__ __forceinline__ uint16_t cvt_e4m3x2(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

// max(a, b, c) / min(a, b, c) in one instruction (sm_100+); a NaN operand
// loses to the others, as with fmaxf / fminf.
__device__ __forceinline__ float max3f(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}
__device__ __forceinline__ float min3f(float a, float b, float c) {
  float d;
  asm("min.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

__device__ __forceinline__ float bf16lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}

}  // namespace loka
