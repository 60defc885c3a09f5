// Fused FP8 GEMM + dequant + bias + LayerNorm/RMSNorm + store, for sm_103a.
//
// Defined by "LoKA: Low-precision Kernel Applications for Recommendation
// Models at Scale": section II-C (the FP8 linear y = Wx + b whose error and
// speed the probe measures), section III-B "Block-wise Normalization" (fuse
// the normalization into the GEMM epilogue while the output tile is on chip;
// case 1: large batch, small N, a whole output row lives in one thread block,
// so the statistics are local and (de)quantization fuses in too) and
// section I (LRMs are wide ensembles of small GEMMs: several independent
// layers share one launch here).
//
// Design (one CTA per SM, persistent, warp-specialized, 320 threads):
//   warp 0      TMA producer: A and B tiles of 128-byte K slices into a
//               shared-memory ring, 128B-swizzled, one mbarrier per stage.
//   warp 1      allocates tensor memory and issues tcgen05.mma (one thread);
//               the fp32 accumulator of a 128 x N tile lives in TMEM, double
//               buffered when 2N <= 512 columns so the epilogue of tile i
//               overlaps the MMAs of tile i+1.
//   warps 2..9  epilogue: two threads per output row (TMEM lane), each owning
//               half of the row's 32-column chunks; they read the row with
//               tcgen05.ld, apply the dequant scales and bias, compute the row
//               statistics in fp32 (Chan/Welford merge of 32-column chunks for
//               LayerNorm, sum of squares for RMSNorm), merge the two halves
//               through shared memory, normalize, pack bf16 into a swizzled
//               staging slab, and one thread TMA-stores each 64-column slab.
// The output makes no extra HBM round trip: Y is written once.
#include <cudaTypedefs.h>

#include <atomic>

#include "loka_internal.h"
#include "ptx.cuh"

namespace loka {

namespace {

constexpr int kBM = 128;                 // rows per tile (= TMEM lanes)
constexpr int kSliceBytes = 128;         // bytes of K per stage per row
constexpr uint32_t kABytes = kBM * kSliceBytes;
constexpr uint32_t kStagingBytes = kBM * 128;   // one 128-byte-wide output slab
constexpr int kTmemCols = 512;
constexpr int kThreads = 320;
constexpr int kEpiThreads = 256;
constexpr int kEpiBar = 1;               // named barrier id for the epilogue warps
constexpr size_t kSmemBudget = 225 * 1024;

template <int N>
struct Cfg {
  static constexpr int N_MMA = N > 256 ? 256 : N;
  static constexpr int N_SPLIT = N / N_MMA;
  static constexpr uint32_t B_BYTES = static_cast<uint32_t>(N) * kSliceBytes;
  static constexpr uint32_t STAGE = kABytes + B_BYTES;
  static constexpr int NBUF = (2 * N <= kTmemCols) ? 2 : 1;
  static constexpr size_t FIXED = 1024 /*align*/ + 2 * kStagingBytes + 4 * N * sizeof(float) +
                               2 * kBM * sizeof(float2) /*row statistics*/ + 512 /*barriers*/;
  static constexpr int STAGES_RAW = static_cast<int>((kSmemBudget - FIXED) / STAGE);
  static constexpr int STAGES = STAGES_RAW > 8 ? 8 : STAGES_RAW;
  static_assert(STAGES >= 2, "not enough shared memory for two stages");
  static constexpr size_t SMEM = FIXED + static_cast<size_t>(STAGES) * STAGE;
};

__device__ __forceinline__ int group_of(const GemmParams& p, int tile) {
  int g = 0;
  while (g + 1 < p.num_groups && p.g[g + 1].tile_begin <= tile) ++g;
  return g;
}

__device__ __forceinline__ float bf16_to_f(uint16_t h) { return __uint_as_float(static_cast<uint32_t>(h) << 16); }

template <int N, int OP, int OUT>
__global__ void __launch_bounds__(kThreads, 1) gemm_norm_kernel(const __grid_constant__ GemmParams p) {
  using C = Cfg<N>;
  constexpr int STAGES = C::STAGES;
  constexpr int NBUF = C::NBUF;
  // K elements per 128-byte slice and per MMA instruction (32 bytes each)
  constexpr int KE = OP == static_cast<int>(OperandKind::kBf16) ? 64 : 128;
  constexpr uint32_t IDESC = OP == static_cast<int>(OperandKind::kBf16)
                                 ? idesc_dense(1, 1, kBM, C::N_MMA)    // bf16 x bf16 -> f32
                                 : idesc_dense(0, 0, kBM, C::N_MMA);   // e4m3 x e4m3 -> f32
  constexpr int OUT_COLS = OUT == static_cast<int>(OutKind::kBf16) ? 64 : 32;   // columns per 128-byte slab

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* ring = smem;                                         // STAGES x (A | B)
  uint8_t* staging = ring + static_cast<size_t>(STAGES) * C::STAGE;   // 2 x 16 KB
  float* vec_sw = reinterpret_cast<float*>(staging + 2 * kStagingBytes);
  float* vec_b = vec_sw + N;
  float* vec_g = vec_b + N;
  float* vec_be = vec_g + N;
  float2* stat_part = reinterpret_cast<float2*>(vec_be + N);   // [2][128] partial row statistics
  uint64_t* bars = reinterpret_cast<uint64_t*>(stat_part + 2 * kBM);
  uint64_t* full = bars;
  uint64_t* empty = full + STAGES;
  uint64_t* tfull = empty + STAGES;
  uint64_t* tempty = tfull + NBUF;
  uint64_t* mma_done = tempty + NBUF;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(mma_done + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(smem_u32(&full[s]), 1);
      mbar_init(smem_u32(&empty[s]), 1);
    }
    for (int b = 0; b < NBUF; ++b) {
      mbar_init(smem_u32(&tfull[b]), 1);
      mbar_init(smem_u32(&tempty[b]), kEpiThreads / 32);
    }
    mbar_init(smem_u32(mma_done), 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    for (int g = 0; g < p.num_groups; ++g) {
      if (p.g[g].M == 0) continue;   // no tiles, descriptors not encoded
      tma_prefetch_desc(&p.g[g].tm_a);
      tma_prefetch_desc(&p.g[g].tm_b);
      tma_prefetch_desc(&p.g[g].tm_y);
    }
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const Watchdog wd{abort_flag, p.status, p.wait_limit_ns};
  const int num_kb = p.K / KE;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      uint32_t issued = 0, last_parity = 0;
      bool ok = true;
      for (int tile = blockIdx.x; ok && tile < p.total_tiles; tile += gridDim.x) {
        const int g = group_of(p, tile);
        const int m0 = (tile - p.g[g].tile_begin) * kBM;
        for (int kb = 0; kb < num_kb; ++kb) {
          if (!wait_parity(wd, smem_u32(&empty[stage]), phase ^ 1u, kErrProducerWait)) {
            ok = false;
            break;
          }
          uint8_t* a_dst = ring + static_cast<size_t>(stage) * C::STAGE;
          uint8_t* b_dst = a_dst + kABytes;
          const uint32_t fb = smem_u32(&full[stage]);
          mbar_arrive_expect_tx(fb, C::STAGE);
          tma_load_2d(smem_u32(a_dst), &p.g[g].tm_a, fb, kb * KE, m0);
#pragma unroll
          for (int s = 0; s < C::N_SPLIT; ++s)
            tma_load_2d(smem_u32(b_dst + s * C::N_MMA * kSliceBytes), &p.g[g].tm_b, fb, kb * KE, s * C::N_MMA);
          issued |= 1u << stage;
          last_parity = (last_parity & ~(1u << stage)) | (phase << stage);
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      if (!ok) {
        // let the copies already in flight land before the CTA exits
        for (int s = 0; s < STAGES; ++s)
          if (issued & (1u << s)) wait_parity_drain(wd, smem_u32(&full[s]), (last_parity >> s) & 1u);
      }
    }
  } else if (warp == 1) {
    // ----------------------------------------------------------------- MMA
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      int local = 0;
      bool ok = true;
      for (int tile = blockIdx.x; ok && tile < p.total_tiles; tile += gridDim.x, ++local) {
        const int buf = NBUF == 2 ? (local & 1) : 0;
        const uint32_t use = NBUF == 2 ? (local >> 1) : local;
        if (!wait_parity(wd, smem_u32(&tempty[buf]), (use & 1u) ^ 1u, kErrMmaWait)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(buf * N);
        for (int kb = 0; kb < num_kb; ++kb) {
          if (!wait_parity(wd, smem_u32(&full[stage]), phase, kErrMmaWait)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a_addr = smem_u32(ring + static_cast<size_t>(stage) * C::STAGE);
          const uint32_t b_addr = a_addr + kABytes;
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const uint64_t adesc = sdesc_k128_sw128(a_addr + k * 32);
#pragma unroll
            for (int s = 0; s < C::N_SPLIT; ++s) {
              const uint64_t bdesc = sdesc_k128_sw128(b_addr + s * C::N_MMA * kSliceBytes + k * 32);
              const uint32_t acc = (kb | k) != 0 ? 1u : 0u;
              if (OP == static_cast<int>(OperandKind::kBf16))
                mma_f16(d_tmem + s * C::N_MMA, adesc, bdesc, IDESC, acc);
              else
                mma_f8f6f4(d_tmem + s * C::N_MMA, adesc, bdesc, IDESC, acc);
            }
          }
          mma_commit(smem_u32(&empty[stage]));   // frees the slot once these MMAs finish
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        mma_commit(smem_u32(&tfull[buf]));
      }
      // all MMAs issued by this thread complete before tensor memory is freed
      mma_commit(smem_u32(mma_done));
      wait_parity_drain(wd, smem_u32(mma_done), 0);
    }
  } else {
    // ------------------------------------------------------------ epilogue
    // Eight warps: two per TMEM lane quadrant.  Warp pair (q, q+4) shares
    // rows 32q..32q+31; half h = 0/1 takes the interleaved 32-column chunks
    // c = 2i + h, so each 64-column output slab is written by both halves.
    const int et = threadIdx.x - 64;         // 0..255
    const int half = et >> 7;                // column half
    const int quad = warp & 3;               // TMEM lane quadrant this warp may access
    const int row = quad * 32 + lane;        // row of the tile owned by this thread
    const uint32_t lane_addr = static_cast<uint32_t>(quad * 32) << 16;
    constexpr int NCHUNK = N / 32;           // 32-column chunks, NCHUNK / 2 per half
    int cur_group = -1;
    int local = 0;
    int step_count = 0;
    for (int tile = blockIdx.x; tile < p.total_tiles; tile += gridDim.x, ++local) {
      const int g = group_of(p, tile);
      const GemmGroup& G = p.g[g];
      if (g != cur_group) {
        named_bar_sync(kEpiBar, kEpiThreads);
        for (int n = et; n < N; n += kEpiThreads) {
          vec_sw[n] = G.sw == nullptr ? 1.0f : (G.sw_per_row ? G.sw[n] : G.sw[0]);
          vec_b[n] = G.bias == nullptr ? 0.0f : bf16_to_f(G.bias[n]);
          vec_g[n] = G.gamma == nullptr ? 1.0f : bf16_to_f(G.gamma[n]);
          vec_be[n] = G.beta == nullptr ? 0.0f : bf16_to_f(G.beta[n]);
        }
        named_bar_sync(kEpiBar, kEpiThreads);
        cur_group = g;
      }
      const int buf = NBUF == 2 ? (local & 1) : 0;
      const uint32_t use = NBUF == 2 ? (local >> 1) : local;
      wait_parity(wd, smem_u32(&tfull[buf]), use & 1u, kErrEpilogueWait);
      // every epilogue thread takes the same decision, so none is left at a
      // named barrier that the others have abandoned
      named_bar_sync(kEpiBar, kEpiThreads);
      if (*abort_flag) break;
      tc_fence_after();
      const int m0 = (tile - G.tile_begin) * kBM;
      const int64_t m = static_cast<int64_t>(m0) + row;
      float sxm = 1.0f;
      if (G.sx != nullptr) sxm = G.sx_per_row ? (m < G.M ? G.sx[m] : 0.0f) : G.sx[0];
      const uint32_t t_row = tmem_base + lane_addr + static_cast<uint32_t>(buf * N);

      // pass 1: statistics of this half's N/2 columns, 32-column chunks
      // merged with Chan et al.'s pairwise update; then the two halves merge
      float mean = 0.0f, m2 = 0.0f;
      if (p.norm != kNormNone) {
#pragma unroll 1
        for (int i = 0; i < NCHUNK / 2; ++i) {
          const int c0 = (2 * i + half) * 32;
          uint32_t r[32];
          tmem_ld_32x32b_x32(t_row + c0, r);
          tmem_ld_wait();
          float v[32];
#pragma unroll
          for (int j = 0; j < 32; j += 4) {
            const float4 sw4 = *reinterpret_cast<const float4*>(vec_sw + c0 + j);
            const float4 b4 = *reinterpret_cast<const float4*>(vec_b + c0 + j);
            v[j + 0] = fmaf(__uint_as_float(r[j + 0]) * sxm, sw4.x, b4.x);
            v[j + 1] = fmaf(__uint_as_float(r[j + 1]) * sxm, sw4.y, b4.y);
            v[j + 2] = fmaf(__uint_as_float(r[j + 2]) * sxm, sw4.z, b4.z);
            v[j + 3] = fmaf(__uint_as_float(r[j + 3]) * sxm, sw4.w, b4.w);
          }
          if (p.norm == kNormRms) {
            float s = 0.0f;
#pragma unroll
            for (int j = 0; j < 32; ++j) s = fmaf(v[j], v[j], s);
            m2 += s;
          } else {
            float s = 0.0f;
#pragma unroll
            for (int j = 0; j < 32; ++j) s += v[j];
            const float cm = s * (1.0f / 32.0f);
            float cq = 0.0f;
#pragma unroll
            for (int j = 0; j < 32; ++j) {
              const float d = v[j] - cm;
              cq = fmaf(d, d, cq);
            }
            if (i == 0) {
              mean = cm;
              m2 = cq;
            } else {   // merge (32 i, mean, m2) with (32, cm, cq)
              const float na = static_cast<float>(32 * i);
              const float nt = na + 32.0f;
              const float delta = cm - mean;
              mean = fmaf(delta, 32.0f / nt, mean);
              m2 += cq + delta * delta * (na * 32.0f / nt);
            }
          }
        }
        stat_part[half * kBM + row] = make_float2(mean, m2);
        named_bar_sync(kEpiBar, kEpiThreads);
        // both threads of the row evaluate the same expression in the same
        // order, so they agree bit for bit
        const float2 lo = stat_part[row];
        const float2 hi = stat_part[kBM + row];
        if (p.norm == kNormRms) {
          m2 = lo.y + hi.y;
        } else {   // two halves of N/2 elements each
          const float delta = hi.x - lo.x;
          m2 = (lo.y + hi.y) + delta * delta * (0.25f * static_cast<float>(N));
          mean = 0.5f * (lo.x + hi.x);
        }
      }
      float rstd = 1.0f;
      if (p.norm == kNormLayer) rstd = rsqrtf(m2 / static_cast<float>(N) + p.eps);
      if (p.norm == kNormRms) {
        rstd = rsqrtf(m2 / static_cast<float>(N) + p.eps);
        mean = 0.0f;
      }
      const float shift = p.norm == kNormNone ? 0.0f : mean;
      const bool use_beta = p.norm == kNormLayer;
      const bool normed = p.norm != kNormNone;

      // pass 2: normalize, pack, stage and TMA-store.  Step i covers columns
      // [64 i, 64 i + 64): this half writes chunk 2 i + half of it.
#pragma unroll 1
      for (int i = 0; i < NCHUNK / 2; ++i) {
        const int c0 = (2 * i + half) * 32;
        uint32_t r[32];
        tmem_ld_32x32b_x32(t_row + c0, r);
        tmem_ld_wait();
        if (i == NCHUNK / 2 - 1) {   // last read of this accumulator: hand it back to the MMA warp
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(smem_u32(&tempty[buf]));
        }
        float y[32];
#pragma unroll
        for (int j = 0; j < 32; j += 4) {
          const float4 sw4 = *reinterpret_cast<const float4*>(vec_sw + c0 + j);
          const float4 b4 = *reinterpret_cast<const float4*>(vec_b + c0 + j);
          const float4 g4 = *reinterpret_cast<const float4*>(vec_g + c0 + j);
          const float4 be4 = *reinterpret_cast<const float4*>(vec_be + c0 + j);
          const float swv[4] = {sw4.x, sw4.y, sw4.z, sw4.w};
          const float bv[4] = {b4.x, b4.y, b4.z, b4.w};
          const float gv[4] = {g4.x, g4.y, g4.z, g4.w};
          const float bev[4] = {be4.x, be4.y, be4.z, be4.w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float v = fmaf(__uint_as_float(r[j + e]) * sxm, swv[e], bv[e]);
            y[j + e] = normed ? fmaf((v - shift) * rstd, gv[e], use_beta ? bev[e] : 0.0f) : v;
          }
        }
        // staging: bf16 -> one 64-column slab per step (double-buffered);
        // fp32 -> two 32-column slabs per step (single buffer)
        constexpr bool kBf16Out = OUT == static_cast<int>(OutKind::kBf16);
        uint8_t* buf_base;
        if (kBf16Out) {
          buf_base = staging + (step_count & 1) * kStagingBytes;
          if (step_count >= 2) {
            if (et == 0) bulk_wait_read<1>();
            named_bar_sync(kEpiBar, kEpiThreads);
          }
          uint8_t* srow = buf_base + row * 128;
#pragma unroll
          for (int u = 0; u < 4; ++u) {   // 4 units of 8 bf16; this half owns units 4h..4h+3
            const uint4 pk = make_uint4(pack_bf16x2(y[8 * u + 0], y[8 * u + 1]), pack_bf16x2(y[8 * u + 2], y[8 * u + 3]),
                                        pack_bf16x2(y[8 * u + 4], y[8 * u + 5]), pack_bf16x2(y[8 * u + 6], y[8 * u + 7]));
            const int unit = half * 4 + u;
            *reinterpret_cast<uint4*>(srow + ((unit ^ (row & 7)) << 4)) = pk;
          }
        } else {
          buf_base = staging;
          if (step_count >= 1) {
            if (et == 0) bulk_wait_read<0>();
            named_bar_sync(kEpiBar, kEpiThreads);
          }
          uint8_t* srow = buf_base + half * kStagingBytes + row * 128;
#pragma unroll
          for (int u = 0; u < 8; ++u) {   // 8 units of 4 floats: the whole 128-byte row of this half's slab
            const uint4 pk = make_uint4(__float_as_uint(y[4 * u + 0]), __float_as_uint(y[4 * u + 1]),
                                        __float_as_uint(y[4 * u + 2]), __float_as_uint(y[4 * u + 3]));
            *reinterpret_cast<uint4*>(srow + ((u ^ (row & 7)) << 4)) = pk;
          }
        }
        fence_proxy_async_smem();
        named_bar_sync(kEpiBar, kEpiThreads);
        if (et == 0) {
          if (kBf16Out) {
            tma_store_2d(&G.tm_y, smem_u32(buf_base), 64 * i, m0);
          } else {
            tma_store_2d(&G.tm_y, smem_u32(buf_base), 64 * i, m0);
            tma_store_2d(&G.tm_y, smem_u32(buf_base + kStagingBytes), 64 * i + 32, m0);
          }
          bulk_commit();
        }
        ++step_count;
      }
    }
    if (et == 0) bulk_wait<0>();
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem_base, kTmemCols);
}

template <int N, int OP, int OUT>
cudaError_t launch_one(const GemmParams& p, int sms, cudaStream_t stream) {
  constexpr size_t smem = Cfg<N>::SMEM;
  auto kern = gemm_norm_kernel<N, OP, OUT>;
  // the shared-memory opt-in is set once per device (it is not a stream
  // operation, so it also stays out of captured CUDA graphs)
  static std::atomic<uint64_t> configured{0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const uint64_t bit = uint64_t(1) << (dev & 63);
  if (!(configured.load() & bit)) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    configured.fetch_or(bit);
  }
  int grid = p.total_tiles < sms ? p.total_tiles : sms;
  if (grid < 1) return cudaSuccess;
  kern<<<grid, kThreads, smem, stream>>>(p);
  return cudaGetLastError();
}

template <int N>
cudaError_t launch_n(const GemmParams& p, OperandKind op, OutKind out, int sms, cudaStream_t stream) {
  if (op == OperandKind::kE4M3 && out == OutKind::kBf16) return launch_one<N, 0, 0>(p, sms, stream);
  if (op == OperandKind::kE4M3 && out == OutKind::kF32) return launch_one<N, 0, 1>(p, sms, stream);
  if (op == OperandKind::kBf16 && out == OutKind::kBf16) return launch_one<N, 1, 0>(p, sms, stream);
  if (op == OperandKind::kBf16 && out == OutKind::kF32) return launch_one<N, 1, 1>(p, sms, stream);
  return cudaErrorInvalidValue;
}

}  // namespace

size_t gemm_smem_bytes(int N, OperandKind) {
  switch (N) {
    case 64: return Cfg<64>::SMEM;
    case 128: return Cfg<128>::SMEM;
    case 192: return Cfg<192>::SMEM;
    case 256: return Cfg<256>::SMEM;
    case 512: return Cfg<512>::SMEM;
    default: return 0;
  }
}

cudaError_t launch_gemm_norm(const GemmParams& p, int N, OperandKind op, OutKind out, int sms, cudaStream_t stream) {
  if (op == OperandKind::kMxE4M3) return cudaErrorNotSupported;
  switch (N) {
    case 64: return launch_n<64>(p, op, out, sms, stream);
    case 128: return launch_n<128>(p, op, out, sms, stream);
    case 192: return launch_n<192>(p, op, out, sms, stream);
    case 256: return launch_n<256>(p, op, out, sms, stream);
    case 512: return launch_n<512>(p, op, out, sms, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace loka
