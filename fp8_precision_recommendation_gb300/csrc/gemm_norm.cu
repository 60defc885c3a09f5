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
// Design (one CTA per SM, persistent, warp-specialized, 192 threads):
//   warp 0      TMA producer: A and B tiles of 128-byte K slices into a
//               shared-memory ring, 128B-swizzled, one mbarrier per stage.
//   warp 1      allocates tensor memory and issues tcgen05.mma (one thread);
//               the fp32 accumulator of a 128 x N tile lives in TMEM, double
//               buffered when 2N <= 512 columns so the epilogue of tile i
//               overlaps the MMAs of tile i+1.
//   warps 2..5  epilogue: thread t owns output row t of the tile (TMEM lane
//               t); it reads its row with tcgen05.ld, applies the dequant
//               scales and bias, computes the row statistics in fp32 (chunked
//               Chan/Welford merge for LayerNorm, sum of squares for RMSNorm),
//               normalizes, packs bf16 into a swizzled staging tile and one
//               thread TMA-stores 128-byte-wide column slabs to HBM.
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
constexpr int kThreads = 192;
constexpr int kEpiThreads = 128;
constexpr int kEpiBar = 1;               // named barrier id for the epilogue warps
constexpr size_t kSmemBudget = 225 * 1024;

template <int N>
struct Cfg {
  static constexpr int N_MMA = N > 256 ? 256 : N;
  static constexpr int N_SPLIT = N / N_MMA;
  static constexpr uint32_t B_BYTES = static_cast<uint32_t>(N) * kSliceBytes;
  static constexpr uint32_t STAGE = kABytes + B_BYTES;
  static constexpr int NBUF = (2 * N <= kTmemCols) ? 2 : 1;
  static constexpr size_t FIXED = 1024 /*align*/ + 2 * kStagingBytes + 4 * N * sizeof(float) + 512 /*barriers*/;
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
  uint64_t* bars = reinterpret_cast<uint64_t*>(vec_be + N);
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
    const int ep = threadIdx.x - 64;         // 0..127
    const int quad = warp & 3;               // TMEM lane quadrant this warp may access
    const int row = quad * 32 + lane;        // row of the tile owned by this thread
    const uint32_t lane_addr = static_cast<uint32_t>(quad * 32) << 16;
    int cur_group = -1;
    int local = 0;
    int slab = 0;
    for (int tile = blockIdx.x; tile < p.total_tiles; tile += gridDim.x, ++local) {
      const int g = group_of(p, tile);
      const GemmGroup& G = p.g[g];
      if (g != cur_group) {
        named_bar_sync(kEpiBar, kEpiThreads);
        for (int n = ep; n < N; n += kEpiThreads) {
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

      // pass 1: row statistics
      float mean = 0.0f, m2 = 0.0f;
      if (p.norm != kNormNone) {
        for (int c0 = 0; c0 < N; c0 += 64) {
          uint32_t r0[32], r1[32];
          tmem_ld_32x32b_x32(t_row + c0, r0);
          tmem_ld_32x32b_x32(t_row + c0 + 32, r1);
          tmem_ld_wait();
          float v[64];
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            v[j] = fmaf(__uint_as_float(r0[j]) * sxm, vec_sw[c0 + j], vec_b[c0 + j]);
            v[32 + j] = fmaf(__uint_as_float(r1[j]) * sxm, vec_sw[c0 + 32 + j], vec_b[c0 + 32 + j]);
          }
          if (p.norm == kNormRms) {
            float s = 0.0f;
#pragma unroll
            for (int j = 0; j < 64; ++j) s = fmaf(v[j], v[j], s);
            m2 += s;
          } else {
            float s = 0.0f;
#pragma unroll
            for (int j = 0; j < 64; ++j) s += v[j];
            const float cm = s * (1.0f / 64.0f);
            float cq = 0.0f;
#pragma unroll
            for (int j = 0; j < 64; ++j) {
              const float d = v[j] - cm;
              cq = fmaf(d, d, cq);
            }
            if (c0 == 0) {
              mean = cm;
              m2 = cq;
            } else {   // Chan et al. merge of (c0, mean, m2) with (64, cm, cq)
              const float nt = static_cast<float>(c0 + 64);
              const float delta = cm - mean;
              mean = fmaf(delta, 64.0f / nt, mean);
              m2 += cq + delta * delta * (static_cast<float>(c0) * 64.0f / nt);
            }
          }
        }
      }
      float rstd = 1.0f;
      if (p.norm == kNormLayer) rstd = rsqrtf(m2 / static_cast<float>(N) + p.eps);
      if (p.norm == kNormRms) {
        rstd = rsqrtf(m2 / static_cast<float>(N) + p.eps);
        mean = 0.0f;
      }

      // pass 2: normalize, pack, stage, TMA-store 128-byte-wide slabs
      for (int c0 = 0; c0 < N; c0 += OUT_COLS) {
        uint32_t r0[32], r1[32];
        tmem_ld_32x32b_x32(t_row + c0, r0);
        if (OUT_COLS == 64) tmem_ld_32x32b_x32(t_row + c0 + 32, r1);
        tmem_ld_wait();
        if (c0 + OUT_COLS >= N) {   // last read of this accumulator: hand it back to the MMA warp
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(smem_u32(&tempty[buf]));
        }
        const int sb = slab & 1;
        if (slab >= 2) {
          if (ep == 0) bulk_wait_read<1>();
          named_bar_sync(kEpiBar, kEpiThreads);
        }
        uint8_t* srow = staging + sb * kStagingBytes + row * 128;
#pragma unroll
        for (int u = 0; u < 8; ++u) {   // eight 16-byte units of the 128-byte row slab
          uint4 pk;
          if (OUT == static_cast<int>(OutKind::kBf16)) {
            uint32_t w[4];
#pragma unroll
            for (int h = 0; h < 4; ++h) {
              float y2[2];
#pragma unroll
              for (int e = 0; e < 2; ++e) {
                const int j = u * 8 + h * 2 + e;
                const int n = c0 + j;
                const float v = fmaf(__uint_as_float(j < 32 ? r0[j] : r1[j & 31]) * sxm, vec_sw[n], vec_b[n]);
                y2[e] = p.norm == kNormNone ? v : fmaf((v - mean) * rstd, vec_g[n], p.norm == kNormLayer ? vec_be[n] : 0.0f);
              }
              w[h] = pack_bf16x2(y2[0], y2[1]);
            }
            pk = make_uint4(w[0], w[1], w[2], w[3]);
          } else {
            float y4[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const int j = u * 4 + e;
              const int n = c0 + j;
              const float v = fmaf(__uint_as_float(j < 32 ? r0[j] : r1[j & 31]) * sxm, vec_sw[n], vec_b[n]);
              y4[e] = p.norm == kNormNone ? v : fmaf((v - mean) * rstd, vec_g[n], p.norm == kNormLayer ? vec_be[n] : 0.0f);
            }
            pk = make_uint4(__float_as_uint(y4[0]), __float_as_uint(y4[1]), __float_as_uint(y4[2]), __float_as_uint(y4[3]));
          }
          *reinterpret_cast<uint4*>(srow + ((u ^ (row & 7)) << 4)) = pk;
        }
        fence_proxy_async_smem();
        named_bar_sync(kEpiBar, kEpiThreads);
        if (ep == 0) {
          tma_store_2d(&G.tm_y, smem_u32(staging + sb * kStagingBytes), c0, m0);
          bulk_commit();
        }
        ++slab;
      }
    }
    if (ep == 0) bulk_wait<0>();
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
