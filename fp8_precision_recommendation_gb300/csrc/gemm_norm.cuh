// Fused FP8 GEMM + dequant + bias + LayerNorm/RMSNorm + store, for sm_103a
// (private to the gemm_*.cu files: each instantiates the operand and output
// kinds it names, so the instantiations compile in parallel; gemm_norm.cu
// dispatches to them).
//
// Defined by "LoKA: Low-precision Kernel Applications for Recommendation
// Models at Scale": section II-C (the FP8 linear y = Wx + b whose error and
// speed the probe measures), section III-B "Block-wise Normalization" (fuse
// the normalization into the GEMM epilogue while the output tile is on chip;
// case 1: large batch, small N, a whole output row lives in one thread block,
// so the statistics are local and (de)quantization fuses in too) and
// section I (LRMs are wide ensembles of small GEMMs: several independent
// layers share one launch here).  The quantized output kind follows the GEM
// Training page ("Handling Quantization Overhead": activation quantization
// fused into the preceding normalization; "Low Precision Flash Attention":
// the fused kernels emit FP8 activations with their scales): the epilogue
// also writes the normalized rows as E4M3 codes with per-row or MX 1x32
// scales, exactly what the standalone quantizer makes of the bf16 output, so
// the next layer takes them as pre-quantized activations.
//
// Design (one CTA per SM, persistent, warp-specialized, 640 threads):
//   warp 0       TMA producer: 128-byte K slices of A (and of B when W does
//                not stay resident) into a shared-memory ring, 128B-swizzled,
//                one mbarrier per stage.  When N x K of the weights fits in
//                128 KB, W is loaded once per CTA (per group) and stays in
//                shared memory, so each tile streams only its activations.
//   warp 1       allocates tensor memory and issues tcgen05.mma (one thread);
//                the fp32 accumulator of a 128 x N tile lives in TMEM, double
//                buffered when 2N <= 512 columns so the epilogue of tile i
//                overlaps the MMAs of tile i+1.
//   warps 2, 3   idle (they complete warpgroup 0, whose registers the
//                epilogue takes with setmaxnreg).
//   warps 4..19  epilogue, two teams of 8 warps taking alternate tiles (and
//                accumulator buffers); each warp owns 16 whole rows of its
//                team's tile.  tcgen05.ld.16x256b gives every thread 2 rows
//                x 8 columns of a 32-column chunk, so a per-column value
//                (scale, bias, gamma, beta) read from shared memory serves
//                both rows, and the math runs on packed fp32 pairs
//                (fma/mul/add .f32x2); TMEM reads are pipelined one chunk
//                ahead.  Row statistics are fp32 shifted sums (LayerNorm) or
//                sums of squares (RMSNorm), merged across the 4 lanes of a
//                row (shuffles) and, for rows wider than one CTA, across the
//                cluster's CTAs (distributed shared memory); the statistics
//                pass writes v back to TMEM for the output pass.  Normalized rows
//                are rounded, transposed across the 4 lanes and stored as
//                contiguous 16-byte (bf16) or 8-byte (E4M3) pieces.
// The output makes no extra HBM round trip: Y is written once.
#pragma once

#include <cudaTypedefs.h>

#include <atomic>
#include <type_traits>

#include "loka_internal.h"
#include "ptx.cuh"
#include "quant_math.cuh"

namespace loka {

namespace {

constexpr int kBM = 128;                 // rows per tile (= TMEM lanes)
constexpr int kSliceBytes = 128;         // bytes of K per stage per row
constexpr uint32_t kABytes = kBM * kSliceBytes;
constexpr int kTmemCols = 512;
// producer, MMA, two idle warps (so the epilogue starts a warpgroup), 16
// epilogue warps; setmaxnreg moves registers from the first warpgroup to the
// epilogue (4 x 32 x kRegsLow + 16 x 32 x kRegsEpi <= 640 x 96, the launch's)
constexpr int kThreads = 640;
constexpr int kRegsLow = 56;
constexpr int kRegsEpi = 104;
static_assert(4 * 32 * kRegsLow + 16 * 32 * kRegsEpi <= kThreads * 96, "register shares exceed the launch's");
constexpr int kEpiBar = 1;               // named barrier id for the epilogue warps
constexpr int kQxBar = 3;                // named barrier id for the quantizer warps
constexpr int kMaxStages = 8;            // TMA ring stages
constexpr int kQxMaxStages = 12;         // staging slots of in-kernel quantization
constexpr int kBarStages = 12;           // full / empty barriers (the larger of the two)
constexpr int kMaxWSlices = 16;          // resident W: 128 KB / (64 rows x 128 bytes)
constexpr size_t kSmemLimit = 227 * 1024;
constexpr size_t kResidentWLimit = 128 * 1024;

// In-kernel activation quantization (OperandKind::kE4M3Qx): 32 warps.
//   warp 0        W, resident (once per group)
//   warp 1        MMA;  warps 2-3 idle (they fill warpgroup 0)
//   warps 4-15    quantizers: each loads its own rows of X (cp.async into a
//                 private ring of 1 KB slots) and writes their codes into
//                 the A tile
//   warps 16-31   epilogue, as in the 640-thread kernel
// Registers: launched at 64 per thread (32 warps, 8 per sub-partition), then
// warpgroup 0 drops to 40, the quantizers to 48 and the epilogue rises to 80:
// per sub-partition 40 + 3 x 48 + 4 x 80 = 504 of the 512 register slots.
constexpr int kQxThreads = 1024;
constexpr int kQxWarps = 12;             // quantizer warps
// register shares of the in-kernel quantization kernel's warpgroups
// (producer / MMA, quantizers, epilogue), within the launch's 1024 x 64
constexpr int kQxRegsLow = 40;
constexpr int kQxRegsQuant = 48;
constexpr int kQxRegsEpi = 80;
constexpr int kQxFirstWarp = 4;
constexpr int kQxEpiWarp = 16;           // first epilogue warp
constexpr uint32_t kQxSlotBytes = 1024;  // staging slot: one row of K = 512, two of K = 256
constexpr int kQxMaxSlots = 8;           // slots of one quantizer warp's ring

// Shared-memory carve-up (all offsets from a 1024-byte-aligned base):
//   ring     stages x (A slice [| B slice]), or (in-kernel quantization)
//            stages x 8 KB staging slots of bf16 X rows
//   a        in-kernel quantization: a_bufs x 128 x K E4M3 A tiles (128B
//            swizzled K slices, the layout TMA would write)
//   w        resident W: K/KE slices of N rows x 128 bytes (when resident)
//   vectors  2 teams x 4 x N fp32 (weight scale, bias, gamma, beta)
//   sx       in-kernel quantization: 2 x 128 fp32 row scales (per
//            accumulator buffer), then a copy of the row-scale tables
//   stats    clusters: 2 x CL x 128 float2 row statistics of the CTAs
//   barriers
struct Layout {
  uint32_t stage_bytes, ring, a, w, vec, sx, stats, bars, total;
};

// MX scale blocks: 512 bytes per 128 rows per 128-element K slice.
constexpr uint32_t kSfBlock = 512;
__host__ __device__ constexpr int sfb_blocks(int N) { return (N + 127) / 128; }

__host__ __device__ inline Layout make_layout(int N, int K, int elem_bytes, bool resident, int stages, bool mx,
                                              int cl = 1, int a_bufs = 0) {
  Layout L;
  const uint32_t b_slice = static_cast<uint32_t>(N) * kSliceBytes;
  const uint32_t sfa = mx ? kSfBlock : 0u;
  const uint32_t sfb = mx ? kSfBlock * sfb_blocks(N) : 0u;
  // stage: [A slice][B slice, streamed W][A scales][B scales, streamed W];
  // with in-kernel quantization (a_bufs > 0) one staging slot of bf16 rows
  // per quantizer warp (quantizer w's slot s at (w * stages + s) * 1 KB)
  L.stage_bytes = a_bufs > 0 ? kQxWarps * kQxSlotBytes
                             : kABytes + (resident ? 0u : b_slice) + sfa + (resident ? 0u : sfb);
  L.ring = 0;
  L.a = L.ring + static_cast<uint32_t>(stages) * L.stage_bytes;
  L.w = L.a + static_cast<uint32_t>(a_bufs) * kBM * static_cast<uint32_t>(K);
  const int nkb = (K * elem_bytes + kSliceBytes - 1) / kSliceBytes;   // the last slice may be partial
  // resident W: [nkb B slices][nkb x B scale blocks]
  const uint32_t w_bytes = resident ? static_cast<uint32_t>(nkb) * (b_slice + sfb) : 0u;
  L.vec = L.w + w_bytes;
  L.sx = L.vec + 2u * 4u * N * sizeof(float);
  // in-kernel quantization: 2 x 128 row scales, then the scale tables (1 KB)
  L.stats = L.sx + (a_bufs > 0 ? 2u * kBM * sizeof(float) + static_cast<uint32_t>(sizeof(RowScaleTables)) : 0u);
  // [2][cluster][128] row statistics of the cluster's CTAs (written
  // remotely, double-buffered by tile parity)
  L.bars = L.stats + (cl > 1 ? 2u * cl * kBM * sizeof(float2) : 0u);
  L.total = L.bars + 512;
  return L;
}

__device__ __forceinline__ int group_of(const GemmParams& p, int tile) {
  int g = 0;
  while (g + 1 < p.num_groups && p.g[g + 1].tile_begin <= tile) ++g;
  return g;
}

__device__ __forceinline__ float bf16_to_f(uint16_t h) { return __uint_as_float(static_cast<uint32_t>(h) << 16); }

__device__ __forceinline__ float2 dup2(float a) { return make_float2(a, a); }

// N = the columns this CTA owns (<= 256); CL = CTAs per cluster sharing each
// 128-row tile (the layer's output has N * CL columns; CTA r owns columns
// [r N, r N + N) and the CTAs of a cluster merge their row statistics
// through distributed shared memory, so a row wider than one CTA's tensor
// memory is still normalized in the epilogue).
template <int N, int CL, int OP, int OUT, bool RESIDENT>
__global__ void __launch_bounds__(OP == static_cast<int>(OperandKind::kE4M3Qx) ? kQxThreads : kThreads, 1)
    gemm_norm_kernel(const __grid_constant__ GemmParams p) {
  static_assert(N <= 256, "one MMA per K step");
  // in-kernel per-row quantization of bf16 X (one CTA per row, W resident)
  constexpr bool kQx = OP == static_cast<int>(OperandKind::kE4M3Qx);
  static_assert(!kQx || (CL == 1 && RESIDENT), "in-kernel quantization keeps W resident and rows within a CTA");
  constexpr int EPI0 = kQx ? kQxEpiWarp : 4;       // first epilogue warp
  constexpr int SF_COLS_MAX = OP == static_cast<int>(OperandKind::kMxE4M3) ? kMaxStages * (4 + 4 * sfb_blocks(N)) : 0;
  constexpr int NBUF = (2 * N + SF_COLS_MAX <= kTmemCols) ? 2 : 1;
  static_assert(N + SF_COLS_MAX <= kTmemCols, "accumulator and scale factors must fit in tensor memory");
  constexpr int N_MMA = N > 256 ? 256 : N;
  constexpr int N_SPLIT = N / N_MMA;
  constexpr bool kBf16Op = OP == static_cast<int>(OperandKind::kBf16);
  constexpr bool kMx = OP == static_cast<int>(OperandKind::kMxE4M3);
  constexpr int NSFB = sfb_blocks(N);
  constexpr uint32_t SFB_BYTES = kMx ? kSfBlock * NSFB : 0u;
  constexpr uint32_t SF_COLS = kMx ? 4 + 4 * NSFB : 0;    // TMEM columns of one stage's scales
  constexpr int EB = kBf16Op ? 2 : 1;               // operand element bytes
  constexpr int KE = kSliceBytes / EB;              // K elements per 128-byte slice
  constexpr uint32_t IDESC = kBf16Op ? idesc_dense(1, 1, kBM, N_MMA)    // bf16 x bf16 -> f32
                                     : idesc_dense(0, 0, kBM, N_MMA);   // e4m3 x e4m3 -> f32
  constexpr uint32_t B_SLICE = static_cast<uint32_t>(N) * kSliceBytes;

  const int stages = p.stages;
  // K slices of 128 bytes; a partial last slice reads zeros past K (the
  // tensor maps' out-of-range fill), which add nothing to the sums
  const int num_kb = (p.K + KE - 1) / KE;
  const Layout L = make_layout(N, p.K, EB, RESIDENT, stages, kMx, CL, kQx ? p.a_bufs : 0);
  // A tile's N-column slices go to the CTAs of a cluster (CL > 1, row
  // statistics exchanged), or, when no statistic spans the row (CL == 1,
  // p.slices > 1), to p.slices independent consecutive CTAs.  rank = this
  // CTA's slice, cid / ncl = its unit (cluster or slice group) and their count.
  const int slices = CL > 1 ? CL : p.slices;
  const uint32_t rank = CL > 1 ? cluster_ctarank() : static_cast<uint32_t>(blockIdx.x) % static_cast<uint32_t>(slices);
  const int col0 = static_cast<int>(rank) * N;      // first output column of this CTA
  const int cid = static_cast<int>(blockIdx.x) / slices;
  const int ncl = static_cast<int>(gridDim.x) / slices;
  // columns of the whole output row (the row pitch of the outputs), and the
  // ones this CTA holds: the kernel's N columns from col0 on, fewer (down to
  // none) when the row is narrower than the CTAs' columns (rows of any
  // multiple of 32 run on the next wider kernel; the weight rows past the
  // row width read as zeros)
  const int ng = p.n_cols;
  const int nvalid = ng - col0 < 0 ? 0 : (ng - col0 > N ? N : ng - col0);
  const int nvc = nvalid / 32;                      // valid 32-column chunks

  // Pointers are derived from the __shared__ array by plain offsets, so the
  // compiler keeps them in the shared address space (LDS/STS, not generic
  // loads).  The 128B-swizzled TMA/UMMA tiles need the 1024-byte alignment.
  extern __shared__ __align__(1024) uint8_t smem[];
  // uniform over the CTA; a misaligned CTA skips all work but still takes
  // part in the cluster barriers below
  const bool misaligned = (smem_u32(smem) & 1023u) != 0;
  uint8_t* ring = smem + L.ring;
  uint8_t* wres = smem + L.w;
  float* vec_base = reinterpret_cast<float*>(smem + L.vec);        // [2 teams][4][N]
  float2* cl_stats = reinterpret_cast<float2*>(smem + L.stats);     // [2][CL][128] cluster row statistics
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L.bars);
  uint64_t* full = bars;
  uint64_t* empty = full + kBarStages;
  uint64_t* tfull = empty + kBarStages;
  uint64_t* tempty = tfull + 2;
  uint64_t* mma_done = tempty + 2;
  uint64_t* w_free = mma_done + 1;
  uint64_t* cl_bar = w_free + 1;                                    // [2] cluster statistics arrivals
  uint64_t* cl_free = cl_bar + 2;                                   // [2] cluster statistics buffers read
  uint64_t* w_full = cl_free + 2;                                   // [16] resident W, one per K slice
  // in-kernel quantization: A tiles written (quantizers) and read (MMA), row
  // scales written (quantizers) and read (epilogue team of that buffer); the
  // staging ring uses full / empty
  uint64_t* afull = w_full + kMaxWSlices;                           // [2]
  uint64_t* aempty = afull + 2;                                     // [2]
  uint64_t* sxfull = aempty + 2;                                    // [2]
  uint64_t* sxempty = sxfull + 2;                                   // [2]
  uint64_t* team_sync = sxempty + 2;                                // [2] epilogue team barriers (bounded)
  uint64_t* epi_done = team_sync + 2;                               // the epilogue's last TMEM read
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(epi_done + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < stages; ++s) {
      mbar_init(smem_u32(&full[s]), 1);
      // a staging slot is released by every quantizer warp, an A stage by the MMA
      mbar_init(smem_u32(&empty[s]), kQx ? kQxWarps : 1);
    }
    if (kQx) {
      for (int b = 0; b < 2; ++b) {
        mbar_init(smem_u32(&afull[b]), kQxWarps);
        mbar_init(smem_u32(&aempty[b]), 1);
        mbar_init(smem_u32(&sxfull[b]), kQxWarps);
        mbar_init(smem_u32(&sxempty[b]), 8);   // the eight warps of the epilogue team of buffer b
        mbar_init(smem_u32(&team_sync[b]), 8);
      }
      mbar_init(smem_u32(epi_done), 16);
    }
    for (int b = 0; b < NBUF; ++b) {
      mbar_init(smem_u32(&tfull[b]), 1);
      mbar_init(smem_u32(&tempty[b]), 8);   // the eight warps of the team that owns buffer b
    }
    mbar_init(smem_u32(mma_done), 1);
    for (int kb = 0; kb < kMaxWSlices; ++kb) mbar_init(smem_u32(&w_full[kb]), 1);
    mbar_init(smem_u32(w_free), 1);
    // a tile's statistics: one arming arrival plus the bytes sent by the
    // other CTAs; its buffer is freed by 8 warps of every CTA
    mbar_init(smem_u32(&cl_bar[0]), 1);
    mbar_init(smem_u32(&cl_bar[1]), 1);
    mbar_init(smem_u32(&cl_free[0]), 8 * CL);
    mbar_init(smem_u32(&cl_free[1]), 8 * CL);
    *abort_flag = misaligned ? 1 : 0;
    if (misaligned) atomicOr(p.status, kErrMisaligned);
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    for (int g = 0; g < p.num_groups; ++g) {
      if (p.g[g].M == 0) continue;   // no tiles, descriptors not encoded
      if (!kQx) tma_prefetch_desc(&p.g[g].tm_a);   // in-kernel quantization reads X without a tensor map
      tma_prefetch_desc(&p.g[g].tm_b);
    }
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  // no CTA touches a partner's shared memory before the partner has set up
  // its barriers
  if (CL > 1) cluster_sync_all();
  // resident W for this CTA's first group.  When the caller's W was
  // complete before the launch that precedes this one, it loads now, while
  // that launch (the activation quantizer) may still run.
  // Each K slice of W has its own barrier, so the first tile's MMAs start
  // on slice 0 while later slices are still arriving.
  auto load_w_slice = [&](int g, int kb) {
    const uint32_t wb = smem_u32(&w_full[kb]);
    mbar_arrive_expect_tx(wb, B_SLICE + SFB_BYTES);
#pragma unroll
    for (int s = 0; s < N_SPLIT; ++s)
      tma_load_2d(smem_u32(wres + kb * B_SLICE + s * N_MMA * kSliceBytes), &p.g[g].tm_b, wb, kb * KE,
                  col0 + s * N_MMA);
    if (kMx) {
#pragma unroll
      for (int h = 0; h < NSFB; ++h)
        bulk_load_1d(smem_u32(wres + num_kb * B_SLICE + (kb * NSFB + h) * kSfBlock),
                     p.g[g].sfb_tc + (static_cast<int64_t>(rank * NSFB + h) * num_kb + kb) * kSfBlock,
                     kSfBlock, wb);
    }
  };
  auto load_w = [&](int g) {
    for (int kb = 0; kb < num_kb; ++kb) load_w_slice(g, kb);
  };
  int w_early_group = -1;
  if (!kQx && RESIDENT && p.w_ready && !misaligned && warp == 0 && lane == 0 && cid < p.total_tiles) {
    w_early_group = group_of(p, cid);
    load_w(w_early_group);
  }
  // everything above touches only this CTA's own state (and W when it was
  // ready); inputs written by the kernel before this one (the quantized
  // operands) are read below.  With in-kernel quantization the quantizer
  // warps read only the caller's bf16 X: when X was complete before the
  // launch that precedes this one (p.x_ready) they start at once.
  const bool x_early = kQx && p.x_ready && warp >= kQxFirstWarp && warp < kQxEpiWarp;
  if (!x_early) wait_prerequisite_grids();
  const uint32_t tmem_base = *tmem_slot;
  const Watchdog wd{abort_flag, p.status, p.wait_limit_ns};
  // one lane waits, the whole warp follows its result
  auto warp_wait = [&](uint32_t bar, uint32_t parity, bool cluster_scope, unsigned code = kErrEpilogueWait) {
    int okw = 1;
    if (lane == 0)
      okw = (cluster_scope ? wait_parity_cluster(wd, bar, parity, kErrClusterWait)
                           : wait_parity(wd, bar, parity, code)) ? 1 : 0;
    return __shfl_sync(0xffffffffu, okw, 0) != 0;
  };

  auto run_producer = [&]() {
    // ------------------------------------------------------------ producer
    if (kQx && lane == 0) {
      // W only (the quantizer warps load X themselves), after waiting for
      // the launch before, which wrote it: once per group, when the MMAs of
      // the previous group are done with it.
      bool ok = true;
      int cur_group = -1, w_loads = 0;
      for (int tile = cid; ok && tile < p.total_tiles; tile += ncl) {
        const int g = group_of(p, tile);
        if (g == cur_group) continue;
        if (w_loads > 0 && !wait_parity(wd, smem_u32(w_free), (w_loads - 1) & 1, kErrProducerWait)) {
          ok = false;
          break;
        }
        ++w_loads;
        cur_group = g;
        load_w(g);
      }
      if (!ok && w_loads > 0)
        for (int kb = 0; kb < num_kb; ++kb) wait_parity_drain(wd, smem_u32(&w_full[kb]), (w_loads - 1) & 1);
    } else if (!kQx && lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      uint32_t issued = 0, last_parity = 0;
      int cur_group = w_early_group, w_loads = w_early_group >= 0 ? 1 : 0;
      uint32_t w_issued = w_early_group >= 0 ? 0xFFFFFFFFu : 0u;   // slices of the current W load issued
      bool w_pending = false;   // the current group's W slices go out with its first tile's A slices
      bool ok = true;
      for (int tile = cid; ok && tile < p.total_tiles; tile += ncl) {
        const int g = group_of(p, tile);
        const int m0 = (tile - p.g[g].tile_begin) * kBM;
        if (RESIDENT && g != cur_group) {
          // reload the resident weights once the MMAs of the previous group are done with them
          if (w_loads > 0 && !wait_parity(wd, smem_u32(w_free), (w_loads - 1) & 1, kErrProducerWait)) {
            ok = false;
            break;
          }
          w_pending = true;
          w_issued = 0;
          ++w_loads;
          cur_group = g;
        }
        for (int kb = 0; kb < num_kb; ++kb) {
          if (!wait_parity(wd, smem_u32(&empty[stage]), phase ^ 1u, kErrProducerWait)) {
            ok = false;
            break;
          }
          if (RESIDENT && w_pending) {
            load_w_slice(g, kb);
            w_issued |= 1u << kb;
          }
          uint8_t* a_dst = ring + static_cast<size_t>(stage) * L.stage_bytes;
          const uint32_t fb = smem_u32(&full[stage]);
          mbar_arrive_expect_tx(fb, L.stage_bytes);
          tma_load_2d(smem_u32(a_dst), &p.g[g].tm_a, fb, kb * KE, m0);
          if (!RESIDENT) {
            uint8_t* b_dst = a_dst + kABytes;
#pragma unroll
            for (int s = 0; s < N_SPLIT; ++s)
              tma_load_2d(smem_u32(b_dst + s * N_MMA * kSliceBytes), &p.g[g].tm_b, fb, kb * KE, col0 + s * N_MMA);
          }
          if (kMx) {
            uint8_t* sf_dst = a_dst + kABytes + (RESIDENT ? 0u : B_SLICE);
            bulk_load_1d(smem_u32(sf_dst), p.g[g].sfa_tc + (static_cast<int64_t>(m0 >> 7) * num_kb + kb) * kSfBlock,
                         kSfBlock, fb);
            if (!RESIDENT) {
#pragma unroll
              for (int h = 0; h < NSFB; ++h)
                bulk_load_1d(smem_u32(sf_dst + kSfBlock + h * kSfBlock),
                             p.g[g].sfb_tc + (static_cast<int64_t>(rank * NSFB + h) * num_kb + kb) * kSfBlock,
                             kSfBlock, fb);
            }
          }
          issued |= 1u << stage;
          last_parity = (last_parity & ~(1u << stage)) | (phase << stage);
          if (++stage == stages) {
            stage = 0;
            phase ^= 1u;
          }
        }
        w_pending = false;
      }
      if (!ok) {
        // let the copies already in flight land before the CTA exits
        for (int s = 0; s < stages; ++s)
          if (issued & (1u << s)) wait_parity_drain(wd, smem_u32(&full[s]), (last_parity >> s) & 1u);
        if (RESIDENT && w_loads > 0) {
          for (int kb = 0; kb < num_kb; ++kb)
            if (w_issued & (1u << kb)) wait_parity_drain(wd, smem_u32(&w_full[kb]), (w_loads - 1) & 1);
        }
      }
    }
  };

  auto run_mma = [&]() {
    // ----------------------------------------------------------------- MMA
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      int local = 0;
      int cur_group = -1, w_uses = 0;
      bool ok = true;
      for (int tile = cid; ok && tile < p.total_tiles; tile += ncl, ++local) {
        if (RESIDENT) {
          const int g = group_of(p, tile);
          if (g != cur_group) {
            if (w_uses > 0) mma_commit(smem_u32(w_free));   // previous weights free once these MMAs finish
            ++w_uses;
            cur_group = g;
          }
        }
        const int buf = NBUF == 2 ? (local & 1) : 0;
        const uint32_t use = NBUF == 2 ? (local >> 1) : local;
        if (!wait_parity(wd, smem_u32(&tempty[buf]), (use & 1u) ^ 1u, kErrMmaWait)) break;
        // in-kernel quantization: the tile's A, written whole by the quantizers
        const int abuf = kQx && p.a_bufs == 2 ? (local & 1) : 0;
        const uint32_t ause = kQx && p.a_bufs == 2 ? static_cast<uint32_t>(local >> 1) : static_cast<uint32_t>(local);
        if (kQx && !wait_parity(wd, smem_u32(&afull[abuf]), ause & 1u, kErrMmaWait)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(buf * N);
        for (int kb = 0; kb < num_kb; ++kb) {
          // this K slice of the resident W (complete at once after the
          // group's first tile)
          if (RESIDENT && !wait_parity(wd, smem_u32(&w_full[kb]), (w_uses - 1) & 1, kErrMmaWait)) {
            ok = false;
            break;
          }
          if (!kQx && !wait_parity(wd, smem_u32(&full[stage]), phase, kErrMmaWait)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a_addr =
              kQx ? smem_u32(smem + L.a + static_cast<size_t>(abuf) * kBM * p.K + static_cast<size_t>(kb) * kABytes)
                  : smem_u32(ring + static_cast<size_t>(stage) * L.stage_bytes);
          const uint32_t b_addr = RESIDENT ? smem_u32(wres + kb * B_SLICE) : a_addr + kABytes;
          uint32_t sfa_tmem = 0, sfb_tmem = 0;
          if (kMx) {
            // E8M0 codes of this K slice into tensor memory: A's 128 rows to
            // 4 columns, B's rows to 4 columns per 128 rows
            const uint32_t sfa_smem = a_addr + kABytes + (RESIDENT ? 0u : B_SLICE);
            const uint32_t sfb_smem = RESIDENT ? smem_u32(wres + num_kb * B_SLICE + kb * NSFB * kSfBlock)
                                               : sfa_smem + kSfBlock;
            sfa_tmem = tmem_base + static_cast<uint32_t>(NBUF * N + stage * SF_COLS);
            sfb_tmem = sfa_tmem + 4;
            tmem_cp_32x128b_warpx4(sfa_tmem, sdesc_rows16(sfa_smem));
#pragma unroll
            for (int h = 0; h < NSFB; ++h) tmem_cp_32x128b_warpx4(sfb_tmem + 4 * h, sdesc_rows16(sfb_smem + h * kSfBlock));
          }
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const uint64_t adesc = sdesc_k128_sw128(a_addr + k * 32);
#pragma unroll
            for (int s = 0; s < N_SPLIT; ++s) {
              const uint64_t bdesc = sdesc_k128_sw128(b_addr + s * N_MMA * kSliceBytes + k * 32);
              const uint32_t acc = (kb | k) != 0 ? 1u : 0u;
              if (kBf16Op)
                mma_f16(d_tmem + s * N_MMA, adesc, bdesc, IDESC, acc);
              else if (kMx)
                mma_mxf8f6f4(d_tmem + s * N_MMA, adesc, bdesc, idesc_mx(kBM, N_MMA, k), sfa_tmem, sfb_tmem, acc);
              else
                mma_f8f6f4(d_tmem + s * N_MMA, adesc, bdesc, IDESC, acc);
            }
          }
          if (!kQx) {
            mma_commit(smem_u32(&empty[stage]));   // frees the slot once these MMAs finish
            if (++stage == stages) {
              stage = 0;
              phase ^= 1u;
            }
          }
        }
        if (!ok) break;
        if (kQx) mma_commit(smem_u32(&aempty[abuf]));   // the quantizers may refill this A tile
        mma_commit(smem_u32(&tfull[buf]));
      }
      // all MMAs issued by this thread complete before tensor memory is freed
      mma_commit(smem_u32(mma_done));
      wait_parity_drain(wd, smem_u32(mma_done), 0);
    }
  };

  [[maybe_unused]] auto run_quantizer = [&]() {
    // ------------------------------------------------------- quantizers
    // LoKA section III-B case 1: with a whole output row in one CTA, the
    // activation quantization fuses into the GEMM.  A tile's rows come in
    // units of 1 KB (one row of K = 512, two rows of K = 256); quantizer
    // warp q takes units q, q + 12, q + 24, ... of every tile.  Each warp
    // keeps its own ring of `stages` 1 KB slots filled with its next units:
    // every lane copies its two 16-byte pieces of a unit (cp.async through
    // the load/store path, one commit group per unit; rows past M arrive as
    // zeros), so no slot is shared and a slot is refilled as soon as the warp
    // has read it.  Lane l holds the pieces at bytes 16 l and 512 + 16 l of a
    // unit: the two halves of a K = 512 row, or the two K = 256 rows.  Per
    // row: one warp reduction of the amax, the standalone quantizer's scales
    // (quant_math.cuh, tables copied into shared memory), the cast, and the
    // codes written straight into the A tile in the 128B-swizzled layout the
    // MMA descriptors describe (16-byte piece c of row r of a K slice at
    // piece c ^ (r % 8)).
    const int qw = warp - kQxFirstWarp;
    const bool two_rows = p.K == 256;
    const int rps = two_rows ? 2 : 1;                       // rows per unit
    const int units = kBM / rps;                            // units per tile
    const int S = stages;                                   // slots of this warp's ring (5..8)
    const uint32_t ring_base = smem_u32(ring) + static_cast<uint32_t>(qw * S) * kQxSlotBytes;
    RowScaleTables* tab = reinterpret_cast<RowScaleTables*>(smem + L.sx + 2 * kBM * sizeof(float));
    {
      const float* src_tab = &kRowScaleTables.inv[0];
      float* dst_tab = &tab->inv[0];
      for (int i = qw * 32 + lane; i < 256; i += kQxWarps * 32) dst_tab[i] = src_tab[i];
      named_bar_sync(kQxBar, kQxWarps * 32);   // the quantizer warps only, before any wait
    }
    // load cursor: the next unit to load, in the order the warp processes
    // them (every lane follows the same sequence).  The tile's parameters
    // are read once per tile; per unit the cursor only advances.
    const int my_units = (units - qw + kQxWarps - 1) / kQxWarps;   // units of a tile for this warp
    const int64_t step = static_cast<int64_t>(kQxWarps) * rps * p.K;  // elements between its units
    int load_tile = cid - ncl, load_left = 0;
    const uint16_t* lbase = nullptr;   // the group's X (a valid address for zero-size copies)
    const uint16_t* lrow = nullptr;    // first row of the next unit
    int64_t lrows = 0;                 // rows of the group from lrow on
    // piece 0 of a unit: its first row, bytes 16 l; piece 1: the same row's
    // bytes 512 + 16 l (K = 512) or the next row's bytes 16 l (K = 256)
    const int64_t off1 = two_rows ? p.K : 256;
    auto issue = [&](int s) {
      if (load_left == 0) {
        load_tile += ncl;
        if (load_tile < p.total_tiles) {
          const GemmGroup& G = p.g[group_of(p, load_tile)];
          const int64_t r0 = static_cast<int64_t>(load_tile - G.tile_begin) * kBM + qw * rps;
          lbase = G.xbf;
          lrow = G.xbf + r0 * p.K + lane * 8;
          lrows = G.M - r0;
          load_left = my_units;
        }
      }
      if (load_left > 0) {
        const uint32_t dst = ring_base + static_cast<uint32_t>(s) * kQxSlotBytes + static_cast<uint32_t>(lane) * 16u;
        const bool ok0 = lrows > 0, ok1 = two_rows ? lrows > 1 : lrows > 0;
        cp_async_16(dst, ok0 ? lrow : lbase, ok0 ? 16u : 0u);
        cp_async_16(dst + 512u, ok1 ? lrow + off1 : lbase, ok1 ? 16u : 0u);
        lrow += step;
        lrows -= kQxWarps * rps;
        --load_left;
      }
      cp_async_commit();   // one group per slot, empty when nothing is left to load
    };
    // waits for the oldest of the S groups in flight
    auto wait_oldest = [&]() {
      switch (S) {
        case 5: cp_async_wait<4>(); break;
        case 6: cp_async_wait<5>(); break;
        case 7: cp_async_wait<6>(); break;
        default: cp_async_wait<7>(); break;
      }
    };
    for (int s = 0; s < S; ++s) issue(s);
    int slot = 0;
    int local = 0;
    bool okq = true;
    for (int tile = cid; okq && tile < p.total_tiles; tile += ncl, ++local) {
      const int ab = p.a_bufs == 2 ? (local & 1) : 0;
      const uint32_t ause = p.a_bufs == 2 ? static_cast<uint32_t>(local >> 1) : static_cast<uint32_t>(local);
      const int sb = local & 1;   // row-scale buffer = the tile's accumulator buffer
      bool a_free = false;
      const uint32_t abase = smem_u32(smem + L.a + static_cast<size_t>(ab) * kBM * p.K);
      float* sxo = reinterpret_cast<float*>(smem + L.sx) + sb * kBM;
      for (int u = qw; u < units; u += kQxWarps) {
        wait_oldest();
        __syncwarp();   // every lane's pieces of the unit are visible to the warp
        const uint32_t src = ring_base + static_cast<uint32_t>(slot) * kQxSlotBytes + static_cast<uint32_t>(lane) * 16u;
        const uint4 d0 = ld_shared_v4(src);
        const uint4 d1 = ld_shared_v4(src + 512u);
        const float a0 = abs_max8(d0, 0.0f), a1 = abs_max8(d1, 0.0f);
        float inv0, inv1, sc0, sc1;
        if (two_rows) {
          row_scales(warp_max(a0), inv0, sc0, *tab);
          row_scales(warp_max(a1), inv1, sc1, *tab);
        } else {
          row_scales(warp_max(fmaxf(a0, a1)), inv0, sc0, *tab);
          inv1 = inv0;
          sc1 = sc0;
        }
        // the slot's data are in registers (the reductions above used every
        // lane's): refill it with this warp's next unit
        __syncwarp();
        issue(slot);
        if (++slot == S) slot = 0;
        if (!a_free) {
          // the A tile and row-scale buffer of this tile are written from here on
          if (!warp_wait(smem_u32(&aempty[ab]), (ause & 1u) ^ 1u, false, kErrQuantWait) ||
              !warp_wait(smem_u32(&sxempty[sb]), ((local >> 1) & 1u) ^ 1u, false, kErrQuantWait)) {
            okq = false;
            break;
          }
          a_free = true;
        }
        // vector 0: row r0, piece idx0; vector 1: row r1, piece idx1
        const int r0 = u * rps, r1 = two_rows ? r0 + 1 : r0;
        const int idx0 = lane, idx1 = two_rows ? lane : lane + 32;
        st_shared_v2(abase + static_cast<uint32_t>(idx0 >> 4) * kABytes + static_cast<uint32_t>(r0) * 128u +
                         ((static_cast<uint32_t>((idx0 & 15) >> 1) ^ static_cast<uint32_t>(r0 & 7)) << 4) +
                         static_cast<uint32_t>(idx0 & 1) * 8u,
                     cast8(d0, inv0));
        st_shared_v2(abase + static_cast<uint32_t>(idx1 >> 4) * kABytes + static_cast<uint32_t>(r1) * 128u +
                         ((static_cast<uint32_t>((idx1 & 15) >> 1) ^ static_cast<uint32_t>(r1 & 7)) << 4) +
                         static_cast<uint32_t>(idx1 & 1) * 8u,
                     cast8(d1, inv1));
        if (lane == 0) {
          sxo[r0] = sc0;
          if (two_rows) sxo[r1] = sc1;
        }
      }
      if (!okq) break;
      // the codes are read by the tensor core (async proxy)
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(smem_u32(&afull[ab]));
        mbar_arrive(smem_u32(&sxfull[sb]));
      }
    }
    // copies still in flight into this warp's ring land before it leaves
    cp_async_wait<0>();
  };

  auto run_epilogue = [&]() {
    // ------------------------------------------------------------ epilogue
    // Sixteen warps in two teams of eight.  Team e takes the tiles whose
    // local index is e (mod 2), i.e. accumulator buffer e, so two tiles are
    // normalized at once (with one accumulator buffer team 0 takes every
    // tile).  In a team, warp (quad q, row half h) owns rows
    // 32q + 16h .. 32q + 16h + 15 of the tile over all of this CTA's N
    // columns, so its row statistics need only 4-lane shuffles and no
    // barrier couples the warps of a tile.  The 16x256b load shape gives
    // thread t rows t/4 + {0, 8} of the 16 and column pairs 8i + 2(t%4) of
    // each 32-column chunk; a per-column value read from shared memory serves
    // both rows.  Chunk reads are pipelined one ahead.
    const int ew = warp - EPI0;                     // 0..15
    const int team = NBUF == 2 ? (ew >> 3) : 0;
    const bool active = NBUF == 2 || ew < 8;
    const int tstep = NBUF == 2 ? 2 : 1;            // a team's tiles are tstep apart
    const uint32_t team_bar = kEpiBar + static_cast<uint32_t>(team);
    const int quad = warp & 3;                      // TMEM lane quadrant this warp may access
    const int rh = (ew >> 2) & 1;                   // row half of the quadrant
    const int g4 = lane >> 2;                       // row within each 8-row group
    const int cp = lane & 3;                        // column pair within each 8-column group
    const uint32_t lane_addr = static_cast<uint32_t>(quad * 32 + rh * 16) << 16;
    constexpr int NCHUNK = N / 32;
    constexpr bool kBf16Out = OUT == static_cast<int>(OutKind::kBf16);
    constexpr bool kQOut = OUT == static_cast<int>(OutKind::kQuant);
    const int norm = p.norm;
    const float eps = p.eps;
    const bool act = p.act != 0;
    // BlockNorm: log2 of the chunks (32 columns) per block
    const int lcpb = 31 - __clz(max(p.norm_block >> 5, 1));
    float* vec_sw = vec_base + team * 4 * N;        // this team's copy of the column vectors
    float* vec_b = vec_sw + N;
    float* vec_g = vec_b + N;
    float* vec_be = vec_g + N;
    int rowk[2];
#pragma unroll
    for (int k = 0; k < 2; ++k) rowk[k] = quad * 32 + rh * 16 + g4 + 8 * k;

    // activation scales of a tile's two rows of this thread (per-tensor
    // weight scales fold in); loaded one tile ahead to hide the latency
    auto row_scales = [&](int tile, float (&out)[2]) {
      const int g = group_of(p, tile);
      const GemmGroup& G = p.g[g];
      const int m0 = (tile - G.tile_begin) * kBM;
      const float swc = (G.sw != nullptr && !G.sw_per_row) ? G.sw[0] : 1.0f;
#pragma unroll
      for (int k = 0; k < 2; ++k) {
        const int64_t m = static_cast<int64_t>(m0) + rowk[k];
        float sx = 1.0f;
        if (G.sx != nullptr) sx = G.sx_per_row ? (m < G.M ? G.sx[m] : 0.0f) : G.sx[0];
        out[k] = sx * swc;
      }
    };
    auto vec2 = [&](const float* vec, int c0, int i) {
      return *reinterpret_cast<const float2*>(vec + c0 + 8 * i + 2 * cp);
    };
    auto acc2 = [&](const uint32_t (&r)[16], int k, int i) {
      const int o = 4 * i + 2 * k;
      return make_float2(__uint_as_float(r[o]), __uint_as_float(r[o + 1]));
    };
    // Runs fn(r, c) over the valid chunks c = 0 .. nvc-1, the TMEM read of chunk
    // c + 1 in flight while chunk c is processed.  The loop and its reads
    // run over all NCHUNK chunks (a loop whose trip count is known keeps r in
    // registers); only fn is skipped past the row's end.
    auto for_chunks = [&](uint32_t t_base, auto&& fn) {
      uint32_t r[2][16];
      tmem_ld_16x256b_x4(t_base, r[0]);
      tmem_ld_wait();
      reg_fence(r[0]);
#pragma unroll
      for (int c = 0; c < NCHUNK; ++c) {
        if (c + 1 < NCHUNK) tmem_ld_16x256b_x4(t_base + (c + 1) * 32, r[(c + 1) & 1]);
        if (c < nvc) fn(r[c & 1], c);   // uniform over the warp
        if (c + 1 < NCHUNK) {
          tmem_ld_wait();
          reg_fence(r[(c + 1) & 1]);
        }
      }
    };
    // v = acc * sx * sw + b for the pair: sw is the per-column weight scale
    // (rowwise W; 1 otherwise, a per-tensor weight scale folds into sx).  MX
    // and bf16 operands have no per-column scale (MX scales act inside the
    // MMA): v = acc * sx + b, one instruction, there.
    auto vpair = [&](const uint32_t (&r)[16], int k, int i, float2 sx2, [[maybe_unused]] float2 sw, float2 b) {
      if constexpr (kMx || kBf16Op)
        return __ffma2_rn(acc2(r, k, i), sx2, b);
      else
        return __ffma2_rn(__fmul2_rn(acc2(r, k, i), sx2), sw, b);
    };
    // The statistics pass writes v back over the accumulator chunk it read
    // (same lanes and columns), so the output pass reads v itself and
    // neither recomputes it nor reloads the column scales and bias.
    // v of pair (k, i) replaces the accumulator pair it came from (read
    // once, so no extra registers hold the chunk)
    auto put_v = [&](uint32_t (&r)[16], int k, int i, float2 v) {
      r[4 * i + 2 * k] = __float_as_uint(v.x);
      r[4 * i + 2 * k + 1] = __float_as_uint(v.y);
    };
    int cur_group = -1;
    bool affine = false;
    float sx_next[2] = {1.f, 1.f};
    // in-kernel quantization: the team's barrier is an mbarrier with a time
    // limit (the 896-thread kernel has no wait without one)
    uint32_t team_phase = 0;
    auto team_barrier = [&]() {
      if constexpr (kQx) {
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&team_sync[team]));
        const bool okt = warp_wait(smem_u32(&team_sync[team]), team_phase, false, kErrTeamWait);
        team_phase ^= 1u;
        return okt && *abort_flag == 0;
      } else {
        return !named_bar_or(team_bar, 256, *abort_flag != 0);
      }
    };
    int local = team;
    int tile = cid + team * ncl;
    if (!kQx && active && tile < p.total_tiles) row_scales(tile, sx_next);
    for (; active && tile < p.total_tiles; tile += tstep * ncl, local += tstep) {
      const int g = group_of(p, tile);
      const GemmGroup& G = p.g[g];
      if (g != cur_group) {
        // this team's column vectors for the group; the barrier's OR makes
        // the abort decision the same for all of the team's warps
        if (!team_barrier()) break;
        const bool normed = norm != kNormNone;
        // LayerNorm is unchanged when one constant is added to every column
        // of a row, so the bias enters centred on its own mean: a bias far
        // above the row's spread (LoKA section III-B: LayerNorm's mean
        // cancellation) then never reaches the fp32 statistics or the
        // output's v - mean.  Every warp of every CTA sums the full row in
        // the same order (lane-strided, then a butterfly, whose partners add
        // the same two values), so all columns subtract the same number.
        float mu_b = 0.0f;
        if (norm == kNormLayer && G.bias != nullptr) {
          float s = 0.0f;
          for (int n = lane; n < ng; n += 32) s += bf16_to_f(G.bias[n]);
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
          mu_b = s / static_cast<float>(ng);
        }
        for (int n = (ew & 7) * 32 + lane; n < N; n += 256) {
          const int gn = col0 + n;
          const bool in = n < nvalid;   // the kernel's columns past the row hold nothing
          vec_sw[n] = (in && G.sw != nullptr && G.sw_per_row) ? G.sw[gn] : 1.0f;
          vec_b[n] = (!in || G.bias == nullptr) ? 0.0f : bf16_to_f(G.bias[gn]) - mu_b;
          vec_g[n] = (!in || G.gamma == nullptr || !normed) ? 1.0f : bf16_to_f(G.gamma[gn]);
          vec_be[n] = (!in || G.beta == nullptr || norm != kNormLayer) ? 0.0f : bf16_to_f(G.beta[gn]);
        }
        affine = normed && (G.gamma != nullptr || (G.beta != nullptr && norm == kNormLayer));
        if constexpr (kQx) {
          if (!team_barrier()) break;
        } else {
          named_bar_sync(team_bar, 256);
        }
        cur_group = g;
      }
      float sxr[2] = {sx_next[0], sx_next[1]};
      const int m0 = (tile - G.tile_begin) * kBM;
      // output row addresses and validity, once per tile
      const int64_t Mg = G.M;
      uint8_t* rowp[2];
      uint32_t ok[2];
      // E4M3 codes of row rowk[0]; those of rowk[1] are 8 rows further
      [[maybe_unused]] uint8_t* rowq = nullptr;
      [[maybe_unused]] const bool has_y = G.y != nullptr;
#pragma unroll
      for (int k = 0; k < 2; ++k) {
        const int64_t m = static_cast<int64_t>(m0) + rowk[k];
        ok[k] = m < Mg ? 1u : 0u;
        // bf16: the 4 lanes of a row group store 16 contiguous bytes each
        // after a transpose; fp32: column pairs straight from registers;
        // E4M3 codes: 8 contiguous bytes per lane after a transpose
        constexpr bool kWide = kBf16Out || kQOut;
        rowp[k] = reinterpret_cast<uint8_t*>(reinterpret_cast<uintptr_t>(G.y) +
                                             (m * ng + col0 + (kWide ? 8 : 2) * cp) * (kWide ? 2 : 4));
        if constexpr (kQOut) {
          if (k == 0) rowq = G.yq + m * ng + col0 + 8 * cp;
        }
      }
      const int buf = NBUF == 2 ? team : 0;
      const uint32_t use = NBUF == 2 ? static_cast<uint32_t>(local >> 1) : static_cast<uint32_t>(local);
      if (!warp_wait(smem_u32(&tfull[buf]), use & 1u, false)) break;
      tc_fence_after();
      if constexpr (kQx) {
        // the row scales the quantizers chose for this tile (buffer = the
        // accumulator buffer); the weight scales are per column
        if (!warp_wait(smem_u32(&sxfull[buf]), use & 1u, false, kErrRowScaleWait)) break;
        const float* sxs = reinterpret_cast<const float*>(smem + L.sx) + buf * kBM;
        sxr[0] = sxs[rowk[0]];
        sxr[1] = sxs[rowk[1]];
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&sxempty[buf]));
      } else if (tile + tstep * ncl < p.total_tiles) {
        row_scales(tile + tstep * ncl, sx_next);
      }
      const uint32_t t_base = tmem_base + lane_addr + static_cast<uint32_t>(buf * N);
      const float2 sx2[2] = {dup2(sxr[0]), dup2(sxr[1])};

      // pass 1: row statistics of v = acc * sx * sw + b
      float mean[2] = {0.f, 0.f}, m2[2] = {0.f, 0.f};
      // extremes of v, kept when they decide the E4M3 row scale (see below)
      [[maybe_unused]] float vhi[2] = {-INFINITY, -INFINITY}, vlo[2] = {INFINITY, INFINITY};
      // BlockNorm: sums of squares of the blocks this lane keeps (b % 4 == cp; slot b / 4)
      [[maybe_unused]] float bsq[2][2] = {{0.f, 0.f}, {0.f, 0.f}};
      auto stats_pass = [&](auto trk_tag) {
        if (norm == kNormLayer) {
          // shifted sums: with K the mean of the row's first 8-value piece,
          // s1 += v - K and s2 += (v - K)^2; no division, little cancellation
          float shift[2] = {0.f, 0.f}, s1[2] = {0.f, 0.f};
          for_chunks(t_base, [&](uint32_t (&r)[16], int c) {
            const int c0 = c * 32;
            float2 sw[4], b[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              sw[i] = vec2(vec_sw, c0, i);
              b[i] = vec2(vec_b, c0, i);
            }
#pragma unroll
            for (int k = 0; k < 2; ++k) {
              float2 v[4];
#pragma unroll
              for (int i = 0; i < 4; ++i) {
                v[i] = vpair(r, k, i, sx2[k], sw[i], b[i]);
                put_v(r, k, i, v[i]);
              }
              if constexpr (decltype(trk_tag)::value) {
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                  vhi[k] = max3f(vhi[k], v[i].x, v[i].y);
                  vlo[k] = min3f(vlo[k], v[i].x, v[i].y);
                }
              }
              if (c == 0) {
                const float2 t = __fadd2_rn(__fadd2_rn(v[0], v[1]), __fadd2_rn(v[2], v[3]));
                shift[k] = (t.x + t.y) * 0.125f;
              }
              const float2 nk = dup2(-shift[k]);
              float2 a1 = make_float2(0.f, 0.f), a2 = make_float2(0.f, 0.f);
#pragma unroll
              for (int i = 0; i < 4; ++i) {
                const float2 d = __fadd2_rn(v[i], nk);
                a1 = __fadd2_rn(a1, d);
                a2 = __ffma2_rn(d, d, a2);
              }
              s1[k] += a1.x + a1.y;
              m2[k] += a2.x + a2.y;
            }
            tmem_st_16x256b_x4(t_base + static_cast<uint32_t>(c0), r);
          });
          // each lane holds 8 values of a row per valid chunk
          const float inv_me = nvc > 0 ? 1.0f / (8.0f * static_cast<float>(nvc)) : 0.0f;
#pragma unroll
          for (int k = 0; k < 2; ++k) {
            const float d = s1[k] * inv_me;
            mean[k] = shift[k] + d;
            m2[k] = fmaxf(m2[k] - s1[k] * d, 0.0f);
          }
        } else if (norm == kNormRms) {
          for_chunks(t_base, [&](uint32_t (&r)[16], int c) {
            const int c0 = c * 32;
            float2 sw[4], b[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              sw[i] = vec2(vec_sw, c0, i);
              b[i] = vec2(vec_b, c0, i);
            }
#pragma unroll
            for (int k = 0; k < 2; ++k) {
              float2 q = make_float2(0.f, 0.f);
#pragma unroll
              for (int i = 0; i < 4; ++i) {
                const float2 v = vpair(r, k, i, sx2[k], sw[i], b[i]);
                put_v(r, k, i, v);
                if constexpr (decltype(trk_tag)::value) {
                  vhi[k] = max3f(vhi[k], v.x, v.y);
                  vlo[k] = min3f(vlo[k], v.x, v.y);
                }
                q = __ffma2_rn(v, v, q);
              }
              m2[k] += q.x + q.y;
            }
            tmem_st_16x256b_x4(t_base + static_cast<uint32_t>(c0), r);
          });
        } else if (norm == kNormBlockRms) {
          // BlockNorm: sums of squares per block of the row; the row's 4
          // lanes merge each chunk's sum, and lane (b % 4) keeps block b's
          for_chunks(t_base, [&](uint32_t (&r)[16], int c) {
            const int c0 = c * 32;
            float2 sw[4], b[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              sw[i] = vec2(vec_sw, c0, i);
              b[i] = vec2(vec_b, c0, i);
            }
            const int blk = c >> lcpb;
#pragma unroll
            for (int k = 0; k < 2; ++k) {
              float2 q = make_float2(0.f, 0.f);
#pragma unroll
              for (int i = 0; i < 4; ++i) {
                const float2 v = vpair(r, k, i, sx2[k], sw[i], b[i]);
                put_v(r, k, i, v);
                q = __ffma2_rn(v, v, q);
              }
              float qs = q.x + q.y;
              qs += __shfl_xor_sync(0xffffffffu, qs, 1);
              qs += __shfl_xor_sync(0xffffffffu, qs, 2);
              if ((blk & 3) == cp) {
                if (blk & 4) bsq[k][1] += qs;
                else bsq[k][0] += qs;
              }
            }
            tmem_st_16x256b_x4(t_base + static_cast<uint32_t>(c0), r);
          });
        }
      };
      // E4M3 row output without gamma and beta: the extremes of v give the
      // row's amax (see below), so the statistics pass keeps them
      [[maybe_unused]] const bool track = kQOut && CL == 1 && p.yq_mode == kScaleRow &&
                                          (norm == kNormLayer || norm == kNormRms) && !affine && !act;
      if (kQOut && CL == 1 && track) {
        stats_pass(std::true_type{});
      } else {
        stats_pass(std::false_type{});
      }
      tmem_st_wait();   // v is read back below

      float rstd[2] = {1.f, 1.f};
      // BlockNorm: 1/rms of the blocks this lane keeps
      [[maybe_unused]] float brs[2][2] = {{1.f, 1.f}, {1.f, 1.f}};
      if (norm == kNormLayer || norm == kNormRms) {
        // merge the 4 lanes of a row group (equal counts) with an ordered
        // expression so all four end bit-identical
#pragma unroll
        for (int lvl = 0; lvl < 2; ++lvl) {
          const int off = 1 << lvl;
          const float half_n = 4.0f * static_cast<float>(nvc) * static_cast<float>(off);   // n_a n_b / (n_a + n_b)
          const bool lo_side = (lane & off) == 0;
#pragma unroll
          for (int k = 0; k < 2; ++k) {
            const float om = __shfl_xor_sync(0xffffffffu, mean[k], off);
            const float oq = __shfl_xor_sync(0xffffffffu, m2[k], off);
            const float lm = lo_side ? mean[k] : om, hm = lo_side ? om : mean[k];
            const float lq = lo_side ? m2[k] : oq, hq = lo_side ? oq : m2[k];
            const float delta = hm - lm;
            m2[k] = norm == kNormRms ? lq + hq : (lq + hq) + delta * delta * half_n;
            mean[k] = norm == kNormRms ? 0.0f : 0.5f * (lm + hm);
          }
        }
        if constexpr (CL > 1) {
          // exchange (mean, M2) of this CTA's N columns with the cluster.
          // Buffer cb holds the statistics of every other tile.  A writer
          // waits until every CTA has read the buffer's previous contents
          // (cl_free); the cp == 0 lanes then send their two rows to every
          // other CTA with st.async, which the receiver's cl_bar counts in
          // bytes, so no release (which would wait for this warp's earlier
          // global stores) is needed.  One thread per CTA arms cl_bar with
          // the bytes it receives; a warp's own rows come from registers.
          const int cb = local & 1;
          const uint32_t cphase = static_cast<uint32_t>(local >> 1) & 1u;
          if ((ew & 7) == 0 && lane == 0) mbar_arrive_expect_tx(smem_u32(&cl_bar[cb]), kBM * 8 * (CL - 1));
          if (!warp_wait(smem_u32(&cl_free[cb]), cphase ^ 1u, true)) break;
          if (cp == 0) {
#pragma unroll
            for (int j = 0; j < CL; ++j) {
              if (j == static_cast<int>(rank)) continue;
              const uint32_t bar = mapa_shared(smem_u32(&cl_bar[cb]), j);
#pragma unroll
              for (int k = 0; k < 2; ++k) {
                const uint32_t a = smem_u32(&cl_stats[(cb * CL + static_cast<int>(rank)) * kBM + rowk[k]]);
                st_async_f32x2(mapa_shared(a, j), mean[k], m2[k], bar);
              }
            }
          }
          if (!warp_wait(smem_u32(&cl_bar[cb]), cphase, true)) break;
          // merge the CTAs' statistics in rank order (Chan: CTA j holds the
          // row's valid columns from j N on, possibly none)
#pragma unroll
          for (int k = 0; k < 2; ++k) {
            float mA = 0.f, qA = 0.f;
#pragma unroll
            for (int j = 0; j < CL; ++j) {
              if (j > 0 && p.chan_w[j] == 0.0f) continue;   // CTA j holds none of the row
              const float2 part_j = j == static_cast<int>(rank) ? make_float2(mean[k], m2[k])
                                                                : cl_stats[(cb * CL + j) * kBM + rowk[k]];
              if (norm == kNormRms) {
                qA += part_j.y;
              } else if (j == 0) {
                mA = part_j.x;
                qA = part_j.y;
              } else {
                const float delta = part_j.x - mA;
                mA = fmaf(delta, p.chan_w[j], mA);
                qA += part_j.y + delta * delta * p.chan_c[j];
              }
            }
            mean[k] = norm == kNormRms ? 0.0f : mA;
            m2[k] = qA;
          }
          // this warp's reads of buffer cb are done (their values are
          // consumed above): tell every CTA
          __syncwarp();
          if (lane == 0) {
#pragma unroll
            for (int j = 0; j < CL; ++j) mbar_arrive_cluster_relaxed(mapa_shared(smem_u32(&cl_free[cb]), j));
          }
        }
#pragma unroll
        for (int k = 0; k < 2; ++k) rstd[k] = rsqrtf(m2[k] * p.inv_n_cols + eps);
      } else if (norm == kNormBlockRms) {
        const float inv_b = 1.0f / static_cast<float>(p.norm_block);   // a power of two: exact
#pragma unroll
        for (int k = 0; k < 2; ++k) {
          brs[k][0] = rsqrtf(bsq[k][0] * inv_b + eps);
          brs[k][1] = rsqrtf(bsq[k][1] * inv_b + eps);
        }
      }
      // y = v * rstd - mean * rstd, then * gamma + beta when present
      const float nmr[2] = {-mean[0] * rstd[0], -mean[1] * rstd[1]};   // -0 for RMSNorm and BlockNorm
      const float2 rstd2[2] = {dup2(rstd[0]), dup2(rstd[1])};
      const float2 nmr2[2] = {dup2(nmr[0]), dup2(nmr[1])};
      // the column vectors of pair i of chunk c0 (1, 0 where absent)
      // post_tag: integral_constant<int, P>; P bit 0 = gamma/beta, bit 1 =
      // Hard Swish, bit 2 = BlockNorm
      auto colv = [&](auto post_tag, int c0, int i, float2& sw, float2& b, float2& gm, float2& be) {
        gm = make_float2(1.f, 1.f);
        be = make_float2(0.f, 0.f);
        sw = make_float2(1.f, 1.f);
        b = make_float2(0.f, 0.f);
        if constexpr ((decltype(post_tag)::value & 8) == 0) {
          sw = vec2(vec_sw, c0, i);
          b = vec2(vec_b, c0, i);
        }
        if constexpr ((decltype(post_tag)::value & 1) != 0) {
          gm = vec2(vec_g, c0, i);
          be = vec2(vec_be, c0, i);
        }
      };
      // the normalized pair of row k: the one arithmetic of every pass below
      // (rs: the row's 1/rms pair for this chunk, see chunk_rstd)
      auto ypair = [&](auto post_tag, const uint32_t (&r)[16], int k, int i, float2 rs, float2 sw, float2 b,
                       float2 gm, float2 be) {
        constexpr int POST = decltype(post_tag)::value;
        // bit 3: the chunk holds v already (written by the statistics pass)
        const float2 v = (POST & 8) != 0 ? acc2(r, k, i) : vpair(r, k, i, sx2[k], sw, b);
        float2 y = __ffma2_rn(v, rs, nmr2[k]);
        if constexpr ((POST & 1) != 0) y = __ffma2_rn(y, gm, be);
        if constexpr ((POST & 2) != 0) {
          // Hard Swish: y * min(max(y + 3, 0), 6) / 6
          const float2 t = __fadd2_rn(y, make_float2(3.0f, 3.0f));
          const float2 tc = make_float2(fminf(fmaxf(t.x, 0.0f), 6.0f), fminf(fmaxf(t.y, 0.0f), 6.0f));
          y = __fmul2_rn(__fmul2_rn(y, tc), make_float2(1.0f / 6.0f, 1.0f / 6.0f));
        }
        return y;
      };
      // 1/rms of both rows for chunk c as pairs: the row's, or (BlockNorm)
      // the chunk's block's, from the lane of the row group that keeps it
      auto chunk_rstd = [&](auto post_tag, int c, float2 (&rs)[2]) {
        if constexpr ((decltype(post_tag)::value & 4) != 0) {
          const int blk = c >> lcpb;
          const int src = (lane & ~3) | (blk & 3);
#pragma unroll
          for (int k = 0; k < 2; ++k)
            rs[k] = dup2(__shfl_sync(0xffffffffu, (blk & 4) ? brs[k][1] : brs[k][0], src));
        } else {
          rs[0] = rstd2[0];
          rs[1] = rstd2[1];
        }
      };
      // fn(post_tag) with the tag of this tile's group.  Without a norm there
      // is no statistics pass (v not stored) and no gamma, beta or blocks.
      auto with_tags = [&](auto&& fn) {
        const int post = (affine ? 1 : 0) | (act ? 2 : 0) | (norm == kNormBlockRms ? 4 : 0) | (norm != kNormNone ? 8 : 0);
        switch (post) {
          case 2: fn(std::integral_constant<int, 2>{}); break;
          case 8: fn(std::integral_constant<int, 8>{}); break;
          case 9: fn(std::integral_constant<int, 9>{}); break;
          case 10: fn(std::integral_constant<int, 10>{}); break;
          case 11: fn(std::integral_constant<int, 11>{}); break;
          case 12: fn(std::integral_constant<int, 12>{}); break;
          case 13: fn(std::integral_constant<int, 13>{}); break;
          case 14: fn(std::integral_constant<int, 14>{}); break;
          case 15: fn(std::integral_constant<int, 15>{}); break;
          default: fn(std::integral_constant<int, 0>{}); break;
        }
      };

      // E4M3 output with one scale per row: the row's amax over its bf16
      // outputs, then the standalone quantizer's scale selection, so the
      // codes and scale equal what it makes of the bf16 row (NaN outputs
      // never become the maximum there either).
      [[maybe_unused]] float qinv[2] = {1.f, 1.f};
      if constexpr (kQOut && CL == 1) {
        if (p.yq_mode == kScaleRow) {
          uint32_t am2[2] = {0u, 0u};   // |bf16| maxima, packed
          if (track) {
            // y = fma(v, rstd, -mean rstd) with rstd > 0 rounds a
            // nondecreasing function of v, and bf16 rounding keeps the
            // order: the row's largest and smallest outputs are those of
            // its largest and smallest v
#pragma unroll
            for (int k = 0; k < 2; ++k)
              am2[k] = absmax_bf16x2(0u, pack_bf16x2(__fmaf_rn(vhi[k], rstd[k], nmr[k]),
                                                     __fmaf_rn(vlo[k], rstd[k], nmr[k])));
          } else {
            auto amax_pass = [&](auto post_tag) {
              for_chunks(t_base, [&](const uint32_t (&r)[16], int c) {
                float2 rs[2];
                chunk_rstd(post_tag, c, rs);
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                  float2 sw, b, gm, be;
                  colv(post_tag, c * 32, i, sw, b, gm, be);
#pragma unroll
                  for (int k = 0; k < 2; ++k) {
                    const float2 y = ypair(post_tag, r, k, i, rs[k], sw, b, gm, be);
                    am2[k] = absmax_bf16x2(am2[k], pack_bf16x2(y.x, y.y));
                  }
                }
              });
            };
            with_tags([&](auto post_tag) { amax_pass(post_tag); });
          }
#pragma unroll
          for (int k = 0; k < 2; ++k) {
            // each lane's maximum covers its own columns; merge the row's 4
            float am = fmaxf(bf16lo(am2[k]), bf16hi(am2[k]));
            am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, 1));
            am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, 2));
            float sc;
            loka::row_scales(am, qinv[k], sc);
            if (cp == 0 && ok[k]) static_cast<float*>(G.yq_scales)[static_cast<int64_t>(m0) + rowk[k]] = sc;
          }
        }
      }

      // pass 2: normalize and store from registers (rows of a ragged last
      // tile are masked).  bf16: a chunk's 4 column pairs per row are packed,
      // transposed across the 4 lanes of the row group, and stored as one
      // 16-byte vector per lane (64 contiguous bytes per row per warp store)
      auto out_pass = [&](auto post_tag) {
        for_chunks(t_base, [&](const uint32_t (&r)[16], int c) {
          const int c0 = c * 32;
          float2 rs[2];
          chunk_rstd(post_tag, c, rs);
          [[maybe_unused]] uint32_t pk[2][4];
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            float2 sw, b, gm, be;
            colv(post_tag, c0, i, sw, b, gm, be);
#pragma unroll
            for (int k = 0; k < 2; ++k) {
              const float2 y = ypair(post_tag, r, k, i, rs[k], sw, b, gm, be);
              if constexpr (kBf16Out)
                pk[k][i] = pack_bf16x2(y.x, y.y);
              else
                st_global_pred_v2f32(rowp[k] + (c0 + 8 * i) * 4, y, ok[k]);
            }
          }
          if constexpr (kBf16Out) {
#pragma unroll
            for (int k = 0; k < 2; ++k) {
              transpose4_lanes(pk[k], cp);
              st_global_pred_v4b32(rowp[k] + c0 * 2, pk[k], ok[k]);
            }
          }
        });
      };
      // pass 2 of the quantized output kind: the bf16 pairs (stored too when
      // asked for) times the row's 448/amax, or, for MX, times 2^-e of the
      // chunk's 32 columns (one E8M0 block: the 4 lanes of the row merge
      // their maxima), cast to E4M3 with the quantizer's arithmetic.  The
      // code pairs of both rows ride one 4-lane transpose; each lane then
      // stores 8 contiguous codes per row.
      [[maybe_unused]] auto out_pass_q = [&](auto post_tag, auto mx_tag) {
        constexpr bool MXO = decltype(mx_tag)::value;
        for_chunks(t_base, [&](const uint32_t (&r)[16], int c) {
          const int c0 = c * 32;
          float2 rs[2];
          chunk_rstd(post_tag, c, rs);
          uint32_t pk[2][4];
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            float2 sw, b, gm, be;
            colv(post_tag, c0, i, sw, b, gm, be);
#pragma unroll
            for (int k = 0; k < 2; ++k) {
              const float2 y = ypair(post_tag, r, k, i, rs[k], sw, b, gm, be);
              pk[k][i] = pack_bf16x2(y.x, y.y);
            }
          }
          float mul[2] = {qinv[0], qinv[1]};
          if constexpr (MXO) {
#pragma unroll
            for (int k = 0; k < 2; ++k) {
              const uint32_t a2 = absmax_bf16x2(absmax_bf16x2(pk[k][0], pk[k][1]), absmax_bf16x2(pk[k][2], pk[k][3]));
              float am = fmaxf(0.0f, fmaxf(bf16lo(a2), bf16hi(a2)));
              am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, 1));
              am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, 2));
              const int e = mx_exponent(am);
              mul[k] = pow2_neg(e);
              if (cp == 0 && ok[k])
                static_cast<uint8_t*>(G.yq_scales)[(static_cast<int64_t>(m0) + rowk[k]) * (ng / 32) + (col0 + c0) / 32] =
                    static_cast<uint8_t>(e + 127);
            }
          }
          const float2 mul0 = dup2(mul[0]), mul1 = dup2(mul[1]);
          uint32_t w[4];
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const float2 f0 = __fmul2_rn(make_float2(bf16lo(pk[0][i]), bf16hi(pk[0][i])), mul0);
            const float2 f1 = __fmul2_rn(make_float2(bf16lo(pk[1][i]), bf16hi(pk[1][i])), mul1);
            w[i] = static_cast<uint32_t>(cvt_e4m3x2(f0.x, f0.y)) | (static_cast<uint32_t>(cvt_e4m3x2(f1.x, f1.y)) << 16);
          }
          if (has_y) {   // the bf16 rows too (after the codes: pk is transposed in place)
#pragma unroll
            for (int k = 0; k < 2; ++k) {
              transpose4_lanes(pk[k], cp);
              st_global_pred_v4b32(rowp[0] + k * (8 * ng * 2) + c0 * 2, pk[k], ok[k]);
            }
          }
          // lane cp now holds, in element t, the codes of columns 8 cp + 2t
          // and 8 cp + 2t + 1: row 0 in the low half, row 1 in the high half
          transpose4_lanes(w, cp);
          st_global_pred_v2b32(rowq + c0, (w[0] & 0xFFFFu) | (w[1] << 16), (w[2] & 0xFFFFu) | (w[3] << 16), ok[0]);
          st_global_pred_v2b32(rowq + 8 * ng + c0, (w[0] >> 16) | (w[1] & 0xFFFF0000u), (w[2] >> 16) | (w[3] & 0xFFFF0000u),
                               ok[1]);
        });
      };
      if constexpr (kQOut) {
        const bool mxo = p.yq_mode == kScaleMx32;
        with_tags([&](auto post_tag) {
          // per-row output scales need the whole row in one CTA (the host
          // allows them for CL == 1 only)
          if (CL > 1 || mxo) out_pass_q(post_tag, std::true_type{});
          else if constexpr (CL == 1) out_pass_q(post_tag, std::false_type{});
        });
      } else {
        with_tags([&](auto post_tag) { out_pass(post_tag); });
      }
      // all of this warp's reads of the accumulator are done
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&tempty[buf]));
    }
  };

  if constexpr (kQx) {
    // Each warpgroup takes its register share in its own branch and the
    // branches never meet again: no barrier without a time limit.  The
    // epilogue warps report their last tensor-memory read on epi_done; the
    // MMA warp waits for it (bounded) and frees tensor memory; everyone else
    // just leaves.
    if (warp < kQxFirstWarp) {
      regs_dec<kQxRegsLow>();
      if (!misaligned) {
        if (warp == 0) run_producer();
        else if (warp == 1) run_mma();
      }
      if (warp == 1) {
        if (lane == 0) {
          const bool done = wait_parity_drain(wd, smem_u32(epi_done), 0);
          if (!done) atomicOr(p.status, kErrTeardownWait);
        }
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem_base, kTmemCols);
      }
    } else if (warp < kQxEpiWarp) {
      regs_dec<kQxRegsQuant>();
      if (!misaligned) run_quantizer();
    } else {
      regs_inc<kQxRegsEpi>();
      if (!misaligned) run_epilogue();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(epi_done));
    }
    return;
  } else {
    // every warpgroup takes its register share in its own branch (no
    // barrier in between); a misaligned CTA skips all work but still meets
    // the teardown barriers
    if (warp < EPI0) {
      regs_dec<kRegsLow>();
      if (!misaligned) {
        if (warp == 0) run_producer();
        else if (warp == 1) run_mma();
      }
    } else {
      regs_inc<kRegsEpi>();
      if (!misaligned) run_epilogue();
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem_base, kTmemCols);
  // partners may still write statistics into this CTA's shared memory until
  // they are done: leave together
  if (CL > 1) cluster_sync_all();
}

// Picks resident W when it fits and leaves at least three A stages.
struct Plan {
  bool resident;
  int stages;
  size_t smem;
};

Plan plan_for(int N, int K, int elem_bytes, bool mx, int cl) {
  Plan pl{false, 0, 0};
  const size_t w_bytes = static_cast<size_t>(N) * K * elem_bytes;
  for (int pass = 0; pass < 2; ++pass) {
    const bool resident = pass == 0;
    if (resident && w_bytes > kResidentWLimit) continue;
    const Layout base = make_layout(N, K, elem_bytes, resident, 0, mx, cl);
    const size_t fixed = base.total;
    const size_t per_stage = base.stage_bytes;
    if (fixed + 2 * per_stage > kSmemLimit) continue;
    int st = static_cast<int>((kSmemLimit - fixed) / per_stage);
    if (st > kMaxStages) st = kMaxStages;
    if (resident && st < 3) continue;
    pl.resident = resident;
    pl.stages = st;
    pl.smem = fixed + static_cast<size_t>(st) * per_stage;
    return pl;
  }
  return pl;
}

template <int N, int CL, int OP, int OUT, bool RES>
cudaError_t launch_one(const GemmParams& p, size_t smem, int sms, cudaStream_t stream) {
  auto kern = gemm_norm_kernel<N, CL, OP, OUT, RES>;
  // the shared-memory opt-in is set once per device (it is not a stream
  // operation, so it also stays out of captured CUDA graphs)
  static std::atomic<uint64_t> configured{0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const uint64_t bit = uint64_t(1) << (dev & 63);
  if (!(configured.load() & bit)) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(kSmemLimit));
    if (e != cudaSuccess) return e;
    // the warpgroups' setmaxnreg shares must fit in the registers the CTA
    // is launched with, or an increase would wait forever: refuse instead
    cudaFuncAttributes fa{};
    e = cudaFuncGetAttributes(&fa, kern);
    if (e != cudaSuccess) return e;
    const long launch_regs = static_cast<long>(fa.numRegs) * (OP == static_cast<int>(OperandKind::kE4M3Qx) ? kQxThreads : kThreads);
    const long shares = OP == static_cast<int>(OperandKind::kE4M3Qx)
                            ? 4L * 32 * kQxRegsLow + static_cast<long>(kQxWarps) * 32 * kQxRegsQuant + 16L * 32 * kQxRegsEpi
                            : 4L * 32 * kRegsLow + 16L * 32 * kRegsEpi;
    if (shares > launch_regs) return cudaErrorInvalidConfiguration;
    if (CL > 1) {
      e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 0);
      if (e != cudaSuccess) return e;
    }
    configured.fetch_or(bit);
  }
  // units: clusters of CL CTAs, or groups of p.slices CTAs (one per slice)
  const int per_unit = CL > 1 ? CL : p.slices;
  int clusters = sms / per_unit;
  cudaLaunchConfig_t cfg = {};
  cfg.blockDim = dim3(OP == static_cast<int>(OperandKind::kE4M3Qx) ? kQxThreads : kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = CL;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  // the prologue may overlap the tail of the quantizer launched before
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  if (CL > 1) {
    // a cluster's CTAs share one GPC, so fewer than sms / CL clusters may be
    // resident at once; the persistent grid takes no more than fit (per
    // device and shared-memory size, asked once)
    static std::atomic<uint64_t> fit[64];
    const uint64_t key = static_cast<uint64_t>(smem) << 20;
    uint64_t cached = fit[dev & 63].load();
    if ((cached & ~uint64_t(0xFFFFF)) != key) {
      int n = 0;
      cfg.gridDim = dim3(static_cast<unsigned>(clusters * CL));
      e = cudaOccupancyMaxActiveClusters(&n, kern, &cfg);
      if (e != cudaSuccess) return e;
      cached = key | static_cast<uint64_t>(n > 0 ? n : 1);
      fit[dev & 63].store(cached);
    }
    const int n = static_cast<int>(cached & 0xFFFFF);
    if (n < clusters) clusters = n;
  }
  if (p.total_tiles < clusters) clusters = p.total_tiles;
  if (clusters < 1) return cudaSuccess;
  cfg.gridDim = dim3(static_cast<unsigned>(clusters * per_unit));
  e = cudaLaunchKernelEx(&cfg, kern, p);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

// In-kernel quantization: K = 256 or 512 (a 1 KB staging unit is one row of
// K = 512 or two of K = 256, so a lane's two 16-byte pieces cover it), W
// resident.  Each of the 12 quantizer warps gets `stages` slots, at least 5
// (60 KB of X in flight per SM); two A tiles when they fit beside that, else
// one.
struct QxPlan {
  int a_bufs, stages;
  size_t smem;
};

inline QxPlan plan_qx(int N, int K) {
  QxPlan q{0, 0, 0};
  if ((K != 256 && K != 512) || N > 256) return q;
  if (static_cast<size_t>(N) * K > kResidentWLimit) return q;
  constexpr int kMinSlots = 5;
  const size_t per_slot = static_cast<size_t>(kQxWarps) * kQxSlotBytes;
  for (int a = 2; a >= 1; --a) {
    const Layout base = make_layout(N, K, 1, true, 0, false, 1, a);
    if (base.total + kMinSlots * per_slot > kSmemLimit) continue;
    int st = static_cast<int>((kSmemLimit - base.total) / per_slot);
    if (st > kQxMaxSlots) st = kQxMaxSlots;
    q.a_bufs = a;
    q.stages = st;
    q.smem = base.total + static_cast<size_t>(st) * per_slot;
    return q;
  }
  return q;
}

template <int N, int CL, int OP, int OUT>
cudaError_t launch_res(const GemmParams& p, const Plan& pl, int sms, cudaStream_t stream) {
  return pl.resident ? launch_one<N, CL, OP, OUT, true>(p, pl.smem, sms, stream)
                     : launch_one<N, CL, OP, OUT, false>(p, pl.smem, sms, stream);
}

// (columns per CTA, cluster size) of an output row of N columns (a multiple
// of 32 up to 2048) when its statistics span the row: up to 256 columns one
// CTA of the next instantiated width (64, 128, 192, 256); wider, a cluster of
// 2, 4 or 8 CTAs of 256 columns, the last ones holding the remainder (or
// nothing).
bool split_n(int N, int* local, int* cl) {
  if (N < 32 || N > 2048 || N % 32 != 0) return false;
  if (N <= 256) {
    *local = N <= 64 ? 64 : (N <= 128 ? 128 : (N <= 192 ? 192 : 256));
    *cl = 1;
  } else {
    *local = 256;
    *cl = N <= 512 ? 2 : (N <= 1024 ? 4 : 8);
  }
  return true;
}


// Plans shared memory and launches gemm_norm_kernel<LN, CL, OP, OUT> (LN =
// the columns one CTA owns).
template <int OP, int OUT, int LN, int CL>
cudaError_t launch_planned(GemmParams& p, int sms, cudaStream_t stream) {
  // W's TMA box must be one CTA's columns: the kernel's B slots hold LN rows
  for (int g = 0; g < p.num_groups; ++g)
    if (p.g[g].M > 0 && p.g[g].b_box_rows != LN) return cudaErrorInvalidValue;
  const int eb = OP == static_cast<int>(OperandKind::kBf16) ? 2 : 1;
  const Plan pl = plan_for(LN, p.K, eb, OP == static_cast<int>(OperandKind::kMxE4M3), CL);
  if (pl.stages == 0) return cudaErrorInvalidValue;
  p.stages = pl.stages;
  return launch_res<LN, CL, OP, OUT>(p, pl, sms, stream);
}

// Output rows of at most 256 columns: one CTA per tile.
template <int OP, int OUT>
cudaError_t launch_narrow(GemmParams& p, int N, int sms, cudaStream_t stream) {
  switch (N) {
    case 64: return launch_planned<OP, OUT, 64, 1>(p, sms, stream);
    case 128: return launch_planned<OP, OUT, 128, 1>(p, sms, stream);
    case 192: return launch_planned<OP, OUT, 192, 1>(p, sms, stream);
    case 256: return launch_planned<OP, OUT, 256, 1>(p, sms, stream);
    default: return cudaErrorInvalidValue;
  }
}

// Wider rows: a cluster of N / 256 CTAs per tile.
template <int OP, int OUT>
cudaError_t launch_wide(GemmParams& p, int N, int sms, cudaStream_t stream) {
  switch (N) {
    case 512: return launch_planned<OP, OUT, 256, 2>(p, sms, stream);
    case 1024: return launch_planned<OP, OUT, 256, 4>(p, sms, stream);
    case 2048: return launch_planned<OP, OUT, 256, 8>(p, sms, stream);
    default: return cudaErrorInvalidValue;
  }
}

template <int OP, int OUT>
cudaError_t launch_kind(GemmParams& p, int N, int sms, cudaStream_t stream) {
  return N <= 256 ? launch_narrow<OP, OUT>(p, N, sms, stream) : launch_wide<OP, OUT>(p, N, sms, stream);
}

}  // namespace

// One per instantiation file (gemm_e4m3.cu, gemm_bf16.cu, gemm_mx.cu and
// gemm_qout_{e4m3,mx}{,_wide}.cu).
cudaError_t launch_gemm_e4m3(GemmParams& p, int N, OutKind out, int sms, cudaStream_t stream);
cudaError_t launch_gemm_bf16(GemmParams& p, int N, OutKind out, int sms, cudaStream_t stream);
cudaError_t launch_gemm_mx(GemmParams& p, int N, OutKind out, int sms, cudaStream_t stream);
cudaError_t launch_gemm_qout_e4m3(GemmParams& p, int N, int sms, cudaStream_t stream);
cudaError_t launch_gemm_qout_e4m3_wide(GemmParams& p, int N, int sms, cudaStream_t stream);
cudaError_t launch_gemm_qout_mx(GemmParams& p, int N, int sms, cudaStream_t stream);
cudaError_t launch_gemm_qout_mx_wide(GemmParams& p, int N, int sms, cudaStream_t stream);
cudaError_t launch_gemm_qx(GemmParams& p, int N, int sms, cudaStream_t stream);

}  // namespace loka
