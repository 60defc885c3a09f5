// Dispatch of the fused FP8 GEMM + normalization kernel (gemm_norm.cuh) to
// the files that instantiate it for each operand and output kind, and the
// shared-memory feasibility check the host validation uses.
#include "gemm_norm.cuh"

namespace loka {

bool gemm_supported(int N, int K, OperandKind op) {
  int local = 0, cl = 0;
  if (!split_n(N, &local, &cl)) return false;
  return plan_for(local, K, op == OperandKind::kBf16 ? 2 : 1, op == OperandKind::kMxE4M3, cl).stages > 0;
}

bool split_n_host(int N, int* local, int* cl) { return split_n(N, local, cl); }

bool gemm_qx_supported(int N, int K, int norm, OutKind out) {
  const GemmRoute r = gemm_route(N, norm);
  if (out != OutKind::kBf16 || r.cl != 1 || r.slices != 1) return false;
  // Chosen only where it measured no slower than quantizer + GEMM: W
  // resident beside two A tiles at 256 columns per CTA (K = 256, the
  // ensemble layers: equal in the step, 2% faster with static W).  With one
  // A tile (K = 512) the quantizer warps wait for every tile's MMAs (48 vs
  // 35 us on the rec-MLP layer), and at 64 columns per CTA the quantizer
  // warps outweigh the short epilogue (75.7 vs 63.3 us at M = 262144,
  // K = 256, N = 64).
  const QxPlan q = plan_qx(r.local, K);
  return r.local == 256 && q.stages > 0 && q.a_bufs == 2;
}

GemmRoute gemm_route(int N, int norm) {
  const bool no_row_stat = norm == kNormNone || norm == kNormBlockRms;
  int local = 0, cl = 0;
  if (!split_n(N, &local, &cl)) return GemmRoute{0, 0, 0};
  // Rows wider than one CTA whose epilogue needs no row statistic (no norm,
  // or BlockNorm, whose blocks lie within a CTA's 256 columns) run as
  // independent 256-column slices, the last one partial: no cluster
  // co-scheduling, every SM busy.
  if (N > 256 && no_row_stat) return GemmRoute{256, 1, (N + 255) / 256};
  return GemmRoute{local, cl, 1};
}

cudaError_t launch_gemm_norm(GemmParams& p, int N, OperandKind op, OutKind out, int sms, cudaStream_t stream) {
  const GemmRoute r = gemm_route(N, p.norm);
  if (r.local == 0) return cudaErrorInvalidValue;
  p.slices = r.slices;
  p.n_cols = N;
  p.inv_n_cols = 1.0f / static_cast<float>(N);
  for (int j = 0; j < 8; ++j) {
    const int left = N - j * 256;
    const float na = static_cast<float>(j * 256);
    const float nb = static_cast<float>(left <= 0 ? 0 : (left > 256 ? 256 : left));
    const float w = nb > 0.0f ? nb / (na + nb) : 0.0f;
    p.chan_w[j] = w;
    p.chan_c[j] = na * w;
  }
  // the launchers take the kernel's width: up to 256 one CTA, wider a
  // cluster of r.cl CTAs of 256 columns
  N = r.cl > 1 ? r.cl * 256 : r.local;
  if (out == OutKind::kQuant) {
    const bool wide = N > 256;
    if (op == OperandKind::kE4M3)
      return wide ? launch_gemm_qout_e4m3_wide(p, N, sms, stream) : launch_gemm_qout_e4m3(p, N, sms, stream);
    if (op == OperandKind::kMxE4M3)
      return wide ? launch_gemm_qout_mx_wide(p, N, sms, stream) : launch_gemm_qout_mx(p, N, sms, stream);
    return cudaErrorInvalidValue;
  }
  switch (op) {
    case OperandKind::kE4M3: return launch_gemm_e4m3(p, N, out, sms, stream);
    case OperandKind::kBf16: return launch_gemm_bf16(p, N, out, sms, stream);
    case OperandKind::kMxE4M3: return launch_gemm_mx(p, N, out, sms, stream);
    case OperandKind::kE4M3Qx: return out == OutKind::kBf16 ? launch_gemm_qx(p, N, sms, stream) : cudaErrorInvalidValue;
  }
  return cudaErrorInvalidValue;
}

}  // namespace loka
