// Instantiations of the fused GEMM + normalization kernel that quantizes its
// bf16 activations per row itself (OperandKind::kE4M3Qx: the codes go from
// the quantizer warps straight into the shared-memory A tile), with E4M3
// weights kept resident and bf16 output.  Rows of at most 256 columns.
#include "gemm_norm.cuh"

namespace loka {

namespace {

template <int N>
cudaError_t launch_qx_n(GemmParams& p, int sms, cudaStream_t stream) {
  for (int g = 0; g < p.num_groups; ++g)
    if (p.g[g].M > 0 && p.g[g].b_box_rows != N) return cudaErrorInvalidValue;
  const QxPlan q = plan_qx(N, p.K);
  if (q.stages == 0) return cudaErrorInvalidValue;
  p.stages = q.stages;
  p.a_bufs = q.a_bufs;
  return launch_one<N, 1, static_cast<int>(OperandKind::kE4M3Qx), static_cast<int>(OutKind::kBf16), true>(
      p, q.smem, sms, stream);
}

}  // namespace

cudaError_t launch_gemm_qx(GemmParams& p, int N, int sms, cudaStream_t stream) {
  switch (N) {
    case 64: return launch_qx_n<64>(p, sms, stream);
    case 128: return launch_qx_n<128>(p, sms, stream);
    case 192: return launch_qx_n<192>(p, sms, stream);
    case 256: return launch_qx_n<256>(p, sms, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace loka
