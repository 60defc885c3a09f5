// Instantiations of the fused GEMM + normalization kernel whose epilogue
// also quantizes its bf16 output rows to E4M3 (per-row or MX 1x32 scales)
// for the next layer: MX 1x32 E4M3 operands,
// rows of 512 to 2048 columns (thread-block clusters).
#include "gemm_norm.cuh"

namespace loka {

cudaError_t launch_gemm_qout_mx_wide(GemmParams& p, int N, int sms, cudaStream_t stream) {
  constexpr int op = static_cast<int>(OperandKind::kMxE4M3);
  return launch_wide<op, static_cast<int>(OutKind::kQuant)>(p, N, sms, stream);
}

}  // namespace loka
