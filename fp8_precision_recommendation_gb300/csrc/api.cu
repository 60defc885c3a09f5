// C ABI of the library (declared in include/loka.h): argument validation,
// workspace layout, TMA descriptor encoding and launch sequencing.  Every
// step of the computation runs in the kernels of quantize.cu, gemm_norm.cu
// and probe.cu; this file does host bookkeeping only and has no fallback.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <string>
#include <vector>

#include "loka.h"
#include "loka_internal.h"

namespace loka {
namespace {

// Device status word: kernels OR an error code into it when a wait gives up.
__device__ unsigned g_status_word;

thread_local std::string t_last_error;

loka_status fail(loka_status s, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  t_last_error = buf;
  return s;
}

loka_status cuda_fail(cudaError_t e, const char* what) {
  return fail(LOKA_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

constexpr uint64_t kDefaultWaitLimitNs = 2000000000ull;   // 2 s: far above any legitimate wait

struct DeviceInfo {
  bool ready = false;
  int sms = 0;
  unsigned* status = nullptr;
};

std::mutex g_mu;
DeviceInfo g_dev[64];

loka_status device_info(DeviceInfo** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev < 0 || dev >= 64) return fail(LOKA_ERR_UNSUPPORTED, "device ordinal %d out of range", dev);
  std::lock_guard<std::mutex> lock(g_mu);
  DeviceInfo& d = g_dev[dev];
  if (!d.ready) {
    int major = 0, minor = 0;
    cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
    cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
    if (major != 10 || minor != 3)
      return fail(LOKA_ERR_UNSUPPORTED, "device %d is sm_%d%d; this library is built for sm_103a only", dev, major, minor);
    e = cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceGetAttribute");
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_status_word);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(status)");
    d.status = static_cast<unsigned*>(p);
    d.ready = true;
  }
  *out = &d;
  return LOKA_OK;
}

// Built-in scratch for loka_fp8_linear_norm_static, for callers that cannot
// allocate device memory.  A file-scope __device__ array: every GPU that
// loads this library holds these bytes until the process exits.
constexpr size_t kStaticScratchBytes = size_t(4) << 20;   // 4 MiB
__device__ __align__(256) unsigned char g_static_scratch[kStaticScratchBytes];

void* g_static_scratch_addr[64];

// Device address of the built-in scratch on the current device.  In host code
// the array's name is only a host-side stand-in, so the address is looked up
// once per device, with that device current, and cached.
loka_status static_scratch(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev < 0 || dev >= 64) return fail(LOKA_ERR_UNSUPPORTED, "device ordinal %d out of range", dev);
  std::lock_guard<std::mutex> lock(g_mu);
  if (g_static_scratch_addr[dev] == nullptr) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_static_scratch);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(static scratch)");
    g_static_scratch_addr[dev] = p;
  }
  *out = g_static_scratch_addr[dev];
  return LOKA_OK;
}

// ------------------------------------------------------------ tensor maps
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// 2-D row-major tensor [outer, inner] with a 128-byte-wide, 128B-swizzled box
// (box_inner = 0), or an unswizzled box of box_inner elements.
loka_status encode_2d(CUtensorMap* m, CUtensorMapDataType dt, int elem_bytes, const void* base, uint64_t inner,
                      uint64_t outer, uint32_t box_outer, uint32_t box_inner = 0) {
  auto fn = encode_fn();
  if (fn == nullptr) return fail(LOKA_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {inner * static_cast<uint64_t>(elem_bytes)};
  cuuint32_t box[2] = {box_inner > 0 ? box_inner : static_cast<cuuint32_t>(128 / elem_bytes), box_outer};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(m, dt, 2, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  box_inner > 0 ? CU_TENSOR_MAP_SWIZZLE_NONE : CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(LOKA_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", static_cast<int>(r));
  return LOKA_OK;
}

// ------------------------------------------------------------- workspace
constexpr size_t kAlign = 256;
size_t align_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

size_t scale_bytes(int mode, int64_t rows, int64_t cols) {
  if (mode == kScaleTensor) return sizeof(float);
  if (mode == kScaleRow) return static_cast<size_t>(rows) * sizeof(float);
  if (mode == kScaleMx32) return static_cast<size_t>(rows) * static_cast<size_t>(cols / 32);
  if (mode == kScaleBlock32) return static_cast<size_t>((rows + 31) / 32) * static_cast<size_t>(cols / 32);
  return 0;
}

// Columns the GEMM's CTAs span for an output row of N: the kernel width up
// to 256, else the cluster's (or slices') 256-column CTAs.
int64_t padded_cols(int64_t N) {
  int local = 0, cl = 0;
  if (!split_n_host(static_cast<int>(N), &local, &cl)) return N;
  return N <= 256 ? local : ((N + 255) / 256 > cl ? (N + 255) / 256 : cl) * 256;
}

struct OperandSlots {   // workspace offsets of one group's quantized operands
  size_t xq, sx, wq, sw, amax;
  size_t sx_tc, sw_tc;   // MX: scale codes in the tensor-memory copy layout
};

// Lays out the quantized operands of every group; returns the total bytes.
size_t layout_operands(const loka_linear_desc* d, int n, std::vector<OperandSlots>* slots) {
  size_t off = 0;
  if (slots) slots->assign(n, OperandSlots{0, 0, 0, 0, 0, 0, 0});
  for (int i = 0; i < n; ++i) {
    OperandSlots s{0, 0, 0, 0, 0, 0, 0};
    if (d[i].mode != kBf16) {
      if (!d[i].x_is_fp8) {
        s.xq = off;
        off = align_up(off + static_cast<size_t>(d[i].M) * d[i].K);
        s.sx = off;
        off = align_up(off + scale_bytes(d[i].mode, d[i].M, d[i].K));
      }
      if (!d[i].w_is_fp8) {
        s.wq = off;
        off = align_up(off + static_cast<size_t>(d[i].N) * d[i].K);
        s.sw = off;
        off = align_up(off + scale_bytes(d[i].mode, d[i].N, d[i].K));
      }
      if (d[i].mode == kScaleTensor) {
        s.amax = off;
        off = align_up(off + 2 * sizeof(unsigned));
      }
      if (d[i].mode == kScaleMx32 || d[i].mode == kScaleBlock32) {
        s.sx_tc = off;
        off = align_up(off + static_cast<size_t>(sf_tc_bytes(d[i].M, d[i].K)));
        s.sw_tc = off;
        // the CTAs load whole 128-row blocks of W's codes for all the columns
        // they span, past N when the row does not fill them
        off = align_up(off + static_cast<size_t>(sf_tc_bytes(padded_cols(d[i].N), d[i].K)));
      }
    }
    if (slots) (*slots)[i] = s;
  }
  return off;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

OperandKind operand_kind(int mode) {
  if (mode == kBf16) return OperandKind::kBf16;
  // square 32x32 blocks use the block-scaled MMA like MX: each row takes its block row's scales
  return (mode == kScaleMx32 || mode == kScaleBlock32) ? OperandKind::kMxE4M3 : OperandKind::kE4M3;
}

// The group whose output fields (y_q, y_q_mode) speak for the call: the
// first with rows (an empty group's tensors may have no storage at all).
const loka_linear_desc& output_reference(const loka_linear_desc* d, int n) {
  for (int i = 0; i < n; ++i)
    if (d[i].M > 0) return d[i];
  return d[0];
}

loka_status validate(const loka_linear_desc* d, int n, bool probe) {
  if (d == nullptr) return fail(LOKA_ERR_INVALID_ARG, "descs is NULL");
  if (n < 1 || n > kMaxGroups) return fail(LOKA_ERR_INVALID_ARG, "num_groups %d not in [1, %d]", n, kMaxGroups);
  const loka_linear_desc& a = d[0];
  if (!(a.eps >= 0.0f) || !std::isfinite(a.eps)) return fail(LOKA_ERR_INVALID_ARG, "eps must be finite and >= 0");
  for (int i = 0; i < n; ++i) {
    const loka_linear_desc& g = d[i];
    if (g.N != a.N || g.K != a.K || g.mode != a.mode || g.norm != a.norm || g.eps != a.eps ||
        g.x_is_fp8 != a.x_is_fp8 || g.w_is_fp8 != a.w_is_fp8 || g.act != a.act ||
        (a.norm == kNormBlockRms && g.norm_block != a.norm_block))
      return fail(LOKA_ERR_UNSUPPORTED,
                  "group %d differs from group 0 in N, K, mode, norm, norm_block, eps, act or operand kind", i);
    if (g.M < 0) return fail(LOKA_ERR_INVALID_ARG, "group %d: M = %lld < 0", i, static_cast<long long>(g.M));
    if (g.M > (int64_t(1) << 31)) return fail(LOKA_ERR_UNSUPPORTED, "group %d: M too large", i);
  }
  if (a.mode < 0 || a.mode > kScaleBlock32)
    return fail(LOKA_ERR_INVALID_ARG, "mode %d is not a LOKA_SCALE_* value", a.mode);
  if (a.norm < 0 || a.norm > kNormBlockRms)
    return fail(LOKA_ERR_INVALID_ARG, "norm %d is not a LOKA_NORM_* value", a.norm);
  if (a.act != kActNone && a.act != kActHardSwish)
    return fail(LOKA_ERR_INVALID_ARG, "act %d is not a LOKA_ACT_* value", a.act);
  if (a.norm == kNormBlockRms) {
    const int b = a.norm_block;
    if (b != 32 && b != 64 && b != 128 && b != 256)
      return fail(LOKA_ERR_UNSUPPORTED, "norm_block %d: BlockNorm blocks are 32, 64, 128 or 256 columns", b);
    if (a.N % b != 0)
      return fail(LOKA_ERR_INVALID_ARG, "norm_block %d does not divide N = %lld", b, static_cast<long long>(a.N));
  }
  if (a.K < 32 || a.K % 32 != 0)
    return fail(LOKA_ERR_UNSUPPORTED, "K = %lld: K must be a positive multiple of 32", static_cast<long long>(a.K));
  if (a.K > (int64_t(1) << 20)) return fail(LOKA_ERR_UNSUPPORTED, "K too large");
  if (a.N < 32 || a.N > 2048 || a.N % 32 != 0)
    return fail(LOKA_ERR_UNSUPPORTED, "N = %lld: N must be a multiple of 32 in [32, 2048]", static_cast<long long>(a.N));
  if (!gemm_supported(static_cast<int>(a.N), static_cast<int>(a.K), operand_kind(a.mode)) ||
      (probe && !gemm_supported(static_cast<int>(a.N), static_cast<int>(a.K), OperandKind::kBf16)))
    return fail(LOKA_ERR_UNSUPPORTED, "no shared-memory plan for N = %lld, K = %lld", static_cast<long long>(a.N),
                static_cast<long long>(a.K));
  if (a.mode == kBf16 && (a.x_is_fp8 || a.w_is_fp8))
    return fail(LOKA_ERR_INVALID_ARG, "LOKA_BF16 takes bf16 operands (x_is_fp8 = w_is_fp8 = 0)");
  if (probe && (a.x_is_fp8 || a.w_is_fp8))
    return fail(LOKA_ERR_INVALID_ARG, "the error probe needs bf16 x and w (it runs the high-precision reference too)");
  // quantized output for the next layer (the probe writes its own outputs);
  // empty groups carry no output pointers
  const loka_linear_desc& r = output_reference(d, n);
  const bool qout = !probe && r.y_q != nullptr;
  if (!probe) {
    for (int i = 0; i < n; ++i)
      if (d[i].M > 0 && ((d[i].y_q != nullptr) != qout || (qout && d[i].y_q_mode != r.y_q_mode)))
        return fail(LOKA_ERR_UNSUPPORTED, "group %d: set y_q (with one y_q_mode) in every group or in none", i);
  }
  if (qout) {
    if (a.mode == kBf16) return fail(LOKA_ERR_UNSUPPORTED, "y_q is produced by the FP8 modes, not LOKA_BF16");
    if (r.y_q_mode == kScaleTensor)
      return fail(LOKA_ERR_UNSUPPORTED,
                  "y_q_mode LOKA_SCALE_TENSOR: a tensor-wide scale needs every row's amax before the first code "
                  "(use LOKA_SCALE_ROW or LOKA_SCALE_MX32)");
    if (r.y_q_mode != kScaleRow && r.y_q_mode != kScaleMx32)
      return fail(LOKA_ERR_INVALID_ARG, "y_q_mode %d is not a LOKA_SCALE_* value", r.y_q_mode);
    if (r.y_q_mode == kScaleRow && a.N > 256)
      return fail(LOKA_ERR_UNSUPPORTED, "y_q_mode LOKA_SCALE_ROW needs N <= 256 (a row within one thread block)");
  }
  for (int i = 0; i < n; ++i) {
    const loka_linear_desc& g = d[i];
    if (g.M == 0) continue;
    if (g.x == nullptr || g.w == nullptr || (!probe && !qout && g.y == nullptr))
      return fail(LOKA_ERR_INVALID_ARG, "group %d: x, w and y must not be NULL", i);
    if (!aligned16(g.x) || !aligned16(g.w) || (!probe && !aligned16(g.y)))
      return fail(LOKA_ERR_INVALID_ARG, "group %d: x, w and y must be 16-byte aligned", i);
    if (qout) {
      if (g.y_q_scales == nullptr) return fail(LOKA_ERR_INVALID_ARG, "group %d: y_q_scales is NULL", i);
      if (!aligned16(g.y_q)) return fail(LOKA_ERR_INVALID_ARG, "group %d: y_q must be 16-byte aligned", i);
      if (r.y_q_mode == kScaleRow && (reinterpret_cast<uintptr_t>(g.y_q_scales) & 3u))
        return fail(LOKA_ERR_INVALID_ARG, "group %d: y_q_scales must be 4-byte aligned", i);
    }
    if (g.x_is_fp8 && g.x_scales == nullptr) return fail(LOKA_ERR_INVALID_ARG, "group %d: x_scales is NULL", i);
    if (g.w_is_fp8 && g.w_scales == nullptr) return fail(LOKA_ERR_INVALID_ARG, "group %d: w_scales is NULL", i);
  }
  return LOKA_OK;
}

// Builds the GEMM launch parameters for the groups; `slots` gives the
// workspace locations of operands quantized by this call (bf16 inputs).
loka_status build_gemm(const loka_linear_desc* d, int n, const std::vector<OperandSlots>& slots, uint8_t* ws,
                       bool bf16_operands, OutKind out, void* const* y_override, int norm, DeviceInfo* dev,
                       GemmParams* p) {
  std::memset(p, 0, sizeof(*p));
  const int mode = d[0].mode;
  int tiles = 0;
  for (int i = 0; i < n; ++i) {
    const loka_linear_desc& g = d[i];
    GemmGroup& G = p->g[i];
    G.M = g.M;
    G.tile_begin = tiles;
    tiles += static_cast<int>((g.M + 127) / 128);
    const uint16_t* bias = static_cast<const uint16_t*>(g.bias);
    G.bias = bias;
    G.gamma = static_cast<const uint16_t*>(g.gamma);
    G.beta = static_cast<const uint16_t*>(g.beta);
    void* y = y_override ? y_override[i] : g.y;
    G.y = y;
    if (g.M == 0) continue;
    loka_status s;
    // W's box: the columns one CTA owns under the launch's route
    const int box = gemm_route(static_cast<int>(g.N), norm).local;
    G.b_box_rows = box;
    if (bf16_operands) {
      if ((s = encode_2d(&G.tm_a, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, g.x, g.K, g.M, 128)) != LOKA_OK) return s;
      if ((s = encode_2d(&G.tm_b, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, g.w, g.K, g.N, box)) != LOKA_OK) return s;
    } else {
      const void* xq = g.x_is_fp8 ? g.x : ws + slots[i].xq;
      const void* wq = g.w_is_fp8 ? g.w : ws + slots[i].wq;
      const void* sx = g.x_is_fp8 ? g.x_scales : ws + slots[i].sx;
      const void* sw = g.w_is_fp8 ? g.w_scales : ws + slots[i].sw;
      if ((s = encode_2d(&G.tm_a, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, xq, g.K, g.M, 128)) != LOKA_OK) return s;
      if ((s = encode_2d(&G.tm_b, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, wq, g.K, g.N, box)) != LOKA_OK) return s;
      if (mode == kScaleMx32 || mode == kScaleBlock32) {   // the block scales are applied inside the MMA
        G.sfa_tc = ws + slots[i].sx_tc;
        G.sfb_tc = ws + slots[i].sw_tc;
      } else {
        G.sx = static_cast<const float*>(sx);
        G.sw = static_cast<const float*>(sw);
        G.sx_per_row = mode == kScaleRow;
        G.sw_per_row = mode == kScaleRow;
      }
    }
    if (out == OutKind::kQuant) {
      G.yq = static_cast<uint8_t*>(g.y_q);
      G.yq_scales = g.y_q_scales;
    }
  }
  p->num_groups = n;
  p->total_tiles = tiles;
  p->K = static_cast<int32_t>(d[0].K);
  p->norm = norm;
  p->eps = d[0].eps;
  p->status = dev->status;
  p->wait_limit_ns = kDefaultWaitLimitNs;
  p->yq_mode = out == OutKind::kQuant ? output_reference(d, n).y_q_mode : 0;
  p->norm_block = norm == kNormBlockRms ? d[0].norm_block : 256;
  // the probe's pre-norm (and the statistics') fp32 outputs take no activation
  p->act = (out == OutKind::kF32 && norm == kNormNone) ? kActNone : d[0].act;
  p->slices = 1;
  return LOKA_OK;
}

// Block-scaled operands whose K is not a multiple of 128: the tensor-memory
// copy of their scale codes has a partial last K block, whose codes past K
// must be finite (the MMA multiplies the zeros read past K by them), so the
// whole copy starts as E8M0 127 (2^0) before the real codes are written.
cudaError_t pad_scale_codes(uint8_t* sf_tc, int64_t rows, int64_t cols, cudaStream_t stream) {
  if (sf_tc == nullptr || cols % 128 == 0 || rows == 0) return cudaSuccess;
  return cudaMemsetAsync(sf_tc, 127, static_cast<size_t>(sf_tc_bytes(rows, cols)), stream);
}

// Quantizes every bf16 operand of the groups into the workspace (one launch
// for X and W of all groups; tensorwise scaling takes an amax launch first).
// w_only: the weights alone (the GEMM quantizes X itself).
loka_status quantize_operands(const loka_linear_desc* d, int n, const std::vector<OperandSlots>& slots, uint8_t* ws,
                              DeviceInfo* dev, cudaStream_t stream, bool w_only = false) {
  QuantJobs jobs;
  std::memset(&jobs, 0, sizeof(jobs));
  int64_t rows = 0;
  for (int i = 0; i < n; ++i) {
    const loka_linear_desc& g = d[i];
    if (!w_only && !g.x_is_fp8 && g.M > 0) {
      QuantJob& j = jobs.j[jobs.n++];
      j.x = g.x;
      j.q = ws + slots[i].xq;
      j.scales = ws + slots[i].sx;
      j.amax_slot = reinterpret_cast<unsigned*>(ws + slots[i].amax);
      j.sf_tc = (g.mode == kScaleMx32 || g.mode == kScaleBlock32) ? ws + slots[i].sx_tc : nullptr;
      j.rows = g.M;
      j.cols = g.K;
      j.ld = g.K;
      j.row_begin = rows;
      rows += g.M;
    }
    if (!g.w_is_fp8) {
      QuantJob& j = jobs.j[jobs.n++];
      j.x = g.w;
      j.q = ws + slots[i].wq;
      j.scales = ws + slots[i].sw;
      j.amax_slot = reinterpret_cast<unsigned*>(ws + slots[i].amax) + 1;
      j.sf_tc = (g.mode == kScaleMx32 || g.mode == kScaleBlock32) ? ws + slots[i].sw_tc : nullptr;
      j.rows = g.N;
      j.cols = g.K;
      j.ld = g.K;
      j.row_begin = rows;
      rows += g.N;
    }
  }
  jobs.total_rows = rows;
  if (jobs.n == 0) return LOKA_OK;
  for (int i = 0; i < jobs.n; ++i) {
    cudaError_t e = pad_scale_codes(jobs.j[i].sf_tc, jobs.j[i].rows, jobs.j[i].cols, stream);
    if (e != cudaSuccess) return cuda_fail(e, "scale-code padding");
  }
  cudaError_t e = launch_quantize(jobs, d[0].mode, dev->sms, stream);
  if (e != cudaSuccess) return cuda_fail(e, "quantize launch");
  return LOKA_OK;
}

}  // namespace
}  // namespace loka

using namespace loka;

extern "C" {

int32_t loka_version(void) { return (0 << 16) | 1; }

const char* loka_last_error(void) { return t_last_error.c_str(); }

loka_status loka_device_status(void* stream) {
  DeviceInfo* dev = nullptr;
  loka_status s = device_info(&dev);
  if (s != LOKA_OK) return s;
  cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
  unsigned word = 0;
  e = cudaMemcpy(&word, dev->status, sizeof(word), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_fail(e, "reading the device status word");
  if (word != 0) {
    const unsigned zero = 0;
    e = cudaMemcpy(dev->status, &zero, sizeof(zero), cudaMemcpyHostToDevice);
    if (e != cudaSuccess) return cuda_fail(e, "clearing the device status word");
    return fail(LOKA_ERR_TIMEOUT, "a kernel wait ran out of time (status bits 0x%x)", word);
  }
  return LOKA_OK;
}

loka_status loka_selftest_watchdog(uint64_t limit_ns, void* stream) {
  DeviceInfo* dev = nullptr;
  loka_status s = device_info(&dev);
  if (s != LOKA_OK) return s;
  if (limit_ns == 0 || limit_ns > 10000000000ull) return fail(LOKA_ERR_INVALID_ARG, "limit_ns must be in (0, 1e10]");
  cudaError_t e = launch_watchdog_selftest(dev->status, limit_ns, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "watchdog self-test launch");
  return LOKA_OK;
}

loka_status loka_selftest_mma_peak(int32_t kind, int64_t mmas_per_sm, void* stream) {
  DeviceInfo* dev = nullptr;
  loka_status s = device_info(&dev);
  if (s != LOKA_OK) return s;
  if (kind != 0 && kind != 1) return fail(LOKA_ERR_INVALID_ARG, "kind %d: 0 (E4M3) or 1 (bf16)", kind);
  if (mmas_per_sm < 1 || mmas_per_sm > (int64_t{1} << 32))
    return fail(LOKA_ERR_INVALID_ARG, "mmas_per_sm = %lld is outside [1, 2^32]", static_cast<long long>(mmas_per_sm));
  // the last MMAs drain within microseconds of the issue loop's end
  cudaError_t e = launch_mma_peak(kind, mmas_per_sm, dev->sms, dev->status, 1000000000ull, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "tensor-core peak launch");
  return LOKA_OK;
}

size_t loka_quantize_fp8_workspace_size(int64_t, int64_t, int32_t mode) {
  return mode == LOKA_SCALE_TENSOR ? kAlign : 0;
}

namespace {

loka_status quantize_one(const void* x, int64_t rows, int64_t cols, int64_t ld, int32_t mode, void* q, void* q_t,
                         void* scales, void* workspace, size_t workspace_bytes, void* stream) {
  if (mode != LOKA_SCALE_TENSOR && mode != LOKA_SCALE_ROW && mode != LOKA_SCALE_MX32 && mode != LOKA_SCALE_BLOCK32)
    return fail(LOKA_ERR_INVALID_ARG, "mode %d is not an FP8 scaling mode", mode);
  if (rows < 0 || cols < 0) return fail(LOKA_ERR_INVALID_ARG, "negative size");
  if (cols % 32 != 0) return fail(LOKA_ERR_INVALID_ARG, "cols = %lld is not a multiple of 32", static_cast<long long>(cols));
  if (ld < cols || ld % 8 != 0)
    return fail(LOKA_ERR_INVALID_ARG, "ld = %lld: the row stride must be >= cols and a multiple of 8 (16-byte rows)",
                static_cast<long long>(ld));
  if (rows == 0 || cols == 0) {
    if (mode == LOKA_SCALE_TENSOR && scales != nullptr) {
      const float one = 1.0f;
      cudaError_t e = cudaMemcpyAsync(scales, &one, sizeof(one), cudaMemcpyHostToDevice, static_cast<cudaStream_t>(stream));
      if (e != cudaSuccess) return cuda_fail(e, "writing the unit scale");
    }
    return LOKA_OK;
  }
  if (x == nullptr || q == nullptr || scales == nullptr) return fail(LOKA_ERR_INVALID_ARG, "x, q and scales must not be NULL");
  if (!aligned16(x) || !aligned16(q)) return fail(LOKA_ERR_INVALID_ARG, "x and q must be 16-byte aligned");
  if (q_t != nullptr && (rows % 32 != 0 || !aligned16(q_t)))
    return fail(LOKA_ERR_INVALID_ARG, "the transposed codes need rows %% 32 == 0 and a 16-byte-aligned q_t");
  if ((mode == LOKA_SCALE_TENSOR || mode == LOKA_SCALE_ROW) && (reinterpret_cast<uintptr_t>(scales) & 3u))
    return fail(LOKA_ERR_INVALID_ARG, "scales must be 4-byte aligned");
  const size_t need = loka_quantize_fp8_workspace_size(rows, cols, mode);
  if (need > 0 && (workspace == nullptr || workspace_bytes < need || (reinterpret_cast<uintptr_t>(workspace) & 255u)))
    return fail(LOKA_ERR_WORKSPACE, "workspace must be >= %zu bytes, 256-byte aligned", need);
  DeviceInfo* dev = nullptr;
  loka_status s = device_info(&dev);
  if (s != LOKA_OK) return s;
  QuantJobs jobs;
  std::memset(&jobs, 0, sizeof(jobs));
  jobs.n = 1;
  jobs.j[0].x = x;
  jobs.j[0].q = static_cast<uint8_t*>(q);
  jobs.j[0].q_t = static_cast<uint8_t*>(q_t);
  jobs.j[0].scales = scales;
  jobs.j[0].amax_slot = static_cast<unsigned*>(workspace);
  jobs.j[0].rows = rows;
  jobs.j[0].cols = cols;
  jobs.j[0].ld = ld;
  jobs.total_rows = rows;
  cudaError_t e = launch_quantize(jobs, mode, dev->sms, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "quantize launch");
  return LOKA_OK;
}

}  // namespace

loka_status loka_quantize_fp8(const void* x, int64_t rows, int64_t cols, int64_t ld, int32_t mode, void* q,
                              void* scales, void* workspace, size_t workspace_bytes, void* stream) {
  return quantize_one(x, rows, cols, ld, mode, q, nullptr, scales, workspace, workspace_bytes, stream);
}

loka_status loka_quantize_fp8_block32(const void* x, int64_t rows, int64_t cols, int64_t ld, void* q, void* q_t,
                                      void* scales, void* stream) {
  return quantize_one(x, rows, cols, ld, LOKA_SCALE_BLOCK32, q, q_t, scales, nullptr, 0, stream);
}

size_t loka_fp8_linear_norm_workspace_size(const loka_linear_desc* descs, int32_t num_groups) {
  if (descs == nullptr || num_groups < 1 || num_groups > kMaxGroups) return 0;
  return layout_operands(descs, num_groups, nullptr);
}

loka_status loka_fp8_linear_norm(const loka_linear_desc* descs, int32_t num_groups, void* workspace,
                                 size_t workspace_bytes, void* stream) {
  loka_status s = validate(descs, num_groups, false);
  if (s != LOKA_OK) return s;
  std::vector<OperandSlots> slots;
  const size_t need = layout_operands(descs, num_groups, &slots);
  if (need > 0 && (workspace == nullptr || workspace_bytes < need || (reinterpret_cast<uintptr_t>(workspace) & 255u)))
    return fail(LOKA_ERR_WORKSPACE, "workspace must be >= %zu bytes, 256-byte aligned", need);
  int64_t total_m = 0;
  for (int i = 0; i < num_groups; ++i) total_m += descs[i].M;
  if (total_m == 0) return LOKA_OK;
  DeviceInfo* dev = nullptr;
  if ((s = device_info(&dev)) != LOKA_OK) return s;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  const bool bf16 = descs[0].mode == kBf16;
  const OutKind out = output_reference(descs, num_groups).y_q != nullptr ? OutKind::kQuant : OutKind::kBf16;
  // Per-row scaling of bf16 X with a whole output row per CTA: the GEMM
  // quantizes X itself (LoKA section III-B case 1), so X is read from HBM
  // once and its codes never leave the chip.  Only W is quantized before.
  if (descs[0].mode == kScaleRow && !descs[0].x_is_fp8 &&
      gemm_qx_supported(static_cast<int>(descs[0].N), static_cast<int>(descs[0].K), descs[0].norm, out)) {
    const bool w_launch = !descs[0].w_is_fp8;
    if (w_launch && (s = quantize_operands(descs, num_groups, slots, ws, dev, st, true)) != LOKA_OK) return s;
    static thread_local GemmParams pq;
    if ((s = build_gemm(descs, num_groups, slots, ws, false, out, nullptr, descs[0].norm, dev, &pq)) != LOKA_OK) return s;
    // the quantizer warps read bf16 X rows directly
    for (int i = 0; i < num_groups; ++i) pq.g[i].xbf = static_cast<const uint16_t*>(descs[i].x);
    // X was complete before this call's W quantizer started (a normal
    // launch), so the GEMM may read X before waiting for that launch
    pq.x_ready = w_launch ? 1 : 0;
    pq.w_ready = 0;
    cudaError_t e = launch_gemm_norm(pq, static_cast<int>(descs[0].N), OperandKind::kE4M3Qx, out, dev->sms, st);
    if (e != cudaSuccess) return cuda_fail(e, "GEMM launch");
    return LOKA_OK;
  }
  if (!bf16 && (!descs[0].x_is_fp8 || !descs[0].w_is_fp8)) {
    if ((s = quantize_operands(descs, num_groups, slots, ws, dev, st)) != LOKA_OK) return s;
  }
  if (descs[0].mode == kScaleMx32 || descs[0].mode == kScaleBlock32) {
    // caller-quantized MX / 32x32-block operands: scales into the copy layout
    const int row_div = descs[0].mode == kScaleBlock32 ? 32 : 1;
    for (int i = 0; i < num_groups; ++i) {
      const loka_linear_desc& g = descs[i];
      cudaError_t e = cudaSuccess;
      if (g.x_is_fp8 && g.M > 0) e = pad_scale_codes(ws + slots[i].sx_tc, g.M, g.K, st);
      if (e == cudaSuccess && g.w_is_fp8) e = pad_scale_codes(ws + slots[i].sw_tc, g.N, g.K, st);
      if (e == cudaSuccess && g.x_is_fp8 && g.M > 0)
        e = launch_sf_permute(static_cast<const uint8_t*>(g.x_scales), ws + slots[i].sx_tc, g.M, g.K, row_div, dev->sms,
                              st);
      if (e == cudaSuccess && g.w_is_fp8)
        e = launch_sf_permute(static_cast<const uint8_t*>(g.w_scales), ws + slots[i].sw_tc, g.N, g.K, row_div, dev->sms,
                              st);
      if (e != cudaSuccess) return cuda_fail(e, "scale permute launch");
    }
  }
  static thread_local GemmParams p;
  if ((s = build_gemm(descs, num_groups, slots, ws, bf16, out, nullptr, descs[0].norm, dev, &p)) != LOKA_OK) return s;
  // Caller-quantized W may load before the GEMM waits for the launch that
  // precedes it only when that launch is this call's own activation
  // quantizer: it started after everything the caller queued (W included)
  // had finished.  (MX also permutes W's scales right before the GEMM.)
  p.w_ready = (!bf16 && descs[0].w_is_fp8 && !descs[0].x_is_fp8 && operand_kind(descs[0].mode) != OperandKind::kMxE4M3)
                  ? 1 : 0;
  cudaError_t e = launch_gemm_norm(p, static_cast<int>(descs[0].N), operand_kind(descs[0].mode), out, dev->sms, st);
  if (e != cudaSuccess) return cuda_fail(e, "GEMM launch");
  return LOKA_OK;
}

loka_status loka_fp8_linear_norm_static(const loka_linear_desc* descs, int32_t num_groups, void* stream) {
  loka_status s = validate(descs, num_groups, false);
  if (s != LOKA_OK) return s;
  const size_t need = layout_operands(descs, num_groups, nullptr);
  if (need > kStaticScratchBytes)
    return fail(LOKA_ERR_WORKSPACE,
                "this call needs %zu bytes of scratch; the built-in scratch of loka_fp8_linear_norm_static holds %zu "
                "bytes (use loka_fp8_linear_norm with a caller workspace)",
                need, kStaticScratchBytes);
  // the architecture check first, as in every other entry point
  DeviceInfo* dev = nullptr;
  if ((s = device_info(&dev)) != LOKA_OK) return s;
  void* scratch = nullptr;
  if ((s = static_scratch(&scratch)) != LOKA_OK) return s;
  return loka_fp8_linear_norm(descs, num_groups, scratch, kStaticScratchBytes, stream);
}

size_t loka_quant_error_workspace_size(const loka_linear_desc* desc) {
  if (desc == nullptr) return 0;
  size_t off = layout_operands(desc, 1, nullptr);
  const size_t mn = static_cast<size_t>(desc->M) * static_cast<size_t>(desc->N) * sizeof(float);
  return off + 2 * align_up(mn) + kAlign;
}

loka_status loka_quant_error(const loka_linear_desc* desc, void* workspace, size_t workspace_bytes,
                             loka_error_stats* stats, void* stream) {
  loka_status s = validate(desc, 1, true);
  if (s != LOKA_OK) return s;
  if (stats == nullptr) return fail(LOKA_ERR_INVALID_ARG, "stats is NULL");
  const size_t need = loka_quant_error_workspace_size(desc);
  if (workspace == nullptr || workspace_bytes < need || (reinterpret_cast<uintptr_t>(workspace) & 255u))
    return fail(LOKA_ERR_WORKSPACE, "workspace must be >= %zu bytes, 256-byte aligned", need);
  std::memset(stats, 0, sizeof(*stats));
  stats->count = desc->M * desc->N;
  if (desc->M == 0) return LOKA_OK;
  DeviceInfo* dev = nullptr;
  if ((s = device_info(&dev)) != LOKA_OK) return s;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  std::vector<OperandSlots> slots;
  const size_t ops = layout_operands(desc, 1, &slots);
  const size_t mn = static_cast<size_t>(desc->M) * static_cast<size_t>(desc->N) * sizeof(float);
  float* out = reinterpret_cast<float*>(ws + ops);
  float* ref = reinterpret_cast<float*>(ws + ops + align_up(mn));
  double* acc = reinterpret_cast<double*>(ws + ops + 2 * align_up(mn));
  const bool bf16 = desc->mode == kBf16;
  static thread_local GemmParams p;
  cudaError_t e;
  if (!bf16) {
    if ((s = quantize_operands(desc, 1, slots, ws, dev, st)) != LOKA_OK) return s;
  }
  void* y_out[1] = {out};
  if ((s = build_gemm(desc, 1, slots, ws, bf16, OutKind::kF32, y_out, kNormNone, dev, &p)) != LOKA_OK) return s;
  e = launch_gemm_norm(p, static_cast<int>(desc->N), operand_kind(desc->mode), OutKind::kF32, dev->sms, st);
  if (e != cudaSuccess) return cuda_fail(e, "probe GEMM launch");
  void* y_ref[1] = {ref};
  if ((s = build_gemm(desc, 1, slots, ws, true, OutKind::kF32, y_ref, kNormNone, dev, &p)) != LOKA_OK) return s;
  e = launch_gemm_norm(p, static_cast<int>(desc->N), OperandKind::kBf16, OutKind::kF32, dev->sms, st);
  if (e != cudaSuccess) return cuda_fail(e, "reference GEMM launch");
  e = launch_error_reduce(out, ref, desc->M * desc->N, acc, dev->sms, st);
  if (e != cudaSuccess) return cuda_fail(e, "probe reduction launch");
  // the same two outputs after the layer's normalization (and activation):
  // both GEMMs again with the norm in the epilogue and fp32 output, into the
  // same buffers (stream order), reduced into the second accumulator block
  const bool post = desc->norm != kNormNone || desc->act != kActNone;
  if (post) {
    if ((s = build_gemm(desc, 1, slots, ws, bf16, OutKind::kF32, y_out, desc->norm, dev, &p)) != LOKA_OK) return s;
    e = launch_gemm_norm(p, static_cast<int>(desc->N), operand_kind(desc->mode), OutKind::kF32, dev->sms, st);
    if (e != cudaSuccess) return cuda_fail(e, "probe post-norm GEMM launch");
    if ((s = build_gemm(desc, 1, slots, ws, true, OutKind::kF32, y_ref, desc->norm, dev, &p)) != LOKA_OK) return s;
    e = launch_gemm_norm(p, static_cast<int>(desc->N), OperandKind::kBf16, OutKind::kF32, dev->sms, st);
    if (e != cudaSuccess) return cuda_fail(e, "reference post-norm GEMM launch");
    e = launch_error_reduce(out, ref, desc->M * desc->N, acc + 8, dev->sms, st);
    if (e != cudaSuccess) return cuda_fail(e, "probe post-norm reduction launch");
  }
  double host[13];
  e = cudaMemcpyAsync(host, acc, sizeof(host), cudaMemcpyDeviceToHost, st);
  if (e != cudaSuccess) return cuda_fail(e, "reading probe statistics");
  if ((s = loka_device_status(stream)) != LOKA_OK) return s;
  stats->mere = host[1] > 0 ? host[0] / host[1] : 0.0;
  stats->rel_err_fro = host[3] > 0 ? std::sqrt(host[2]) / std::sqrt(host[3]) : 0.0;
  stats->max_abs = host[4];
  stats->max_abs_post_norm = post ? host[12] : host[4];
  stats->zero_ref_count = desc->M * desc->N - static_cast<int64_t>(host[1]);
  return LOKA_OK;
}

loka_status loka_dispatch_select(const loka_dispatch_entry* table, int64_t n, const loka_problem* p,
                                 const loka_policy* policy, int32_t* choice) {
  if (p == nullptr || policy == nullptr || choice == nullptr) return fail(LOKA_ERR_INVALID_ARG, "NULL argument");
  if (n < 0 || (n > 0 && table == nullptr)) return fail(LOKA_ERR_INVALID_ARG, "bad table");
  if (p->M <= 0) return fail(LOKA_ERR_INVALID_ARG, "problem M must be positive");
  *choice = LOKA_BF16;
  // candidate rows: same N, K, norm; nearest log2(M) (ties: larger M);
  // nearest outlier fraction (ties: larger)
  double best_dm = INFINITY;
  int64_t best_m = -1;
  for (int64_t i = 0; i < n; ++i) {
    const loka_problem& q = table[i].p;
    if (q.N != p->N || q.K != p->K || q.norm != p->norm || q.M <= 0) continue;
    const double dm = std::fabs(std::log2(static_cast<double>(q.M)) - std::log2(static_cast<double>(p->M)));
    if (dm < best_dm || (dm == best_dm && q.M > best_m)) {
      best_dm = dm;
      best_m = q.M;
    }
  }
  if (best_m < 0) return LOKA_OK;
  double best_do = INFINITY, best_o = -INFINITY;
  for (int64_t i = 0; i < n; ++i) {
    const loka_problem& q = table[i].p;
    if (q.N != p->N || q.K != p->K || q.norm != p->norm || q.M != best_m) continue;
    const double d_o = std::fabs(q.outlier_frac - p->outlier_frac);
    if (d_o < best_do || (d_o == best_do && q.outlier_frac > best_o)) {
      best_do = d_o;
      best_o = q.outlier_frac;
    }
  }
  auto is_cand = [&](const loka_dispatch_entry& e) {
    return e.p.N == p->N && e.p.K == p->K && e.p.norm == p->norm && e.p.M == best_m && e.p.outlier_frac == best_o;
  };
  double t_ref = INFINITY;
  bool have_ref = false;
  for (int64_t i = 0; i < n; ++i)
    if (is_cand(table[i]) && table[i].variant == LOKA_BF16) {
      have_ref = true;
      t_ref = std::fmin(t_ref, table[i].time_us);
    }
  const loka_dispatch_entry* best = nullptr;
  for (int64_t i = 0; i < n; ++i) {
    const loka_dispatch_entry& e = table[i];
    if (!is_cand(e)) continue;
    if (!(e.rel_err <= policy->max_rel_err)) continue;
    if (policy->max_mere >= 0 && !(e.mere < policy->max_mere)) continue;
    if (policy->min_speedup >= 0 && e.variant != LOKA_BF16) {
      if (!have_ref || !(t_ref / e.time_us > policy->min_speedup)) continue;
    }
    if (best == nullptr || e.time_us < best->time_us ||
        (e.time_us == best->time_us && (e.rel_err < best->rel_err ||
                                        (e.rel_err == best->rel_err && e.variant < best->variant))))
      best = &e;
  }
  if (best != nullptr) *choice = best->variant;
  return LOKA_OK;
}

}  // extern "C"

namespace {

// Workspace of one statistics update: X^T in G split-K groups of Bg batch
// rows (a multiple of 128, zero-padded), column sums per 128-row tile, the
// fp64 column sums, and the G fp32 [K, K] GEMM partials.
struct StatsLayout {
  int G;
  int64_t Bg, tiles;
  size_t xt, colpart, colsum, partials, total;
};

StatsLayout stats_layout(int64_t B, int64_t K) {
  StatsLayout L{};
  const int64_t chunks = (B + 127) / 128;
  L.G = static_cast<int>(chunks < kMaxGroups ? (chunks < 1 ? 1 : chunks) : kMaxGroups);
  L.Bg = (chunks + L.G - 1) / L.G * 128;
  L.tiles = L.G * L.Bg / 128;
  size_t off = 0;
  L.xt = off;
  off = align_up(off + static_cast<size_t>(L.G) * K * L.Bg * 2);
  L.colpart = off;
  off = align_up(off + static_cast<size_t>(L.tiles) * K * sizeof(float));
  L.colsum = off;   // column-sum chunks and per-column terms: (32 + 3) x K fp64
  off = align_up(off + static_cast<size_t>(35) * K * sizeof(double));
  L.partials = off;
  off = align_up(off + static_cast<size_t>(L.G) * K * K * sizeof(float));
  L.total = off;
  return L;
}

bool probe_k_ok(int64_t K) { return K == 128 || K == 256 || K == 512 || K == 1024 || K == 2048; }

}  // namespace

extern "C" {

size_t loka_probe_stats_workspace_size(int64_t B, int64_t K) {
  if (B <= 0 || !probe_k_ok(K)) return 0;
  return stats_layout(B, K).total;
}

loka_status loka_probe_stats_update(loka_input_stats* stats, const void* x, int64_t B, void* workspace,
                                    size_t workspace_bytes, void* stream) {
  if (stats == nullptr) return fail(LOKA_ERR_INVALID_ARG, "stats is NULL");
  const int64_t K = stats->K;
  if (!probe_k_ok(K))
    return fail(LOKA_ERR_UNSUPPORTED, "K = %lld: the probe statistics take K in {128, 256, 512, 1024, 2048}",
                static_cast<long long>(K));
  if (B < 0 || stats->n < 0) return fail(LOKA_ERR_INVALID_ARG, "negative row count");
  if (B > (int64_t(1) << 24)) return fail(LOKA_ERR_UNSUPPORTED, "B = %lld: at most 2^24 rows per update",
                                          static_cast<long long>(B));
  if (B == 0) return LOKA_OK;
  if (x == nullptr || stats->mu == nullptr || stats->scatter == nullptr)
    return fail(LOKA_ERR_INVALID_ARG, "x, mu and scatter must not be NULL");
  if (!aligned16(x) || (reinterpret_cast<uintptr_t>(stats->mu) & 7u) || (reinterpret_cast<uintptr_t>(stats->scatter) & 7u))
    return fail(LOKA_ERR_INVALID_ARG, "x must be 16-byte aligned, mu and scatter 8-byte aligned");
  const StatsLayout L = stats_layout(B, K);
  if (workspace == nullptr || workspace_bytes < L.total || (reinterpret_cast<uintptr_t>(workspace) & 255u))
    return fail(LOKA_ERR_WORKSPACE, "workspace must be >= %zu bytes, 256-byte aligned", L.total);
  DeviceInfo* dev = nullptr;
  loka_status s = device_info(&dev);
  if (s != LOKA_OK) return s;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  float* colpart = reinterpret_cast<float*>(ws + L.colpart);
  float* partials = reinterpret_cast<float*>(ws + L.partials);
  cudaError_t e = launch_stats_transpose(x, B, K, L.Bg, L.G, ws + L.xt, colpart, st);
  if (e != cudaSuccess) return cuda_fail(e, "statistics transpose launch");
  // the batch's raw scatter, one fp32 [K, K] partial per group: the fused
  // GEMM with bf16 operands X^T_g (as A and as W), no norm, fp32 output
  loka_linear_desc d[kMaxGroups];
  void* yo[kMaxGroups];
  for (int g = 0; g < L.G; ++g) {
    std::memset(&d[g], 0, sizeof(d[g]));
    d[g].M = K;
    d[g].N = K;
    d[g].K = L.Bg;
    d[g].mode = kBf16;
    d[g].norm = kNormNone;
    d[g].x = d[g].w = ws + L.xt + static_cast<size_t>(g) * K * L.Bg * 2;
    yo[g] = partials + static_cast<size_t>(g) * K * K;
    d[g].y = yo[g];
  }
  std::vector<OperandSlots> slots;
  layout_operands(d, L.G, &slots);
  static thread_local GemmParams p;
  if ((s = build_gemm(d, L.G, slots, ws, true, OutKind::kF32, yo, kNormNone, dev, &p)) != LOKA_OK) return s;
  e = launch_gemm_norm(p, static_cast<int>(K), OperandKind::kBf16, OutKind::kF32, dev->sms, st);
  if (e != cudaSuccess) return cuda_fail(e, "statistics GEMM launch");
  e = launch_stats_merge(colpart, L.tiles, partials, L.G, K, reinterpret_cast<double*>(ws + L.colsum), stats->mu,
                         stats->scatter, stats->n, B, dev->sms, st);
  if (e != cudaSuccess) return cuda_fail(e, "statistics merge launch");
  stats->n += B;
  return LOKA_OK;
}

loka_status loka_probe_covariance(const loka_input_stats* stats, double* cov, void* stream) {
  if (stats == nullptr || cov == nullptr) return fail(LOKA_ERR_INVALID_ARG, "stats and cov must not be NULL");
  if (stats->K <= 0) return fail(LOKA_ERR_INVALID_ARG, "K = %lld", static_cast<long long>(stats->K));
  if (stats->n < 2) return fail(LOKA_ERR_INVALID_ARG, "n = %lld: a covariance needs at least two rows",
                                static_cast<long long>(stats->n));
  if (stats->scatter == nullptr) return fail(LOKA_ERR_INVALID_ARG, "scatter is NULL");
  if ((reinterpret_cast<uintptr_t>(cov) & 7u) != 0) return fail(LOKA_ERR_INVALID_ARG, "cov must be 8-byte aligned");
  DeviceInfo* dev = nullptr;
  loka_status s = device_info(&dev);
  if (s != LOKA_OK) return s;
  cudaError_t e = launch_covariance(stats->scatter, stats->K, stats->n, cov, dev->sms, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "covariance launch");
  return LOKA_OK;
}

size_t loka_probe_cholesky_workspace_size(int64_t K) {
  if (!probe_k_ok(K)) return 0;
  return align_up(static_cast<size_t>(K) * K * sizeof(float)) + kAlign;
}

loka_status loka_probe_cholesky(const loka_input_stats* stats, double eps_rel, void* chol, void* mu_out,
                                void* workspace, size_t workspace_bytes, void* stream) {
  if (stats == nullptr || chol == nullptr || mu_out == nullptr)
    return fail(LOKA_ERR_INVALID_ARG, "stats, chol and mu_out must not be NULL");
  const int64_t K = stats->K;
  if (!probe_k_ok(K))
    return fail(LOKA_ERR_UNSUPPORTED, "K = %lld: the probe takes K in {128, 256, 512, 1024, 2048}",
                static_cast<long long>(K));
  if (stats->n < 2) return fail(LOKA_ERR_INVALID_ARG, "n = %lld: a covariance needs at least two rows",
                                static_cast<long long>(stats->n));
  if (!(eps_rel >= 0.0) || !std::isfinite(eps_rel)) return fail(LOKA_ERR_INVALID_ARG, "eps_rel must be finite and >= 0");
  if (stats->mu == nullptr || stats->scatter == nullptr) return fail(LOKA_ERR_INVALID_ARG, "mu and scatter are NULL");
  if (!aligned16(chol)) return fail(LOKA_ERR_INVALID_ARG, "chol must be 16-byte aligned");
  const size_t need = loka_probe_cholesky_workspace_size(K);
  if (workspace == nullptr || workspace_bytes < need || (reinterpret_cast<uintptr_t>(workspace) & 255u))
    return fail(LOKA_ERR_WORKSPACE, "workspace must be >= %zu bytes, 256-byte aligned", need);
  DeviceInfo* dev = nullptr;
  loka_status s = device_info(&dev);
  if (s != LOKA_OK) return s;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  int* status = reinterpret_cast<int*>(ws + align_up(static_cast<size_t>(K) * K * sizeof(float)));
  cudaError_t e = launch_cholesky(stats->scatter, stats->mu, K, stats->n, eps_rel, reinterpret_cast<float*>(ws), chol,
                                  mu_out, status, st);
  if (e != cudaSuccess) return cuda_fail(e, "Cholesky launch");
  int host = 0;
  if ((e = cudaMemcpyAsync(&host, status, sizeof(host), cudaMemcpyDeviceToHost, st)) != cudaSuccess)
    return cuda_fail(e, "reading the Cholesky status");
  if ((e = cudaStreamSynchronize(st)) != cudaSuccess) return cuda_fail(e, "Cholesky");
  if (host != 0) return fail(LOKA_ERR_NUMERIC, "the regularized covariance is not positive definite");
  return LOKA_OK;
}

size_t loka_probe_sample_workspace_size(int64_t B, int64_t K) {
  if (B <= 0 || !probe_k_ok(K)) return 0;
  return align_up(static_cast<size_t>(B) * K * 2);
}

loka_status loka_probe_sample_inputs(const void* mu, const void* chol, int64_t B, int64_t K, uint64_t seed, void* out,
                                     void* workspace, size_t workspace_bytes, void* stream) {
  if (!probe_k_ok(K))
    return fail(LOKA_ERR_UNSUPPORTED, "K = %lld: the sampler takes K in {128, 256, 512, 1024, 2048}",
                static_cast<long long>(K));
  if (B < 0) return fail(LOKA_ERR_INVALID_ARG, "B = %lld < 0", static_cast<long long>(B));
  if (B > (int64_t(1) << 31)) return fail(LOKA_ERR_UNSUPPORTED, "B too large");
  if (B == 0) return LOKA_OK;
  if (mu == nullptr || chol == nullptr || out == nullptr) return fail(LOKA_ERR_INVALID_ARG, "mu, chol and out must not be NULL");
  if (!aligned16(chol) || !aligned16(out)) return fail(LOKA_ERR_INVALID_ARG, "chol and out must be 16-byte aligned");
  const size_t need = loka_probe_sample_workspace_size(B, K);
  if (workspace == nullptr || workspace_bytes < need || (reinterpret_cast<uintptr_t>(workspace) & 255u))
    return fail(LOKA_ERR_WORKSPACE, "workspace must be >= %zu bytes, 256-byte aligned", need);
  DeviceInfo* dev = nullptr;
  loka_status s = device_info(&dev);
  if (s != LOKA_OK) return s;
  cudaError_t e = launch_normals(seed, B * K, workspace, dev->sms, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "normals launch");
  // T' = Z L^T + mu: the bf16 GEMM with L as the weights and mu as the bias
  loka_linear_desc d;
  std::memset(&d, 0, sizeof(d));
  d.M = B;
  d.N = K;
  d.K = K;
  d.mode = kBf16;
  d.norm = kNormNone;
  d.x = workspace;
  d.w = chol;
  d.bias = mu;
  d.y = out;
  return loka_fp8_linear_norm(&d, 1, nullptr, 0, stream);
}

}  // extern "C"

namespace {

// Workspace of the probe's weight model: Wc, W_V, W_U [R, C]; L_U, U' [R, R];
// L_V, V' [C, C] (fp32); 2 fp64 traces; 2 status words.
WeightWork weight_layout(int64_t R, int64_t C, uint8_t* base, size_t* total) {
  WeightWork w{};
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t o = off;
    off = align_up(off + bytes);
    return base + o;
  };
  const size_t rc = static_cast<size_t>(R) * C * sizeof(float);
  w.wc = reinterpret_cast<float*>(take(rc));
  w.wv = reinterpret_cast<float*>(take(rc));
  w.wu = reinterpret_cast<float*>(take(rc));
  w.lu = reinterpret_cast<float*>(take(static_cast<size_t>(R) * R * sizeof(float)));
  w.u1 = reinterpret_cast<float*>(take(static_cast<size_t>(R) * R * sizeof(float)));
  w.lv = reinterpret_cast<float*>(take(static_cast<size_t>(C) * C * sizeof(float)));
  w.v1 = reinterpret_cast<float*>(take(static_cast<size_t>(C) * C * sizeof(float)));
  w.trace = reinterpret_cast<double*>(take(2 * sizeof(double)));
  w.status = reinterpret_cast<int*>(take(2 * sizeof(int)));
  if (total) *total = off;
  return w;
}

bool weight_dims_ok(int64_t R, int64_t C) { return R >= 2 && C >= 2 && R <= 2048 && C <= 2048 && C % 2 == 0; }

loka_status weight_check(const loka_weight_stats* st, void* workspace, size_t workspace_bytes, WeightWork* w) {
  if (st == nullptr) return fail(LOKA_ERR_INVALID_ARG, "stats is NULL");
  if (!weight_dims_ok(st->R, st->C))
    return fail(LOKA_ERR_UNSUPPORTED, "R = %lld, C = %lld: the weight model takes 2 <= R, C <= 2048, C even",
                static_cast<long long>(st->R), static_cast<long long>(st->C));
  if (st->mean == nullptr || st->U == nullptr || st->V == nullptr)
    return fail(LOKA_ERR_INVALID_ARG, "mean, U and V must not be NULL");
  if ((reinterpret_cast<uintptr_t>(st->mean) | reinterpret_cast<uintptr_t>(st->U) | reinterpret_cast<uintptr_t>(st->V)) & 3u)
    return fail(LOKA_ERR_INVALID_ARG, "mean, U and V must be 4-byte aligned");
  size_t need = 0;
  weight_layout(st->R, st->C, nullptr, &need);
  if (workspace == nullptr || workspace_bytes < need || (reinterpret_cast<uintptr_t>(workspace) & 255u))
    return fail(LOKA_ERR_WORKSPACE, "workspace must be >= %zu bytes, 256-byte aligned", need);
  *w = weight_layout(st->R, st->C, static_cast<uint8_t*>(workspace), nullptr);
  return LOKA_OK;
}

// Reads the two factorization status words after the stream has finished.
loka_status weight_status(const WeightWork& w, cudaStream_t st) {
  int host[2] = {0, 0};
  cudaError_t e = cudaMemcpyAsync(host, w.status, sizeof(host), cudaMemcpyDeviceToHost, st);
  if (e != cudaSuccess) return cuda_fail(e, "reading the factorization status");
  if ((e = cudaStreamSynchronize(st)) != cudaSuccess) return cuda_fail(e, "weight model");
  if (host[0] || host[1])
    return fail(LOKA_ERR_NUMERIC, "the regularized %s covariance is not positive definite", host[0] ? "row" : "column");
  return LOKA_OK;
}

}  // namespace

extern "C" {

size_t loka_probe_weight_workspace_size(int64_t R, int64_t C) {
  if (!weight_dims_ok(R, C)) return 0;
  size_t need = 0;
  weight_layout(R, C, nullptr, &need);
  return need;
}

loka_status loka_probe_weight_update(loka_weight_stats* stats, const void* w, double momentum, double eps_rel,
                                     void* workspace, size_t workspace_bytes, void* stream) {
  WeightWork ww{};
  loka_status s = weight_check(stats, workspace, workspace_bytes, &ww);
  if (s != LOKA_OK) return s;
  if (w == nullptr || (reinterpret_cast<uintptr_t>(w) & 1u)) return fail(LOKA_ERR_INVALID_ARG, "w must be a bf16 array");
  if (!(momentum >= 0.0 && momentum < 1.0)) return fail(LOKA_ERR_INVALID_ARG, "momentum must be in [0, 1)");
  if (!(eps_rel >= 0.0) || !std::isfinite(eps_rel)) return fail(LOKA_ERR_INVALID_ARG, "eps_rel must be finite and >= 0");
  if (stats->n < 0) return fail(LOKA_ERR_INVALID_ARG, "negative update count");
  DeviceInfo* dev = nullptr;
  if ((s = device_info(&dev)) != LOKA_OK) return s;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e;
  if (stats->n == 0) {
    e = launch_weight_init(w, stats->R, stats->C, stats->mean, stats->U, stats->V, dev->sms, st);
    if (e != cudaSuccess) return cuda_fail(e, "weight model start");
    stats->n = 1;
    return LOKA_OK;
  }
  e = launch_weight_update(w, stats->R, stats->C, momentum, eps_rel, stats->mean, stats->U, stats->V, ww, dev->sms, st);
  if (e != cudaSuccess) return cuda_fail(e, "weight model update");
  if ((s = weight_status(ww, st)) != LOKA_OK) return s;
  stats->n += 1;
  return LOKA_OK;
}

loka_status loka_probe_sample_weights(const loka_weight_stats* stats, double eps_rel, uint64_t seed, void* out,
                                      void* workspace, size_t workspace_bytes, void* stream) {
  WeightWork ww{};
  loka_status s = weight_check(stats, workspace, workspace_bytes, &ww);
  if (s != LOKA_OK) return s;
  if (stats->n < 1) return fail(LOKA_ERR_INVALID_ARG, "the weight model has no update yet");
  if (out == nullptr || (reinterpret_cast<uintptr_t>(out) & 1u)) return fail(LOKA_ERR_INVALID_ARG, "out must be a bf16 array");
  if (!(eps_rel >= 0.0) || !std::isfinite(eps_rel)) return fail(LOKA_ERR_INVALID_ARG, "eps_rel must be finite and >= 0");
  DeviceInfo* dev = nullptr;
  if ((s = device_info(&dev)) != LOKA_OK) return s;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e = launch_weight_sample(stats->mean, stats->U, stats->V, stats->R, stats->C, eps_rel, seed, out, ww,
                                       dev->sms, st);
  if (e != cudaSuccess) return cuda_fail(e, "weight sampler");
  return weight_status(ww, st);
}

}  // extern "C"
