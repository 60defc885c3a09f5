// Scale selection and E4M3 cast arithmetic shared by the standalone quantizer
// (quantize.cu) and the GEMM that quantizes its activations rows in-kernel
// (gemm_norm.cu), so both produce the same codes and scales bit for bit.
//
// Defined by "LoKA: Low-precision Kernel Applications for Recommendation
// Models at Scale", section II-C (tensorwise / rowwise / blockwise FP8
// scaling of the linear layer's operands), and by the MXFP8 1x32 block
// scaling with E8M0 scales along K on the GEM Training page.
#pragma once

#include "ptx.cuh"

namespace loka {

constexpr float kE4M3Max = 448.0f;

// max(|a|, |b|) per bf16 half; a NaN input loses to the other operand (as
// fmaxf does), so NaN elements never become the maximum.
__device__ __forceinline__ uint32_t absmax_bf16x2(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("max.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a & 0x7FFF7FFFu), "r"(b & 0x7FFF7FFFu));
  return d;
}

// fmaxf(m, |x|) over the 8 bf16 of v.  The maximum of exactly representable
// values is exact in any order, so the packed bf16 reduction equals the
// elementwise fp32 one.
__device__ __forceinline__ float abs_max8(const uint4& v, float m) {
  uint32_t a = absmax_bf16x2(v.x, v.y);
  const uint32_t b = absmax_bf16x2(v.z, v.w);
  asm("max.bf16x2 %0, %0, %1;" : "+r"(a) : "r"(b));
  return fmaxf(m, fmaxf(bf16lo(a), bf16hi(a)));
}

// Maximum over the warp of a non-negative, non-NaN float (an abs maximum):
// such floats order like their bit patterns.
__device__ __forceinline__ float warp_max(float m) {
  return __uint_as_float(__reduce_max_sync(0xffffffffu, __float_as_uint(m)));
}

// inv = 448/amax and scale = amax/448, each the correctly rounded fp32
// quotient; amax 0 -> 1.
//
// A row amax is the magnitude of a bf16 value, m * 2^e with m = 1 + k/128
// (k = 0..127).  Then 448/amax = (448/m) * 2^-e and amax/448 = (m/448) * 2^e
// exactly, and scaling a correctly rounded quotient by a power of two keeps
// it correctly rounded while the result stays a normal float.  So the two
// quotients are a table entry per k (IEEE fp32 division, evaluated when the
// table is built) with e added to the exponent field: no division on the
// per-row critical path.  Exponent fields below 10 (amax < 2^-117, where a
// result leaves the normal range) and Inf/NaN take the divisions.
struct RowScaleTables {
  float inv[128];     // 448 / (1 + k/128)
  float scale[128];   // (1 + k/128) / 448
};
constexpr RowScaleTables make_row_scale_tables() {
  RowScaleTables t{};
  for (int k = 0; k < 128; ++k) {
    const float m = 1.0f + static_cast<float>(k) / 128.0f;   // exact
    t.inv[k] = kE4M3Max / m;
    t.scale[k] = m / kE4M3Max;
  }
  return t;
}
__constant__ RowScaleTables kRowScaleTables = make_row_scale_tables();

// tab: the two 128-entry tables (constant memory, or a copy in shared memory
// for kernels whose constant cache is busy with large parameter blocks).
__device__ __forceinline__ void row_scales(float amax, float& inv, float& scale,
                                           const RowScaleTables& tab = kRowScaleTables) {
  const uint32_t a = __float_as_uint(amax);
  const uint32_t ef = (a >> 23) & 0xFFu;   // exponent field
  if (amax == 0.0f) {
    inv = 1.0f;
    scale = 1.0f;
  } else if (ef >= 10u && ef <= 254u && (a & 0xFFFFu) == 0u) {
    const int k = static_cast<int>((a >> 16) & 0x7Fu);
    // table entries have exponent fields 134/135 (inv) and 118/119 (scale)
    inv = __uint_as_float(__float_as_uint(tab.inv[k]) + ((127u - ef) << 23));
    scale = __uint_as_float(__float_as_uint(tab.scale[k]) + ((ef - 127u) << 23));
  } else {
    inv = __fdiv_rn(kE4M3Max, amax);
    scale = __fdiv_rn(amax, kE4M3Max);
  }
}

// 8 bf16 * mul -> 8 E4M3 codes; each product is one fp32 round-to-nearest
// multiply (two per packed instruction), then RNE + saturation to +-448.
__device__ __forceinline__ uint2 cast8(const uint4& v, float mul) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
  const float2 m2 = make_float2(mul, mul);
  uint32_t c[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 f = __fmul2_rn(make_float2(bf16lo(w[i]), bf16hi(w[i])), m2);
    c[i] = cvt_e4m3x2(f.x, f.y);
  }
  return make_uint2(c[0] | (c[1] << 16), c[2] | (c[3] << 16));
}

// E8M0 exponent of a block from the fp32 exponent field of its amax:
// e = clamp(floor(log2 amax) - 8, -127, 127).  A subnormal or zero amax has
// field 0, which lands below -127 and clamps; Inf/NaN have field 255.
__device__ __forceinline__ int mx_exponent(float amax) {
  const int field = static_cast<int>((__float_as_uint(amax) >> 23) & 0xFFu);
  int e = field - 127 - 8;
  e = e < -127 ? -127 : e;
  e = e > 127 ? 127 : e;
  return e;
}

// 2^-e as an fp32 (exact: e is in [-127, 120], so 127 - e is in [7, 254]).
__device__ __forceinline__ float pow2_neg(int e) { return __uint_as_float(static_cast<uint32_t>(127 - e) << 23); }

}  // namespace loka
