// situ_math.cuh -- FP32 evaluation of one SiTU-GLU output coordinate,
//
//   h(g, u) = [b1 tanh(g / b1) sigmoid(g)] [b2 tanh(u / b2)],
//
// shared by the standalone activation kernel and the GEMM epilogue.  Sources:
// "SiTU-GLU" problem page (ai-engineer-exhaustive.pages.dev), "Implementation
// order" (divide by the cap, tanh, multiply back; sigmoid of the uncapped gate;
// cap the up branch with its own cap; multiply); "DenseFFN and SituGLU - Docs",
// "one split, two softly bounded branches" (math in FP32, cast at the end).
//
// Method (written for this library):
//   * tanh(g / b1) and tanh(u / b2) come from the hardware tanh.approx.f32
//     (documented maximum relative error about 2^-11 over the whole range; no
//     cancellation near zero, since it returns tanh itself, not 1 - something);
//   * the sigmoid is carried scaled by 2^64, in a form with no branch or select:
//         2^64 sigmoid(g) = 1 / (2^-64 + 2^(-g log2(e) - 64)),
//     one FMA, one ex2.approx, one add, one rcp.approx.  It is exact in the
//     negative tail, where 0.5 + 0.5 tanh(g/2) would cancel to zero, and the
//     2^64 scale keeps outputs in the subnormal range (g from about -87 down to
//     -104) correctly rounded instead of flushed: the 2^-64 is applied by the
//     last multiply, and that multiply and the bf16 conversion keep subnormals.
//     For g below about -133 the exponential overflows to +inf and the sigmoid
//     to 0, below any representable output; for g above about 44 the sum is
//     2^-64 and the sigmoid exactly 1.
// Four special-function ops and eight FP32 ops per output.  Relative error: at
// most about 2 * 2^-11 from the two tanh plus about 2^-17 from the sigmoid's
// exponent argument, below a quarter of a bf16 ulp, so after round-to-nearest-
// even the output is within 0.75 bf16 ulp of the exact value (measured: 0.503
// ulp worst case over every bf16 input of either branch).
// Bound: |tanh.approx| <= 1 (it saturates at +-1), the reciprocal is at most
// 2^64 (its argument is at least 2^-64 and its error is under one ulp), and a
// round-to-nearest multiply by a factor of magnitude <= 1 never increases a
// magnitude, so |h| <= b1 b2 holds structurally, with no clamp.  NaN propagates.
//
// situ_glu_f32_accurate is the variant for float32 outputs, where a 2^-11 error
// would be visible: the sigmoid as P / (1 + e^{-|g|}) (P = 1 or e^{-|g|}, the
// latter carried as 2^64 e^{-|g|}), each tanh in exponential form,
// tanh(x) = (1 - e^{-2x}) / (1 + e^{-2x}) for x >= 0, with 1 - e^{-2x} from its
// Taylor series x' - x'^2/2 + x'^3/6 - x'^4/24 + x'^5/120 (x' = 2x) below x' = 1/16
// (where 1 - e^{-x'} cancels) and one reciprocal for the product of the three
// denominators.  Relative error a few 2^-20.
#pragma once

#include <cstdint>

namespace situ {

struct SituParams {
  float inv_b1;  // 1 / beta1
  float inv_b2;  // 1 / beta2
  float b1b2;    // beta1 * beta2, the bound on |h|
  float limit;   // beta1 * beta2 * 2^64: the bound before the final 2^-64 scale
};

__host__ __device__ inline SituParams make_situ_params(float beta, float linear_beta) {
  SituParams p;
  p.inv_b1 = 1.0f / beta;
  p.inv_b2 = 1.0f / linear_beta;
  p.b1b2 = beta * linear_beta;
  p.limit = p.b1b2 * 0x1p64f;
  return p;
}

__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ float rcp_approx(float x) {
  float y;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ float tanh_approx(float x) {
  float y;
  asm("tanh.approx.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// One SiTU-GLU output in FP32 (see the header comment for the method).
__device__ __forceinline__ float situ_glu_f32(float g, float u, const SituParams& p) {
  constexpr float kLog2e = 1.4426950408889634f;
  const float t1 = tanh_approx(g * p.inv_b1);  // tanh(g / b1), carries sign(g)
  const float t2 = tanh_approx(u * p.inv_b2);  // tanh(u / b2), carries sign(u)
  // 2^64 sigmoid(g) = 1 / (2^-64 + e^{-g} 2^-64)
  const float s = rcp_approx(0x1p-64f + ex2_approx(fmaf(-g, kLog2e, -64.0f)));
  float h = p.b1b2 * s;
  h = h * t1;
  h = h * t2;
  return h * 0x1p-64f;  // correctly rounded, subnormals kept
}

// 1 - exp(-x) for x >= 0: Taylor series below 1/16, else 1 - e (e = exp(-x)).
__device__ __forceinline__ float one_minus_exp_neg(float x, float e) {
  float q = fmaf(x, 1.0f / 120.0f, -1.0f / 24.0f);
  q = fmaf(x, q, 1.0f / 6.0f);
  q = fmaf(x, q, -0.5f);
  q = fmaf(x, q, 1.0f);
  const float series = x * q;
  return x < 0.0625f ? series : 1.0f - e;
}

// One SiTU-GLU output in FP32 for float32 outputs (see the header comment).
__device__ __forceinline__ float situ_glu_f32_accurate(float g, float u, const SituParams& p) {
  constexpr float kLog2e = 1.4426950408889634f;
  const float ag = fabsf(g);
  const float au = fabsf(u);
  const float x1 = 2.0f * ag * p.inv_b1;  // 2|g|/b1
  const float x2 = 2.0f * au * p.inv_b2;  // 2|u|/b2
  const float e1 = ex2_approx(-x1 * kLog2e);
  const float f = ex2_approx(-x2 * kLog2e);
  const float n1 = one_minus_exp_neg(x1, e1);
  const float n2 = one_minus_exp_neg(x2, f);
  const bool gneg = g < 0.0f;
  const float r = ex2_approx(fmaf(-ag, kLog2e, gneg ? 64.0f : 0.0f));
  const float e0 = gneg ? r * 0x1p-64f : r;
  const float ps = gneg ? r : 0x1p64f;
  const float den = (1.0f + e1) * (1.0f + f) * (1.0f + e0);
  float mag = p.b1b2 * ps;
  mag = mag * rcp_approx(den);
  mag = mag * n1;
  mag = mag * n2;
  mag = mag > p.limit ? p.limit : mag;
  const float h = mag * 0x1p-64f;
  const uint32_t sign = (__float_as_uint(g) ^ __float_as_uint(u)) & 0x80000000u;
  return __uint_as_float(__float_as_uint(h) | sign);
}

}  // namespace situ
