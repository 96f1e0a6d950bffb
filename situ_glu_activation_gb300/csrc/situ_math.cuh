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
// Method (exponential form, written for this library).  With
//   E1 = exp(-2|g|/b1), F = exp(-2|u|/b2), E0 = exp(-|g|),
//   tanh(|g|/b1) = (1 - E1) / (1 + E1),  tanh(|u|/b2) = (1 - F) / (1 + F),
//   sigmoid(g)   = P / (1 + E0),  P = 1 for g >= 0 and P = E0 for g < 0,
// so that
//   |h| = b1 b2 (1 - E1)(1 - F) P / ((1 + E1)(1 + F)(1 + E0)),
//   sign(h) = sign(g) sign(u).
// Three ex2 and one reciprocal on the special-function unit; the rest is FMA.
//   * 1 - exp(-x) loses relative accuracy for small x (cancellation), so for
//     x < 1/16 it is taken from its Taylor series x - x^2/2 + x^3/6 - x^4/24 +
//     x^5/120 (truncation below 2^-29 relative there); above, 1 - E has
//     relative error below 2^-17.
//   * For g < 0 the factor P = e^g is evaluated as 2^64 e^g and the product is
//     scaled back by 2^-64 in its last multiply, so outputs in the subnormal
//     range (g from about -87 down to -104) come out correctly rounded instead of
//     flushed: the final multiply and the bf16 conversion keep subnormals.
//   * Every factor is at most 1, so |h| <= b1 b2 holds after rounding; an explicit
//     min keeps the bound structural even for caps whose product rounds.
// The ex2 and rcp used are the hardware approximations (ex2.approx.ftz,
// rcp.approx.ftz); their inputs and outputs that matter stay normal.  Overall
// relative error is a few 2^-20, far inside half a bf16 ulp (2^-9 relative).
#pragma once

#include <cstdint>

namespace situ {

struct SituParams {
  float two_inv_b1;  // 2 / beta1
  float two_inv_b2;  // 2 / beta2
  float b1b2;        // beta1 * beta2, the bound on |h|
  float limit;       // beta1 * beta2 * 2^64: the bound before the final 2^-64 scale
};

__host__ __device__ inline SituParams make_situ_params(float beta, float linear_beta) {
  SituParams p;
  p.two_inv_b1 = 2.0f / beta;
  p.two_inv_b2 = 2.0f / linear_beta;
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

// 1 - exp(-x) for x >= 0: Taylor series below 1/16, else 1 - e (e = exp(-x)).
__device__ __forceinline__ float one_minus_exp_neg(float x, float e) {
  float q = fmaf(x, 1.0f / 120.0f, -1.0f / 24.0f);
  q = fmaf(x, q, 1.0f / 6.0f);
  q = fmaf(x, q, -0.5f);
  q = fmaf(x, q, 1.0f);
  const float series = x * q;
  return x < 0.0625f ? series : 1.0f - e;
}

// One SiTU-GLU output in FP32 (see the header comment for the method).
__device__ __forceinline__ float situ_glu_f32(float g, float u, const SituParams& p) {
  constexpr float kLog2e = 1.4426950408889634f;
  const float ag = fabsf(g);
  const float au = fabsf(u);
  const float x1 = ag * p.two_inv_b1;  // 2|g|/b1
  const float x2 = au * p.two_inv_b2;  // 2|u|/b2
  const float e1 = ex2_approx(-x1 * kLog2e);
  const float f = ex2_approx(-x2 * kLog2e);
  const float n1 = one_minus_exp_neg(x1, e1);
  const float n2 = one_minus_exp_neg(x2, f);
  const bool gneg = g < 0.0f;
  // r = 2^64 e^{-|g|} for g < 0, e^{-|g|} otherwise.
  const float r = ex2_approx(fmaf(-ag, kLog2e, gneg ? 64.0f : 0.0f));
  const float e0 = gneg ? r * 0x1p-64f : r;  // e^{-|g|}
  const float ps = gneg ? r : 0x1p64f;       // 2^64 P
  const float den = (1.0f + e1) * (1.0f + f) * (1.0f + e0);
  // |h| 2^64 = b1 b2 (2^64 P) rcp(den) n1 n2; the scale is dropped last.
  float mag = p.b1b2 * ps;
  mag = mag * rcp_approx(den);
  mag = mag * n1;
  mag = mag * n2;
  mag = mag > p.limit ? p.limit : mag;  // NaN passes through
  const float h = mag * 0x1p-64f;       // correctly rounded, subnormals kept
  const uint32_t sign = (__float_as_uint(g) ^ __float_as_uint(u)) & 0x80000000u;
  return __uint_as_float(__float_as_uint(h) | sign);
}

}  // namespace situ
