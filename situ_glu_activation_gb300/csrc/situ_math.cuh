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
// situ_act_accurate is the variant for float32 outputs, where a 2^-11 error would
// be visible: the sigmoid as P / (1 + e^{-|g|}) (P = 1 or e^{-|g|}, the latter
// carried as 2^64 e^{-|g|}), each tanh in exponential form,
// tanh(x) = (1 - e^{-2x}) / (1 + e^{-2x}) for x >= 0, with 1 - e^{-2x} from its
// Taylor series x' - x'^2/2 + x'^3/6 - x'^4/24 + x'^5/120 (x' = 2x) below x' = 1/16
// (where 1 - e^{-x'} cancels).  Relative error a few 2^-18 (the exponent
// argument's rounding dominates in the negative tail).
#pragma once

#include <cstdint>

namespace situ {

// Which branches carry a soft cap.  A cap of +infinity stands for "no cap":
// beta tanh(x / beta) -> x as beta -> infinity, so the uncapped up branch is the
// activation module's linear_beta = None ("Kimi K3 - Bound the up branch", code
// excerpt of SituAndMul) and both caps infinite give SwiGLU exactly (the
// "SiTU-GLU" chapter, "Les proprietes": SwiGLU again as beta1, beta2 -> infinity).
enum class Caps : int {
  kBoth = 0,      // SiTU-GLU: beta1 on the gate, beta2 on the up branch
  kGateOnly = 1,  // up branch uncapped (linear_beta unset)
  kUpOnly = 2,    // gate branch uncapped (Swish gate), up branch capped
  kNone = 3       // SwiGLU
};

struct SituParams {
  float b1, b2;          // the caps (finite ones only are used)
  float inv_b1, inv_b2;  // 1 / beta1, 1 / beta2
  float b1b2;            // beta1 * beta2, the bound on |h| when both are finite
};

__host__ __device__ inline SituParams make_situ_params(float beta, float linear_beta) {
  SituParams p;
  p.b1 = beta;
  p.b2 = linear_beta;
  p.inv_b1 = 1.0f / beta;
  p.inv_b2 = 1.0f / linear_beta;
  p.b1b2 = beta * linear_beta;
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

constexpr float kLog2e = 1.4426950408889634f;

// 2^64 sigmoid(g) = 1 / (2^-64 + e^{-g} 2^-64), select-free (see the header).
__device__ __forceinline__ float sigmoid_x2p64(float g) {
  return rcp_approx(0x1p-64f + ex2_approx(fmaf(-g, kLog2e, -64.0f)));
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

// tanh(x) in exponential form, for float32 outputs: sign(x) (1 - e)/(1 + e),
// e = exp(-2|x|), with 1 - e from the series where it cancels.
__device__ __forceinline__ float tanh_accurate(float x) {
  const float x2 = 2.0f * fabsf(x);
  const float e = ex2_approx(-x2 * kLog2e);
  const float t = one_minus_exp_neg(x2, e) * rcp_approx(1.0f + e);
  return __uint_as_float(__float_as_uint(t) | (__float_as_uint(x) & 0x80000000u));
}

// 2^64 sigmoid(g) as P / (1 + e^{-|g|}), P = 1 or e^{-|g|} (carried as
// 2^64 e^{-|g|}), for float32 outputs.
__device__ __forceinline__ float sigmoid_x2p64_accurate(float g) {
  const bool gneg = g < 0.0f;
  const float r = ex2_approx(fmaf(-fabsf(g), kLog2e, gneg ? 64.0f : 0.0f));
  const float e0 = gneg ? r * 0x1p-64f : r;
  return (gneg ? r : 0x1p64f) * rcp_approx(1.0f + e0);
}

// Combine tanh values t1 = tanh(g/b1), t2 = tanh(u/b2) and s = 2^64 sigmoid(g)
// into h for the cap configuration kC.  The 2^64 scale is dropped by the last
// multiply, so subnormal outputs are correctly rounded.  For the uncapped
// branches the scale is applied where no intermediate can overflow: a gate value
// above 2^40 is used unscaled (its sigmoid is exactly 1), and an up value above
// 2^20 in magnitude is scaled down instead of the product.
template <Caps kC>
__device__ __forceinline__ float situ_combine(float g, float u, float t1, float t2, float s,
                                              const SituParams& p) {
  if constexpr (kC == Caps::kBoth) {
    float h = p.b1b2 * s;
    h = h * t1;
    h = h * t2;
    return h * 0x1p-64f;
  } else {
    constexpr bool kCapGate = kC == Caps::kGateOnly;
    constexpr bool kCapUp = kC == Caps::kUpOnly;
    float a_s, scale;
    if constexpr (kCapGate) {
      a_s = (p.b1 * s) * t1;  // 2^64 * b1 tanh(g/b1) sigmoid(g)
      scale = 0x1p-64f;
    } else {
      const bool big = g > 0x1p40f;
      a_s = big ? g : g * s;  // 2^64 * g sigmoid(g), or g itself when sigmoid(g) = 1
      scale = big ? 1.0f : 0x1p-64f;
    }
    const float b = kCapUp ? p.b2 * t2 : u;
    return fabsf(b) <= 0x1p20f ? (a_s * b) * scale : a_s * (b * scale);
  }
}

// One activation output in FP32, fast form (bf16 outputs): hardware tanh.approx
// for the caps (see the header comment for the method and its error).
template <Caps kC>
__device__ __forceinline__ float situ_act(float g, float u, const SituParams& p) {
  const bool cap_g = kC == Caps::kBoth || kC == Caps::kGateOnly;
  const bool cap_u = kC == Caps::kBoth || kC == Caps::kUpOnly;
  const float t1 = cap_g ? tanh_approx(g * p.inv_b1) : 0.0f;
  const float t2 = cap_u ? tanh_approx(u * p.inv_b2) : 0.0f;
  return situ_combine<kC>(g, u, t1, t2, sigmoid_x2p64(g), p);
}

// Same, accurate form (float32 outputs): exponential-form tanh and sigmoid.
template <Caps kC>
__device__ __forceinline__ float situ_act_accurate(float g, float u, const SituParams& p) {
  const bool cap_g = kC == Caps::kBoth || kC == Caps::kGateOnly;
  const bool cap_u = kC == Caps::kBoth || kC == Caps::kUpOnly;
  const float t1 = cap_g ? tanh_accurate(g * p.inv_b1) : 0.0f;
  const float t2 = cap_u ? tanh_accurate(u * p.inv_b2) : 0.0f;
  return situ_combine<kC>(g, u, t1, t2, sigmoid_x2p64_accurate(g), p);
}

// tanh(x) and sech^2(x) = 1 - tanh^2(x) for the backward pass: tanh from the hardware
// tanh.approx (relative error about 2^-11 everywhere, no cancellation near zero), and
// sech^2 = 4 e / (1 + e)^2 with e = exp(-2|x|), which keeps its relative accuracy where
// 1 - tanh^2 would cancel (|x| large).  4e is one ex2 of an argument shifted by 2.
// Three special-function ops and five FP32 ops.
__device__ __forceinline__ void tanh_sech2(float x, float& t, float& sech2) {
  t = tanh_approx(x);
  const float e4 = ex2_approx(fmaf(fabsf(x), -2.0f * kLog2e, 2.0f));  // 4 exp(-2|x|)
  const float r = rcp_approx(fmaf(0.25f, e4, 1.0f));                   // 1 / (1 + e)
  sech2 = e4 * r * r;
}

// Partial derivatives of one output h = a(g) b(u) for the backward pass:
//   dh/dg = b(u) a'(g),  a'(g) = sech^2(g/b1) sigmoid(g) + b1 tanh(g/b1) sigmoid(g) sigmoid(-g)
//   dh/du = a(g) b'(u),  b'(u) = sech^2(u/b2)
// (uncapped: a = g sigmoid(g), a' = sigmoid(g) + g sigmoid(g) sigmoid(-g); b = u, b' = 1).
// sigmoid(g) and sigmoid(-g) come from one e^{-|g|} as 1/(1+e) and e/(1+e).
template <Caps kC>
__device__ __forceinline__ void situ_act_grad(float g, float u, const SituParams& p, float& pg,
                                              float& pu) {
  const float e0 = ex2_approx(-fabsf(g) * kLog2e);
  const float r0 = rcp_approx(1.0f + e0);
  const float s_hi = r0, s_lo = e0 * r0;  // sigmoid(|g|), sigmoid(-|g|)
  const bool gpos = g >= 0.0f;
  const float sg = gpos ? s_hi : s_lo;    // sigmoid(g)
  const float sgm = gpos ? s_lo : s_hi;   // sigmoid(-g)
  float a, da;
  if constexpr (kC == Caps::kBoth || kC == Caps::kGateOnly) {
    float t, sech2;
    tanh_sech2(g * p.inv_b1, t, sech2);
    a = p.b1 * t * sg;
    da = sech2 * sg + p.b1 * t * sg * sgm;
  } else {
    a = g * sg;
    da = sg + g * sg * sgm;
  }
  float b, db;
  if constexpr (kC == Caps::kBoth || kC == Caps::kUpOnly) {
    float t, sech2;
    tanh_sech2(u * p.inv_b2, t, sech2);
    b = p.b2 * t;
    db = sech2;
  } else {
    b = u;
    db = 1.0f;
  }
  pg = b * da;
  pu = a * db;
}

// Two FP32 lanes in one 64-bit register pair, for the paired FP32 instructions
// (add/mul/fma .rn.f32x2): one issue slot for two elements.
__device__ __forceinline__ uint64_t f2_pack(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ void f2_unpack(uint64_t v, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ uint64_t f2_add(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ uint64_t f2_mul(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ uint64_t f2_fma(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}

// tanh and sech^2 of two arguments (as tanh_sech2, the FP32 arithmetic paired).
__device__ __forceinline__ void tanh_sech2_x2(uint64_t x, uint64_t& t, uint64_t& sech2) {
  float x0, x1;
  f2_unpack(x, x0, x1);
  t = f2_pack(tanh_approx(x0), tanh_approx(x1));
  const uint64_t e4 = f2_pack(ex2_approx(fmaf(fabsf(x0), -2.0f * kLog2e, 2.0f)),
                              ex2_approx(fmaf(fabsf(x1), -2.0f * kLog2e, 2.0f)));
  float d0, d1;
  f2_unpack(f2_fma(f2_pack(0.25f, 0.25f), e4, f2_pack(1.0f, 1.0f)), d0, d1);
  const uint64_t r = f2_pack(rcp_approx(d0), rcp_approx(d1));
  sech2 = f2_mul(f2_mul(e4, r), r);
}

// d(g, u) of two adjacent outputs: dh * (dh/dg, dh/du) at (g0, u0) and (g1, u1), the
// partial derivatives as in situ_act_grad, with the FP32 products and sums on pairs.
// dh holds the two dh values; returns dg (lo, hi) in og and du in ou.
template <Caps kC>
__device__ __forceinline__ void situ_act_grad_x2(float g0, float g1, float u0, float u1,
                                                 uint64_t dh, const SituParams& p, uint64_t& og,
                                                 uint64_t& ou) {
  const uint64_t one = f2_pack(1.0f, 1.0f);
  const uint64_t e0 = f2_pack(ex2_approx(-fabsf(g0) * kLog2e), ex2_approx(-fabsf(g1) * kLog2e));
  float den0, den1;
  f2_unpack(f2_add(e0, one), den0, den1);
  const float r00 = rcp_approx(den0), r01 = rcp_approx(den1);
  float lo0, lo1;
  f2_unpack(f2_mul(e0, f2_pack(r00, r01)), lo0, lo1);  // sigmoid(-|g|)
  const uint64_t sg = f2_pack(g0 >= 0.0f ? r00 : lo0, g1 >= 0.0f ? r01 : lo1);   // sigmoid(g)
  const uint64_t sgm = f2_pack(g0 >= 0.0f ? lo0 : r00, g1 >= 0.0f ? lo1 : r01);  // sigmoid(-g)
  const uint64_t g = f2_pack(g0, g1), u = f2_pack(u0, u1);
  uint64_t a, da;
  if constexpr (kC == Caps::kBoth || kC == Caps::kGateOnly) {
    uint64_t t, sech2;
    tanh_sech2_x2(f2_mul(g, f2_pack(p.inv_b1, p.inv_b1)), t, sech2);
    a = f2_mul(f2_mul(f2_pack(p.b1, p.b1), t), sg);
    da = f2_fma(a, sgm, f2_mul(sech2, sg));
  } else {
    a = f2_mul(g, sg);
    da = f2_fma(a, sgm, sg);
  }
  uint64_t pg, pu;
  if constexpr (kC == Caps::kBoth || kC == Caps::kUpOnly) {
    uint64_t t, sech2;
    tanh_sech2_x2(f2_mul(u, f2_pack(p.inv_b2, p.inv_b2)), t, sech2);
    pg = f2_mul(f2_mul(f2_pack(p.b2, p.b2), t), da);
    pu = f2_mul(a, sech2);
  } else {
    pg = f2_mul(u, da);
    pu = a;
  }
  og = f2_mul(dh, pg);
  ou = f2_mul(dh, pu);
}

// SiTU-GLU with both caps (the hot path).
__device__ __forceinline__ float situ_glu_f32(float g, float u, const SituParams& p) {
  return situ_act<Caps::kBoth>(g, u, p);
}

}  // namespace situ
