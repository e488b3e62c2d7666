// Expert activations of the grouped GEMM epilogue, two columns per packed fp32x2
// operation. Kept in a header of their own so that a test kernel can run the very
// same device code over a dense sweep of inputs.
//
// Pages: "Mixture of Experts" (aigrafen.se) MoE code and "MoE Architecture"
// (vanos001.github.io) StandardExpert: GELU, the exact erf form of nn.GELU;
// "MoE Architecture" SwiGLUExpert: silu(W1 x) * (W3 x), silu(a) = a / (1 + e^-a).
#pragma once

#include <cuda_runtime.h>

namespace moe {
namespace act {

__device__ __forceinline__ float ex2_ftz(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ float rcp_ftz(float x) {
  float y;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// GELU(u) = u * Phi(u) = 0.5 u (1 + erf(u / sqrt 2)), with erf from Abramowitz &
// Stegun, Handbook of Mathematical Functions, formula 7.1.28 (after Hastings):
// erf(z) = 1 - 1 / (1 + a1 z + ... + a6 z^6)^16, z >= 0, |error| <= 3e-7 -- far
// below the bf16 rounding of the stored result. With z = |u| / sqrt 2 and the
// factor 1/2 of Phi taken into the polynomial as 2^(1/16):
//   Phi(-|u|) = 1 / q(|u|)^16,  q(y) = c0 + c1 y + ... + c6 y^6,  c_i = 2^(1/16) a_i 2^(-i/2), a0 = 1,
// and GELU(u) = max(u, 0) - |u| Phi(-|u|) for either sign of u (no select): six
// FMAs, four squarings and one reciprocal per value (q^16 overflows to infinity
// for |u| > ~20, where the reciprocal's zero is the exact limit). Two values per
// packed fp32x2 multiply / FMA.
__device__ __forceinline__ float2 gelu2_as7128(float2 u) {
  constexpr double kR = 1.0442737824274138;  // 2^(1/16)
  constexpr double kH = 0.7071067811865476;  // 2^(-1/2)
  constexpr float kC0 = (float)kR, kC1 = (float)(kR * 0.0705230784 * kH),
                  kC2 = (float)(kR * 0.0422820123 * kH * kH), kC3 = (float)(kR * 0.0092705272 * kH * kH * kH),
                  kC4 = (float)(kR * 0.0001520143 * kH * kH * kH * kH),
                  kC5 = (float)(kR * 0.0002765672 * kH * kH * kH * kH * kH),
                  kC6 = (float)(kR * 0.0000430638 * kH * kH * kH * kH * kH * kH);
  const float2 y = make_float2(fabsf(u.x), fabsf(u.y));
  float2 q = __ffma2_rn(make_float2(kC6, kC6), y, make_float2(kC5, kC5));
  q = __ffma2_rn(q, y, make_float2(kC4, kC4));
  q = __ffma2_rn(q, y, make_float2(kC3, kC3));
  q = __ffma2_rn(q, y, make_float2(kC2, kC2));
  q = __ffma2_rn(q, y, make_float2(kC1, kC1));
  q = __ffma2_rn(q, y, make_float2(kC0, kC0));
  q = __fmul2_rn(q, q);  // q^2
  q = __fmul2_rn(q, q);  // q^4
  q = __fmul2_rn(q, q);  // q^8
  q = __fmul2_rn(q, q);  // q^16
  const float2 nphi = make_float2(rcp_ftz(-q.x), rcp_ftz(-q.y));  // -Phi(-|u|)
  return __ffma2_rn(y, nphi, make_float2(fmaxf(u.x, 0.f), fmaxf(u.y, 0.f)));
}

// SwiGLU's hidden value silu(a) * b = a / (1 + 2^(-a log2 e)) * b, two columns per
// packed operation (for a < ~ -88 the power overflows to infinity and the
// reciprocal's zero is the limit).
__device__ __forceinline__ float2 silu_mul2(float2 a, float2 b) {
  const float2 m = __fmul2_rn(a, make_float2(-1.4426950408889634f, -1.4426950408889634f));
  const float2 den = __fadd2_rn(make_float2(ex2_ftz(m.x), ex2_ftz(m.y)), make_float2(1.f, 1.f));
  return __fmul2_rn(__fmul2_rn(a, make_float2(rcp_ftz(den.x), rcp_ftz(den.y))), b);
}

}  // namespace act
}  // namespace moe
