// Elementwise math of the epilogues, fp32.
//   GELU(x)  = x * Phi(x) = x * 1/2 [1 + erf(x / sqrt 2)]      (exact erf form)
//   GELU'(x) = Phi(x) + x * phi(x),  phi(x) = exp(-x^2/2) / sqrt(2 pi)
//   SiLU(x)  = x * s(x), s(x) = 1 / (1 + e^-x);  SiLU'(x) = s(x) (1 + x (1 - s(x)))
// GELU is the formula of the 张量并行 notes (§MLP 层的并行化); SiLU is the gate of
// the SwiGLU named (not written out) in 20260402-parallelism, §1 TP.
#pragma once
#include <cuda_bf16.h>

namespace tp {

__device__ __forceinline__ float gelu_f(float x) {
  return 0.5f * x * (1.0f + erff(x * 0.70710678118654752f));
}

__device__ __forceinline__ float gelu_prime_f(float x) {
  const float cdf = 0.5f * (1.0f + erff(x * 0.70710678118654752f));
  const float pdf = 0.39894228040143268f * expf(-0.5f * x * x);
  return cdf + x * pdf;
}

__device__ __forceinline__ float sigmoid_f(float x) { return 1.0f / (1.0f + expf(-x)); }

__device__ __forceinline__ float silu_f(float x) { return x * sigmoid_f(x); }

// returns dG, writes dU:  a = dA, g = gate pre-activation, u = up pre-activation
__device__ __forceinline__ float dswiglu_of(float a, float g, float u, float s, float& du) {
  du = a * g * s;
  return a * u * s * (1.0f + g * (1.0f - s));
}
__device__ __forceinline__ float dswiglu_f(float a, float g, float u, float& du) {
  return dswiglu_of(a, g, u, sigmoid_f(g), du);
}

// The same on the special-function unit, for epilogues whose results are rounded to
// bf16: e^-x = 2^(-x log2 e) by ex2.approx and the reciprocal by rcp.approx, each
// within a few fp32 ulp (about 1e-6 relative in all), where bf16 keeps 8 bits. The
// full-precision forms above cost an accurate exponential and an IEEE division per
// element, which made the epilogue warps, not the tensor core, the limit of the
// SwiGLU GEMMs. Large |x| saturate correctly: e^-x = inf gives 0, e^-x = 0 gives 1.
__device__ __forceinline__ float sigmoid_sfu(float x) {
  float e, r;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(e) : "f"(x * -1.4426950408889634f));
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(1.0f + e));
  return r;
}
__device__ __forceinline__ float silu_sfu(float x) { return x * sigmoid_sfu(x); }
__device__ __forceinline__ float dswiglu_sfu(float a, float g, float u, float& du) {
  return dswiglu_of(a, g, u, sigmoid_sfu(g), du);
}

}  // namespace tp
