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

// Phi and phi for the bf16 epilogues, after Abramowitz & Stegun, Handbook of
// Mathematical Functions, 7.1.26 (Hastings' approximation):
//   erfc(z) = t (a1 + t (a2 + t (a3 + t (a4 + t a5)))) e^(-z^2),  t = 1 / (1 + p z),  z >= 0,
// absolute error below 1.5e-7 (CUDA's erff is within ~1e-7). With z = |x| / sqrt 2,
// e^(-z^2) = e^(-x^2 / 2) = sqrt(2 pi) phi(x), so GELU' = Phi + x phi takes one
// exponential for both terms; the exponential (2^(-x^2 log2(e) / 2)) and the reciprocal
// run on the SFU. Phi is formed from the small tail erfc(|x| / sqrt 2) / 2 on either side.
__device__ __forceinline__ void normal_sfu(float x, float& Phi, float& phi) {
  float t, e;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(t) : "f"(fmaf(0.3275911f * 0.70710678118654752f, fabsf(x), 1.0f)));
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(e) : "f"(x * x * -0.72134752044448170f));
  const float poly =
      t * fmaf(t, fmaf(t, fmaf(t, fmaf(t, 1.061405429f, -1.453152027f), 1.421413741f), -0.284496736f),
               0.254829592f);
  const float tail = 0.5f * poly * e;  // P(N(0,1) > |x|)
  Phi = x >= 0.0f ? 1.0f - tail : tail;
  phi = 0.39894228040143268f * e;
}
__device__ __forceinline__ float gelu_sfu(float x) {
  float Phi, phi;
  normal_sfu(x, Phi, phi);
  return x * Phi;
}
__device__ __forceinline__ float gelu_prime_sfu(float x) {
  float Phi, phi;
  normal_sfu(x, Phi, phi);
  return fmaf(x, phi, Phi);
}
__device__ __forceinline__ float dswiglu_sfu(float a, float g, float u, float& du) {
  return dswiglu_of(a, g, u, sigmoid_sfu(g), du);
}

}  // namespace tp
