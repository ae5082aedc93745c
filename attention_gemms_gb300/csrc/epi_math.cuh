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
__device__ __forceinline__ float dswiglu_f(float a, float g, float u, float& du) {
  const float s = sigmoid_f(g);
  du = a * g * s;
  return a * u * s * (1.0f + g * (1.0f - s));
}

}  // namespace tp
