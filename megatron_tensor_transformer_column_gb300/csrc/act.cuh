// act.cuh -- the activations of the MLP block and their derivatives, fp32.
//
// GeLU is the exact (erf) form, GeLU(a) = a * Phi(a); its derivative is
// Phi(a) + a * phi(a).  Swish is Swish_1(g) = g * sigmoid(g) (SiLU), with
// derivative s + g s (1 - s).  Block definition: "Parallelism" tag page of
// Jiang Yi's homepage, post "megatron-lm", Method / FFN and the SwiGLU
// listing (silu on the W1 projection, times the W3 projection).
#pragma once

namespace tpmlp {
namespace act {

constexpr float kInvSqrt2 = 0.70710678118654752440f;
constexpr float kInvSqrt2Pi = 0.39894228040143267794f;

__device__ __forceinline__ float norm_cdf(float a) { return 0.5f * (1.0f + erff(a * kInvSqrt2)); }

__device__ __forceinline__ float gelu(float a) { return a * norm_cdf(a); }

__device__ __forceinline__ float gelu_grad(float a) {
  return norm_cdf(a) + a * (kInvSqrt2Pi * expf(-0.5f * a * a));
}

__device__ __forceinline__ float sigmoid(float g) { return 1.0f / (1.0f + expf(-g)); }

__device__ __forceinline__ float swish(float g) { return g * sigmoid(g); }

// dG and dU of H = U * Swish(G) given dH.
__device__ __forceinline__ void swiglu_grads(float dh, float g, float u, float& dg, float& du) {
  const float s = sigmoid(g);
  du = dh * (g * s);
  dg = dh * u * (s + g * s * (1.0f - s));
}

}  // namespace act
}  // namespace tpmlp
