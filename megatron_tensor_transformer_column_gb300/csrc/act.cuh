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

// Faster forms for the bf16 tensor-core epilogues, whose outputs are rounded
// to bf16 (relative step 2^-8): Phi from the rational approximation of erf
// by Hastings given as formula 7.1.26 in Abramowitz & Stegun (|error of erf|
// <= 1.5e-7), with exp(-a^2/2) shared between Phi and the density in GeLU'.
struct NormTerms {
  float cdf;  // Phi(a)
  float e;    // exp(-a^2 / 2)
};

__device__ __forceinline__ NormTerms norm_terms_fast(float a) {
  constexpr float p = 0.3275911f * kInvSqrt2;  // t = 1 / (1 + p |a| / sqrt 2)
  constexpr float a1 = 0.254829592f, a2 = -0.284496736f, a3 = 1.421413741f, a4 = -1.453152027f,
                  a5 = 1.061405429f;
  const float t = __fdividef(1.0f, fmaf(p, fabsf(a), 1.0f));
  const float poly = t * fmaf(t, fmaf(t, fmaf(t, fmaf(t, a5, a4), a3), a2), a1);
  const float e = __expf(-0.5f * a * a);
  const float q = 0.5f * poly * e;  // Phi(-|a|)
  NormTerms r;
  r.cdf = a >= 0.0f ? 1.0f - q : q;
  r.e = e;
  return r;
}

__device__ __forceinline__ float gelu_fast(float a) { return a * norm_terms_fast(a).cdf; }

__device__ __forceinline__ float gelu_grad_fast(float a) {
  const NormTerms n = norm_terms_fast(a);
  return fmaf(a * kInvSqrt2Pi, n.e, n.cdf);
}

__device__ __forceinline__ float sigmoid_fast(float g) { return __fdividef(1.0f, 1.0f + __expf(-g)); }

__device__ __forceinline__ float swish_fast(float g) { return g * sigmoid_fast(g); }

__device__ __forceinline__ void swiglu_grads_fast(float dh, float g, float u, float& dg, float& du) {
  const float s = sigmoid_fast(g);
  du = dh * (g * s);
  dg = dh * u * (s + g * s * (1.0f - s));
}

}  // namespace act
}  // namespace tpmlp
