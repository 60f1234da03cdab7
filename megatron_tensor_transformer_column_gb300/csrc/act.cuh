// act.cuh -- the activations of the MLP block and their derivatives, fp32.
//
// GeLU is the exact (erf) form, GeLU(a) = a * Phi(a); its derivative is
// Phi(a) + a * phi(a).  Swish is Swish_1(g) = g * sigmoid(g) (SiLU), with
// derivative s + g s (1 - s).  Block definition: "Parallelism" tag page of
// Jiang Yi's homepage, post "megatron-lm", Method / FFN and the SwiGLU
// listing (silu on the W1 projection, times the W3 projection).
#pragma once

#include <stdint.h>

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

// ---- fast packed forms for the bf16 tensor-core epilogues, whose outputs
// are rounded to bf16 (relative step 2^-8): Phi from the rational
// approximation of erf by Hastings given as formula 7.1.26 in Abramowitz &
// Stegun (|error of erf| <= 1.5e-7), with e = exp(-a^2/2) shared between Phi
// and the density in GeLU', the exponentials taken as ex2.approx of an
// argument that carries the log2(e) scale (so e = 1 exactly at a = 0, and
// GeLU'(0) = 1/2 exactly), and the reciprocals from the fast reciprocal.  Two
// elements per fp32x2 instruction (fma/mul/add.rn.f32x2): every step but the
// special-function calls (reciprocal, exponential) acts on a pair:
//   q = Phi(-|a|) = 0.5 * poly(t) * e, t = 1 / (1 + p |a|), e = 2^(a^2 (-log2(e) / 2));
//   GeLU(a) = a Phi(a) = max(a, 0) - |a| q;
//   Phi(a) = 0.5 + copysign(0.5 - q, a),  GeLU'(a) = Phi(a) + a phi(a).
namespace x2 {

__device__ __forceinline__ uint64_t pk(float a, float b) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
  return r;
}
__device__ __forceinline__ void upk(uint64_t v, float& a, float& b) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(v));
}
__device__ __forceinline__ uint64_t fma2(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t r;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
  return r;
}
__device__ __forceinline__ uint64_t mul2(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ uint64_t add2(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ uint64_t splat(float a) { return pk(a, a); }

// 2^y, the hardware approximation (PTX ex2.approx.ftz: relative error about
// 2^-22; results below 2^-126 flush to zero).
__device__ __forceinline__ float ex2(float y) {
  float r;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(y));
  return r;
}
__device__ __forceinline__ uint64_t ex2_pair(uint64_t y) {
  float y0, y1;
  upk(y, y0, y1);
  return pk(ex2(y0), ex2(y1));
}

constexpr float kLog2E = 1.44269504088896340736f;

// q = Phi(-|a|) and e = exp(-a^2/2) for a pair; nx = -|a|.
__device__ __forceinline__ void norm_q(uint64_t a, uint64_t& nx, uint64_t& q, uint64_t& e) {
  constexpr float p = 0.3275911f * kInvSqrt2;
  // Abramowitz & Stegun 7.1.26 coefficients, halved: q = poly * e
  constexpr float c1 = 0.5f * 0.254829592f, c2 = 0.5f * -0.284496736f, c3 = 0.5f * 1.421413741f,
                  c4 = 0.5f * -1.453152027f, c5 = 0.5f * 1.061405429f;
  float a0, a1;
  upk(a, a0, a1);
  nx = pk(-fabsf(a0), -fabsf(a1));
  const uint64_t den = fma2(splat(-p), nx, splat(1.0f));  // 1 + p |a|
  float d0, d1;
  upk(den, d0, d1);
  const uint64_t t = pk(__fdividef(1.0f, d0), __fdividef(1.0f, d1));
  uint64_t poly = fma2(t, splat(c5), splat(c4));
  poly = fma2(t, poly, splat(c3));
  poly = fma2(t, poly, splat(c2));
  poly = fma2(t, poly, splat(c1));
  poly = mul2(t, poly);
  e = ex2_pair(mul2(mul2(a, a), splat(-0.5f * kLog2E)));
  q = mul2(poly, e);
}

// h = GeLU(a) for v[0..N-1] in place (N even).
template <int N>
__device__ __forceinline__ void gelu_xn(float (&v)[N]) {
#pragma unroll
  for (int j = 0; j < N; j += 2) {
    const uint64_t a = pk(v[j], v[j + 1]);
    uint64_t nx, q, e;
    norm_q(a, nx, q, e);
    const uint64_t h = fma2(nx, q, pk(fmaxf(v[j], 0.0f), fmaxf(v[j + 1], 0.0f)));
    upk(h, v[j], v[j + 1]);
  }
}

// dA = dH * GeLU'(A): acc holds dH, a holds A on entry and dA on exit; with
// kWithH, h receives GeLU(A) as well.
template <bool kWithH, int N>
__device__ __forceinline__ void gelu_bwd_xn(const float (&acc)[N], float (&a)[N], float (&h)[N]) {
#pragma unroll
  for (int j = 0; j < N; j += 2) {
    const uint64_t av = pk(a[j], a[j + 1]);
    uint64_t nx, q, e;
    norm_q(av, nx, q, e);
    float m0, m1;
    upk(fma2(q, splat(-1.0f), splat(0.5f)), m0, m1);  // 0.5 - q, then its sign from a
    const uint64_t cdf = add2(splat(0.5f), pk(copysignf(m0, a[j]), copysignf(m1, a[j + 1])));
    const uint64_t grad = fma2(av, mul2(e, splat(kInvSqrt2Pi)), cdf);
    if (kWithH) {
      const uint64_t hv = fma2(nx, q, pk(fmaxf(a[j], 0.0f), fmaxf(a[j + 1], 0.0f)));
      upk(hv, h[j], h[j + 1]);
    }
    upk(mul2(pk(acc[j], acc[j + 1]), grad), a[j], a[j + 1]);
  }
}

// s = sigmoid(g) for a pair: 1 / (1 + 2^(-g log2(e))).
__device__ __forceinline__ uint64_t sigmoid2(float g0, float g1) {
  const uint64_t den = add2(splat(1.0f), ex2_pair(mul2(pk(g0, g1), splat(-kLog2E))));
  float d0, d1;
  upk(den, d0, d1);
  return pk(__fdividef(1.0f, d0), __fdividef(1.0f, d1));
}

// h = u * Swish(g) for N pairs of (g, u).
template <int N>
__device__ __forceinline__ void swiglu_xn(const float (&g)[N], const float (&u)[N], float (&h)[N]) {
#pragma unroll
  for (int j = 0; j < N; j += 2) {
    const uint64_t gv = pk(g[j], g[j + 1]);
    const uint64_t s = sigmoid2(g[j], g[j + 1]);
    upk(mul2(pk(u[j], u[j + 1]), mul2(gv, s)), h[j], h[j + 1]);
  }
}

// dG = dH * U * Swish'(G), dU = dH * Swish(G); g, u hold G, U on entry and
// dG, dU on exit; with kWithH, h receives U * Swish(G).
template <bool kWithH, int N>
__device__ __forceinline__ void swiglu_bwd_xn(const float (&acc)[N], float (&g)[N], float (&u)[N], float (&h)[N]) {
#pragma unroll
  for (int j = 0; j < N; j += 2) {
    const uint64_t gv = pk(g[j], g[j + 1]), uv = pk(u[j], u[j + 1]), dh = pk(acc[j], acc[j + 1]);
    const uint64_t s = sigmoid2(g[j], g[j + 1]);
    const uint64_t gs = mul2(gv, s);                                      // Swish(G)
    if (kWithH) upk(mul2(uv, gs), h[j], h[j + 1]);
    const uint64_t ds = fma2(gs, fma2(s, splat(-1.0f), splat(1.0f)), s);  // s + g s (1 - s)
    upk(mul2(mul2(dh, uv), ds), g[j], g[j + 1]);
    upk(mul2(dh, gs), u[j], u[j + 1]);
  }
}

}  // namespace x2

}  // namespace act
}  // namespace tpmlp
