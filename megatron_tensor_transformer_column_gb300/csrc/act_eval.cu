// act_eval.cu -- runs the epilogues' activation code on plain device arrays,
// so that the exact instruction sequences the GEMM epilogues use (act.cuh)
// can be compared, element by element, with a reference over a dense grid
// of inputs.  Nothing here is on the hot path.
#include <cuda_runtime.h>

#include "act.cuh"
#include "tpmlp.h"
#include "tpmlp_internal.h"

namespace tpmlp {
namespace {

// Each thread evaluates 32 consecutive elements through the same entry
// points the tensor-core epilogues call (their arithmetic is element-wise, so
// the chunk width does not change a result) (elements past n are padded with
// zeros and not stored); the fp32 forms are evaluated per element, as the
// fp32 path's epilogue does.
__global__ void __launch_bounds__(128) tpmlp_act_eval(int fn, const float* __restrict__ x,
                                                      const float* __restrict__ y, const float* __restrict__ dh,
                                                      float* __restrict__ o0, float* __restrict__ o1,
                                                      float* __restrict__ o2, int64_t n) {
  const int64_t base = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) * 32;
  if (base >= n) return;
  const int cnt = n - base < 32 ? static_cast<int>(n - base) : 32;
  float a[32], b[32], c[32], h[32];
#pragma unroll
  for (int j = 0; j < 32; ++j) {
    const bool ok = j < cnt;
    a[j] = ok ? x[base + j] : 0.0f;
    b[j] = (ok && y) ? y[base + j] : 0.0f;
    c[j] = (ok && dh) ? dh[base + j] : 0.0f;
    h[j] = 0.0f;
  }
  switch (fn) {
    case TPMLP_ACT_EVAL_GELU:  // o0 = GeLU(x)
      act::x2::gelu_xn(a);
      for (int j = 0; j < cnt; ++j) o0[base + j] = a[j];
      break;
    case TPMLP_ACT_EVAL_GELU_BWD:  // o0 = dh * GeLU'(x)
      act::x2::gelu_bwd_xn<false>(c, a, h);
      for (int j = 0; j < cnt; ++j) o0[base + j] = a[j];
      break;
    case TPMLP_ACT_EVAL_GELU_BWD_H:  // o0 = dh * GeLU'(x), o1 = GeLU(x)
      act::x2::gelu_bwd_xn<true>(c, a, h);
      for (int j = 0; j < cnt; ++j) {
        o0[base + j] = a[j];
        o1[base + j] = h[j];
      }
      break;
    case TPMLP_ACT_EVAL_SWIGLU:  // o0 = y * Swish(x)
      act::x2::swiglu_xn(a, b, h);
      for (int j = 0; j < cnt; ++j) o0[base + j] = h[j];
      break;
    case TPMLP_ACT_EVAL_SWIGLU_BWD:  // o0 = dG, o1 = dU
    case TPMLP_ACT_EVAL_SWIGLU_BWD_H:  // and o2 = y * Swish(x)
      if (fn == TPMLP_ACT_EVAL_SWIGLU_BWD_H)
        act::x2::swiglu_bwd_xn<true>(c, a, b, h);
      else
        act::x2::swiglu_bwd_xn<false>(c, a, b, h);
      for (int j = 0; j < cnt; ++j) {
        o0[base + j] = a[j];
        o1[base + j] = b[j];
        if (fn == TPMLP_ACT_EVAL_SWIGLU_BWD_H) o2[base + j] = h[j];
      }
      break;
    case TPMLP_ACT_EVAL_FP32_GELU:  // the fp32 path: o0 = GeLU(x), o1 = dh * GeLU'(x)
      for (int j = 0; j < cnt; ++j) {
        o0[base + j] = act::gelu(a[j]);
        o1[base + j] = c[j] * act::gelu_grad(a[j]);
      }
      break;
    case TPMLP_ACT_EVAL_FP32_SWIGLU:  // o0 = y * Swish(x), o1 = dG, o2 = dU
      for (int j = 0; j < cnt; ++j) {
        float dg, du;
        act::swiglu_grads(c[j], a[j], b[j], dg, du);
        o0[base + j] = b[j] * act::swish(a[j]);
        o1[base + j] = dg;
        o2[base + j] = du;
      }
      break;
    default:
      break;
  }
}

}  // namespace

cudaError_t launch_act_eval(int fn, const float* x, const float* y, const float* dh, float* o0, float* o1,
                            float* o2, int64_t n, cudaStream_t stream) {
  if (n <= 0) return cudaSuccess;
  const int64_t threads = (n + 31) / 32;
  const int64_t blocks = (threads + 127) / 128;
  tpmlp_act_eval<<<static_cast<unsigned>(blocks), 128, 0, stream>>>(fn, x, y, dh, o0, o1, o2, n);
  return cudaGetLastError();
}

}  // namespace tpmlp
