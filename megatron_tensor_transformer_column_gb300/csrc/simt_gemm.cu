// simt_gemm.cu -- fp32 path of the t-sharded MLP block (exact fp32 FFMA,
// fp32 accumulation), for problems stored in fp32.
//
// It runs the same problem lists as the tensor-core path (same segments, so
// the g-sum and the f-sum are K loops into one register accumulator here
// too, and the same epilogues), one 32x32 output tile per CTA.  The
// tensor-core path is bf16-only; fp32 storage with a 1e-4 relative bound
// rules out the tf32 tensor-core kind, whose per-product error is too close
// to that bound.
#include <cuda_runtime.h>

#include "act.cuh"
#include "tpmlp_internal.h"

namespace tpmlp {
namespace {

constexpr int kT = 32;        // tile edge (M and N)
constexpr int kK = 32;        // K chunk
constexpr int kThreads = 256; // 32 columns x 8 row groups of 4 rows

// Element (row, col) of a stored row-major array, or of the launch's striped
// input (token stripes) when `striped`.
__device__ __forceinline__ float load_elem(const GemmParams& p, const void* base, int64_t ld, bool striped,
                                           int64_t row, int64_t col) {
  if (striped) {
    const Stripes& st = p.stripes;
    int j = 0;
    while (j + 1 < st.num && row >= st.row0[j + 1]) ++j;
    return static_cast<const float*>(st.in[j])[(row - st.row0[j]) * st.in_ld + col];
  }
  return static_cast<const float*>(base)[row * ld + col];
}

__device__ __forceinline__ float load_a(const GemmParams& p, const Seg& S, int major, int64_t m, int64_t k) {
  return major == MAJOR_MN ? load_elem(p, S.a, S.lda, S.a_striped, k, m) : load_elem(p, S.a, S.lda, S.a_striped, m, k);
}

__device__ __forceinline__ float load_b(const GemmParams& p, const void* b, int64_t ldb, bool striped, int major,
                                        int64_t k, int64_t n) {
  return major == MAJOR_MN ? load_elem(p, b, ldb, striped, k, n) : load_elem(p, b, ldb, striped, n, k);
}

__global__ void __launch_bounds__(kThreads) tpmlp_fp32_simt_gemm(const __grid_constant__ GemmParams p) {
  __shared__ float As[kK][kT + 1];   // [k][m]
  __shared__ float Bs[kK][kT + 1];   // [k][n]
  __shared__ float B2s[kK][kT + 1];  // [k][n] (SwiGLU up projection)

  // tile decode (same raster as the tensor-core path, tile_m = 32)
  const int tile = blockIdx.x;
  int g = 0;
  while (g + 1 < p.num_groups && tile >= p.groups[g + 1].tile_start) ++g;
  const Group& G = p.groups[g];
  int mt, n_lin;
  group_tile(G, tile - G.tile_start, mt, n_lin);
  int pi = G.first_prob;
  while (n_lin >= p.probs[pi].tiles_n) {
    n_lin -= p.probs[pi].tiles_n;
    ++pi;
  }
  const Prob& P = p.probs[pi];
  const int64_t m0 = static_cast<int64_t>(mt) * kT;
  const int64_t n0 = static_cast<int64_t>(n_lin) * P.tile_n;
  const bool dual = P.epi == EPI_SWIGLU_FWD;

  const int tx = threadIdx.x & 31;   // output column in tile
  const int ty = threadIdx.x >> 5;   // rows 4*ty .. 4*ty+3
  float acc[4] = {0.f, 0.f, 0.f, 0.f};
  float acc2[4] = {0.f, 0.f, 0.f, 0.f};

  for (int s = P.seg_begin; s < P.seg_begin + P.seg_count; ++s) {
    const Seg& S = p.segs[s];
    for (int k0 = 0; k0 < S.K; k0 += kK) {
      for (int e = threadIdx.x; e < kT * kK; e += kThreads) {
        // coalesce along the contiguous dimension of each operand
        int mm, kk, nn, kb;
        if (P.a_major == MAJOR_MN) { mm = e & 31; kk = e >> 5; } else { kk = e & 31; mm = e >> 5; }
        if (P.b_major == MAJOR_MN) { nn = e & 31; kb = e >> 5; } else { kb = e & 31; nn = e >> 5; }
        const int64_t gm = m0 + mm, gk = k0 + kk, gn = n0 + nn, gkb = k0 + kb;
        As[kk][mm] = (gm < P.M && gk < S.K) ? load_a(p, S, P.a_major, gm, gk) : 0.f;
        const bool bin = gn < P.N && gkb < S.K;
        Bs[kb][nn] = bin ? load_b(p, S.b, S.ldb, S.b_striped, P.b_major, gkb, gn) : 0.f;
        if (dual) B2s[kb][nn] = bin ? load_b(p, S.b2, S.ldb, false, P.b_major, gkb, gn) : 0.f;
      }
      __syncthreads();
#pragma unroll 8
      for (int kk = 0; kk < kK; ++kk) {
        const float b = Bs[kk][tx];
        const float b2 = dual ? B2s[kk][tx] : 0.f;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float a = As[kk][4 * ty + i];
          acc[i] = fmaf(a, b, acc[i]);
          if (dual) acc2[i] = fmaf(a, b2, acc2[i]);
        }
      }
      __syncthreads();
    }
  }

  const int64_t col = n0 + tx;
  if (col >= P.N) return;
  for (int i = 0; i < 4; ++i) {
    const int64_t row = m0 + 4 * ty + i;
    if (row >= P.M) continue;
    const int64_t o = row * P.ldo + col;
    float v = acc[i];
    switch (P.epi) {
      case EPI_STORE:
        if (P.aux0) v += static_cast<const float*>(P.aux0)[col];
        if (P.out_striped) {  // token stripes of the sequence-parallel layout
          const Stripes& st = p.stripes;
          int j = 0;
          while (j + 1 < st.num && row >= st.row0[j + 1]) ++j;
          static_cast<float*>(st.out[j])[(row - st.row0[j]) * st.out_ld + col] = v;
        } else {
          static_cast<float*>(P.out0)[o] = v;
        }
        break;
      case EPI_GELU_FWD:
        if (P.aux0) v += static_cast<const float*>(P.aux0)[col];
        static_cast<float*>(P.out0)[o] = v;
        static_cast<float*>(P.out1)[o] = act::gelu(v);
        break;
      case EPI_SWIGLU_FWD: {
        float u = acc2[i];
        if (P.aux0) v += static_cast<const float*>(P.aux0)[col];
        if (P.aux1) u += static_cast<const float*>(P.aux1)[col];
        static_cast<float*>(P.out0)[o] = v;
        static_cast<float*>(P.out1)[o] = u;
        static_cast<float*>(P.out2)[o] = u * act::swish(v);
        break;
      }
      case EPI_GELU_BWD: {
        const float a = static_cast<const float*>(P.aux0)[o];
        static_cast<float*>(P.out0)[o] = v * act::gelu_grad(a);
        if (P.out1) static_cast<float*>(P.out1)[o] = act::gelu(a);  // recomputed H
        break;
      }
      case EPI_SWIGLU_BWD: {
        float dg, du;
        const float gg = static_cast<const float*>(P.aux0)[o], uu = static_cast<const float*>(P.aux1)[o];
        act::swiglu_grads(v, gg, uu, dg, du);
        static_cast<float*>(P.out0)[o] = dg;
        static_cast<float*>(P.out1)[o] = du;
        if (P.out2) static_cast<float*>(P.out2)[o] = uu * act::swish(gg);  // recomputed H
        break;
      }
      default:
        break;
    }
  }
}

}  // namespace

cudaError_t launch_simt_gemm(const GemmParams& p, cudaStream_t stream) {
  if (p.total_tiles <= 0) return cudaSuccess;
  tpmlp_fp32_simt_gemm<<<p.total_tiles, kThreads, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace tpmlp
