// colsum.cu -- column sums over the token dimension, for the bias gradients
// of the MLP block: db2 = sum over tokens of dY, db1_i = sum over tokens of
// dA_i (SwiGLU: dG_i), db3_i = sum over tokens of dU_i.  ("Tensor
// parallelism", brunomaga.github.io, Megatron_FeedForward: fc1 carries a bias,
// fc2's bias is added once after the all-reduce, so its gradient is that of
// the whole Y.)
//
// HBM-bound: every input byte is read once.  A cluster of 8 CTAs owns one
// column strip of one matrix and splits its rows into 8 chunks.  In a CTA of
// 256 threads, kLaneThreads threads cover a strip row with 16-byte loads
// (strips of 128, 64 or 32 bytes) and the other factor, the row lanes, walk
// the chunk kUnroll rows at a time (independent loads in flight per thread);
// the lane partials of a column are added in a fixed tree order in shared
// memory; CTA 0 of the cluster then adds the 8 chunk partials in rank order
// through distributed shared memory.  The result is the same on every run: no
// atomics, no global scratch.  The host picks the widest strip that still
// gives the launch enough CTAs to fill the GPU (colsum_lane_threads).  A job
// without a source reads the launch's token stripes (the dY stripes of the
// sequence-parallel layout) as one tensor.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "ptx.cuh"
#include "tpmlp_internal.h"

namespace tpmlp {
namespace {

constexpr int kThreads = 256;
constexpr int kChunks = 8;  // CTAs per cluster (row chunks of a strip)

template <bool kBf16, int kPer>
__device__ __forceinline__ void accumulate_row(const void* src, int64_t off, float (&acc)[kPer]) {
  if (kBf16) {
    const uint4 q = __ldg(reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(src) + off));
    const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w[e]));
      acc[2 * e] += f.x;
      acc[2 * e + 1] += f.y;
    }
  } else {
    const float4 q = __ldg(reinterpret_cast<const float4*>(static_cast<const float*>(src) + off));
    acc[0] += q.x;
    acc[1] += q.y;
    acc[2] += q.z;
    acc[3] += q.w;
  }
}

template <bool kBf16, int kLaneThreads, int kUnroll>
__global__ void __launch_bounds__(kThreads) tpmlp_bias_grad_colsum(const __grid_constant__ ColsumParams p) {
  constexpr int kPer = kBf16 ? 8 : 4;  // elements per 16-byte load
  constexpr int kRowLanes = kThreads / kLaneThreads;
  constexpr int kStripCols = kLaneThreads * kPer;
  __shared__ float part[kRowLanes][kStripCols + 1];

  const int strip_global = blockIdx.x / kChunks;
  const uint32_t chunk = ptx::cluster_ctarank();
  int j = 0;
  while (j + 1 < p.num_jobs && strip_global >= p.jobs[j + 1].strip_begin) ++j;
  const ColsumJob& J = p.jobs[j];
  const int strip = strip_global - J.strip_begin;
  const int lane_row = threadIdx.x / kLaneThreads;
  const int lane_col = threadIdx.x % kLaneThreads;
  const int64_t col0 = static_cast<int64_t>(strip) * kStripCols + lane_col * kPer;
  const bool col_ok = col0 < J.cols;  // cols is a multiple of kPer
  const int64_t per_chunk = (J.rows + kChunks - 1) / kChunks;
  const int64_t r_begin = per_chunk * chunk;
  const int64_t r_end = min(J.rows, r_begin + per_chunk);

  float acc[kPer];
#pragma unroll
  for (int e = 0; e < kPer; ++e) acc[e] = 0.f;
  if (col_ok && !J.src) {
    // token stripes (sequence-parallel layout): walk the rows stripe by stripe
    int sj = 0;
    for (int64_t r = r_begin + lane_row; r < r_end; r += kRowLanes) {
      while (sj + 1 < p.num_stripes && r >= p.stripe_row0[sj + 1]) ++sj;
      accumulate_row<kBf16, kPer>(p.stripe_src[sj], (r - p.stripe_row0[sj]) * J.cols + col0, acc);
    }
  } else if (col_ok) {
    int64_t r = r_begin + lane_row;
    for (; r + (kUnroll - 1) * kRowLanes < r_end; r += kUnroll * kRowLanes) {
      float a[kUnroll][kPer];
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) {
#pragma unroll
        for (int e = 0; e < kPer; ++e) a[u][e] = 0.f;
        accumulate_row<kBf16, kPer>(J.src, (r + u * kRowLanes) * J.cols + col0, a[u]);
      }
#pragma unroll
      for (int u = 0; u < kUnroll; ++u)
#pragma unroll
        for (int e = 0; e < kPer; ++e) acc[e] += a[u][e];
    }
    for (; r < r_end; r += kRowLanes) accumulate_row<kBf16, kPer>(J.src, r * J.cols + col0, acc);
  }
#pragma unroll
  for (int e = 0; e < kPer; ++e) part[lane_row][lane_col * kPer + e] = acc[e];
  __syncthreads();
  // Fixed-order tree over the 32 row lanes of this chunk.
  for (int half = kRowLanes / 2; half > 0; half >>= 1) {
    for (int i = threadIdx.x; i < half * kStripCols; i += kThreads) {
      const int rr = i / kStripCols, cc = i % kStripCols;
      part[rr][cc] += part[rr + half][cc];
    }
    __syncthreads();
  }
  ptx::cluster_sync();  // every chunk's partial is in its shared memory
  if (chunk == 0) {
    for (int c = threadIdx.x; c < kStripCols; c += kThreads) {
      float s = part[0][c];
      const uint32_t local = ptx::smem_u32(&part[0][c]);
      for (uint32_t k = 1; k < kChunks; ++k) {
        float v;
        asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(ptx::map_to_cta(local, k)) : "memory");
        s += v;
      }
      const int64_t col = static_cast<int64_t>(strip) * kStripCols + c;
      if (col < J.cols) {
        if (kBf16)
          static_cast<__nv_bfloat16*>(J.dst)[col] = __float2bfloat16_rn(s);
        else
          static_cast<float*>(J.dst)[col] = s;
      }
    }
  }
  ptx::cluster_sync();  // peers keep their shared memory until CTA 0 has read it
}

}  // namespace

int colsum_strip_cols(bool bf16, int lane_threads) { return lane_threads * (bf16 ? 8 : 4); }

// The launch shape of a set of jobs: lane threads per strip row (strips of
// 128, 64 or 32 bytes) and rows in flight per thread.  128-byte strips read
// best (measured on GB300: C5's db2, the column sums of dY, 29 us with 64-byte
// strips against 23 us with 128-byte ones, both 8 rows ahead); narrower ones
// only for launches too small to give the GPU a fifth of its slots (8 CTAs
// per SM) otherwise.  8 rows ahead while the launch leaves slots empty, 4
// when it fills most of them (C5's db1: 73 us with 4, 76 us with 8).
ColsumShape colsum_shape(const ColsumJob* jobs, int num_jobs, bool bf16, int sms) {
  const int64_t slots = int64_t{8} * sms;
  auto ctas = [&](int lt) {
    int64_t n = 0;
    for (int j = 0; j < num_jobs; ++j) n += kChunks * ((jobs[j].cols + colsum_strip_cols(bf16, lt) - 1) / colsum_strip_cols(bf16, lt));
    return n;
  };
  int lt = 2;
  for (int c : {8, 4})
    if (ctas(c) * 5 >= slots) {
      lt = c;
      break;
    }
  return ColsumShape{lt, ctas(lt) * 5 >= slots * 4 ? 4 : 8};
}

cudaError_t launch_colsum(const ColsumParams& p, bool bf16, ColsumShape shape, cudaStream_t stream) {
  if (p.total_strips <= 0) return cudaSuccess;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.total_strips * kChunks, 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = kChunks;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const int key = (bf16 ? 100 : 0) + 10 * shape.lane_threads + shape.unroll;
  switch (key) {
    case 184: return cudaLaunchKernelEx(&cfg, tpmlp_bias_grad_colsum<true, 8, 4>, p);
    case 188: return cudaLaunchKernelEx(&cfg, tpmlp_bias_grad_colsum<true, 8, 8>, p);
    case 148: return cudaLaunchKernelEx(&cfg, tpmlp_bias_grad_colsum<true, 4, 8>, p);
    case 128: return cudaLaunchKernelEx(&cfg, tpmlp_bias_grad_colsum<true, 2, 8>, p);
    case 84: return cudaLaunchKernelEx(&cfg, tpmlp_bias_grad_colsum<false, 8, 4>, p);
    case 88: return cudaLaunchKernelEx(&cfg, tpmlp_bias_grad_colsum<false, 8, 8>, p);
    case 48: return cudaLaunchKernelEx(&cfg, tpmlp_bias_grad_colsum<false, 4, 8>, p);
    case 28: return cudaLaunchKernelEx(&cfg, tpmlp_bias_grad_colsum<false, 2, 8>, p);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace tpmlp
