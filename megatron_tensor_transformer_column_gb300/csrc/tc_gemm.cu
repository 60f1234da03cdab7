// tc_gemm.cu -- persistent, warp-specialised tcgen05 GEMM for sm_103a with
// the MLP block's fused epilogues.
//
// One CTA per SM.  Warp 0 (one lane) streams 64x64 bf16 boxes of A and B
// into a 4-stage shared-memory ring with TMA; warp 1 (one lane) allocates
// 512 TMEM columns and issues tcgen05.mma into one of two 128x256 fp32
// accumulators; warps 2..9 drain the other accumulator through tcgen05.ld,
// apply the epilogue (store, GeLU / SwiGLU forward, GeLU' / SwiGLU'
// backward) and write bf16 rows straight to HBM.  The two accumulators let
// the epilogue of one tile run under the main loop of the next.
//
// The shard sums of the tensor-parallel MLP are K loops here: a problem
// with several segments (one per shard) accumulates every segment's product
// into the same TMEM tile before the epilogue reads it, so the g-sum of the
// forward row-parallel GEMM and the f-sum of the dX GEMM never leave the
// chip.  ("Parallelism" tag page of Jiang Yi's homepage, post "megatron-lm",
// Method / FFN: the partial-sum identity [H1, H2][W21; W22] = H1 W21 + H2 W22
// and the f/g table.)
//
// Every wait is bounded: after GemmParams::timeout_ns a waiting role records
// a status code in the workspace, raises a shared abort flag that makes the
// other roles leave their loops, waits (again bounded) for its own copies
// and MMAs in flight, and the CTA frees its TMEM and exits.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "act.cuh"
#include "ptx.cuh"
#include "tpmlp_internal.h"

namespace tpmlp {
namespace {

constexpr int kBM = 128;                        // tile rows (MMA M)
constexpr int kBK = 64;                         // K per stage (one 128-byte swizzle row of bf16)
constexpr int kStages = 4;
constexpr int kBoxBytes = 64 * 64 * 2;          // one TMA box: 64 x 64 bf16
constexpr int kStageBytes = 6 * kBoxBytes;      // 2 A boxes + 4 B boxes
constexpr int kNumEpiWarps = 8;
constexpr int kThreads = 32 * (2 + kNumEpiWarps);
constexpr int kTmemCols = 512;
constexpr int kAccCols = 256;
constexpr int kNumAcc = 2;
constexpr int kNumBars = 2 * kStages + 2 * kNumAcc + 1;
constexpr int kSmemBytes = 1024 + kStages * kStageBytes + 8 * kNumBars + 16;
constexpr uint64_t kDrainTimeoutNs = 200ull * 1000 * 1000;

static_assert(kSmemBytes <= 227 * 1024, "shared memory budget");
static_assert(kNumAcc * kAccCols <= kTmemCols, "TMEM budget");

struct TileInfo {
  int prob, m0, n0, valid_m, valid_n;
};

__device__ __forceinline__ TileInfo decode_tile(const GemmParams& p, int tile) {
  int g = 0;
  while (g + 1 < p.num_groups && tile >= p.groups[g + 1].tile_start) ++g;
  const Group& G = p.groups[g];
  const int local = tile - G.tile_start;
  const int full_band = G.band_m * G.tiles_per_row;
  const int band = local / full_band;
  const int m_first = band * G.band_m;
  const int bm = min(G.band_m, G.tiles_m - m_first);
  const int r = local - band * full_band;
  int n_lin = r / bm;
  const int mt = m_first + (r - n_lin * bm);
  int pi = G.first_prob;
  while (n_lin >= p.probs[pi].tiles_n) {
    n_lin -= p.probs[pi].tiles_n;
    ++pi;
  }
  const Prob& P = p.probs[pi];
  TileInfo t;
  t.prob = pi;
  t.m0 = mt * kBM;
  t.n0 = n_lin * P.tile_n;
  t.valid_m = min(kBM, P.M - t.m0);
  t.valid_n = min(P.tile_n, P.N - t.n0);
  return t;
}

struct Ctl {
  volatile int32_t* abort_flag;
  int32_t* status;
  uint64_t timeout_ns;
};

// Wait for the phase of `bar` with the given parity; false if the wait
// timed out (status recorded) or another role aborted.
__device__ __forceinline__ bool bounded_wait(uint32_t bar, uint32_t parity, const Ctl& c, int32_t code) {
  if (ptx::mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = ptx::globaltimer_ns();
  while (true) {
    if (ptx::mbar_try_wait(bar, parity)) return true;
    if (*c.abort_flag) return false;
    if (ptx::globaltimer_ns() - t0 > c.timeout_ns) {
      *c.abort_flag = 1;
      if (c.status) atomicCAS(c.status, 0, code);
      return false;
    }
  }
}

// Wait used while draining after an abort: bounded, ignores the abort flag.
__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity) {
  const uint64_t t0 = ptx::globaltimer_ns();
  while (!ptx::mbar_try_wait(bar, parity)) {
    if (ptx::globaltimer_ns() - t0 > kDrainTimeoutNs) return;
  }
}

__device__ __forceinline__ uint32_t pack_bf16x2(float a, float b) {
  __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&v);
}

__device__ __forceinline__ float2 unpack_bf16x2(uint32_t v) {
  __nv_bfloat162 h = *reinterpret_cast<__nv_bfloat162*>(&v);
  return __bfloat1622float2(h);
}

// Store 32 consecutive values of one row (nvalid of them, a multiple of 8)
// as bf16 with 16-byte stores.
__device__ __forceinline__ void store_row32(void* out, int64_t ldo, int64_t row, int col, int nvalid,
                                            const float (&v)[32]) {
  __nv_bfloat16* dst = reinterpret_cast<__nv_bfloat16*>(out) + row * ldo + col;
#pragma unroll
  for (int g = 0; g < 4; ++g) {
    if (8 * g < nvalid) {
      uint4 o;
      o.x = pack_bf16x2(v[8 * g + 0], v[8 * g + 1]);
      o.y = pack_bf16x2(v[8 * g + 2], v[8 * g + 3]);
      o.z = pack_bf16x2(v[8 * g + 4], v[8 * g + 5]);
      o.w = pack_bf16x2(v[8 * g + 6], v[8 * g + 7]);
      *reinterpret_cast<uint4*>(dst + 8 * g) = o;
    }
  }
}

__device__ __forceinline__ void load_row32(const void* src, int64_t ld, int64_t row, int col, int nvalid,
                                           float (&v)[32]) {
  const __nv_bfloat16* s = reinterpret_cast<const __nv_bfloat16*>(src) + row * ld + col;
#pragma unroll
  for (int g = 0; g < 4; ++g) {
    uint4 q = make_uint4(0, 0, 0, 0);
    if (8 * g < nvalid) q = __ldg(reinterpret_cast<const uint4*>(s + 8 * g));
    float2 f;
    f = unpack_bf16x2(q.x); v[8 * g + 0] = f.x; v[8 * g + 1] = f.y;
    f = unpack_bf16x2(q.y); v[8 * g + 2] = f.x; v[8 * g + 3] = f.y;
    f = unpack_bf16x2(q.z); v[8 * g + 4] = f.x; v[8 * g + 5] = f.y;
    f = unpack_bf16x2(q.w); v[8 * g + 6] = f.x; v[8 * g + 7] = f.y;
  }
}

// Epilogue of one 32-column chunk of one accumulator row (single accumulator).
__device__ __forceinline__ void epilogue_chunk(const Prob& P, int64_t row, int col, int nvalid,
                                               const uint32_t (&r)[32]) {
  float acc[32];
#pragma unroll
  for (int j = 0; j < 32; ++j) acc[j] = __uint_as_float(r[j]);
  switch (P.epi) {
    case EPI_STORE:
      store_row32(P.out0, P.ldo, row, col, nvalid, acc);
      break;
    case EPI_GELU_FWD: {
      store_row32(P.out0, P.ldo, row, col, nvalid, acc);  // A (pre-activation)
      float h[32];
#pragma unroll
      for (int j = 0; j < 32; ++j) h[j] = act::gelu(acc[j]);
      store_row32(P.out1, P.ldo, row, col, nvalid, h);
      break;
    }
    case EPI_GELU_BWD: {
      float a[32];
      load_row32(P.aux0, P.ldo, row, col, nvalid, a);
#pragma unroll
      for (int j = 0; j < 32; ++j) a[j] = acc[j] * act::gelu_grad(a[j]);
      store_row32(P.out0, P.ldo, row, col, nvalid, a);
      break;
    }
    case EPI_SWIGLU_BWD: {
      float g[32], u[32];
      load_row32(P.aux0, P.ldo, row, col, nvalid, g);
      load_row32(P.aux1, P.ldo, row, col, nvalid, u);
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        float dg, du;
        act::swiglu_grads(acc[j], g[j], u[j], dg, du);
        g[j] = dg;
        u[j] = du;
      }
      store_row32(P.out0, P.ldo, row, col, nvalid, g);
      store_row32(P.out1, P.ldo, row, col, nvalid, u);
      break;
    }
    default:
      break;
  }
}

__device__ __forceinline__ void tc_gemm_body(const GemmParams& p, uint8_t* smem_raw) {
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kStages * kStageBytes);
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(bars + kNumBars);
  volatile int32_t* abort_flag = reinterpret_cast<volatile int32_t*>(tmem_holder + 1);

  const uint32_t smem_base = ptx::smem_u32(smem);
  const uint32_t bar0 = ptx::smem_u32(bars);
  auto full_bar = [&](int s) { return bar0 + 8u * s; };
  auto empty_bar = [&](int s) { return bar0 + 8u * (kStages + s); };
  auto tfull_bar = [&](int a) { return bar0 + 8u * (2 * kStages + a); };
  auto tempty_bar = [&](int a) { return bar0 + 8u * (2 * kStages + kNumAcc + a); };
  const uint32_t drain_bar = bar0 + 8u * (2 * kStages + 2 * kNumAcc);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      ptx::mbar_init(full_bar(s), 1);
      ptx::mbar_init(empty_bar(s), 1);
    }
    for (int a = 0; a < kNumAcc; ++a) {
      ptx::mbar_init(tfull_bar(a), 1);
      ptx::mbar_init(tempty_bar(a), kNumEpiWarps);
    }
    ptx::mbar_init(drain_bar, 1);
    *abort_flag = 0;
    ptx::fence_mbarrier_init();
  }
  if (warp == 0 && lane == 0) {
    for (int i = 0; i < p.num_maps; ++i) ptx::prefetch_tmap(&p.maps[i]);
  }
  if (warp == 1) {
    ptx::tmem_alloc(ptx::smem_u32(tmem_holder), kTmemCols);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem_base = *tmem_holder;
  const Ctl ctl{abort_flag, p.status, p.timeout_ns};

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      int armed_parity[kStages];
#pragma unroll
      for (int s = 0; s < kStages; ++s) armed_parity[s] = -1;
      bool ok = true;
      for (int tile = blockIdx.x; ok && tile < p.total_tiles; tile += gridDim.x) {
        const TileInfo ti = decode_tile(p, tile);
        const Prob& P = p.probs[ti.prob];
        const bool dual = P.epi == EPI_SWIGLU_FWD;
        const int nA = ti.valid_m > 64 ? 2 : 1;
        const int nB = (ti.valid_n + 63) / 64;
        const uint32_t bytes = static_cast<uint32_t>((nA + nB * (dual ? 2 : 1)) * kBoxBytes);
        for (int s = P.seg_begin; ok && s < P.seg_begin + P.seg_count; ++s) {
          const Seg& S = p.segs[s];
          const void* ma = &p.maps[S.a_map];
          const void* mb = &p.maps[S.b_map];
          const void* mb2 = dual ? static_cast<const void*>(&p.maps[S.b2_map]) : nullptr;
          const int kblocks = (S.K + kBK - 1) / kBK;
          for (int kb = 0; kb < kblocks; ++kb) {
            if (!bounded_wait(empty_bar(stage), phase ^ 1u, ctl, kDevTimeoutProducer)) {
              ok = false;
              break;
            }
            const uint32_t fb = full_bar(stage);
            ptx::mbar_arrive_expect_tx(fb, bytes);
            armed_parity[stage] = static_cast<int>(phase);
            const uint32_t sb = smem_base + stage * kStageBytes;
            const int k0 = kb * kBK;
            for (int b = 0; b < nA; ++b) {
              if (P.a_major == MAJOR_MN)
                ptx::tma_load_2d(sb + b * kBoxBytes, ma, ti.m0 + 64 * b, k0, fb);
              else
                ptx::tma_load_2d(sb + b * kBoxBytes, ma, k0, ti.m0 + 64 * b, fb);
            }
            for (int j = 0; j < nB; ++j) {
              if (P.b_major == MAJOR_MN)
                ptx::tma_load_2d(sb + (2 + j) * kBoxBytes, mb, ti.n0 + 64 * j, k0, fb);
              else
                ptx::tma_load_2d(sb + (2 + j) * kBoxBytes, mb, k0, ti.n0 + 64 * j, fb);
            }
            if (dual) {
              for (int j = 0; j < nB; ++j) ptx::tma_load_2d(sb + (4 + j) * kBoxBytes, mb2, ti.n0 + 64 * j, k0, fb);
            }
            if (++stage == kStages) {
              stage = 0;
              phase ^= 1u;
            }
          }
        }
      }
      if (!ok) {
        // Let every copy already issued land before the CTA can exit.
        for (int s = 0; s < kStages; ++s)
          if (armed_parity[s] >= 0) drain_wait(full_bar(s), static_cast<uint32_t>(armed_parity[s]));
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      bool ok = true;
      bool issued = false;
      for (int tile = blockIdx.x; ok && tile < p.total_tiles; tile += gridDim.x) {
        const TileInfo ti = decode_tile(p, tile);
        const Prob& P = p.probs[ti.prob];
        const bool dual = P.epi == EPI_SWIGLU_FWD;
        const int n_cap = dual ? 128 : 256;
        const int n_mma = min(n_cap, (ti.valid_n + 15) & ~15);
        const uint32_t idesc = ptx::make_idesc_bf16(kBM, n_mma, P.a_major, P.b_major);
        if (!bounded_wait(tempty_bar(acc), acc_phase ^ 1u, ctl, kDevTimeoutMma)) {
          ok = false;
          break;
        }
        ptx::tc_fence_after();
        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * kAccCols);
        uint32_t accumulate = 0;
        for (int s = P.seg_begin; ok && s < P.seg_begin + P.seg_count; ++s) {
          const Seg& S = p.segs[s];
          const int kblocks = (S.K + kBK - 1) / kBK;
          for (int kb = 0; kb < kblocks; ++kb) {
            if (!bounded_wait(full_bar(stage), phase, ctl, kDevTimeoutMma)) {
              ok = false;
              break;
            }
            ptx::tc_fence_after();
            const uint32_t sa = smem_base + stage * kStageBytes;
            const uint32_t sb = sa + 2 * kBoxBytes;
            const int rem = S.K - kb * kBK;
            const int nk = min(kBK / 16, (rem + 15) / 16);
            for (int j = 0; j < nk; ++j) {
              const uint64_t ad = P.a_major == MAJOR_MN ? ptx::make_sdesc_sw128(sa + 2048u * j, kBoxBytes, 1024)
                                                        : ptx::make_sdesc_sw128(sa + 32u * j, 16, 1024);
              const uint64_t bd = P.b_major == MAJOR_MN ? ptx::make_sdesc_sw128(sb + 2048u * j, kBoxBytes, 1024)
                                                        : ptx::make_sdesc_sw128(sb + 32u * j, 16, 1024);
              ptx::mma_bf16(d_tmem, ad, bd, idesc, accumulate);
              if (dual) {
                const uint64_t bd2 = ptx::make_sdesc_sw128(sb + 2 * kBoxBytes + 2048u * j, kBoxBytes, 1024);
                ptx::mma_bf16(d_tmem + 128u, ad, bd2, idesc, accumulate);
              }
              accumulate = 1;
              issued = true;
            }
            ptx::mma_commit(empty_bar(stage));  // frees the stage once these MMAs have read it
            if (++stage == kStages) {
              stage = 0;
              phase ^= 1u;
            }
          }
        }
        if (!ok) break;
        ptx::mma_commit(tfull_bar(acc));  // accumulator ready for the epilogue
        if (++acc == kNumAcc) {
          acc = 0;
          acc_phase ^= 1u;
        }
      }
      if (!ok && issued) {
        // Every MMA issued so far must finish before TMEM is released.
        ptx::mma_commit(drain_bar);
        drain_wait(drain_bar, 0);
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;              // TMEM lane quarter this warp may read
    const int half = (warp - 2) >> 2;    // which half of the tile's columns
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int tile = blockIdx.x; tile < p.total_tiles; tile += gridDim.x) {
      const TileInfo ti = decode_tile(p, tile);
      const Prob& P = p.probs[ti.prob];
      if (!bounded_wait(tfull_bar(acc), acc_phase, ctl, kDevTimeoutEpilogue)) break;
      ptx::tc_fence_after();
      const int row = q * 32 + lane;
      const bool row_ok = row < ti.valid_m;
      const int64_t grow = static_cast<int64_t>(ti.m0) + row;
      const uint32_t tacc = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(acc * kAccCols);
      if (P.epi == EPI_SWIGLU_FWD) {
#pragma unroll 1
        for (int c = 0; c < 2; ++c) {
          const int col = half * 64 + c * 32;
          if (col >= ti.valid_n) break;
          uint32_t rg[32], ru[32];
          ptx::tmem_ld_32x32b_x32(tacc + col, rg);
          ptx::tmem_ld_32x32b_x32(tacc + 128u + col, ru);
          ptx::tmem_wait_ld();
          if (row_ok) {
            const int nvalid = min(32, ti.valid_n - col);
            float g[32], u[32], h[32];
#pragma unroll
            for (int j = 0; j < 32; ++j) {
              g[j] = __uint_as_float(rg[j]);
              u[j] = __uint_as_float(ru[j]);
              h[j] = u[j] * act::swish(g[j]);
            }
            store_row32(P.out0, P.ldo, grow, ti.n0 + col, nvalid, g);
            store_row32(P.out1, P.ldo, grow, ti.n0 + col, nvalid, u);
            store_row32(P.out2, P.ldo, grow, ti.n0 + col, nvalid, h);
          }
        }
      } else {
#pragma unroll 1
        for (int c = 0; c < 4; ++c) {
          const int col = half * 128 + c * 32;
          if (col >= ti.valid_n) break;
          uint32_t r[32];
          ptx::tmem_ld_32x32b_x32(tacc + col, r);
          ptx::tmem_wait_ld();
          if (row_ok) epilogue_chunk(P, grow, ti.n0 + col, min(32, ti.valid_n - col), r);
        }
      }
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(tempty_bar(acc));
      if (++acc == kNumAcc) {
        acc = 0;
        acc_phase ^= 1u;
      }
    }
  }

  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem_base, kTmemCols);
  }
}

}  // namespace

// One kernel symbol per launch kind of a training step (same body).
#define TPMLP_TC_KERNEL(name)                                                          \
  __global__ void __launch_bounds__(kThreads, 1) name(const __grid_constant__ GemmParams p) { \
    extern __shared__ __align__(1024) uint8_t smem_raw[];                              \
    tc_gemm_body(p, smem_raw);                                                         \
  }

TPMLP_TC_KERNEL(tpmlp_fwd_column_gemm_act)
TPMLP_TC_KERNEL(tpmlp_fwd_row_gemm_gsum)
TPMLP_TC_KERNEL(tpmlp_bwd_dgrad_act_wgrad2)
TPMLP_TC_KERNEL(tpmlp_bwd_dx_fsum_wgrad1)

int tc_gemm_max_smem_bytes() { return kSmemBytes; }

cudaError_t launch_tc_gemm(const GemmParams& p, int kernel_tag, int grid, cudaStream_t stream) {
  void (*k)(GemmParams) = nullptr;
  switch (kernel_tag) {
    case TAG_FWD_COLUMN: k = tpmlp_fwd_column_gemm_act; break;
    case TAG_FWD_ROW: k = tpmlp_fwd_row_gemm_gsum; break;
    case TAG_BWD_DGRAD: k = tpmlp_bwd_dgrad_act_wgrad2; break;
    case TAG_BWD_FSUM: k = tpmlp_bwd_dx_fsum_wgrad1; break;
    default: return cudaErrorInvalidValue;
  }
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
  if (e != cudaSuccess) return e;
  k<<<grid, kThreads, kSmemBytes, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace tpmlp
