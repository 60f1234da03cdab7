// tc_gemm_common.cuh -- device building blocks of the persistent 2-SM
// tcgen05 GEMM (tc_gemm.cu): tile geometry, bounded waits, the per-pair load
// shape, the straight-line MMA issue of a stage and the fused epilogue of a
// 32-column chunk.
#pragma once
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <climits>

#include "act.cuh"
#include "ptx.cuh"
#include "tpmlp_internal.h"

namespace tpmlp {
namespace {

constexpr int kBM = 128;                        // rows of A / D per CTA
constexpr int kPairM = 2 * kBM;                 // rows of a pair's tile
// A stage holds, per CTA, a 128 x kBK slice of A and of its half of B, each
// as 128-byte-swizzled rows.  A K-major slice is kBK/64 boxes of 128 rows x
// 64 K; an MN-major one is two boxes of 64 MN columns x kBK K rows.
constexpr int kBK = kTcBK;                      // K per stage
constexpr int kRowBytes = 128;                  // one swizzle row: 64 bf16
constexpr int kKBoxBytes = 128 * kRowBytes;     // K-major box: 128 rows x 64 K (16 KB)
constexpr int kMNBoxBytes = kBK * kRowBytes;    // MN-major box: kBK K rows x 64 MN
constexpr int kOperandBytes = 128 * kBK * 2;    // one operand slice per stage
constexpr int kStageBytes = 2 * kOperandBytes;  // A + B
constexpr int kStages = (224 * 1024) / kStageBytes;
static_assert(kBK % 64 == 0, "stage depth is a whole number of 64-wide boxes");
static_assert(kOperandBytes == (kBK / 64) * kKBoxBytes && kOperandBytes == 2 * kMNBoxBytes, "stage layout");
// Epilogue configurations: kEW epilogue warps per CTA, 8 (chunks of 32
// accumulator columns) or 16 (chunks of 16, so that a thread's registers stay
// within 65,536 / (32 x 18) = 113).  The warps of a TMEM lane quarter split a
// tile's 256 columns between them (2 x 128 or 4 x 64), which is four chunks
// per warp and tile in both, and both use 32 KB of staging.
constexpr int chunk_cols(int ew) { return ew == 8 ? 32 : 16; }
constexpr int threads_for(int ew) { return 32 * (2 + ew); }
constexpr int kMaxEpiWarps = 16;
constexpr int kTmemCols = 512;
constexpr int kAccCols = 256;
constexpr int kNumAcc = 2;
constexpr int kNumBars = 2 * kStages + 2 * kNumAcc + 1;
// Epilogue staging: each epilogue warp owns two 32 x kCW bf16 blocks (its 32
// TMEM lanes x kCW columns), written row by row with a swizzle and stored by
// TMA while the other block is being filled.
constexpr int kEpiBytes = 32 * 1024;
static_assert(8 * 2 * 32 * chunk_cols(8) * 2 == kEpiBytes && 16 * 2 * 32 * chunk_cols(16) * 2 == kEpiBytes,
              "staging");
constexpr int kSmemBytes = 1024 + kStages * kStageBytes + kEpiBytes + 8 * kNumBars + 16;
constexpr uint64_t kDrainTimeoutNs = 200ull * 1000 * 1000;
constexpr uint64_t kPeerDrainNs = 2ull * 1000 * 1000;
constexpr uint16_t kPairMask = 0x3;

static_assert(kSmemBytes <= 227 * 1024, "shared memory budget");
static_assert(kNumAcc * kAccCols <= kTmemCols, "TMEM budget");

struct TileInfo {
  int prob, m0, n0, valid_m, valid_n;
  int rev;  // walk the K blocks last to first (see Prob::k_rev)
};

// wave: the pairs of the launch, or 0 for a stream-K part (never reversed).
__device__ __forceinline__ TileInfo decode_tile(const GemmParams& p, int tile, int wave) {
  int g = 0;
  while (g + 1 < p.num_groups && tile >= p.groups[g + 1].tile_start) ++g;
  const Group& G = p.groups[g];
  const int local = tile - G.tile_start;
  int mt, n_lin;
  group_tile(G, local, mt, n_lin);
  int pi = G.first_prob;
  while (n_lin >= p.probs[pi].tiles_n) {
    n_lin -= p.probs[pi].tiles_n;
    ++pi;
  }
  const Prob& P = p.probs[pi];
  TileInfo t;
  t.prob = pi;
  t.m0 = mt * kPairM;
  t.n0 = n_lin * P.tile_n;
  t.valid_m = min(kPairM, P.M - t.m0);
  t.valid_n = min(P.tile_n, P.N - t.n0);
  t.rev = 0;
  if (P.k_rev && wave > 0) t.rev = (local / wave) & 1;  // long-K tiles only: a division per tile
  return t;
}

// Stripe of a token row (sequence-parallel layout): the last j with
// row0[j] <= row.  Empty stripes are never selected.
__device__ __forceinline__ int stripe_of(const Stripes& st, int64_t row) {
  int j = 0;
  while (j + 1 < st.num && row >= st.row0[j + 1]) ++j;
  return j;
}

struct Ctl {
  volatile int32_t* abort_flag;
  uint32_t peer_abort;  // cluster address of the peer CTA's abort flag
  int32_t* status;
  uint64_t timeout_ns;
};

__device__ __forceinline__ void raise_abort(const Ctl& c, int32_t code) {
  *c.abort_flag = 1;
  ptx::st_cluster_u32(c.peer_abort, 1u);
  if (c.status) atomicCAS(c.status, 0, code);
}

// Wait for the phase of `bar` with the given parity; false if the wait
// timed out (status recorded, both CTAs aborted) or an abort was raised.
__device__ __forceinline__ bool bounded_wait(uint32_t bar, uint32_t parity, const Ctl& c, int32_t code) {
  if (ptx::mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = ptx::globaltimer_ns();
  while (true) {
    if (ptx::mbar_try_wait(bar, parity)) return true;
    if (*c.abort_flag) return false;
    if (ptx::globaltimer_ns() - t0 > c.timeout_ns) {
      raise_abort(c, code);
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

__device__ __forceinline__ void spin_ns(uint64_t ns) {
  const uint64_t t0 = ptx::globaltimer_ns();
  while (ptx::globaltimer_ns() - t0 < ns) {
  }
}

// What CTA `rank` of the pair loads and computes for one tile.  MN-major
// boxes wholly outside the valid rows / columns are not loaded (nor are the
// A boxes of a CTA with no valid rows): the MMA rows / columns they would
// feed are never stored.
struct PairShape {
  int n_mma;        // MMA N (multiple of 32, covers the tile's valid columns)
  int half;         // B columns held by each CTA (n_mma / 2)
  int nA[2];        // A copies each CTA issues
  int nB[2];        // B copies (per B operand) each CTA issues
  uint32_t bytes[2];  // bytes each CTA loads per K block
};

// TMA copies of one operand slice: K-major, kBK/64 boxes covering all 128
// rows; MN-major, one box per 64 valid columns.
__device__ __forceinline__ int copies_for(int major, int valid) {
  if (valid <= 0) return 0;
  return major == MAJOR_K ? kBK / 64 : (valid + 63) / 64;
}

__device__ __forceinline__ int box_bytes(int major) { return major == MAJOR_K ? kKBoxBytes : kMNBoxBytes; }

__device__ __forceinline__ PairShape pair_shape(const TileInfo& ti, bool dual, int a_major, int b_major) {
  PairShape s;
  const int cap = dual ? 128 : 256;
  s.n_mma = min(cap, (ti.valid_n + 31) & ~31);
  s.half = s.n_mma >> 1;
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    const int vm = max(0, min(kBM, ti.valid_m - kBM * r));
    const int vb = max(0, min(s.half, ti.valid_n - s.half * r));
    s.nA[r] = copies_for(a_major, vm);
    s.nB[r] = copies_for(b_major, vb);
    s.bytes[r] = static_cast<uint32_t>(s.nA[r] * box_bytes(a_major) + (dual ? 2 : 1) * s.nB[r] * box_bytes(b_major));
  }
  return s;
}

// The MMAs of one stage: K steps j = 0 .. nk-1 of 16, each one (SwiGLU:
// two, gate and up projection into the two 128-column halves) pair MMA.
// Descriptors advance by offsets in 16-byte units: K-major, +32 B per K step
// inside a 64-wide box and +16 KB per box; MN-major, +2048 B per K step.
// A full stage is straight-line code.  A branch between two tcgen05.mma
// instructions delays the issue of the second one (about 45 cycles per MMA
// on GB300, against 128 cycles of tensor work for a 256 x 256 x 16 pair
// MMA), so every choice -- SwiGLU or not, full or partial stage -- is made
// once, before the sequence.
template <bool kDual, bool kAmn, bool kBmn>
__device__ __forceinline__ void issue_stage(uint32_t d_tmem, uint32_t a_lo0, uint32_t a_hi, uint32_t b_lo0,
                                            uint32_t b_hi, uint32_t idesc, int nk, uint32_t& accumulate) {
  if (nk == kBK / 16) {
#pragma unroll
    for (int j = 0; j < kBK / 16; ++j) {
      constexpr uint32_t kBoxOff = kMNBoxBytes >> 4;
      const uint32_t koff = static_cast<uint32_t>(((j >> 2) * kKBoxBytes + (j & 3) * 32) >> 4);
      const uint32_t moff = static_cast<uint32_t>((j * 2048) >> 4);
      const uint32_t al = a_lo0 + (kAmn ? moff : koff);
      const uint32_t bl = b_lo0 + (kBmn ? moff : koff);
      if (j == 0) {
        ptx::mma_bf16_pair_lohi(d_tmem, al, a_hi, bl, b_hi, idesc, accumulate);
        if (kDual) ptx::mma_bf16_pair_lohi(d_tmem + 128u, al, a_hi, bl + kBoxOff, b_hi, idesc, accumulate);
      } else {
        ptx::mma_bf16_pair_lohi_acc(d_tmem, al, a_hi, bl, b_hi, idesc);
        if (kDual) ptx::mma_bf16_pair_lohi_acc(d_tmem + 128u, al, a_hi, bl + kBoxOff, b_hi, idesc);
      }
    }
    accumulate = 1;
    return;
  }
  for (int j = 0; j < nk; ++j) {  // the last, partial stage of a segment
    const uint32_t koff = static_cast<uint32_t>(((j >> 2) * kKBoxBytes + (j & 3) * 32) >> 4);
    const uint32_t moff = static_cast<uint32_t>((j * 2048) >> 4);
    const uint32_t al = a_lo0 + (kAmn ? moff : koff);
    const uint32_t bl = b_lo0 + (kBmn ? moff : koff);
    ptx::mma_bf16_pair_lohi(d_tmem, al, a_hi, bl, b_hi, idesc, accumulate);
    if (kDual) ptx::mma_bf16_pair_lohi(d_tmem + 128u, al, a_hi, bl + (kMNBoxBytes >> 4), b_hi, idesc, accumulate);
    accumulate = 1;
  }
}

// One stage's MMAs, with every choice (SwiGLU split pair, operand majors)
// resolved by a single switch ahead of the straight-line sequence.
__device__ __forceinline__ void issue_stage_any(int kind, uint32_t d_tmem, uint32_t a_lo0, uint32_t a_hi,
                                                uint32_t b_lo0, uint32_t b_hi, uint32_t idesc, int nk,
                                                uint32_t& accumulate) {
  switch (kind) {
    case 0: issue_stage<false, false, false>(d_tmem, a_lo0, a_hi, b_lo0, b_hi, idesc, nk, accumulate); break;
    case 1: issue_stage<false, false, true>(d_tmem, a_lo0, a_hi, b_lo0, b_hi, idesc, nk, accumulate); break;
    case 2: issue_stage<false, true, false>(d_tmem, a_lo0, a_hi, b_lo0, b_hi, idesc, nk, accumulate); break;
    case 3: issue_stage<false, true, true>(d_tmem, a_lo0, a_hi, b_lo0, b_hi, idesc, nk, accumulate); break;
    case 4: issue_stage<true, false, false>(d_tmem, a_lo0, a_hi, b_lo0, b_hi, idesc, nk, accumulate); break;
    case 5: issue_stage<true, false, true>(d_tmem, a_lo0, a_hi, b_lo0, b_hi, idesc, nk, accumulate); break;
    case 6: issue_stage<true, true, false>(d_tmem, a_lo0, a_hi, b_lo0, b_hi, idesc, nk, accumulate); break;
    default: issue_stage<true, true, true>(d_tmem, a_lo0, a_hi, b_lo0, b_hi, idesc, nk, accumulate); break;
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

// One epilogue warp's output path: 32 rows (its TMEM lanes) x N columns of
// bf16 at a time (N = 32 or 16, the chunk width of the kernel's epilogue
// configuration) go through one of its two shared-memory blocks and out with
// a TMA store.  A thread writes its row as N / 8 16-byte pieces, piece g at
// position g ^ ((row / 2) % 4) for 64-byte rows (N = 32) or g ^ ((row / 4) % 2)
// for 32-byte rows (N = 16) -- the 64- / 32-byte swizzle of the output maps --
// so every 8 consecutive rows fill all 32 banks once.  Rows and columns past
// the tensor's end are clipped by the TMA unit.  Compared with each thread
// storing its own row to global memory (32 cache lines per warp store), this
// moves a warp's block in a few shared-memory wavefronts and one bulk copy.
struct EpiStore {
  uint32_t buf;  // this warp's two blocks
  uint32_t next; // the block the next store uses (every bulk group reads one block)
  int rows;      // rows of the current problem's outputs
  int sj, sy0;   // striped out0: the stripe of this warp's rows and its first row
};

template <int N>
constexpr int epi_block_bytes() { return 32 * N * 2; }

// The swizzled position of 16-byte piece g of row r in a staging block (the
// output maps' 64- or 32-byte swizzle).
template <int N>
__device__ __forceinline__ uint32_t stage_off(int r, int g) {
  const uint32_t sw = N == 32 ? (static_cast<uint32_t>(r) >> 1) & 3u : (static_cast<uint32_t>(r) >> 2) & 1u;
  return static_cast<uint32_t>(r) * (2u * N) + ((static_cast<uint32_t>(g) ^ sw) << 4);
}

// Rows grow0 .. grow0 + 31 (valid_rows of them), columns x .. x + N - 1
// (nvalid of them) of a row-major bf16 array into staging block blk,
// coalesced: a warp instruction covers 32 / (N / 8) whole rows.
template <int N>
__device__ __forceinline__ void stage_rows(const void* src, int64_t ld, int64_t grow0, int valid_rows, int x,
                                           int nvalid, uint32_t blk, int lane) {
  constexpr int P = N / 8;
  constexpr int RPI = 32 / P;
  const int g = lane % P;
#pragma unroll
  for (int i = 0; i < P; ++i) {
    const int r = i * RPI + lane / P;
    uint4 q = make_uint4(0, 0, 0, 0);
    if (r < valid_rows && 8 * g < nvalid)
      q = __ldg(reinterpret_cast<const uint4*>(reinterpret_cast<const __nv_bfloat16*>(src) + (grow0 + r) * ld + x + 8 * g));
    ptx::st_shared_v4(blk + stage_off<N>(r, g), q);
  }
}

// This thread's row of a staging block as floats.
template <int N>
__device__ __forceinline__ void read_row(uint32_t blk, int lane, float (&v)[N]) {
#pragma unroll
  for (int g = 0; g < N / 8; ++g) {
    const uint4 q = ptx::ld_shared_v4(blk + stage_off<N>(lane, g));
    float2 f;
    f = unpack_bf16x2(q.x); v[8 * g + 0] = f.x; v[8 * g + 1] = f.y;
    f = unpack_bf16x2(q.y); v[8 * g + 2] = f.x; v[8 * g + 3] = f.y;
    f = unpack_bf16x2(q.z); v[8 * g + 4] = f.x; v[8 * g + 5] = f.y;
    f = unpack_bf16x2(q.w); v[8 * g + 6] = f.x; v[8 * g + 7] = f.y;
  }
}

// This thread's row of a staging block from floats (bf16, swizzled).
template <int N>
__device__ __forceinline__ void write_row(uint32_t blk, int lane, const float (&v)[N]) {
#pragma unroll
  for (int g = 0; g < N / 8; ++g) {
    uint4 o;
    o.x = pack_bf16x2(v[8 * g + 0], v[8 * g + 1]);
    o.y = pack_bf16x2(v[8 * g + 2], v[8 * g + 3]);
    o.z = pack_bf16x2(v[8 * g + 4], v[8 * g + 5]);
    o.w = pack_bf16x2(v[8 * g + 6], v[8 * g + 7]);
    ptx::st_shared_v4(blk + stage_off<N>(lane, g), o);
  }
}

// Output k (0..2) of problem P: columns x .. x + N - 1 (nvalid of them inside
// the tensor) of this warp's rows y .. y + 31.
template <int N>
__device__ __forceinline__ void store_block(EpiStore& es, const GemmParams& p, const Prob& P, int k, int x, int y,
                                            int nvalid, const float (&v)[N], int lane) {
  static_assert(N == 32 || N == 16, "chunk width");
  if (y >= es.rows) return;  // every row of this warp is past the end: no store starts out of range
  (void)nvalid;              // the TMA unit clips columns past the end
  int map = P.out_map[k];
  if (k == 0 && P.out_striped) {  // token stripes: the stripe's own map, stripe-local rows
    map += es.sj;
    y -= es.sy0;
  }
  const uint32_t b = es.buf + es.next * epi_block_bytes<N>();
  if (lane == 0) ptx::bulk_wait_group_read<1>();  // the store that last used block b has read it
  __syncwarp();
  write_row<N>(b, lane, v);
  ptx::fence_proxy_async_smem();
  __syncwarp();
  if (lane == 0) {
    ptx::tma_store_2d(&p.maps[map], b, x, y);
    ptx::bulk_commit_group();
  }
  es.next ^= 1u;
}

// Outputs k0 and k1 of the same chunk through both of the warp's blocks,
// behind one async-proxy fence.  Measured on GB300: the GeLU forward's A and
// H in the short-K configuration (N = 16), 3 % off the GPT-2-small column
// launch, but 1-2 % slower with N = 32 on the larger shapes (the wait for both
// blocks outweighing the fence saved); the SwiGLU backward's dG and dU, whose
// chunks already wait on two loads, 1.1 % off C4's dgrad launch.
template <int N>
__device__ __forceinline__ void store_pair(EpiStore& es, const GemmParams& p, const Prob& P, int k0, int k1, int x,
                                           int y, const float (&v0)[N], const float (&v1)[N], int lane) {
  if (y >= es.rows) return;  // every row of this warp is past the end: no store starts out of range
  if (lane == 0) ptx::bulk_wait_group_read<0>();  // both blocks have been read by their last stores
  __syncwarp();
  write_row<N>(es.buf, lane, v0);
  write_row<N>(es.buf + epi_block_bytes<N>(), lane, v1);
  ptx::fence_proxy_async_smem();
  __syncwarp();
  if (lane == 0) {  // one bulk group per block, block 1 last, as two single stores would leave them
    ptx::tma_store_2d(&p.maps[P.out_map[k0]], es.buf, x, y);
    ptx::bulk_commit_group();
    ptx::tma_store_2d(&p.maps[P.out_map[k1]], es.buf + epi_block_bytes<N>(), x, y);
    ptx::bulk_commit_group();
  }
  es.next = 0;
}

// N bf16 values of row `row` of a row-major array from column col on (the
// nvalid first of them; the others read as zero).
template <int N>
__device__ __forceinline__ void load_row(const void* src, int64_t ld, int64_t row, int col, int nvalid,
                                         float (&v)[N]) {
  const __nv_bfloat16* s = reinterpret_cast<const __nv_bfloat16*>(src) + row * ld + col;
#pragma unroll
  for (int g = 0; g < N / 8; ++g) {
    uint4 q = make_uint4(0, 0, 0, 0);
    if (8 * g < nvalid) q = __ldg(reinterpret_cast<const uint4*>(s + 8 * g));
    float2 f;
    f = unpack_bf16x2(q.x); v[8 * g + 0] = f.x; v[8 * g + 1] = f.y;
    f = unpack_bf16x2(q.y); v[8 * g + 2] = f.x; v[8 * g + 3] = f.y;
    f = unpack_bf16x2(q.z); v[8 * g + 4] = f.x; v[8 * g + 5] = f.y;
    f = unpack_bf16x2(q.w); v[8 * g + 6] = f.x; v[8 * g + 7] = f.y;
  }
}

// v[j] += bias[col + j] for the chunk's valid columns (bias may be null).
template <int N>
__device__ __forceinline__ void add_bias(const void* bias, int col, int nvalid, float (&v)[N]) {
  if (!bias) return;
  float b[N];
  load_row<N>(bias, 0, 0, col, nvalid, b);
#pragma unroll
  for (int j = 0; j < N; ++j) v[j] += b[j];
}

// Epilogue of one N-column chunk (columns x .. x+N-1 of rows y .. y+31, this
// thread's row grow) of a single accumulator.  Every lane takes part (the
// stores are per warp); inputs are read only for valid rows and columns.
template <int N>
__device__ __forceinline__ void epilogue_chunk(const GemmParams& p, const Prob& P, EpiStore& es, int64_t grow,
                                               bool row_ok, int x, int y, int nvalid, const uint32_t (&r)[N],
                                               int lane) {
  float acc[N];
#pragma unroll
  for (int j = 0; j < N; ++j) acc[j] = __uint_as_float(r[j]);
  const int nload = row_ok ? nvalid : 0;
  switch (P.epi) {
    case EPI_STORE:
      add_bias<N>(P.aux0, x, nvalid, acc);
      store_block<N>(es, p, P, 0, x, y, nvalid, acc, lane);
      break;
    case EPI_GELU_FWD: {
      add_bias<N>(P.aux0, x, nvalid, acc);
      if (N == 16 && !P.out_striped) {  // A and H behind one fence
        float h[N];
#pragma unroll
        for (int j = 0; j < N; ++j) h[j] = acc[j];
        act::x2::gelu_xn(h);
        store_pair<N>(es, p, P, 0, 1, x, y, acc, h, lane);
        break;
      }
      store_block<N>(es, p, P, 0, x, y, nvalid, acc, lane);  // A (pre-activation)
      act::x2::gelu_xn(acc);
      store_block<N>(es, p, P, 1, x, y, nvalid, acc, lane);
      break;
    }
    case EPI_GELU_BWD: {
      if (N == 32 && !P.out1 && y < es.rows) {  // A staged through the output block, dA written over it
        const uint32_t b = es.buf + es.next * epi_block_bytes<N>();
        if (lane == 0) ptx::bulk_wait_group_read<1>();  // the store that last used block b has read it
        __syncwarp();
        stage_rows<N>(P.aux0, P.ldo, grow - lane, es.rows - y, x, nvalid, b, lane);
        __syncwarp();
        float a[N];
        read_row<N>(b, lane, a);
        act::x2::gelu_bwd_xn<false>(acc, a, acc);
        write_row<N>(b, lane, a);
        ptx::fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          ptx::tma_store_2d(&p.maps[P.out_map[0]], b, x, y);
          ptx::bulk_commit_group();
        }
        es.next ^= 1u;
        break;
      }
      float a[N];
      load_row<N>(P.aux0, P.ldo, grow, x, nload, a);
      if (P.out1) {  // recompute H = GeLU(A) for the weight gradient of W2
        float h[N];
        act::x2::gelu_bwd_xn<true>(acc, a, h);
        store_block<N>(es, p, P, 1, x, y, nvalid, h, lane);
      } else {
        act::x2::gelu_bwd_xn<false>(acc, a, acc);
      }
      store_block<N>(es, p, P, 0, x, y, nvalid, a, lane);
      break;
    }
    case EPI_SWIGLU_BWD: {
      if (N == 32 && !P.out2 && y < es.rows) {  // G and U staged through both blocks, dG and dU written over them
        if (lane == 0) ptx::bulk_wait_group_read<0>();
        __syncwarp();
        const uint32_t b0 = es.buf, b1 = es.buf + epi_block_bytes<N>();
        stage_rows<N>(P.aux0, P.ldo, grow - lane, es.rows - y, x, nvalid, b0, lane);
        stage_rows<N>(P.aux1, P.ldo, grow - lane, es.rows - y, x, nvalid, b1, lane);
        __syncwarp();
        float g[N], u[N];
        read_row<N>(b0, lane, g);
        read_row<N>(b1, lane, u);
        act::x2::swiglu_bwd_xn<false>(acc, g, u, acc);
        write_row<N>(b0, lane, g);
        write_row<N>(b1, lane, u);
        ptx::fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {  // one bulk group per block, as in store_pair
          ptx::tma_store_2d(&p.maps[P.out_map[0]], b0, x, y);
          ptx::bulk_commit_group();
          ptx::tma_store_2d(&p.maps[P.out_map[1]], b1, x, y);
          ptx::bulk_commit_group();
        }
        es.next = 0;
        break;
      }
      float g[N], u[N];
      load_row<N>(P.aux0, P.ldo, grow, x, nload, g);
      load_row<N>(P.aux1, P.ldo, grow, x, nload, u);
      if (P.out2) {  // recompute H = U * Swish(G) for the weight gradient of W2
        float h[N];
        act::x2::swiglu_bwd_xn<true>(acc, g, u, h);
        store_block<N>(es, p, P, 2, x, y, nvalid, h, lane);
        store_block<N>(es, p, P, 0, x, y, nvalid, g, lane);
        store_block<N>(es, p, P, 1, x, y, nvalid, u, lane);
      } else {  // dG and dU behind one fence (C4's dgrad launch: -1.1 % on GB300)
        act::x2::swiglu_bwd_xn<false>(acc, g, u, acc);
        store_pair<N>(es, p, P, 0, 1, x, y, g, u, lane);
      }
      break;
    }
    default:
      break;
  }
}

// Whether a SwiGLU forward tile was computed with merged N = 256 MMAs: full
// tiles (128 output columns, 64 per CTA of the pair).  Each CTA's B stage
// holds 64 gate columns then 64 up columns (two MN-major blocks), so the
// accumulator columns are, per CTA-half h of B (h = 0, 1): gate columns
// 64 h .. 64 h + 63 of the tile at 128 h .. 128 h + 63, the matching up
// columns at 128 h + 64 .. 128 h + 127.  Partial tiles use two MMAs of
// N = 2 x 64-or-fewer columns: gate at 0 .., up at 128 ...
__device__ __forceinline__ bool swiglu_merged(const TileInfo& ti, const Prob& P) {
  return pair_shape(ti, true, P.a_major, P.b_major).n_mma == 128;
}

}  // namespace
}  // namespace tpmlp
