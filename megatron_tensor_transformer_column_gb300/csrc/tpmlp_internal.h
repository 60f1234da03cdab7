// tpmlp_internal.h -- work description shared by the host launcher and the
// kernels of the t-sharded MLP library.
//
// Every launch of the library is a list of GEMM problems
//     C[M x N] = sum over segments s of A_s[M x K_s] * B_s[K_s x N]
// followed by a fused epilogue.  A segment list longer than one is how the
// cross-shard sums are done on chip: the row-parallel forward GEMM has one
// segment per shard (H_i, W2_i) and its K loop walks them into one fp32
// accumulator (the g operator); the dX GEMM does the same with (dA_i, W1_i)
// (the f operator's backward sum).  See tpmlp.h for the algebra and sources.
#pragma once

#include <cuda.h>  // CUtensorMap (type only; the driver entry point is fetched at run time)
#include <stdint.h>

namespace tpmlp {

constexpr int kMaxShards = 16;

// K depth of one shared-memory stage of the tensor-core GEMM (a multiple of
// 64).  TMA boxes are 64 columns wide: 128 rows for K-major operand tiles,
// kTcBK K rows for MN-major ones.
#ifndef TPMLP_TC_BK
#define TPMLP_TC_BK 128
#endif
constexpr int kTcBK = TPMLP_TC_BK;
// A tensor used both K-major (128-row boxes) and MN-major (64-row boxes) in
// one launch needs two maps: the SwiGLU f-sum launch has X, dG_i and dU_i
// twice each, W1_i and W3_i (6t + 1).
// Output tensors get maps of their own (32 x 32 boxes, 64-byte swizzle) for
// the tensor-core epilogue's TMA stores: the SwiGLU f-sum launch adds dW1_i,
// dW3_i and dX (2t + 1), the SwiGLU dgrad launch dG_i, dU_i, dW2_i and, when
// H is recomputed, H_i (4t).
// Problems, segments and groups: the largest launch is the SwiGLU f-sum
// launch of the recompute backward, which also carries dW2_i = H_i^T dY:
// 3t + 1 problems (dW2_i, dW1_i, dW3_i, dX), 5t segments (one each for the
// weight gradients, 2t for dX) and t + 2 groups.  Its tensor maps (10t + 3)
// exceed kMaxMaps for t > 12; the host then moves dW2 to a launch of its own.
// The host checks every table bound while it builds a launch.
constexpr int kMaxMaps = 8 * kMaxShards + 4;
constexpr int kMaxProbs = 3 * kMaxShards + 2;
constexpr int kMaxGroups = kMaxShards + 2;
constexpr int kMaxSegs = 5 * kMaxShards + 2;

// Fused epilogues.  acc is the fp32 accumulator tile; bias vectors are
// optional (null = none) and indexed by output column.
enum EpiKind : int32_t {
  EPI_STORE = 0,       // out0 = acc (+ aux0[n]: b2, added once after the g-sum)
  EPI_GELU_FWD = 1,    // A = acc (+ aux0[n]: b1_i); out0 = A (kept for backward), out1 = H = GeLU(A)
  EPI_SWIGLU_FWD = 2,  // two accumulators (B = W1_i, B2 = W3_i): G = acc_G (+ aux0[n]: b1_i),
                       // U = acc_U (+ aux1[n]: b3_i); out0 = G, out1 = U, out2 = H = U * Swish(G)
  EPI_GELU_BWD = 3,    // acc = dH; aux0 = A: out0 = dA = dH * GeLU'(A)
                       //   (+ out1, if set: H = GeLU(A) recomputed from the saved A)
  EPI_SWIGLU_BWD = 4,  // acc = dH; aux0 = G, aux1 = U:
                       // out0 = dG = dH * U * Swish'(G), out1 = dU = dH * Swish(G)
                       //   (+ out2, if set: H = U * Swish(G) recomputed)
};

// Operand majors.  A(m, k) is K-major when a[m][k] is contiguous in k,
// MN-major when a[k][m] is contiguous in m; B(k, n) likewise.
enum Major : int32_t { MAJOR_K = 0, MAJOR_MN = 1 };

struct Seg {
  const void* a;   // raw pointers (used by the SIMT path)
  const void* b;
  const void* b2;  // second B (SwiGLU up projection), else null
  int64_t lda;     // row stride of the stored 2-D array behind A, in elements
  int64_t ldb;
  int32_t a_map;   // tensor-map indices (used by the tensor-core path)
  int32_t b_map;
  int32_t b2_map;
  int32_t K;
  // Sequence-parallel layout: the operand is the launch's striped input
  // (GemmParams::in_stripe), stored as token stripes; its map index is the
  // first of num_stripes consecutive maps and its raw pointer is unused.
  int32_t a_striped;
  int32_t b_striped;
};

struct Prob {
  int32_t M, N;
  int32_t tile_n;    // tile width along N for this problem
  int32_t tiles_n;
  int32_t seg_begin, seg_count;
  int32_t a_major, b_major;
  int32_t epi;
  int32_t out_map[3];  // tensor maps of out0..out2 for TMA stores (-1: none)
  int32_t out_striped; // out0 is the launch's striped output (token stripes)
  int32_t kblocks;     // K blocks of a tile, over all segments (tensor-core path)
  // Long K (tensor-core path): the group's tiles walk their K blocks first to
  // last in even waves (group-local tile / pairs) and last to first in odd
  // ones, so a wave starts on the K blocks the previous one read last, which
  // are still in L2.
  int32_t k_rev;
  int64_t ldo;       // row stride of out*/aux*, in elements
  void* out0;
  void* out1;
  void* out2;
  const void* aux0;
  const void* aux1;
};

// Problems with the same M that are rastered together: tiles are ordered in
// bands of band_m M-tiles; inside a band, N-tiles (across every problem of
// the group, in order) are the slow index and M-tiles the fast one, so the
// CTAs that run at the same time share operand panels in L2.  (Chunking the
// N-tiles as well, so that a chunk's B panels stay in L2 while the bands walk
// down M, was measured on GB300 to raise DRAM reads: C5's column launch 715
// -> 779 MB, its dgrad launch 2.81 -> 3.13 GB.)
struct Group {
  int32_t first_prob, num_probs;
  int32_t tiles_m;
  int32_t tiles_per_row;  // sum of tiles_n over the group's problems
  int32_t band_m;
  int32_t tile_start;     // first global tile index of the group
};

// The M-tile and the linear N-tile (across the group's problems) of a
// group's local-th tile, in the order described at Group; the one raster of
// the host planner and both kernels.
__host__ __device__ inline void group_tile(const Group& G, int local, int& mt, int& n_lin) {
  const int full_band = G.band_m * G.tiles_per_row;
  const int b = local / full_band;
  const int r = local - b * full_band;
  const int m_first = b * G.band_m;
  const int bm = G.tiles_m - m_first < G.band_m ? G.tiles_m - m_first : G.band_m;
  const int nl = r / bm;
  mt = m_first + (r - nl * bm);
  n_lin = nl;
}

// The deal of a launch's data-parallel tiles [0, dp_end) to its P pairs.  A
// launch that mixes K = T weight-gradient tiles with short ones places the
// long tiles first, tiles [0, nl): they go round robin over all pairs, so
// pairs r = nl mod P .. P - 1 draw one long tile fewer.  Of the short tiles
// after them, the first s0 go round robin over those pairs only, the rest
// round robin over all pairs from pair r on.  With s0 = 0 this is the plain
// round robin, tile i to pair i mod P.  One pair walks its tiles with a Deal
// cursor; the host planner runs the same walk to cost a choice of s0.
struct Deal {
  int phase;  // 0: long tiles, 1: the head of the short tiles, 2: the rest, 3: done
  int next;   // the phase's next index
};

__host__ __device__ inline void deal_init(Deal& d, int pair) {
  d.phase = pair < 0 ? 3 : 0;
  d.next = pair;
}

// This pair's next tile, or -1 (r = nl mod npairs, computed once: this runs
// on the kernel's critical path between tiles, where an integer division
// costs a visible bubble).
__host__ __device__ inline int deal_next(Deal& d, int nl, int r, int s0, int pair, int npairs, int dp_end) {
  if (d.phase == 0) {
    if (d.next < nl && d.next < dp_end) {
      const int t = d.next;
      d.next += npairs;
      return t;
    }
    d.phase = 1;
    d.next = pair - r;  // negative: this pair drew one long tile more, no head tiles
  }
  if (d.phase == 1) {
    if (d.next >= 0 && d.next < s0 && nl + d.next < dp_end) {
      const int t = nl + d.next;
      d.next += npairs - r;
      return t;
    }
    d.phase = 2;
    d.next = s0 + (pair >= r ? pair - r : pair - r + npairs);
  }
  if (d.phase == 2 && nl + d.next < dp_end) {
    const int t = nl + d.next;
    d.next += npairs;
    return t;
  }
  d.phase = 3;
  return -1;
}

// Token stripes of the sequence-parallel layout: stripe j holds rows
// [row0[j], row0[j+1]) of a [T x cols] tensor in its own buffer.  Internal
// boundaries are multiples of 128 rows, so no TMA box (128 rows of A, 128 K
// rows of an MN-major operand, 32 rows of an output block) crosses one.
constexpr int kMaxStripes = kMaxShards;
struct Stripes {
  int32_t num;                      // 0: the launch has no striped tensor
  int32_t pad_;
  int64_t row0[kMaxStripes + 1];
  const void* in[kMaxStripes];      // striped input (X or dY), raw pointers (fp32 path)
  void* out[kMaxStripes];           // striped output (Y or dX), raw pointers (fp32 path)
  int64_t in_ld, out_ld;            // row strides of the stripes, in elements
};

// Stream-K schedule (tensor-core path).  Tiles [0, dp_tiles) are dealt out
// round robin, tile i to pair i mod pairs.  The K blocks of the remaining
// tiles, concatenated in tile order, are cut into one contiguous range per
// pair: range r (held by pair pairs - 1 - r) starts at (start_tile[r],
// start_kb[r]) and ends where range r + 1 starts.  A range may end inside a
// tile, span whole tiles and start inside another, so it holds at most two
// parts of split tiles: its first item (partial slot 2r) and its last item
// (slot 2r + 1).  Every part leaves its fp32 accumulator in its slot and takes
// a ticket from a per-tile counter (one per epilogue warp position, in the
// counter block, keyed by the range holding the tile's K block 0 and tagged
// with the launch's epoch, so that a count left by an aborted launch reads as
// zero); the part with the last ticket adds all parts in range order and runs
// the tile's epilogue.  Nobody waits for another pair, and the fixed order
// makes the result the same on every run.
constexpr int kMaxSkPairs = 80;
constexpr int kSkWarpsPerPair = 32;                        // epilogue warps of a pair, at most
constexpr size_t kStatusBytes = 256;                       // workspace: status word block
constexpr size_t kSkFlagsOffset = kStatusBytes;            // kMaxSkPairs x kSkWarpsPerPair uint32 counters
constexpr size_t kSkSlotsOffset = 16384;                   // partial accumulators, two slots per range
constexpr size_t kSkSlotBytes = 256 * 256 * sizeof(float);
constexpr size_t kSkWorkspaceBytes = kSkSlotsOffset + 2 * kMaxSkPairs * kSkSlotBytes;
static_assert(kSkFlagsOffset + kMaxSkPairs * kSkWarpsPerPair * sizeof(uint32_t) <= kSkSlotsOffset, "flags fit");
struct StreamK {
  int32_t on;
  int32_t dp_tiles;  // data-parallel tiles (all of them when on == 0)
  int32_t pairs;     // pairs the ranges were made for (the launched pairs)
  uint32_t epoch;    // tag of this launch's ticket counts (24 bits, never 0)
  int32_t start_tile[kMaxSkPairs + 1];
  int32_t start_kb[kMaxSkPairs + 1];
  // Per range, for the tile of its first item (head) and of its last item
  // (tail), when that tile is split: the first range covering the tile and
  // the number of (non-empty) ranges that do.
  int16_t head_q0[kMaxSkPairs], head_n[kMaxSkPairs];
  int16_t tail_q0[kMaxSkPairs], tail_n[kMaxSkPairs];
};

struct GemmParams {
  CUtensorMap maps[kMaxMaps];
  Stripes stripes;
  StreamK sk;
  Prob probs[kMaxProbs];
  Group groups[kMaxGroups];
  Seg segs[kMaxSegs];
  int32_t num_maps, num_probs, num_groups, num_segs;
  int32_t total_tiles;
  int32_t deal_long, deal_s0;  // the deal of the data-parallel tiles (see Deal); 0, 0: round robin
  int32_t deal_r;              // deal_long mod the launch's pairs
  int32_t tile_m;
  int32_t* status;          // device status word (workspace)
  uint64_t timeout_ns;      // bound on every wait inside the kernel
  int32_t stall_injection;  // test hook: 1, producers load nothing; 2, stream-K parts but a tile's first run late
};

// Column sums over tokens (bias gradients): dst[c] = sum_r src[r][c].
constexpr int kMaxColsumJobs = 2 * kMaxShards + 1;
struct ColsumJob {
  const void* src;  // [rows x cols] row-major, the plan's dtype
  void* dst;        // [cols], the plan's dtype
  int64_t rows;
  int32_t cols;
  int32_t strip_begin;  // first CTA of this job
};
struct ColsumParams {
  ColsumJob jobs[kMaxColsumJobs];
  int32_t num_jobs;
  int32_t total_strips;
  // A job whose src is null reads the stripes below as one [rows x cols]
  // tensor (db2 of the sequence-parallel layout, from the dY stripes).
  int32_t num_stripes;
  int64_t stripe_row0[kMaxStripes + 1];
  const void* stripe_src[kMaxStripes];
};
// Columns of a strip with lane_threads 16-byte loads per strip row, and the
// launch shape (lane threads 8, 4 or 2; rows in flight per thread 4 or 8) of
// a set of jobs on sms SMs.
struct ColsumShape {
  int lane_threads, unroll;
};
int colsum_strip_cols(bool bf16, int lane_threads);
ColsumShape colsum_shape(const ColsumJob* jobs, int num_jobs, bool bf16, int sms);
cudaError_t launch_colsum(const ColsumParams& p, bool bf16, ColsumShape shape, cudaStream_t stream);

// Kernel parameters live in the 32 KB parameter space (__grid_constant__).
static_assert(sizeof(GemmParams) <= 32000, "kernel parameter block too large");

// Status codes written to the device status word.
constexpr int32_t kDevOk = 0;
constexpr int32_t kDevTimeoutProducer = 1;
constexpr int32_t kDevTimeoutMma = 2;
constexpr int32_t kDevTimeoutEpilogue = 3;

// Launchers (defined next to their kernels).
int tc_gemm_max_smem_bytes();
// Launches clusters of two CTAs: p.sk.pairs of them when the stream-K tail is
// on (the kernel's stream-K instance), else as many as fit on the device (at
// most one per tile), with epi_warps epilogue warps per CTA; max_pairs_hint is
// used if the occupancy query fails.
cudaError_t launch_tc_gemm(const GemmParams& p, int kernel_tag, int epi_warps, int max_pairs_hint,
                           cudaStream_t stream);
// Pairs (clusters of two CTAs) of a launch kind that can be resident at once
// on the current device (0 if the query fails).
int tc_gemm_max_pairs(int kernel_tag);
// The pairs launch_tc_gemm launches for p when the stream-K tail is off.
int tc_gemm_grid_pairs(const GemmParams& p, int kernel_tag, int max_pairs_hint);
// Epilogue warps per CTA for a launch (8: 32-column chunks and 32 x 32
// output boxes; 16: 16-column chunks and 32-row x 16-column boxes): 16 for a
// column or dgrad launch whose activation problems have at most
// kShortKBlocks K blocks (p.probs[].kblocks must be set).
constexpr int kShortKBlocks = 8;  // K <= 1024
// Problems of at least this many K blocks alternate their K direction by wave
// (Prob::k_rev).
constexpr int kRevKBlocks = 48;  // K > 6016
int tc_epi_warps_for(const GemmParams& p, int kernel_tag);
cudaError_t launch_simt_gemm(const GemmParams& p, cudaStream_t stream);
// The epilogues' activation forms on plain arrays (tpmlp_eval_activation).
cudaError_t launch_act_eval(int fn, const float* x, const float* y, const float* dh, float* o0, float* o1,
                            float* o2, int64_t n, cudaStream_t stream);

// Kernel tags: one kernel symbol per launch kind, so that profiles tell the
// launches of a training step apart.
enum KernelTag : int {
  TAG_FWD_COLUMN = 0,   // column-parallel GEMM + activation
  TAG_FWD_ROW = 1,      // row-parallel GEMM with the g-sum
  TAG_BWD_DGRAD = 2,    // dH_i -> dA_i (act') and dW2_i
  TAG_BWD_FSUM = 3,     // dX with the f-sum, and dW1_i (dW3_i)
  TAG_ATTN_QKV = 4,     // attention: column-parallel QKV projection
  TAG_ATTN_OUT = 5,     // attention: row-parallel output projection with the g-sum
  TAG_ATTN_OUT_BWD = 6, // attention: dO_i and dWO_i
  TAG_ATTN_QKV_BWD = 7, // attention: dX with the f-sum, and dW_QKV,i
  kNumKernelTags = 8,
};

}  // namespace tpmlp
