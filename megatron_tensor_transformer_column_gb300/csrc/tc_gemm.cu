// tc_gemm.cu -- persistent, warp-specialised 2-SM tcgen05 GEMM for sm_103a
// with the MLP block's fused epilogues.
//
// CTAs run in pairs (clusters of two, one CTA per SM).  A pair owns a
// 256 x 256 output tile: each CTA holds 128 rows of A and half of B's columns
// in its shared memory; the even CTA issues tcgen05.mma.cta_group::2, which
// reads both CTAs' operands and writes each CTA's 128 rows of D into that
// CTA's TMEM.  Per CTA:
//   * warp 0 (one lane): TMA producer -- per 128-deep K stage, this CTA's
//     128 x 128 slice of A and of its half of B (boxes of 64 columns x 128
//     rows, 64 KB) into a 3-stage ring; the completion of both CTAs' copies
//     is counted on the even CTA's "full" barrier;
//   * warp 1 (one lane, even CTA): allocates 512 TMEM columns in both CTAs,
//     issues the MMAs into one of two 256-column accumulators and multicasts
//     its commits (stage free, accumulator ready) to both CTAs;
//   * warps 2..9 (or 2..17, see tc_epi_warps_for): drain the other
//     accumulator through tcgen05.ld, apply the epilogue (store, GeLU /
//     SwiGLU forward, GeLU' / SwiGLU' backward, whose saved pre-activations
//     come in through the warp's staging blocks) and write bf16 rows to HBM
//     with TMA stores from those blocks; the two accumulators let the
//     epilogue of one tile run under the main loop of the next.
// The MMAs of a stage are issued as straight-line code (issue_stage): on
// GB300 a branch between two tcgen05.mma instructions cost about a third of
// the tensor throughput.
//
// The shard sums of the tensor-parallel MLP are K loops here: a problem
// with several segments (one per shard) accumulates every segment's product
// into the same TMEM tile before the epilogue reads it, so the g-sum of the
// forward row-parallel GEMM and the f-sum of the dX GEMM never leave the
// chip.  ("Parallelism" tag page of Jiang Yi's homepage, post "megatron-lm",
// Method / FFN: the partial-sum identity [H1, H2][W21; W22] = H1 W21 + H2 W22
// and the f/g table.)
//
// One body, two schedules (template parameter kSK):
//   * data-parallel: pair q computes tiles q, q + pairs, q + 2 pairs, ...,
//     or, in a launch that places long-K weight-gradient tiles first, the
//     deal described at Deal (tpmlp_internal.h), which hands the pairs that
//     drew one long tile fewer a head of short tiles first; a long-K tile
//     (Prob::k_rev) walks its K blocks backwards in odd waves;
//   * stream-K tail: round robin for the launch's full waves, then each pair
//     takes one item of the last, partial wave: a range of one tile's K
//     blocks (a part).  Every part leaves its fp32 accumulator in the
//     workspace and takes a ticket; the part whose ticket is the last one
//     adds all parts, in range order, into its own accumulator and runs the
//     tile's epilogue.  No pair ever waits for another pair, so the result
//     does not depend on which pairs are resident or when they run, and the
//     fixed order makes it the same on every run.
//
// Every wait is bounded: after GemmParams::timeout_ns a waiting role records
// a status code in the workspace, raises the abort flag of both CTAs, which
// makes the other roles leave their loops, waits (again bounded) for its own
// copies and MMAs in flight, and the pair frees its TMEM and exits.
#include <mutex>

#include "tc_gemm_common.cuh"

namespace tpmlp {
namespace {

// ------------------------------------------------------------------ schedules
// An item is a tile and a range [kb0, kb1) of its K blocks, counted over all
// of its segments: the whole tile, or (stream-K) a part of a split tile.
struct Item {
  TileInfo ti;
  int tile;      // -1: no more items
  int kb0, kb1;
  bool split;    // a part of a tile split between stream-K ranges
};

template <bool kSK>
struct Sched {
  Item it;
  Deal deal;           // this pair's walk over the data-parallel tiles
  int pair;
  int r;               // stream-K: this pair's range
  int sk_tile, sk_kb;  // stream-K: next position in that range
  bool in_dp;
};

template <bool kSK>
__device__ __forceinline__ void sched_next(Sched<kSK>& s, const GemmParams& p, int npairs) {
  const int dp_end = kSK ? p.sk.dp_tiles : p.total_tiles;
  if (!kSK || s.in_dp) {
    const int t = deal_next(s.deal, p.deal_long, p.deal_r, p.deal_s0, s.pair, npairs, dp_end);
    if (t >= 0) {
      s.it.tile = t;
      s.it.ti = decode_tile(p, s.it.tile, npairs);
      s.it.kb0 = 0;
      s.it.kb1 = p.probs[s.it.ti.prob].kblocks;
      s.it.split = false;
      return;
    }
    if (!kSK) {
      s.it.tile = -1;
      return;
    }
    s.in_dp = false;
    if (s.r < 0 || s.r >= p.sk.pairs) {
      s.it.tile = -1;
      return;
    }
    s.sk_tile = p.sk.start_tile[s.r];
    s.sk_kb = p.sk.start_kb[s.r];
  }
  const int end_tile = p.sk.start_tile[s.r + 1], end_kb = p.sk.start_kb[s.r + 1];
  while (s.sk_tile < end_tile || (s.sk_tile == end_tile && s.sk_kb < end_kb)) {
    const int t = s.sk_tile;
    const TileInfo ti = decode_tile(p, t, 0);
    const int kbt = p.probs[ti.prob].kblocks;
    const int kb0 = s.sk_kb, kb1 = t == end_tile ? end_kb : kbt;
    s.sk_tile = t + 1;
    s.sk_kb = 0;
    if (kb1 > kb0) {
      s.it.tile = t;
      s.it.ti = ti;
      s.it.kb0 = kb0;
      s.it.kb1 = kb1;
      s.it.split = kb0 > 0 || kb1 < kbt;
      return;
    }
  }
  s.it.tile = -1;
}

// pair < 0: an empty schedule.
template <bool kSK>
__device__ __forceinline__ void sched_init(Sched<kSK>& s, const GemmParams& p, int pair, int npairs) {
  deal_init(s.deal, pair);
  s.pair = pair;
  s.r = pair < 0 ? -1 : npairs - 1 - pair;
  s.in_dp = true;
  sched_next(s, p, npairs);
}

// ------------------------------------------------------------------ producer cursor
// Walks the (item, segment, K block) sequence of one CTA of a pair in the
// order the main loop consumes it.
template <bool kSK>
struct Cursor {
  Sched<kSK> s;        // the current item
  const void* ma;      // tensor maps of the current segment
  const void* mb;
  const void* mb2;
  int seg, kb, kblocks, left;  // segment, K block in it, its K blocks; K blocks left in the item
  int dir;                     // +1, or -1 for a reversed walk (TileInfo::rev)
  int a_major, b_major, dual;
  int a_striped, b_striped;  // operand read from the launch's token stripes
  int a_sj, b_sj;            // its current stripe,
  int a_y0, b_y0;            //   that stripe's first token row,
  int a_next, b_next;        //   and the next stripe's (an MN-major K walk crosses it)
  int m0, n0;          // this CTA's first row of A and first column of B
  int nA, nB;          // boxes this CTA loads per operand
  uint32_t bytes_pair; // bytes both CTAs load per K block (counted on the even CTA)
};

template <bool kSK>
__device__ __forceinline__ void cursor_segment(Cursor<kSK>& c, const GemmParams& p) {
  const Seg& S = p.segs[c.seg];
  c.kb = 0;
  c.kblocks = (S.K + kBK - 1) / kBK;
  c.ma = &p.maps[S.a_map];
  c.mb = &p.maps[S.b_map];
  c.mb2 = c.dual ? static_cast<const void*>(&p.maps[S.b2_map]) : nullptr;
  c.a_striped = S.a_striped;
  c.b_striped = S.b_striped;
  // The stripe of the first box: K-major operands keep it for the whole
  // segment (their token rows are this CTA's M or N rows); MN-major ones walk
  // the tokens along K and move to the next stripe in cursor_next.
  if (c.a_striped) {
    const int j = stripe_of(p.stripes, c.a_major == MAJOR_MN ? 0 : c.m0);
    c.a_sj = j;
    c.a_y0 = static_cast<int>(p.stripes.row0[j]);
    c.a_next = j + 1 < p.stripes.num ? static_cast<int>(p.stripes.row0[j + 1]) : INT_MAX;
  }
  if (c.b_striped) {
    const int j = stripe_of(p.stripes, c.b_major == MAJOR_MN ? 0 : c.n0);
    c.b_sj = j;
    c.b_y0 = static_cast<int>(p.stripes.row0[j]);
    c.b_next = j + 1 < p.stripes.num ? static_cast<int>(p.stripes.row0[j + 1]) : INT_MAX;
  }
}

__device__ __forceinline__ void stripe_advance(const GemmParams& p, int k0, int& sj, int& y0, int& next) {
  while (k0 >= next) {
    ++sj;
    y0 = next;
    next = sj + 1 < p.stripes.num ? static_cast<int>(p.stripes.row0[sj + 1]) : INT_MAX;
  }
}

// The stripe holding token row k0, from scratch (a reversed K walk).
__device__ __forceinline__ void stripe_at(const GemmParams& p, int k0, int& sj, int& y0, int& next) {
  sj = stripe_of(p.stripes, k0);
  y0 = static_cast<int>(p.stripes.row0[sj]);
  next = sj + 1 < p.stripes.num ? static_cast<int>(p.stripes.row0[sj + 1]) : INT_MAX;
}

template <bool kSK>
__device__ __forceinline__ void cursor_stripes(Cursor<kSK>& c, const GemmParams& p) {
  const bool rev = c.s.it.ti.rev;
  if (c.a_striped && c.a_major == MAJOR_MN) {
    if (rev) stripe_at(p, c.kb * kBK, c.a_sj, c.a_y0, c.a_next);
    else stripe_advance(p, c.kb * kBK, c.a_sj, c.a_y0, c.a_next);
  }
  if (c.b_striped && c.b_major == MAJOR_MN) {
    if (rev) stripe_at(p, c.kb * kBK, c.b_sj, c.b_y0, c.b_next);
    else stripe_advance(p, c.kb * kBK, c.b_sj, c.b_y0, c.b_next);
  }
}

// A reversed walk enters a segment at its last K block.
template <bool kSK>
__device__ __forceinline__ void cursor_segment_last(Cursor<kSK>& c, const GemmParams& p) {
  cursor_segment(c, p);
  c.kb = c.kblocks - 1;
  cursor_stripes(c, p);
}

// Set the cursor on the first K block of its schedule's current item.
template <bool kSK>
__device__ __forceinline__ void cursor_item(Cursor<kSK>& c, const GemmParams& p, uint32_t rank) {
  if (c.s.it.tile < 0) return;
  const TileInfo& ti = c.s.it.ti;
  const Prob& P = p.probs[ti.prob];
  c.dual = P.epi == EPI_SWIGLU_FWD;
  const PairShape ps = pair_shape(ti, c.dual, P.a_major, P.b_major);
  c.nA = rank ? ps.nA[1] : ps.nA[0];
  c.nB = rank ? ps.nB[1] : ps.nB[0];
  c.bytes_pair = ps.bytes[0] + ps.bytes[1];
  c.m0 = ti.m0 + kBM * static_cast<int>(rank);
  c.n0 = ti.n0 + ps.half * static_cast<int>(rank);
  c.a_major = P.a_major;
  c.b_major = P.b_major;
  c.left = c.s.it.kb1 - c.s.it.kb0;
  c.dir = ti.rev ? -1 : 1;
  if (ti.rev) {  // a whole tile (kb0 = 0), its segments and K blocks last to first
    c.seg = P.seg_begin + P.seg_count - 1;
    cursor_segment_last(c, p);
    return;
  }
  c.seg = P.seg_begin;
  int skip = c.s.it.kb0;
  cursor_segment(c, p);
  if (kSK) {
    while (skip >= c.kblocks) {  // a stream-K part may start in a later segment
      skip -= c.kblocks;
      ++c.seg;
      cursor_segment(c, p);
    }
    if (skip > 0) {
      c.kb = skip;
      cursor_stripes(c, p);
    }
  }
}

template <bool kSK>
__device__ __forceinline__ void cursor_next(Cursor<kSK>& c, const GemmParams& p, int npairs, uint32_t rank) {
  if (--c.left == 0) {
    sched_next(c.s, p, npairs);
    cursor_item(c, p, rank);
    return;
  }
  c.kb += c.dir;
  if (static_cast<unsigned>(c.kb) < static_cast<unsigned>(c.kblocks)) {
    cursor_stripes(c, p);
    return;
  }
  c.seg += c.dir;
  if (c.dir < 0) cursor_segment_last(c, p);
  else cursor_segment(c, p);
}

// Issue this CTA's box copies for the cursor's K block.
template <bool kSK>
__device__ __forceinline__ void cursor_issue(const GemmParams& p, const Cursor<kSK>& c, uint32_t sb, uint32_t fb) {
  const int k0 = c.kb * kBK;
  const uint32_t sbB = sb + kOperandBytes;
  for (int b = 0; b < c.nA; ++b) {
    // K-major: box b covers K [k0 + 64 b, +64) of the 128 rows;
    // MN-major: box b covers columns [m0 + 64 b, +64) of K rows [k0, k0 + kBK).
    const bool mn = c.a_major == MAJOR_MN;
    const int x = mn ? c.m0 + 64 * b : k0 + 64 * b;
    int y = mn ? k0 : c.m0;
    const CUtensorMap* ma = static_cast<const CUtensorMap*>(c.ma);
    if (c.a_striped) {  // the stored rows are tokens: the stripe's map, stripe-local y
      ma += c.a_sj;
      y -= c.a_y0;
    }
    ptx::tma_load_2d_pair(sb + b * (mn ? kMNBoxBytes : kKBoxBytes), ma, x, y, fb);
  }
  for (int j = 0; j < c.nB; ++j) {
    const bool mn = c.b_major == MAJOR_MN;
    const int x = mn ? c.n0 + 64 * j : k0 + 64 * j;
    int y = mn ? k0 : c.n0;
    const CUtensorMap* mb = static_cast<const CUtensorMap*>(c.mb);
    if (c.b_striped) {
      mb += c.b_sj;
      y -= c.b_y0;
    }
    ptx::tma_load_2d_pair(sbB + j * (mn ? kMNBoxBytes : kKBoxBytes), mb, x, y, fb);
  }
  if (c.dual && c.nB > 0)  // SwiGLU up projection (MN-major like the gate), second B box
    ptx::tma_load_2d_pair(sbB + kMNBoxBytes, c.mb2, c.n0, k0, fb);
}

// ------------------------------------------------------------------ stream-K parts
// A range's first split item leaves its partial in slot 2r, its last one in
// slot 2r + 1 (a range holds at most those two parts: the items between them
// are whole tiles).  A slot holds, per epilogue warp wi of the pair
// (rank * kEW + warp - 2), the four 32 x N fp32 accumulator chunks that warp
// drains (the same TMEM lanes and columns in every pair), laid out so that
// each 16-byte store / load of a warp covers 512 contiguous bytes.  The
// ticket counter of a split tile, one per epilogue warp position, is the
// counter word of the range holding the tile's K block 0.
__device__ __forceinline__ uint32_t* sk_counter(const GemmParams& p, int q0, int wi) {
  return reinterpret_cast<uint32_t*>(reinterpret_cast<char*>(p.status) + kSkFlagsOffset) + q0 * kSkWarpsPerPair + wi;
}

template <int N>
__device__ __forceinline__ char* sk_chunk(const GemmParams& p, int slot, int wi, int cslot) {
  return reinterpret_cast<char*>(p.status) + kSkSlotsOffset + static_cast<size_t>(slot) * kSkSlotBytes +
         static_cast<size_t>(wi * 4 + cslot) * (32 * N * sizeof(float));
}

// The slot of range q's part of tile j: its first item starts in j.
__device__ __forceinline__ int sk_slot(const GemmParams& p, int q, int j) {
  return 2 * q + (p.sk.start_tile[q] == j ? 0 : 1);
}

__device__ __forceinline__ bool sk_range_empty(const GemmParams& p, int r) {
  return p.sk.start_tile[r] == p.sk.start_tile[r + 1] && p.sk.start_kb[r] == p.sk.start_kb[r + 1];
}

// TMEM column of this warp's chunk cslot (0..3) of a tile -- the chunks the
// epilogue reads, in its order -- or -1 past the tile's valid columns.  The
// warp covers columns part * 256 / parts .. of the accumulator (parts = the
// warps per lane quarter).  SwiGLU forward: the warp's output columns are
// part * 128 / parts ..; chunk 2c is the gate, 2c + 1 the up projection of
// output columns oc = part * 128 / parts + c N .. (see swiglu_cols).
template <int N>
__device__ __forceinline__ void swiglu_cols(bool merged, int oc, uint32_t& g_col, uint32_t& u_col) {
  // merged: CTA-half h = oc / 64 of B holds gate columns at 128 h + oc % 64
  // and the matching up columns 64 further; split: gate at oc, up at 128 + oc
  const int h = oc >> 6, w = oc & 63;
  g_col = merged ? static_cast<uint32_t>(128 * h + w) : static_cast<uint32_t>(oc);
  u_col = merged ? g_col + 64u : 128u + static_cast<uint32_t>(oc);
}

template <int N>
__device__ __forceinline__ int sk_chunk_col(const Prob& P, const TileInfo& ti, int part, int parts, int cslot) {
  if (P.epi == EPI_SWIGLU_FWD) {
    const int oc = part * (128 / parts) + (cslot >> 1) * N;
    if (oc >= ti.valid_n) return -1;
    uint32_t g, u;
    swiglu_cols<N>(swiglu_merged(ti, P), oc, g, u);
    return static_cast<int>((cslot & 1) ? u : g);
  }
  const int col = part * (256 / parts) + cslot * N;
  return col < ti.valid_n ? col : -1;
}

// This warp's chunks of a part, raw fp32, to its slot.
template <int N>
__device__ __forceinline__ void sk_part_store(const GemmParams& p, const Prob& P, const Item& it, int slot,
                                              uint32_t tacc, int part, int parts, int wi, int lane) {
#pragma unroll 1
  for (int cs = 0; cs < 4; ++cs) {
    const int tc = sk_chunk_col<N>(P, it.ti, part, parts, cs);
    if (tc < 0) continue;
    uint32_t v[N];
    ptx::tmem_ld_32x32b(tacc + static_cast<uint32_t>(tc), v);
    ptx::tmem_wait_ld();
    char* dst = sk_chunk<N>(p, slot, wi, cs) + lane * 16;
#pragma unroll
    for (int j4 = 0; j4 < N / 4; ++j4)
      ptx::st_cg_v4(dst + j4 * 512, v[4 * j4], v[4 * j4 + 1], v[4 * j4 + 2], v[4 * j4 + 3]);
  }
}

// After its stores: take this warp's ticket of the tile.  A counter holds
// the launch's epoch (low 24 bits) above an 8-bit count of the parts that
// arrived; a value from another launch (an aborted one) counts as zero, so
// no reset is needed.  The compare-and-swap loop retries only when another
// part arrived in between: at most nparts + 1 rounds, and it never waits for
// a part that has not arrived.  True for the warp holding the last ticket;
// that warp then acquires every other part's stores.
__device__ __forceinline__ bool sk_ticket(const GemmParams& p, int q0, int nparts, int wi, int lane) {
  __threadfence();
  __syncwarp();
  uint32_t* ctr = sk_counter(p, q0, wi);
  uint32_t count = 0;
  if (lane == 0) {
    const uint32_t tag = (p.sk.epoch & 0xFFFFFFu) << 8;
    uint32_t cur = tag;
    for (int round = 0; round <= kMaxSkPairs + 1; ++round) {
      const uint32_t want = ((cur & ~0xFFu) == tag ? cur : tag) + 1u;
      const uint32_t seen = ptx::atom_cas_acq_rel_gpu_u32(ctr, cur, want);
      if (seen == cur) {
        count = want & 0xFFu;
        break;
      }
      cur = seen;
    }
  }
  count = __shfl_sync(0xffffffffu, count, 0);
  if (count != static_cast<uint32_t>(nparts)) return false;
  (void)ptx::ld_acquire_gpu_u32(ctr);  // every lane acquires the other parts' stores
  __syncwarp();
  return true;
}

// Add range q's chunk (N / 4 16-byte loads in flight per lane) to v.
template <int N>
__device__ __forceinline__ void sk_add_slot(const char* src, uint32_t (&v)[N]) {
  float4 f[N / 4];
#pragma unroll
  for (int j4 = 0; j4 < N / 4; ++j4) f[j4] = ptx::ld_cg_v4f(src + j4 * 512);
#pragma unroll
  for (int j4 = 0; j4 < N / 4; ++j4) {
    v[4 * j4 + 0] = __float_as_uint(__uint_as_float(v[4 * j4 + 0]) + f[j4].x);
    v[4 * j4 + 1] = __float_as_uint(__uint_as_float(v[4 * j4 + 1]) + f[j4].y);
    v[4 * j4 + 2] = __float_as_uint(__uint_as_float(v[4 * j4 + 2]) + f[j4].z);
    v[4 * j4 + 3] = __float_as_uint(__uint_as_float(v[4 * j4 + 3]) + f[j4].w);
  }
}

// Add this pair's own chunk, from TMEM, to v.
template <int N>
__device__ __forceinline__ void sk_add_tmem(uint32_t taddr, uint32_t (&v)[N]) {
  uint32_t t[N];
  ptx::tmem_ld_32x32b(taddr, t);
  ptx::tmem_wait_ld();
#pragma unroll
  for (int j = 0; j < N; ++j) v[j] = __float_as_uint(__uint_as_float(v[j]) + __uint_as_float(t[j]));
}

// The last part: the sum of all parts, added in range order (its own from
// TMEM, the others from their slots), written back into its accumulator, on
// which the tile's normal epilogue then runs.  The parts of tile j are the
// non-empty ranges from q0 (the one holding its K block 0) on that start in
// j.
template <int N>
__device__ __forceinline__ void sk_fold(const GemmParams& p, const Prob& P, const Item& it, int r, int q0,
                                        uint32_t tacc, int part, int parts, int wi, int lane) {
#pragma unroll 1
  for (int cs = 0; cs < 4; ++cs) {
    const int tc = sk_chunk_col<N>(P, it.ti, part, parts, cs);
    if (tc < 0) continue;
    const uint32_t taddr = tacc + static_cast<uint32_t>(tc);
    uint32_t v[N];
    if (q0 == r) {
      ptx::tmem_ld_32x32b(taddr, v);
      ptx::tmem_wait_ld();
    } else {
      const char* src = sk_chunk<N>(p, sk_slot(p, q0, it.tile), wi, cs) + lane * 16;
#pragma unroll
      for (int j4 = 0; j4 < N / 4; ++j4) {
        const float4 f = ptx::ld_cg_v4f(src + j4 * 512);
        v[4 * j4 + 0] = __float_as_uint(f.x);
        v[4 * j4 + 1] = __float_as_uint(f.y);
        v[4 * j4 + 2] = __float_as_uint(f.z);
        v[4 * j4 + 3] = __float_as_uint(f.w);
      }
    }
#pragma unroll 1
    for (int q = q0 + 1; q < p.sk.pairs && p.sk.start_tile[q] == it.tile; ++q) {
      if (sk_range_empty(p, q)) continue;
      if (q == r)
        sk_add_tmem<N>(taddr, v);
      else
        sk_add_slot<N>(sk_chunk<N>(p, sk_slot(p, q, it.tile), wi, cs) + lane * 16, v);
    }
    ptx::tmem_st_32x32b(taddr, v);
  }
  ptx::tmem_wait_st();
}

// ------------------------------------------------------------------ the kernel body
template <bool kSK, int kEW>
__device__ __forceinline__ void tc_gemm_body(const GemmParams& p, uint8_t* smem_raw) {
  constexpr int N = chunk_cols(kEW);  // accumulator columns per epilogue chunk
  constexpr int kParts = kEW / 4;      // epilogue warps per TMEM lane quarter
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kStages * kStageBytes + kEpiBytes);
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(bars + kNumBars);
  volatile int32_t* abort_flag = reinterpret_cast<volatile int32_t*>(tmem_holder + 1);

  const uint32_t smem_base = ptx::smem_u32(smem);
  const uint32_t bar0 = ptx::smem_u32(bars);
  auto full_bar = [&](int s) { return bar0 + 8u * s; };                        // even CTA: copies landed
  auto empty_bar = [&](int s) { return bar0 + 8u * (kStages + s); };           // both: stage consumed
  auto tfull_bar = [&](int a) { return bar0 + 8u * (2 * kStages + a); };       // both: accumulator ready
  auto tempty_bar = [&](int a) { return bar0 + 8u * (2 * kStages + kNumAcc + a); };  // even CTA: drained
  const uint32_t drain_bar = bar0 + 8u * (2 * kStages + 2 * kNumAcc);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = ptx::cluster_ctarank();
  const bool leader = rank == 0;
  const int pair = blockIdx.x >> 1;
  const int npairs = gridDim.x >> 1;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      ptx::mbar_init(full_bar(s), 1);
      ptx::mbar_init(empty_bar(s), 1);
    }
    for (int a = 0; a < kNumAcc; ++a) {
      ptx::mbar_init(tfull_bar(a), 1);
      ptx::mbar_init(tempty_bar(a), 2 * kEW);
    }
    ptx::mbar_init(drain_bar, 1);
    *abort_flag = 0;
    ptx::fence_mbarrier_init();
  }
  if (warp == 0 && lane == 0) {
    for (int i = 0; i < p.num_maps; ++i) ptx::prefetch_tmap(&p.maps[i]);
  }
  if (warp == 1) {
    ptx::tmem_alloc_pair(ptx::smem_u32(tmem_holder), kTmemCols);
    ptx::tmem_relinquish_pair();
  }
  ptx::tc_fence_before();
  ptx::cluster_sync();  // barriers of both CTAs initialised, TMEM allocated
  ptx::tc_fence_after();
  const uint32_t tmem_base = *tmem_holder;
  const Ctl ctl{abort_flag, ptx::map_to_cta(ptx::smem_u32(const_cast<int32_t*>(abort_flag)), rank ^ 1u), p.status,
                p.timeout_ns};

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer (both CTAs)
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      int armed_parity[kStages];
#pragma unroll
      for (int s = 0; s < kStages; ++s) armed_parity[s] = -1;
      bool ok = true;
      bool issued = false;
      Cursor<kSK> ld;
      sched_init(ld.s, p, p.stall_injection == 1 ? -1 : pair, npairs);  // injected stall: nothing to load
      cursor_item(ld, p, rank);
      while (ld.s.it.tile >= 0) {
        if (!bounded_wait(empty_bar(stage), phase ^ 1u, ctl, kDevTimeoutProducer)) {
          ok = false;
          break;
        }
        if (leader) {
          ptx::mbar_arrive_expect_tx(full_bar(stage), ld.bytes_pair);
          armed_parity[stage] = static_cast<int>(phase);
        }
        cursor_issue(p, ld, smem_base + stage * kStageBytes, ptx::map_to_cta(full_bar(stage), 0));
        issued = true;
        cursor_next(ld, p, npairs, rank);
        if (++stage == kStages) {
          stage = 0;
          phase ^= 1u;
        }
      }
      if (!ok && issued) {
        // Let every copy already issued land before the CTA can exit.
        if (leader) {
          for (int s = 0; s < kStages; ++s)
            if (armed_parity[s] >= 0) drain_wait(full_bar(s), static_cast<uint32_t>(armed_parity[s]));
        }
        spin_ns(kPeerDrainNs);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer (even CTA)
    if (leader && lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      bool ok = true;
      bool issued = false;
      // Descriptors of stage 0 for each operand layout; a stage and a K step
      // are added to the start-address field (16-byte units, no carry: the
      // ring lies below 256 KB).  K-major: 8-row groups 1024 B apart; K16
      // step j is +32 B inside a 64-wide box, box j/4 is +16 KB.  MN-major:
      // the two 64-column blocks are kMNBoxBytes apart (leading offset), 8-row
      // K groups 1024 B apart, K16 step j is +2048 B.
      const uint64_t a_k_desc = ptx::make_sdesc_sw128(smem_base, 16, 1024);
      const uint64_t a_mn_desc = ptx::make_sdesc_sw128(smem_base, kMNBoxBytes, 1024);
      const uint64_t b_k_desc = ptx::make_sdesc_sw128(smem_base + kOperandBytes, 16, 1024);
      const uint64_t b_mn_desc = ptx::make_sdesc_sw128(smem_base + kOperandBytes, kMNBoxBytes, 1024);
      Sched<kSK> s;
      for (sched_init(s, p, pair, npairs); ok && s.it.tile >= 0; sched_next(s, p, npairs)) {
        const Item& it = s.it;
        const TileInfo& ti = it.ti;
        const Prob& P = p.probs[ti.prob];
        const int a_major = P.a_major, b_major = P.b_major;
        const bool dual = P.epi == EPI_SWIGLU_FWD;
        const PairShape ps = pair_shape(ti, dual, a_major, b_major);
        // A full SwiGLU tile issues one N = 256 MMA over each CTA's [gate | up]
        // column blocks instead of two N = 128 MMAs (the wider MMA runs at the
        // full tensor rate, N = 128 at about 88 %); see swiglu_merged().
        const bool merged = dual && ps.n_mma == 128;
        const uint32_t idesc = ptx::make_idesc_bf16(kPairM, merged ? 256 : ps.n_mma, a_major, b_major);
        const uint64_t a_desc0 = a_major == MAJOR_MN ? a_mn_desc : a_k_desc;
        const uint64_t b_desc0 = b_major == MAJOR_MN ? b_mn_desc : b_k_desc;
        const uint32_t a_lo = static_cast<uint32_t>(a_desc0), a_hi = static_cast<uint32_t>(a_desc0 >> 32);
        const uint32_t b_lo = static_cast<uint32_t>(b_desc0), b_hi = static_cast<uint32_t>(b_desc0 >> 32);
        const int kind = (dual && !merged ? 4 : 0) | (a_major == MAJOR_MN ? 2 : 0) | (b_major == MAJOR_MN ? 1 : 0);
        if (!bounded_wait(tempty_bar(acc), acc_phase ^ 1u, ctl, kDevTimeoutMma)) {
          ok = false;
          break;
        }
        ptx::tc_fence_after();
        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * kAccCols);
        uint32_t accumulate = 0;
        // The item's K blocks [kb0, kb1), counted over the tile's segments.
        int sg = P.seg_begin;
        int K = p.segs[sg].K;
        int skip = it.kb0;
        if (kSK) {
          while (skip >= (K + kBK - 1) / kBK) {
            skip -= (K + kBK - 1) / kBK;
            K = p.segs[++sg].K;
          }
        }
        int k0 = skip * kBK;
        const int kstep = ti.rev ? -kBK : kBK;
        if (ti.rev) {  // a whole tile walked last to first: start at the last segment's last block
          sg = P.seg_begin + P.seg_count - 1;
          K = p.segs[sg].K;
          k0 = (K - 1) / kBK * kBK;
        }
        for (int left = it.kb1 - it.kb0; left > 0; --left) {
          if (!bounded_wait(full_bar(stage), phase, ctl, kDevTimeoutMma)) {
            ok = false;
            break;
          }
          ptx::tc_fence_after();
          const uint32_t st = static_cast<uint32_t>((stage * kStageBytes) >> 4);
          const int nk = min(kBK / 16, (K - k0 + 15) >> 4);
          issue_stage_any(kind, d_tmem, a_lo + st, a_hi, b_lo + st, b_hi, idesc, nk, accumulate);
          issued = true;
          ptx::mma_commit_pair_mc(empty_bar(stage), kPairMask);  // stage free in both CTAs
          if (++stage == kStages) {
            stage = 0;
            phase ^= 1u;
          }
          k0 += kstep;
          if (static_cast<unsigned>(k0) >= static_cast<unsigned>(K) && left > 1) {  // past either end
            sg += kstep > 0 ? 1 : -1;
            K = p.segs[sg].K;
            k0 = kstep > 0 ? 0 : (K - 1) / kBK * kBK;
          }
        }
        if (!ok) break;
        ptx::mma_commit_pair_mc(tfull_bar(acc), kPairMask);  // accumulator ready in both CTAs
        if (++acc == kNumAcc) {
          acc = 0;
          acc_phase ^= 1u;
        }
      }
      if (!ok && issued) {
        // Every MMA issued so far must finish before TMEM is released.
        ptx::mma_commit_pair(drain_bar);
        drain_wait(drain_bar, 0);
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue (both CTAs)
    const int q = warp & 3;              // TMEM lane quarter this warp may read
    const int part = (warp - 2) >> 2;    // which of the kParts column ranges of a tile
    constexpr int kCols = 256 / kParts;  // accumulator columns per warp (4 chunks of N)
    EpiStore es{smem_base + static_cast<uint32_t>(kStages * kStageBytes + (warp - 2) * 2 * epi_block_bytes<N>()), 0u,
                0, 0, 0};
    const int wi = static_cast<int>(rank) * kEW + (warp - 2);  // stream-K slot position of this warp
    int acc = 0;
    uint32_t acc_phase = 0;
    Sched<kSK> s;
    for (sched_init(s, p, pair, npairs); s.it.tile >= 0; sched_next(s, p, npairs)) {
      const Item& it = s.it;
      const TileInfo ti = it.ti;
      const Prob& P = p.probs[ti.prob];
      const int row = q * 32 + lane;
      const int vm = max(0, min(kBM, ti.valid_m - kBM * static_cast<int>(rank)));
      const bool row_ok = row < vm;
      const int64_t grow = static_cast<int64_t>(ti.m0) + kBM * static_cast<int>(rank) + row;
      const int wrow = ti.m0 + kBM * static_cast<int>(rank) + q * 32;  // this warp's first row
      es.rows = P.M;
      if (P.out_striped && wrow < P.M) {  // a warp's 32 rows never cross a stripe boundary
        es.sj = stripe_of(p.stripes, wrow);
        es.sy0 = static_cast<int>(p.stripes.row0[es.sj]);
      }
      if (row_ok && (P.epi == EPI_GELU_BWD || P.epi == EPI_SWIGLU_BWD)) {
        // Pull this thread's row of the saved pre-activation(s) into L2
        // while the accumulator is still being computed.
        const int c0 = part * kCols;
        const int cn = min(kCols, ti.valid_n - c0);
        if (cn > 0) {
          const int64_t off = grow * P.ldo + ti.n0 + c0;
          const __nv_bfloat16* a0 = static_cast<const __nv_bfloat16*>(P.aux0) + off;
          for (int b = 0; b < 2 * cn; b += 128) ptx::prefetch_l2(reinterpret_cast<const char*>(a0) + b);
          ptx::prefetch_l2(reinterpret_cast<const char*>(a0) + 2 * cn - 1);
          if (P.epi == EPI_SWIGLU_BWD) {
            const __nv_bfloat16* a1 = static_cast<const __nv_bfloat16*>(P.aux1) + off;
            for (int b = 0; b < 2 * cn; b += 128) ptx::prefetch_l2(reinterpret_cast<const char*>(a1) + b);
            ptx::prefetch_l2(reinterpret_cast<const char*>(a1) + 2 * cn - 1);
          }
        }
      }
      if (!bounded_wait(tfull_bar(acc), acc_phase, ctl, kDevTimeoutEpilogue)) break;
      ptx::tc_fence_after();
      const uint32_t tacc = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(acc * kAccCols);
      bool finish = true;
      if (kSK && it.split) {
        // A part of a split tile: publish it; the last part to arrive adds
        // them all and runs the epilogue.  (Test hook, stall injection 2:
        // every part but the tile's first runs late, so that another part
        // than the first finishes the tile.)
        const bool head = p.sk.start_tile[s.r] == it.tile;  // the range's first item, else its last
        if (vm > 0) sk_part_store<N>(p, P, it, 2 * s.r + (head ? 0 : 1), tacc, part, kParts, wi, lane);
        const int q0 = head ? p.sk.head_q0[s.r] : p.sk.tail_q0[s.r];
        if (p.stall_injection == 2 && s.r != q0) spin_ns(20ull * 1000 * 1000);
        finish = sk_ticket(p, q0, head ? p.sk.head_n[s.r] : p.sk.tail_n[s.r], wi, lane);
        if (finish && vm > 0) sk_fold<N>(p, P, it, s.r, q0, tacc, part, kParts, wi, lane);
      }
      if (finish && vm > 0) {
        if (P.epi == EPI_SWIGLU_FWD) {
          const bool merged = swiglu_merged(ti, P);
#pragma unroll 1
          for (int c = 0; c < 2; ++c) {
            const int oc = part * (128 / kParts) + c * N;  // output columns oc .. oc + N - 1 of the tile
            if (oc >= ti.valid_n) break;
            uint32_t g_col, u_col;
            swiglu_cols<N>(merged, oc, g_col, u_col);
            uint32_t rg[N], ru[N];
            ptx::tmem_ld_32x32b(tacc + g_col, rg);
            ptx::tmem_ld_32x32b(tacc + u_col, ru);
            ptx::tmem_wait_ld();
            const int nvalid = min(N, ti.valid_n - oc);
            float g[N], u[N], h[N];
#pragma unroll
            for (int j = 0; j < N; ++j) {
              g[j] = __uint_as_float(rg[j]);
              u[j] = __uint_as_float(ru[j]);
            }
            add_bias<N>(P.aux0, ti.n0 + oc, nvalid, g);
            add_bias<N>(P.aux1, ti.n0 + oc, nvalid, u);
            act::x2::swiglu_xn(g, u, h);
            store_block<N>(es, p, P, 0, ti.n0 + oc, wrow, nvalid, g, lane);
            store_block<N>(es, p, P, 1, ti.n0 + oc, wrow, nvalid, u, lane);
            store_block<N>(es, p, P, 2, ti.n0 + oc, wrow, nvalid, h, lane);
          }
        } else {
#pragma unroll 1
          for (int c = 0; c < 4; ++c) {
            const int col = part * kCols + c * N;
            if (col >= ti.valid_n) break;
            uint32_t r[N];
            ptx::tmem_ld_32x32b(tacc + col, r);
            ptx::tmem_wait_ld();
            epilogue_chunk<N>(p, P, es, grow, row_ok, ti.n0 + col, wrow, min(N, ti.valid_n - col), r, lane);
          }
        }
      }
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive_cluster(ptx::map_to_cta(tempty_bar(acc), 0));
      if (++acc == kNumAcc) {
        acc = 0;
        acc_phase ^= 1u;
      }
    }
    if (lane == 0) ptx::bulk_wait_group_all();  // this warp's TMA stores are complete
    __syncwarp();
  }

  ptx::tc_fence_before();
  ptx::cluster_sync();  // no CTA leaves while its peer may still signal it
  if (warp == 1) {
    __syncwarp();
    ptx::tc_fence_after();
    ptx::tmem_dealloc_pair(tmem_base, kTmemCols);
  }
}

}  // namespace

// Two kernel symbols per launch kind (same body): the data-parallel schedule
// and, with the suffix _sk, the one with a stream-K tail; EW is the number
// of epilogue warps (kernel_for).
#define TPMLP_TC_KERNELS(name, EW)                                                                       \
  __global__ void __launch_bounds__(threads_for(EW), 1) name(const __grid_constant__ GemmParams p) {     \
    extern __shared__ __align__(1024) uint8_t smem_raw[];                                                \
    tc_gemm_body<false, EW>(p, smem_raw);                                                                \
  }                                                                                                      \
  __global__ void __launch_bounds__(threads_for(EW), 1) name##_sk(const __grid_constant__ GemmParams p) { \
    extern __shared__ __align__(1024) uint8_t smem_raw[];                                                \
    tc_gemm_body<true, EW>(p, smem_raw);                                                                 \
  }

// Launch kinds whose epilogues carry the activation (the column GEMM, the
// dgrad GEMM) also exist with 16 epilogue warps (suffix _w16).  The host
// takes them where the tiles' K is short (tc_epi_warps_for): there the
// epilogue of a tile lasts longer than its main loop and is bound by each
// warp's chain of TMEM load, arithmetic and store, which more warps overlap.
// With longer K the epilogue hides under the next tile's main loop and the
// extra warps only compete with the producer and the MMA issuer for issue
// slots (measured on GB300: C2's column and dgrad launches -7 % and -5 % with
// 16 warps; C3 to C5's +1 to +3 %).
TPMLP_TC_KERNELS(tpmlp_fwd_column_gemm_act, 8)
TPMLP_TC_KERNELS(tpmlp_fwd_column_gemm_act_w16, 16)
TPMLP_TC_KERNELS(tpmlp_fwd_row_gemm_gsum, 8)
TPMLP_TC_KERNELS(tpmlp_bwd_dgrad_act_wgrad2, 8)
TPMLP_TC_KERNELS(tpmlp_bwd_dgrad_act_wgrad2_w16, 16)
TPMLP_TC_KERNELS(tpmlp_bwd_dx_fsum_wgrad1, 8)
TPMLP_TC_KERNELS(tpmlp_attn_qkv_proj, 8)
TPMLP_TC_KERNELS(tpmlp_attn_out_proj_gsum, 8)
TPMLP_TC_KERNELS(tpmlp_attn_out_proj_bwd, 8)
TPMLP_TC_KERNELS(tpmlp_attn_qkv_bwd_dx_fsum, 8)

int tc_gemm_max_smem_bytes() { return kSmemBytes; }

int tc_epi_warps_for(const GemmParams& p, int tag) {
  if (tag != TAG_FWD_COLUMN && tag != TAG_BWD_DGRAD) return 8;
  for (int i = 0; i < p.num_probs; ++i) {
    const Prob& P = p.probs[i];
    if (P.epi != EPI_STORE && P.kblocks > kShortKBlocks) return 8;
  }
  return 16;
}

using KernelFn = void (*)(GemmParams);

KernelFn kernel_for(int tag, bool stream_k, int epi_warps) {
  const bool w16 = epi_warps == 16;
  switch (tag) {
    case TAG_FWD_COLUMN:
      return w16 ? (stream_k ? tpmlp_fwd_column_gemm_act_w16_sk : tpmlp_fwd_column_gemm_act_w16)
                 : (stream_k ? tpmlp_fwd_column_gemm_act_sk : tpmlp_fwd_column_gemm_act);
    case TAG_FWD_ROW: return stream_k ? tpmlp_fwd_row_gemm_gsum_sk : tpmlp_fwd_row_gemm_gsum;
    case TAG_BWD_DGRAD:
      return w16 ? (stream_k ? tpmlp_bwd_dgrad_act_wgrad2_w16_sk : tpmlp_bwd_dgrad_act_wgrad2_w16)
                 : (stream_k ? tpmlp_bwd_dgrad_act_wgrad2_sk : tpmlp_bwd_dgrad_act_wgrad2);
    case TAG_BWD_FSUM: return stream_k ? tpmlp_bwd_dx_fsum_wgrad1_sk : tpmlp_bwd_dx_fsum_wgrad1;
    case TAG_ATTN_QKV: return stream_k ? tpmlp_attn_qkv_proj_sk : tpmlp_attn_qkv_proj;
    case TAG_ATTN_OUT: return stream_k ? tpmlp_attn_out_proj_gsum_sk : tpmlp_attn_out_proj_gsum;
    case TAG_ATTN_OUT_BWD: return stream_k ? tpmlp_attn_out_proj_bwd_sk : tpmlp_attn_out_proj_bwd;
    case TAG_ATTN_QKV_BWD: return stream_k ? tpmlp_attn_qkv_bwd_dx_fsum_sk : tpmlp_attn_qkv_bwd_dx_fsum;
    default: return nullptr;
  }
}

// Pairs (clusters of two CTAs) that can be resident at once on this device
// (every kernel has one CTA per SM: the same shared memory).
int tc_gemm_max_pairs(int tag) {
  static std::mutex mu;
  static int cache[64][kNumKernelTags] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64 || tag < 0 || tag >= kNumKernelTags) return 0;
  std::lock_guard<std::mutex> lk(mu);
  if (cache[dev][tag] > 0) return cache[dev][tag];
  KernelFn k = kernel_for(tag, false, 8);
  if (cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes) != cudaSuccess) return 0;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2, 1, 1);
  cfg.blockDim = dim3(threads_for(8), 1, 1);
  cfg.dynamicSmemBytes = kSmemBytes;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, k, &cfg) != cudaSuccess || n <= 0) return 0;
  cache[dev][tag] = n;
  return n;
}

int tc_gemm_grid_pairs(const GemmParams& p, int kernel_tag, int max_pairs_hint) {
  int pairs = tc_gemm_max_pairs(kernel_tag);
  if (pairs <= 0) pairs = max_pairs_hint > 0 ? max_pairs_hint : 1;
  return pairs < p.total_tiles ? pairs : p.total_tiles;
}

cudaError_t launch_tc_gemm(const GemmParams& p, int kernel_tag, int epi_warps, int max_pairs_hint,
                           cudaStream_t stream) {
  KernelFn k = kernel_for(kernel_tag, p.sk.on != 0, epi_warps);
  if (!k) return cudaErrorInvalidValue;
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
  if (e != cudaSuccess) return e;
  // the stream-K ranges were cut for exactly p.sk.pairs pairs
  const int pairs = p.sk.on ? p.sk.pairs : tc_gemm_grid_pairs(p, kernel_tag, max_pairs_hint);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * pairs, 1, 1);
  cfg.blockDim = dim3(threads_for(epi_warps), 1, 1);
  cfg.dynamicSmemBytes = kSmemBytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, k, p);
}

}  // namespace tpmlp
