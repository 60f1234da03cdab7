// tpmlp_api.cu -- host side of the C ABI declared in include/tpmlp.h:
// argument checks, the shard table, TMA tensor maps, the per-launch problem
// lists and the launches.  No device memory is allocated here.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <atomic>
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <new>
#include <vector>

#include "tpmlp.h"
#include "tpmlp_internal.h"

using namespace tpmlp;

enum PlanKind : int32_t { PLAN_MLP = 0, PLAN_ATTN = 1 };

struct tpmlp_plan {
  PlanKind kind;
  int64_t T, d;
  int32_t t;
  std::vector<int64_t> d_i;  // MLP: shard widths; attention: fused QKV widths n_i = dq_i + 2 dkv_i
  std::vector<int64_t> o_i;
  int64_t dff;
  std::vector<int64_t> dq_i, dkv_i;  // attention only
  tpmlp_act act;
  tpmlp_dtype dtype;
  uint64_t timeout_ns;
  int32_t stall_injection;
  int32_t stream_k;  // TPMLP_STREAM_K_OFF / _AUTO / _ALWAYS
  std::vector<int64_t> stripe_rows;  // sequence-parallel token stripes (empty: not set)
};

namespace {

thread_local int g_last_cuda_error = 0;
thread_local int g_last_launches = 0;
// Tiles the stream-K schedule split in the last launch of each kind on this
// thread: (problem, first row, first column, address of the problem's first
// output) per tile.
thread_local std::vector<int64_t> g_last_split[kNumKernelTags];
thread_local char g_last_error[256] = "";

tpmlp_status fail(tpmlp_status st, const char* fmt, ...) __attribute__((format(printf, 2, 3)));
tpmlp_status fail(tpmlp_status st, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_last_error, sizeof(g_last_error), fmt, ap);
  va_end(ap);
  return st;
}

constexpr int kTileM = 256;  // rows of a CTA pair's tile
constexpr int kSimtTile = 32;
constexpr uint64_t kDefaultTimeoutNs = 2000ull * 1000 * 1000;  // 2 s

tpmlp_status cuda_fail(cudaError_t e) {
  g_last_cuda_error = static_cast<int>(e);
  return fail(TPMLP_ERR_CUDA, "CUDA error %d (%s)", static_cast<int>(e), cudaGetErrorString(e));
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// ------------------------------------------------------------------ device
struct DeviceInfo {
  bool ok = false;
  int sms = 0;
  int cc_major = 0, cc_minor = 0;
};

tpmlp_status device_info(DeviceInfo* out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e);
  static std::mutex mu;
  static DeviceInfo cache[64];
  std::lock_guard<std::mutex> lk(mu);
  if (dev < 0 || dev >= 64) return TPMLP_ERR_UNSUPPORTED;
  if (!cache[dev].ok) {
    DeviceInfo di;
    if ((e = cudaDeviceGetAttribute(&di.sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return cuda_fail(e);
    if ((e = cudaDeviceGetAttribute(&di.cc_major, cudaDevAttrComputeCapabilityMajor, dev)) != cudaSuccess)
      return cuda_fail(e);
    if ((e = cudaDeviceGetAttribute(&di.cc_minor, cudaDevAttrComputeCapabilityMinor, dev)) != cudaSuccess)
      return cuda_fail(e);
    di.ok = true;
    cache[dev] = di;
  }
  *out = cache[dev];
  // Bind the device's primary context to this thread (threads that only ran
  // runtime calls without a context, such as autograd's worker, have none
  // current; the tensor-map encoder is a driver call and needs one).
  if ((e = cudaSetDevice(dev)) != cudaSuccess) return cuda_fail(e);
  // The kernels are built for sm_103a only (GB300).
  if (out->cc_major != 10 || out->cc_minor != 3)
    return fail(TPMLP_ERR_UNSUPPORTED, "device %d is sm_%d%d; the kernels are built for sm_103a", dev, out->cc_major,
                out->cc_minor);
  return TPMLP_OK;
}

// ------------------------------------------------------------------ tensor maps
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// 2-D row-major bf16 [rows x cols] with row stride ld elements.
// Operand maps (box_rows > 0): boxes of 64 columns (128 bytes, the swizzle
// span) by box_rows rows, 128-byte swizzle, out-of-range elements read as
// zero.  K-major operand tiles use 128-row boxes (128 M/N rows x 64 K),
// MN-major ones kTcBK-row boxes (kTcBK K rows of a 64-wide M/N block).
// Output maps, for the epilogue's TMA stores (out-of-range elements are not
// written): box_rows == kOutputMap32, 32 rows x 32 columns with a 64-byte
// swizzle (epilogues of 8 warps); kOutputMap16, 32 rows x 16 columns with a
// 32-byte swizzle (epilogues of 16 warps).
// Returns 0 on success, the CUresult otherwise (-1: entry point unavailable).
constexpr int kOutputMap32 = -1;
constexpr int kOutputMap16 = -2;
int encode_map(CUtensorMap* m, const void* ptr, int64_t rows, int64_t cols, int64_t ld, int box_rows) {
  auto fn = encode_fn();
  if (!fn) return -1;
  const bool out = box_rows < 0;
  const bool narrow = box_rows == kOutputMap16;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(ld) * 2};
  cuuint32_t box[2] = {out ? (narrow ? 16u : 32u) : 64u, out ? 32u : static_cast<cuuint32_t>(box_rows)};
  cuuint32_t es[2] = {1, 1};
  const CUtensorMapSwizzle swz =
      out ? (narrow ? CU_TENSOR_MAP_SWIZZLE_32B : CU_TENSOR_MAP_SWIZZLE_64B) : CU_TENSOR_MAP_SWIZZLE_128B;
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides, box, es,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, swz,
                  out ? CU_TENSOR_MAP_L2_PROMOTION_NONE : CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return static_cast<int>(r);
}

// ------------------------------------------------------------------ problem lists
// Stand-ins passed for an operand (or out0) that is the launch's striped
// input (output) in the sequence-parallel layout; never dereferenced.
const void* const kStripedIn = reinterpret_cast<const void*>(uintptr_t{16});
void* const kStripedOut = reinterpret_cast<void*>(uintptr_t{32});

struct Builder {
  GemmParams* p;
  bool tc;  // tensor-core path (tensor maps) or fp32 SIMT path
  int tile_m;
  std::vector<const void*> map_ptr;
  std::vector<int64_t> map_rows, map_cols;
  std::vector<int> map_box;
  std::vector<int64_t> map_ld;
  bool map_error = false;
  int cur_group = -1;
  int long_from = -1;  // first tile of the long-K groups placed last (balanced stream-K), or -1
  int long_end = 0;    // tiles [0, long_end) are long-K groups placed first (see Deal)

  explicit Builder(GemmParams* params, bool tensor_cores) : p(params), tc(tensor_cores) {
    std::memset(static_cast<void*>(p), 0, sizeof(GemmParams));
    tile_m = tc ? kTileM : kSimtTile;
    p->tile_m = tile_m;
  }

  // Sequence-parallel layout: this launch's token-striped input (X or dY,
  // in_cols wide) and output (Y or dX, out_cols wide), stripes as the plan set.
  int stripe_map_base[3] = {-1, -1, -1};  // input K-major, input MN-major, output
  void set_stripes(const tpmlp_plan* pl, const void* const* in, int64_t in_cols, void* const* out,
                   int64_t out_cols) {
    Stripes& st = p->stripes;
    st.num = static_cast<int32_t>(pl->stripe_rows.size());
    st.row0[0] = 0;
    for (int j = 0; j < st.num; ++j) {
      st.row0[j + 1] = st.row0[j] + pl->stripe_rows[j];
      st.in[j] = in ? in[j] : nullptr;
      st.out[j] = out ? out[j] : nullptr;
    }
    st.in_ld = in_cols;
    st.out_ld = out_cols;
  }

  // num consecutive maps, one per stripe (an empty stripe reuses a non-empty
  // stripe's map: no box ever selects it).
  int stripe_maps(bool output, int box_rows) {
    if (!tc) return -1;
    const int slot = output ? 2 : (box_rows == 128 ? 0 : 1);  // one output box shape per launch
    if (stripe_map_base[slot] >= 0) return stripe_map_base[slot];
    const Stripes& st = p->stripes;
    int ref = 0;
    while (ref < st.num && st.row0[ref + 1] == st.row0[ref]) ++ref;
    if (ref == st.num || p->num_maps + st.num > kMaxMaps) {
      map_error = true;
      fail(TPMLP_ERR_INVALID_ARG, ref == st.num ? "every stripe is empty" : "more than %d tensor maps in one launch",
           kMaxMaps);
      return 0;
    }
    const int base = p->num_maps;
    for (int j = 0; j < st.num; ++j) {
      const int jj = st.row0[j + 1] > st.row0[j] ? j : ref;
      const void* ptr = output ? st.out[jj] : st.in[jj];
      const int64_t cols = output ? st.out_ld : st.in_ld;
      const int idx = p->num_maps++;
      const int r = encode_map(&p->maps[idx], ptr, st.row0[jj + 1] - st.row0[jj], cols, cols, box_rows);
      if (r != 0) {
        map_error = true;
        fail(TPMLP_ERR_INVALID_ARG, "cuTensorMapEncodeTiled failed (%d) for stripe %d", r, j);
      }
      // keep the dedupe tables aligned with the map array (never matched: null pointer)
      map_ptr.push_back(nullptr);
      map_rows.push_back(0);
      map_cols.push_back(0);
      map_box.push_back(0);
      map_ld.push_back(0);
    }
    stripe_map_base[slot] = base;
    return base;
  }

  int map(const void* ptr, int64_t rows, int64_t cols, int box_rows, int64_t ld = -1) {
    if (!tc) return -1;
    if (ld < 0) ld = cols;
    for (size_t i = 0; i < map_ptr.size(); ++i)
      if (map_ptr[i] == ptr && map_rows[i] == rows && map_cols[i] == cols && map_box[i] == box_rows &&
          map_ld[i] == ld)
        return static_cast<int>(i);
    if (p->num_maps >= kMaxMaps) {
      map_error = true;
      fail(TPMLP_ERR_INVALID_ARG, "more than %d tensor maps in one launch", kMaxMaps);
      return 0;
    }
    const int idx = p->num_maps++;
    const int r = encode_map(&p->maps[idx], ptr, rows, cols, ld, box_rows);
    if (r != 0) {
      map_error = true;
      fail(TPMLP_ERR_INVALID_ARG, "cuTensorMapEncodeTiled failed (%d) for %p [%lld x %lld]", r, ptr,
           static_cast<long long>(rows), static_cast<long long>(cols));
    }
    map_ptr.push_back(ptr);
    map_rows.push_back(rows);
    map_cols.push_back(cols);
    map_box.push_back(box_rows);
    map_ld.push_back(ld);
    return idx;
  }

  // Table overflow (too many problems, segments or groups for one launch):
  // sticky like map_error; the entries past the end go to a dummy slot that
  // is never launched.
  bool table_error = false;
  Prob dummy_prob{};
  Seg dummy_seg{};
  Group dummy_group{};
  bool table_full(int used, int cap, const char* what) {
    if (used < cap) return false;
    if (!table_error) fail(TPMLP_ERR_UNSUPPORTED, "more than %d %s in one launch", cap, what);
    table_error = true;
    return true;
  }
  Group& group_at(int g) { return g >= 0 && g < kMaxGroups ? p->groups[g] : dummy_group; }

  void begin_group(int64_t M, int band_m) {
    if (table_full(p->num_groups, kMaxGroups, "problem groups")) {
      cur_group = -1;
      return;
    }
    Group& G = p->groups[p->num_groups];
    cur_group = p->num_groups++;
    G.first_prob = p->num_probs;
    G.num_probs = 0;
    G.tiles_m = static_cast<int32_t>((M + tile_m - 1) / tile_m);
    G.tiles_per_row = 0;
    G.band_m = std::max(1, std::min(band_m, G.tiles_m));
    G.tile_start = p->total_tiles;
  }

  Prob& add_prob(int64_t M, int64_t N, int tile_n, int a_major, int b_major, int epi, int64_t ldo) {
    if (cur_group < 0 || table_full(p->num_probs, kMaxProbs, "GEMM problems")) {
      table_error = true;
      dummy_prob = Prob{};
      return dummy_prob;
    }
    Prob& P = p->probs[p->num_probs++];
    P.M = static_cast<int32_t>(M);
    P.N = static_cast<int32_t>(N);
    P.tile_n = tc ? tile_n : kSimtTile;
    P.tiles_n = static_cast<int32_t>((N + P.tile_n - 1) / P.tile_n);
    P.seg_begin = p->num_segs;
    P.seg_count = 0;
    P.a_major = a_major;
    P.b_major = b_major;
    P.epi = epi;
    P.out_map[0] = P.out_map[1] = P.out_map[2] = -1;
    P.out_striped = 0;
    P.ldo = ldo;
    Group& G = group_at(cur_group);
    G.num_probs++;
    G.tiles_per_row += P.tiles_n;
    return P;
  }

  void add_seg(Prob& P, const void* a, int64_t a_rows, int64_t a_cols, const void* b, int64_t b_rows,
               int64_t b_cols, const void* b2, int64_t K) {
    if (&P == &dummy_prob || table_full(p->num_segs, kMaxSegs, "K segments")) return;
    Seg& S = p->segs[p->num_segs++];
    S.a = a;
    S.b = b;
    S.b2 = b2;
    S.lda = a_cols;
    S.ldb = b_cols;
    const int a_box = P.a_major == MAJOR_K ? 128 : kTcBK;
    const int b_box = P.b_major == MAJOR_K ? 128 : kTcBK;
    S.a_striped = a == kStripedIn ? 1 : 0;
    S.b_striped = b == kStripedIn ? 1 : 0;
    if (S.a_striped) S.a = nullptr;
    if (S.b_striped) S.b = nullptr;
    S.a_map = S.a_striped ? stripe_maps(false, a_box) : map(a, a_rows, a_cols, a_box);
    S.b_map = S.b_striped ? stripe_maps(false, b_box) : map(b, b_rows, b_cols, b_box);
    S.b2_map = b2 ? map(b2, b_rows, b_cols, b_box) : -1;
    S.K = static_cast<int32_t>(K);
    P.seg_count++;
  }

  void end_group() {
    if (cur_group < 0) return;
    Group& G = p->groups[cur_group];
    p->total_tiles += G.tiles_m * G.tiles_per_row;
  }
};

GemmParams* scratch_params() {
  thread_local GemmParams* params = nullptr;
  if (!params) params = new (std::align_val_t(64)) GemmParams;
  return params;
}

int band_for(int sms) {
  // The pairs running at the same time cover about a square block of tiles.
  const int pairs = sms / 2;
  int b = 1;
  while ((b + 1) * (b + 1) <= pairs) ++b;
  return b;
}

// Band height of a weight-gradient group (K = T): the whole M (d, or a
// shard's width) when it is at most 16 tiles, so that every wave shares the
// same A panels and the backward K walk of odd waves finds them in L2;
// measured on GB300: C5's f-sum launch (dW1, 12 M-tiles) 1326 -> 1314 us,
// C4's (16 M-tiles) 1680 -> 1672 us (bands of 12 there: 1693 us).
int band_wgrad(int sms, int64_t M) {
  const int64_t tiles = (M + kTileM - 1) / kTileM;
  return tiles <= 16 ? static_cast<int>(tiles) : band_for(sms);
}

// Band height of a short-K group (K = d: the column GEMM, dgrad, the QKV
// projection, dO): taller bands read each B panel fewer times (once per
// band), as long as the band's A panels (256 rows x K each) stay in L2 while
// the band sweeps N: about 24 MB of them, between the square band and 32.
// Measured on GB300: C5's column launch (K = 3072) reads 724 MB from DRAM
// with bands of 8, 477 MB with 16, 538 MB with 24, 945 MB with 32.
int band_short(int sms, int64_t K) {
  const int64_t panel = int64_t{kTileM} * K * 2;  // a pair's 256 rows of A, bf16
  const int64_t fit = (int64_t{24} << 20) / std::max<int64_t>(panel, 1);
  return std::max(band_for(sms), static_cast<int>(std::min<int64_t>(32, fit)));
}

// Tile -> problem and its first output row and column, as the kernel's
// decode_tile maps it.
int tile_prob(const GemmParams& p, int tile, int* m0 = nullptr, int* n0 = nullptr) {
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
  if (m0) *m0 = mt * p.tile_m;
  if (n0) *n0 = n_lin * p.probs[pi].tile_n;
  return pi;
}

std::atomic<uint32_t> g_sk_epoch{0};  // tags of the stream-K launches' ticket counts

// Range bookkeeping shared by both ways of cutting (see StreamK): from the
// ranges' starts, the head / tail split information of every range, and the
// tiles that more than one range covers (reported by tpmlp_last_split_tiles).
void finish_ranges(GemmParams& p, int pairs, const std::vector<int32_t>& kb, std::vector<int>* split_tiles) {
  StreamK& sk = p.sk;
  const int n = p.total_tiles;
  auto empty = [&](int q) { return sk.start_tile[q] == sk.start_tile[q + 1] && sk.start_kb[q] == sk.start_kb[q + 1]; };
  // covering ranges of each tile of the split region: first and count
  std::vector<int> first(n, -1), count(n, 0);
  for (int q = 0; q < pairs; ++q) {
    if (empty(q)) continue;
    int t = sk.start_tile[q];
    const int end_t = sk.start_tile[q + 1], end_kb = sk.start_kb[q + 1];
    // tiles touched: start_tile .. (end_kb > 0 ? end_t : end_t - 1)
    const int last = end_kb > 0 ? end_t : end_t - 1;
    for (; t <= last && t < n; ++t) {
      if (first[t] < 0) first[t] = q;
      ++count[t];
    }
  }
  for (int q = 0; q < pairs; ++q) {
    sk.head_q0[q] = sk.tail_q0[q] = static_cast<int16_t>(q);
    sk.head_n[q] = sk.tail_n[q] = 1;
    if (empty(q)) continue;
    const int th = sk.start_tile[q];
    const int tt = sk.start_kb[q + 1] > 0 ? sk.start_tile[q + 1] : sk.start_tile[q + 1] - 1;
    if (th < n) {
      sk.head_q0[q] = static_cast<int16_t>(first[th]);
      sk.head_n[q] = static_cast<int16_t>(count[th]);
    }
    if (tt >= 0 && tt < n) {
      sk.tail_q0[q] = static_cast<int16_t>(first[tt]);
      sk.tail_n[q] = static_cast<int16_t>(count[tt]);
    }
  }
  if (split_tiles) {
    split_tiles->clear();
    for (int t = sk.dp_tiles; t < n; ++t)
      if (count[t] > 1) split_tiles->push_back(t);
  }
  (void)kb;
}

// Estimated cost of a tile in K blocks: its main loop, or its epilogue when
// that is longer (about 14 K blocks for an activation epilogue of a 256 x 256
// tile, 4 for a plain store; measured on GB300 on the short-K launches of the
// GPT-2-small shape: a column tile every 9 us, a K block every 0.67 us).
int64_t tile_cost(const Prob& P, int kb) {
  const int64_t epi = P.epi == EPI_STORE ? 4 : 14;
  return std::max<int64_t>(kb, epi);
}

// Estimated cost (tile_cost) of every tile of a launch.
std::vector<int64_t> tile_costs(const GemmParams& p) {
  std::vector<int64_t> cost(p.total_tiles);
  for (int t = 0; t < p.total_tiles; ++t) {
    const Prob& P = p.probs[tile_prob(p, t)];
    cost[t] = tile_cost(P, P.kblocks);
  }
  return cost;
}

// Each pair's load (tile_cost) under the deal (long_end, r, s0) of tiles
// [0, dp_end), walked with the kernel's own deal_next; returns the largest.
int64_t deal_loads(int pairs, int long_end, int r, int s0, int dp_end, const std::vector<int64_t>& cost,
                   std::vector<int64_t>* loads = nullptr) {
  int64_t worst = 0;
  if (loads) loads->assign(pairs, 0);
  for (int q = 0; q < pairs; ++q) {
    Deal d;
    deal_init(d, q);
    int64_t load = 0;
    for (int t = deal_next(d, long_end, r, s0, q, pairs, dp_end); t >= 0;
         t = deal_next(d, long_end, r, s0, q, pairs, dp_end))
      load += cost[t];
    if (loads) (*loads)[q] = load;
    worst = std::max(worst, load);
  }
  return worst;
}

// The deal of the data-parallel tiles [0, dp_end) (see Deal) for a launch
// whose first long_end tiles are long-K weight-gradient tiles.  The plain
// round robin leaves pairs 0 .. r - 1 (r = long_end mod P) one long tile
// ahead; a head of s0 short tiles dealt to the other pairs first evens that
// out.  s0 runs over whole rounds of those pairs, up to the ratio of the tile
// costs, and the one with the smallest largest pair load is taken if it saves
// at least kMinDealSaving K blocks and 1 % of the round robin's (else s0 = 0:
// the round robin).  Any s0 gives the same results: every tile is computed
// once, by one pair, with the same K order.
struct DealChoice {
  int long_end = 0, r = 0, s0 = 0;
  int64_t makespan = 0;  // the largest pair load
};
DealChoice choose_deal(int pairs, int long_end, int dp_end, const std::vector<int64_t>& cost) {
  DealChoice c;
  c.makespan = deal_loads(pairs, 0, 0, 0, dp_end, cost);  // round robin
  if (long_end <= 0 || long_end >= dp_end || pairs < 2 || dp_end <= pairs) return c;
  const int r = long_end % pairs;
  if (r == 0) return c;  // every pair drew the same number of long tiles
  int64_t long_max = 0, short_min = INT64_MAX;
  for (int t = 0; t < dp_end; ++t) {
    if (t < long_end) long_max = std::max(long_max, cost[t]);
    else short_min = std::min(short_min, cost[t]);
  }
  constexpr int64_t kMinDealSaving = 4;
  const int64_t rr = c.makespan;
  int64_t best = rr;
  int best_s0 = 0;
  const int rounds = static_cast<int>(long_max / std::max<int64_t>(short_min, 1)) + 1;
  for (int k = 1; k <= rounds && k * (pairs - r) <= dp_end - long_end; ++k) {
    const int64_t m = deal_loads(pairs, long_end, r, k * (pairs - r), dp_end, cost);
    if (m < best) {
      best = m;
      best_s0 = k * (pairs - r);
    }
  }
  if (rr - best < std::max<int64_t>(kMinDealSaving, rr / 100)) return c;
  c.long_end = long_end;
  c.r = r;
  c.s0 = best_s0;
  c.makespan = best;
  return c;
}

void set_deal(GemmParams& p, const DealChoice& c) {
  p.deal_long = c.long_end;
  p.deal_r = c.r;
  p.deal_s0 = c.s0;
}

void plan_deal(GemmParams& p, int pairs, int long_end) {
  set_deal(p, DealChoice{});
  if (long_end <= 0 || long_end >= p.total_tiles || pairs < 2 || p.total_tiles <= pairs) return;
  set_deal(p, choose_deal(pairs, long_end, p.total_tiles, tile_costs(p)));
}

// The water level of pair loads `load` after adding L K blocks where the
// loads are lowest: sum over pairs of max(0, lambda - load) = L (integers).
int64_t water_level(const std::vector<int64_t>& load, int64_t L) {
  std::vector<int64_t> sorted(load);
  std::sort(sorted.begin(), sorted.end());
  const int pairs = static_cast<int>(sorted.size());
  int64_t rest = L;
  for (int i = 0; i < pairs; ++i) {
    const int64_t cnt = i + 1;  // pairs at or below this level
    if (i + 1 == pairs || rest <= (sorted[i + 1] - sorted[i]) * cnt) return sorted[i] + rest / cnt;
    rest -= (sorted[i + 1] - sorted[i]) * cnt;
  }
  return sorted.empty() ? 0 : sorted.back();
}

// Cut the K blocks of tiles [dp_tiles, n), concatenated in tile order, into
// one range per pair that fills the pair up to the common water level over
// its data-parallel load (range r belongs to pair pairs - 1 - r).  False if
// there is nothing to cut.
bool water_fill(StreamK& sk, int pairs, int dp_tiles, int n, const std::vector<int32_t>& kb,
                const std::vector<int64_t>& load) {
  int64_t L = 0;
  for (int t = dp_tiles; t < n; ++t) L += kb[t];
  if (L == 0) return false;
  const int64_t lambda = water_level(load, L);
  std::vector<int64_t> size(pairs, 0);
  int64_t given = 0;
  for (int q = 0; q < pairs; ++q) {
    size[q] = std::max<int64_t>(0, lambda - load[q]);
    given += size[q];
  }
  for (int q = 0; given < L; q = (q + 1) % pairs)  // the remainder, one K block at a time, to the lowest loads
    if (load[q] + size[q] <= lambda) {
      ++size[q];
      ++given;
    }
  int t = dp_tiles, k = 0;
  for (int r = 0; r < pairs; ++r) {
    sk.start_tile[r] = t;
    sk.start_kb[r] = k;
    int64_t want = size[pairs - 1 - r];
    while (want > 0 && t < n) {
      const int64_t take = std::min<int64_t>(want, kb[t] - k);
      want -= take;
      k += static_cast<int>(take);
      if (k == kb[t]) {
        ++t;
        k = 0;
      }
    }
  }
  sk.start_tile[pairs] = n;
  sk.start_kb[pairs] = 0;
  sk.dp_tiles = dp_tiles;
  return true;
}

// Cut the stream-K schedule of a tensor-core launch (see StreamK).  Two ways:
//
// Last wave (modes AUTO and ALWAYS, long_from < 0).  Every full wave of tiles
// stays data-parallel: the pairs of a wave start together and walk their
// tiles' K loops in step, so tiles that share a row block of A or a column
// block of B read it from L2 once.  (Cutting more than the last wave was
// measured slower on the large launches: parts that run out of step lose that
// sharing and become bound by HBM.)  Only the last, partial wave of R tiles
// is cut, and only when every pair carries the same data-parallel load and
// the R tiles have the same depth KB: each tile is then split into k parts of
// KB / k K blocks (rounded), on k ranges, with k <= pairs / R chosen to
// minimise KB / k + kPartCost (k - 1).  kPartCost, in K blocks, is what one
// more part costs the finisher: reading a 256 KB partial accumulator per pair
// back from L2 (about 2.8 us each on GB300, about five K blocks).  Auto mode
// keeps the plain round robin unless the cut saves at least max(16, 2 %) of
// a pair's K blocks: measured on GB300, smaller savings were lost to the
// launch's fixed costs and, under the power cap, to lower clocks in the
// following launches.  (Cutting the last wave of a mixed launch -- dealt full
// waves, the tail water-filled over the dealt loads -- was also measured
// slower, although the load model promised 1-2 %: C5's f-sum launch 1316 ->
// 1324 us, C4's 1671 -> 1749 us.)
//
// Balanced (long_from >= 0: the host placed the launch's long-K weight-
// gradient tiles last, from tile long_from on; mode BALANCE, or AUTO when
// those tiles' operands fit in L2).  The short tiles before long_from are
// dealt out round robin; the long tiles' K blocks are cut into ranges that
// fill every pair up to the same estimated load (water filling over the
// round-robin loads, tile_cost).  With the operands resident in L2, parts
// that run out of step cost no HBM traffic, and the pairs no longer wait on
// the few that drew a long tile.
void plan_stream_k(GemmParams& p, int pairs, int mode, int long_from, std::vector<int>* split_tiles) {
  StreamK& sk = p.sk;
  sk.on = 0;
  sk.dp_tiles = p.total_tiles;
  sk.pairs = 0;
  sk.epoch = 0;
  if (split_tiles) split_tiles->clear();
  const int n = p.total_tiles;
  if (mode == TPMLP_STREAM_K_OFF || pairs < 2 || pairs > kMaxSkPairs || n <= 0) return;
  std::vector<int32_t> kb(n, p.probs[0].kblocks);
  bool same_depth = true;
  for (int i = 1; i < p.num_probs; ++i) same_depth = same_depth && p.probs[i].kblocks == p.probs[0].kblocks;
  std::vector<int> prob_of(n, 0);
  if (!same_depth || long_from >= 0 || mode == TPMLP_STREAM_K_BALANCE)
    for (int t = 0; t < n; ++t) {
      prob_of[t] = tile_prob(p, t);
      kb[t] = p.probs[prob_of[t]].kblocks;
    }

  if (long_from >= 0 || mode == TPMLP_STREAM_K_BALANCE) {
    const int dp_tiles = long_from >= 0 ? long_from : 0;
    std::vector<int64_t> load(pairs, 0);
    for (int t = 0; t < dp_tiles; ++t) load[t % pairs] += tile_cost(p.probs[prob_of[t]], kb[t]);
    if (!water_fill(sk, pairs, dp_tiles, n, kb, load)) return;
    sk.dp_tiles = dp_tiles;
  } else {
    const int dp_tiles = (n / pairs) * pairs;
    const int R = n - dp_tiles;
    if (R == 0) return;  // no partial wave
    // Auto mode needs tiles of one depth; that holds exactly when every
    // problem has the same K blocks, which spares the per-tile walk above.
    if (!same_depth && mode == TPMLP_STREAM_K_AUTO) return;
    std::vector<int64_t> dp(pairs, 0);
    for (int t = 0; t < dp_tiles; ++t) dp[t % pairs] += kb[t];
    const int64_t dp_lo = *std::min_element(dp.begin(), dp.end());
    const int64_t dp_hi = *std::max_element(dp.begin(), dp.end());
    int kb_lo = kb[dp_tiles], kb_hi = kb[dp_tiles];
    for (int t = dp_tiles; t < n; ++t) {
      kb_lo = std::min(kb_lo, kb[t]);
      kb_hi = std::max(kb_hi, kb[t]);
    }
    const bool uniform = dp_lo == dp_hi && kb_lo == kb_hi;
    if (!uniform && mode == TPMLP_STREAM_K_AUTO) return;
    constexpr int64_t kPartCost = 5;
    constexpr int64_t kMinSaving = 16;  // K blocks (about 9 us): below that, launch and power effects dominate
    const int k_max = std::max(1, pairs / R);
    int kparts = 1;
    int64_t best = kb_hi;
    for (int c = 2; c <= k_max; ++c) {
      const int64_t m = (kb_hi + c - 1) / c + kPartCost * (c - 1);
      if (m < best) {
        best = m;
        kparts = c;
      }
    }
    if (mode == TPMLP_STREAM_K_ALWAYS) kparts = std::min(k_max, kb_hi);  // as many parts as fit: a stress test
    if (mode == TPMLP_STREAM_K_AUTO) {
      const int64_t rr = dp_hi + kb_hi, cut = dp_hi + best;
      if (kparts == 1 || rr - cut < std::max<int64_t>(kMinSaving, rr / 50)) return;
    }
    if (kparts < 2) return;
    // Range r = j k + i (held by pair pairs - 1 - r) is part i of tail tile j;
    // ranges from R k on are empty.
    for (int r = 0; r <= pairs; ++r) {
      const int j = r / kparts, i = r % kparts;
      if (j >= R) {
        sk.start_tile[r] = n;
        sk.start_kb[r] = 0;
      } else {
        sk.start_tile[r] = dp_tiles + j;
        sk.start_kb[r] = static_cast<int32_t>(static_cast<int64_t>(kb[dp_tiles + j]) * i / kparts);
      }
    }
    sk.dp_tiles = dp_tiles;
  }
  finish_ranges(p, pairs, kb, split_tiles);
  uint32_t e = ++g_sk_epoch & 0xFFFFFFu;  // 24-bit tag of this launch's ticket counts
  if (e == 0) e = ++g_sk_epoch & 0xFFFFFFu;
  sk.on = 1;
  sk.pairs = pairs;
  sk.epoch = e;
}

// sk_workspace: the workspace holds the stream-K flags and partial slots
// (tpmlp_workspace_size bytes); false for the library's status-only scratch.
tpmlp_status launch(Builder& B, int tag, const DeviceInfo& di, const tpmlp_plan* plan, void* workspace,
                    cudaStream_t stream, bool sk_workspace = true) {
  GemmParams& p = *B.p;
  if (p.total_tiles == 0) return TPMLP_OK;
  if (B.tc) {
    for (int i = 0; i < p.num_probs; ++i) {
      Prob& P = p.probs[i];
      P.kblocks = 0;
      for (int sg = P.seg_begin; sg < P.seg_begin + P.seg_count; ++sg) P.kblocks += (p.segs[sg].K + kTcBK - 1) / kTcBK;
      // Alternate the K direction by wave where a wave's operands outgrow L2
      // (measured on GB300, C5: the row launch reads 1.49 -> 1.22 GB from DRAM,
      // the f-sum launch 2.85 -> 2.51 GB; short-K launches gain nothing).
      P.k_rev = P.kblocks >= kRevKBlocks ? 1 : 0;
    }
  }
  const int epi_warps = B.tc ? tc_epi_warps_for(p, tag) : 0;
  const int out_box = epi_warps == 16 ? kOutputMap16 : kOutputMap32;
  for (int i = 0; i < p.num_probs; ++i) {  // token-striped output (sequence-parallel layout)
    Prob& P = p.probs[i];
    if (P.out0 == kStripedOut) {
      P.out0 = nullptr;
      P.out_striped = 1;
      P.out_map[0] = B.stripe_maps(true, out_box);
    }
  }
  if (B.tc) {  // the tensor-core epilogue writes every output with TMA stores
    for (int i = 0; i < p.num_probs; ++i) {
      Prob& P = p.probs[i];
      void* outs[3] = {P.out0, P.out1, P.out2};
      for (int k = 0; k < 3; ++k)
        if (outs[k]) P.out_map[k] = B.map(outs[k], P.M, P.N, out_box, P.ldo);
    }
  }
  if (B.table_error) return TPMLP_ERR_UNSUPPORTED;  // message set by Builder::table_full
  if (B.map_error) return TPMLP_ERR_INVALID_ARG;  // message set by Builder::map
  p.status = static_cast<int32_t*>(workspace);
  p.timeout_ns = plan->timeout_ns;
  p.stall_injection = plan->stall_injection;
  p.sk.on = 0;
  p.sk.dp_tiles = p.total_tiles;
  std::vector<int> split_tiles;
  if (B.tc && sk_workspace) plan_stream_k(p, tc_gemm_max_pairs(tag), plan->stream_k, B.long_from, &split_tiles);
  if (B.tc && !p.sk.on) plan_deal(p, tc_gemm_grid_pairs(p, tag, di.sms / 2), B.long_end);
  std::vector<int64_t>& split = g_last_split[tag];
  split.clear();
  for (int t : split_tiles) {
    int m0 = 0, n0 = 0;
    const int pi = tile_prob(p, t, &m0, &n0);
    split.insert(split.end(), {pi, m0, n0, static_cast<int64_t>(reinterpret_cast<uintptr_t>(p.probs[pi].out0))});
  }
  cudaError_t e;
  if (B.tc) {
    e = launch_tc_gemm(p, tag, epi_warps, di.sms / 2, stream);
  } else {
    e = launch_simt_gemm(p, stream);
  }
  if (e != cudaSuccess) return cuda_fail(e);
  ++g_last_launches;
  return TPMLP_OK;
}

// ------------------------------------------------------------------ checks
#define TPMLP_TRY(expr)                   \
  do {                                    \
    tpmlp_status st_ = (expr);            \
    if (st_ != TPMLP_OK) return st_;      \
  } while (0)

tpmlp_status check_ptr(const char* name, const void* q, bool may_be_null) {
  if (!q) return may_be_null ? TPMLP_OK : fail(TPMLP_ERR_INVALID_ARG, "%s is NULL", name);
  if (!aligned16(q)) return fail(TPMLP_ERR_ALIGNMENT, "%s (%p) is not 16-byte aligned", name, q);
  return TPMLP_OK;
}

tpmlp_status check_array(const char* name, const void* const* arr, int n, bool may_be_null_entries) {
  if (!arr) return fail(TPMLP_ERR_INVALID_ARG, "pointer array %s is NULL", name);
  for (int i = 0; i < n; ++i) {
    if (!arr[i]) {
      if (may_be_null_entries) continue;
      return fail(TPMLP_ERR_INVALID_ARG, "%s[%d] is NULL", name, i);
    }
    if (!aligned16(arr[i])) return fail(TPMLP_ERR_ALIGNMENT, "%s[%d] (%p) is not 16-byte aligned", name, i, arr[i]);
  }
  return TPMLP_OK;
}

bool swiglu(const tpmlp_plan* pl) { return pl->act == TPMLP_ACT_SWIGLU; }
int nsaved(const tpmlp_plan* pl) { return swiglu(pl) ? 2 * pl->t : pl->t; }

tpmlp_status check_kind(const tpmlp_plan* pl, PlanKind kind) {
  if (pl->kind == kind) return TPMLP_OK;
  return fail(TPMLP_ERR_INVALID_ARG, kind == PLAN_MLP ? "an attention plan was passed to an MLP entry point"
                                                      : "an MLP plan was passed to an attention entry point");
}

tpmlp_status common_checks(const tpmlp_plan* pl, void* workspace, DeviceInfo* di, PlanKind kind = PLAN_MLP) {
  g_last_error[0] = 0;
  if (!pl) return fail(TPMLP_ERR_INVALID_ARG, "plan is NULL");
  TPMLP_TRY(check_kind(pl, kind));
  TPMLP_TRY(check_ptr("workspace", workspace, false));
  return device_info(di);
}

// ------------------------------------------------------------------ bias gradients
// dst_j[c] = sum over the T rows of src_j[r][c], one launch for all jobs.
struct ColsumBuilder {
  ColsumParams p{};
  bool bf16;
  explicit ColsumBuilder(bool is_bf16) : bf16(is_bf16) {}
  void set_stripes(const tpmlp_plan* pl, const void* const* src) {
    p.num_stripes = static_cast<int32_t>(pl->stripe_rows.size());
    p.stripe_row0[0] = 0;
    for (int j = 0; j < p.num_stripes; ++j) {
      p.stripe_row0[j + 1] = p.stripe_row0[j] + pl->stripe_rows[j];
      p.stripe_src[j] = src[j];
    }
  }
  void add(const void* src, void* dst, int64_t rows, int64_t cols) {
    ColsumJob& J = p.jobs[p.num_jobs++];
    J.src = src;
    J.dst = dst;
    J.rows = rows;
    J.cols = static_cast<int32_t>(cols);
  }
  // Cut every job into strips of the width the launch uses.
  ColsumShape finish(int sms) {
    const ColsumShape shape = colsum_shape(p.jobs, p.num_jobs, bf16, sms);
    const int strip_cols = colsum_strip_cols(bf16, shape.lane_threads);
    p.total_strips = 0;
    for (int j = 0; j < p.num_jobs; ++j) {
      p.jobs[j].strip_begin = p.total_strips;
      p.total_strips += (p.jobs[j].cols + strip_cols - 1) / strip_cols;
    }
    return shape;
  }
};

tpmlp_status launch_colsums(ColsumBuilder& C, const DeviceInfo& di, cudaStream_t st) {
  if (C.p.num_jobs == 0) return TPMLP_OK;
  const ColsumShape shape = C.finish(di.sms);
  cudaError_t e = launch_colsum(C.p, C.bf16, shape, st);
  if (e != cudaSuccess) return cuda_fail(e);
  ++g_last_launches;
  return TPMLP_OK;
}

// ------------------------------------------------------------------ phases
// Whether a launch places its long-K weight-gradient tiles last and lets the
// stream-K planner spread them evenly over the pairs (plan_stream_k,
// balanced): in TPMLP_STREAM_K_BALANCE mode.  Auto mode does not: measured on
// GB300 on the GPT-2-small shape (whose weight-gradient operands stay in L2),
// the parts' partial stores (4-7 us) and the last part's read-back of the
// others (8-11 us) cost more than the balance gained (f-sum launch 65 -> 70
// us; dgrad 98 -> 92 us).  long_bytes (those tiles' operands and outputs) is
// kept for that decision.
bool balance_long(const tpmlp_plan* pl, int64_t long_bytes) {
  (void)long_bytes;
  return pl->dtype == TPMLP_BF16 && pl->stream_k == TPMLP_STREAM_K_BALANCE;
}

tpmlp_status fwd_column(const tpmlp_plan* pl, const DeviceInfo& di, const void* X, const void* const* W1,
                        const void* const* W3, const void* const* b1, const void* const* b3, void* const* saved,
                        void* const* H, void* ws, cudaStream_t st, const void* const* X_stripes = nullptr) {
  if (pl->T == 0) return TPMLP_OK;
  const bool tc = pl->dtype == TPMLP_BF16;
  const bool sw = swiglu(pl);
  Builder B(scratch_params(), tc);
  if (X_stripes) {  // all-gather of the X stripes: every shard reads all of them
    B.set_stripes(pl, X_stripes, pl->d, nullptr, 0);
    X = kStripedIn;
  }
  B.begin_group(pl->T, band_short(di.sms, pl->d));
  for (int i = 0; i < pl->t; ++i) {
    const int64_t di_ = pl->d_i[i];
    Prob& P = B.add_prob(pl->T, di_, sw ? 128 : 256, MAJOR_K, MAJOR_MN, sw ? EPI_SWIGLU_FWD : EPI_GELU_FWD, di_);
    P.out0 = saved[i];
    P.out1 = sw ? saved[pl->t + i] : H[i];
    P.out2 = sw ? H[i] : nullptr;
    P.aux0 = b1 ? b1[i] : nullptr;
    P.aux1 = (sw && b3) ? b3[i] : nullptr;
    B.add_seg(P, X, pl->T, pl->d, W1[i], pl->d, di_, sw ? W3[i] : nullptr, pl->d);
  }
  B.end_group();
  return launch(B, TAG_FWD_COLUMN, di, pl, ws, st);
}

tpmlp_status fwd_row(const tpmlp_plan* pl, const DeviceInfo& di, const void* const* W2, const void* b2, void* Y,
                     void* const* H, void* ws, cudaStream_t st, void* const* Y_stripes = nullptr,
                     bool sk_workspace = true) {
  if (pl->T == 0) return TPMLP_OK;
  Builder B(scratch_params(), pl->dtype == TPMLP_BF16);
  if (Y_stripes) {  // reduce-scatter: the summed rows of stripe j go to Y_j
    B.set_stripes(pl, nullptr, 0, Y_stripes, pl->d);
    Y = kStripedOut;
  }
  B.begin_group(pl->T, band_for(di.sms));
  Prob& P = B.add_prob(pl->T, pl->d, 256, MAJOR_K, MAJOR_MN, EPI_STORE, pl->d);
  P.out0 = Y;
  P.aux0 = b2;  // added once, after the whole g-sum
  // g operator: every shard's H_i W2_i accumulates into the same tile.
  for (int i = 0; i < pl->t; ++i) B.add_seg(P, H[i], pl->T, pl->d_i[i], W2[i], pl->d_i[i], pl->d, nullptr, pl->d_i[i]);
  B.end_group();
  return launch(B, TAG_FWD_ROW, di, pl, ws, st, sk_workspace);
}

// With recompute, H is an output: the dgrad epilogue writes H_i = act(saved_i)
// and dW2 moves to the f-sum launch (bwd_fsum's dW2 problems).
tpmlp_status bwd_dgrad(const tpmlp_plan* pl, const DeviceInfo& di, const void* const* W2,
                       const void* const* saved, const void* const* H, const void* dY, void* const* dact,
                       void* const* dW2, void* db2, void* ws, cudaStream_t st, bool recompute = false,
                       const void* const* dY_stripes = nullptr) {
  const bool sw = swiglu(pl);
  if (pl->T == 0) {
    const size_t es = pl->dtype == TPMLP_BF16 ? 2 : 4;
    for (int i = 0; i < pl->t; ++i) {
      cudaError_t e = cudaMemsetAsync(dW2[i], 0, static_cast<size_t>(pl->d_i[i] * pl->d) * es, st);
      if (e != cudaSuccess) return cuda_fail(e);
    }
    if (db2) {
      cudaError_t e = cudaMemsetAsync(db2, 0, static_cast<size_t>(pl->d) * es, st);
      if (e != cudaSuccess) return cuda_fail(e);
    }
    return TPMLP_OK;
  }
  Builder B(scratch_params(), pl->dtype == TPMLP_BF16);
  const void* dY_dense = dY;
  if (dY_stripes) {  // all-gather of the dY stripes (backward of the reduce-scatter)
    B.set_stripes(pl, dY_stripes, pl->d, nullptr, 0);
    dY = kStripedIn;
  }
  // dW2_i = H_i^T dY (K = T): the long tiles go first, or last when the
  // stream-K planner spreads them over the pairs
  const bool balanced = !recompute && balance_long(pl, 2 * (pl->T * pl->dff + pl->T * pl->d + pl->dff * pl->d));
  auto add_dw2 = [&] {
    for (int i = 0; i < pl->t && !recompute; ++i) {
      const int64_t di_ = pl->d_i[i];
      B.begin_group(di_, band_wgrad(di.sms, di_));
      Prob& P = B.add_prob(di_, pl->d, 256, MAJOR_MN, MAJOR_MN, EPI_STORE, pl->d);
      P.out0 = dW2[i];
      B.add_seg(P, H[i], pl->T, di_, dY, pl->T, pl->d, nullptr, pl->T);
      B.end_group();
    }
  };
  if (!balanced) {
    add_dw2();
    B.long_end = B.p->total_tiles;
  }
  // dH_i = dY W2_i^T with act' fused (g backward = identity: every shard reads dY)
  B.begin_group(pl->T, band_short(di.sms, pl->d));
  for (int i = 0; i < pl->t; ++i) {
    const int64_t di_ = pl->d_i[i];
    Prob& P = B.add_prob(pl->T, di_, 256, MAJOR_K, MAJOR_K, sw ? EPI_SWIGLU_BWD : EPI_GELU_BWD, di_);
    P.aux0 = saved[i];
    P.aux1 = sw ? saved[pl->t + i] : nullptr;
    P.out0 = dact[i];
    P.out1 = sw ? dact[pl->t + i] : (recompute ? const_cast<void*>(H[i]) : nullptr);
    P.out2 = (sw && recompute) ? const_cast<void*>(H[i]) : nullptr;
    B.add_seg(P, dY, pl->T, pl->d, W2[i], di_, pl->d, nullptr, pl->d);
  }
  B.end_group();
  if (balanced) {
    B.long_from = B.p->total_tiles;
    add_dw2();
  }
  TPMLP_TRY(launch(B, TAG_BWD_DGRAD, di, pl, ws, st));
  if (db2) {  // g backward is the identity: b2's gradient is that of Y
    ColsumBuilder C(pl->dtype == TPMLP_BF16);
    if (dY_stripes) C.set_stripes(pl, dY_stripes);
    C.add(dY_stripes ? nullptr : dY_dense, db2, pl->T, pl->d);
    TPMLP_TRY(launch_colsums(C, di, st));
  }
  return TPMLP_OK;
}

tpmlp_status bwd_fsum(const tpmlp_plan* pl, const DeviceInfo& di, const void* X, const void* const* W1,
                      const void* const* W3, const void* const* dact, void* dX, void* const* dW1,
                      void* const* dW3, void* const* db1, void* const* db3, void* ws, cudaStream_t st,
                      const void* const* H_for_dW2 = nullptr, const void* dY = nullptr, void* const* dW2 = nullptr,
                      const void* const* X_stripes = nullptr, void* const* dX_stripes = nullptr) {
  const bool sw = swiglu(pl);
  if (pl->T == 0) {
    const size_t es = pl->dtype == TPMLP_BF16 ? 2 : 4;
    for (int i = 0; i < pl->t; ++i) {
      const size_t n = static_cast<size_t>(pl->d * pl->d_i[i]) * es;
      const size_t nb = static_cast<size_t>(pl->d_i[i]) * es;
      cudaError_t e = cudaMemsetAsync(dW1[i], 0, n, st);
      if (e == cudaSuccess && sw) e = cudaMemsetAsync(dW3[i], 0, n, st);
      if (e == cudaSuccess && db1) e = cudaMemsetAsync(db1[i], 0, nb, st);
      if (e == cudaSuccess && sw && db3) e = cudaMemsetAsync(db3[i], 0, nb, st);
      if (e != cudaSuccess) return cuda_fail(e);
    }
    return TPMLP_OK;
  }
  const bool tc = pl->dtype == TPMLP_BF16;
  const int band = band_for(di.sms);
  // Recompute mode: dW2_i = H_i^T dY from the H the dgrad launch rewrote.  It
  // shares the f-sum launch unless that launch's tables would overflow (the
  // SwiGLU tensor maps, 10t + 3, for t > 12); it then runs as a launch of its
  // own just before.
  auto add_dw2 = [&](Builder& B) {
    for (int i = 0; i < pl->t; ++i) {
      const int64_t di_ = pl->d_i[i];
      B.begin_group(di_, band_wgrad(di.sms, di_));
      Prob& P = B.add_prob(di_, pl->d, 256, MAJOR_MN, MAJOR_MN, EPI_STORE, pl->d);
      P.out0 = dW2[i];
      B.add_seg(P, H_for_dW2[i], pl->T, di_, dY, pl->T, pl->d, nullptr, pl->T);
      B.end_group();
    }
  };
  const int t = pl->t;
  const bool dw2_fits = (!tc || (sw ? 10 : 6) * t + 3 <= kMaxMaps) && (sw ? 3 : 2) * t + 1 <= kMaxProbs &&
                        (sw ? 5 : 3) * t <= kMaxSegs && t + 2 <= kMaxGroups;
  const int64_t dw2_bytes = 2 * (pl->T * pl->dff + pl->T * pl->d + pl->dff * pl->d);
  if (H_for_dW2 && !dw2_fits) {
    Builder B2(scratch_params(), tc);
    if (balance_long(pl, dw2_bytes)) B2.long_from = 0;
    add_dw2(B2);
    TPMLP_TRY(launch(B2, TAG_BWD_FSUM, di, pl, ws, st));
  }
  Builder B(scratch_params(), tc);
  if (X_stripes || dX_stripes) {  // X gathered from its stripes; dX reduce-scattered into stripes
    B.set_stripes(pl, X_stripes, pl->d, dX_stripes, pl->d);
    if (X_stripes) X = kStripedIn;
    if (dX_stripes) dX = kStripedOut;
  }
  // The weight gradients (K = T) go first, or last when the stream-K planner
  // spreads them over the pairs.
  const int64_t nact = sw ? 2 : 1;
  const bool with_dw2 = H_for_dW2 && dw2_fits;
  const bool balanced =
      balance_long(pl, 2 * (pl->T * pl->d + nact * (pl->T * pl->dff + pl->d * pl->dff)) + (with_dw2 ? dw2_bytes : 0));
  auto add_wgrads = [&] {
    if (with_dw2) add_dw2(B);
    // dW1_i = X^T dA_i (SwiGLU: X^T dG_i) and dW3_i = X^T dU_i
    B.begin_group(pl->d, band_wgrad(di.sms, pl->d));
    for (int i = 0; i < pl->t; ++i) {
      const int64_t di_ = pl->d_i[i];
      Prob& P = B.add_prob(pl->d, di_, 256, MAJOR_MN, MAJOR_MN, EPI_STORE, di_);
      P.out0 = dW1[i];
      B.add_seg(P, X, pl->T, pl->d, dact[i], pl->T, di_, nullptr, pl->T);
    }
    if (sw) {
      for (int i = 0; i < pl->t; ++i) {
        const int64_t di_ = pl->d_i[i];
        Prob& P = B.add_prob(pl->d, di_, 256, MAJOR_MN, MAJOR_MN, EPI_STORE, di_);
        P.out0 = dW3[i];
        B.add_seg(P, X, pl->T, pl->d, dact[pl->t + i], pl->T, di_, nullptr, pl->T);
      }
    }
    B.end_group();
  };
  if (!balanced) {
    add_wgrads();
    B.long_end = B.p->total_tiles;
  }
  // dX = sum_i dA_i W1_i^T (+ dU_i W3_i^T): the f operator's backward sum.
  B.begin_group(pl->T, band);
  Prob& P = B.add_prob(pl->T, pl->d, 256, MAJOR_K, MAJOR_K, EPI_STORE, pl->d);
  P.out0 = dX;
  for (int i = 0; i < pl->t; ++i)
    B.add_seg(P, dact[i], pl->T, pl->d_i[i], W1[i], pl->d, pl->d_i[i], nullptr, pl->d_i[i]);
  if (sw)
    for (int i = 0; i < pl->t; ++i)
      B.add_seg(P, dact[pl->t + i], pl->T, pl->d_i[i], W3[i], pl->d, pl->d_i[i], nullptr, pl->d_i[i]);
  B.end_group();
  if (balanced) {
    B.long_from = B.p->total_tiles;
    add_wgrads();
  }
  TPMLP_TRY(launch(B, TAG_BWD_FSUM, di, pl, ws, st));
  if (db1 || (sw && db3)) {
    ColsumBuilder C(pl->dtype == TPMLP_BF16);
    for (int i = 0; i < pl->t; ++i) {
      if (db1) C.add(dact[i], db1[i], pl->T, pl->d_i[i]);
      if (sw && db3) C.add(dact[pl->t + i], db3[i], pl->T, pl->d_i[i]);
    }
    TPMLP_TRY(launch_colsums(C, di, st));
  }
  return TPMLP_OK;
}

// ------------------------------------------------------------------ attention projections
// Shard i: W_QKV,i [d x n_i] = [WQ_i | WK_i | WV_i], n_i = dq_i + 2 dkv_i;
// O_i [T x dq_i]; WO_i [dq_i x d].  Every epilogue is a plain store.
tpmlp_status attn_qkv_fwd(const tpmlp_plan* pl, const DeviceInfo& di, const void* X, const void* const* Wqkv,
                          void* const* QKV, void* ws, cudaStream_t st) {
  if (pl->T == 0) return TPMLP_OK;
  Builder B(scratch_params(), pl->dtype == TPMLP_BF16);
  B.begin_group(pl->T, band_short(di.sms, pl->d));
  for (int i = 0; i < pl->t; ++i) {  // f forward is the identity: every shard reads X
    const int64_t n = pl->d_i[i];
    Prob& P = B.add_prob(pl->T, n, 256, MAJOR_K, MAJOR_MN, EPI_STORE, n);
    P.out0 = QKV[i];
    B.add_seg(P, X, pl->T, pl->d, Wqkv[i], pl->d, n, nullptr, pl->d);
  }
  B.end_group();
  return launch(B, TAG_ATTN_QKV, di, pl, ws, st);
}

tpmlp_status attn_out_fwd(const tpmlp_plan* pl, const DeviceInfo& di, const void* const* WO, const void* const* O,
                          void* Z, void* ws, cudaStream_t st) {
  if (pl->T == 0) return TPMLP_OK;
  Builder B(scratch_params(), pl->dtype == TPMLP_BF16);
  B.begin_group(pl->T, band_for(di.sms));
  Prob& P = B.add_prob(pl->T, pl->d, 256, MAJOR_K, MAJOR_MN, EPI_STORE, pl->d);
  P.out0 = Z;
  // g operator: every shard's O_i WO_i accumulates into the same tile.
  for (int i = 0; i < pl->t; ++i)
    B.add_seg(P, O[i], pl->T, pl->dq_i[i], WO[i], pl->dq_i[i], pl->d, nullptr, pl->dq_i[i]);
  B.end_group();
  return launch(B, TAG_ATTN_OUT, di, pl, ws, st);
}

tpmlp_status attn_out_bwd(const tpmlp_plan* pl, const DeviceInfo& di, const void* const* WO, const void* const* O,
                          const void* dZ, void* const* dO, void* const* dWO, void* ws, cudaStream_t st) {
  if (pl->T == 0) {
    const size_t es = pl->dtype == TPMLP_BF16 ? 2 : 4;
    for (int i = 0; i < pl->t; ++i) {
      cudaError_t e = cudaMemsetAsync(dWO[i], 0, static_cast<size_t>(pl->dq_i[i] * pl->d) * es, st);
      if (e != cudaSuccess) return cuda_fail(e);
    }
    return TPMLP_OK;
  }
  Builder B(scratch_params(), pl->dtype == TPMLP_BF16);
  int64_t dq = 0;
  for (int i = 0; i < pl->t; ++i) dq += pl->dq_i[i];
  // dWO_i = O_i^T dZ (K = T): the long tiles go first, or last when the
  // stream-K planner spreads them over the pairs
  const bool balanced = balance_long(pl, 2 * (pl->T * dq + pl->T * pl->d + dq * pl->d));
  auto add_dwo = [&] {
    for (int i = 0; i < pl->t; ++i) {
      const int64_t w = pl->dq_i[i];
      B.begin_group(w, band_wgrad(di.sms, w));
      Prob& P = B.add_prob(w, pl->d, 256, MAJOR_MN, MAJOR_MN, EPI_STORE, pl->d);
      P.out0 = dWO[i];
      B.add_seg(P, O[i], pl->T, w, dZ, pl->T, pl->d, nullptr, pl->T);
      B.end_group();
    }
  };
  if (!balanced) {
    add_dwo();
    B.long_end = B.p->total_tiles;
  }
  // dO_i = dZ WO_i^T (g backward is the identity: every shard reads dZ)
  B.begin_group(pl->T, band_short(di.sms, pl->d));
  for (int i = 0; i < pl->t; ++i) {
    const int64_t w = pl->dq_i[i];
    Prob& P = B.add_prob(pl->T, w, 256, MAJOR_K, MAJOR_K, EPI_STORE, w);
    P.out0 = dO[i];
    B.add_seg(P, dZ, pl->T, pl->d, WO[i], w, pl->d, nullptr, pl->d);
  }
  B.end_group();
  if (balanced) {
    B.long_from = B.p->total_tiles;
    add_dwo();
  }
  return launch(B, TAG_ATTN_OUT_BWD, di, pl, ws, st);
}

tpmlp_status attn_qkv_bwd(const tpmlp_plan* pl, const DeviceInfo& di, const void* X, const void* const* Wqkv,
                          const void* const* dQKV, void* dX, void* const* dWqkv, void* ws, cudaStream_t st) {
  if (pl->T == 0) {
    const size_t es = pl->dtype == TPMLP_BF16 ? 2 : 4;
    for (int i = 0; i < pl->t; ++i) {
      cudaError_t e = cudaMemsetAsync(dWqkv[i], 0, static_cast<size_t>(pl->d * pl->d_i[i]) * es, st);
      if (e != cudaSuccess) return cuda_fail(e);
    }
    return TPMLP_OK;
  }
  Builder B(scratch_params(), pl->dtype == TPMLP_BF16);
  const int band = band_for(di.sms);
  // dW_QKV,i = X^T dQKV_i (K = T): first, or last when the stream-K planner
  // spreads them over the pairs
  const bool balanced = balance_long(pl, 2 * (pl->T * pl->d + pl->T * pl->dff + pl->d * pl->dff));
  auto add_dwqkv = [&] {
    B.begin_group(pl->d, band_wgrad(di.sms, pl->d));
    for (int i = 0; i < pl->t; ++i) {
      const int64_t n = pl->d_i[i];
      Prob& P = B.add_prob(pl->d, n, 256, MAJOR_MN, MAJOR_MN, EPI_STORE, n);
      P.out0 = dWqkv[i];
      B.add_seg(P, X, pl->T, pl->d, dQKV[i], pl->T, n, nullptr, pl->T);
    }
    B.end_group();
  };
  if (!balanced) {
    add_dwqkv();
    B.long_end = B.p->total_tiles;
  }
  // dX = sum_i dQKV_i W_QKV,i^T (= dQ_i WQ_i^T + dK_i WK_i^T + dV_i WV_i^T): the f-sum.
  B.begin_group(pl->T, band);
  Prob& P = B.add_prob(pl->T, pl->d, 256, MAJOR_K, MAJOR_K, EPI_STORE, pl->d);
  P.out0 = dX;
  for (int i = 0; i < pl->t; ++i) B.add_seg(P, dQKV[i], pl->T, pl->d_i[i], Wqkv[i], pl->d, pl->d_i[i], nullptr, pl->d_i[i]);
  B.end_group();
  if (balanced) {
    B.long_from = B.p->total_tiles;
    add_dwqkv();
  }
  return launch(B, TAG_ATTN_QKV_BWD, di, pl, ws, st);
}

}  // namespace

// ------------------------------------------------------------------ library-owned scratch
// Scratch of tpmlp_forward_row_noalloc: a file-scope device array instead of
// a caller workspace.  Every device that loads the library holds it until
// the process exits; all calls on a device share it.
constexpr size_t kStaticScratchBytes = 256;
static __device__ __align__(256) unsigned char g_static_scratch[kStaticScratchBytes];

// Device address of g_static_scratch on the current device, looked up once
// per device (the host-side name is only a stand-in for the symbol).
tpmlp_status static_scratch(int32_t** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e);
  if (dev < 0 || dev >= 64) return fail(TPMLP_ERR_UNSUPPORTED, "device ordinal %d out of range", dev);
  static std::mutex mu;
  static void* addr[64] = {};
  std::lock_guard<std::mutex> lk(mu);
  if (!addr[dev]) {
    void* ptr = nullptr;
    e = cudaGetSymbolAddress(&ptr, g_static_scratch);
    if (e != cudaSuccess) return cuda_fail(e);
    addr[dev] = ptr;
  }
  *out = static_cast<int32_t*>(addr[dev]);
  return TPMLP_OK;
}

// ====================================================================== C ABI
extern "C" {

tpmlp_status tpmlp_plan_create(const tpmlp_desc* desc, tpmlp_plan** out) {
  g_last_error[0] = 0;
  if (!out) return fail(TPMLP_ERR_INVALID_ARG, "out is NULL");
  *out = nullptr;
  if (!desc || !desc->d_i) return fail(TPMLP_ERR_INVALID_ARG, "desc or desc->d_i is NULL");
  if (desc->act != TPMLP_ACT_GELU && desc->act != TPMLP_ACT_SWIGLU)
    return fail(TPMLP_ERR_INVALID_ARG, "unknown act %d", static_cast<int>(desc->act));
  if (desc->dtype != TPMLP_BF16 && desc->dtype != TPMLP_FP32)
    return fail(TPMLP_ERR_INVALID_ARG, "unknown dtype %d", static_cast<int>(desc->dtype));
  if (desc->T < 0 || desc->d < 1 || desc->t < 1 || desc->t > TPMLP_MAX_SHARDS)
    return fail(TPMLP_ERR_SHAPE, "need T >= 0, d >= 1, 1 <= t <= %d (got T=%lld d=%lld t=%d)", TPMLP_MAX_SHARDS,
                static_cast<long long>(desc->T), static_cast<long long>(desc->d), desc->t);
  const int64_t mult = desc->dtype == TPMLP_BF16 ? 8 : 4;
  const int64_t kMax32 = (int64_t(1) << 31) - 1;
  int64_t dff = 0;
  for (int i = 0; i < desc->t; ++i) {
    if (desc->d_i[i] < 1) return fail(TPMLP_ERR_SHAPE, "d_i[%d] = %lld < 1", i, static_cast<long long>(desc->d_i[i]));
    dff += desc->d_i[i];
  }
  if (desc->d % mult)
    return fail(TPMLP_ERR_ALIGNMENT, "d = %lld is not a multiple of %lld", static_cast<long long>(desc->d),
                static_cast<long long>(mult));
  for (int i = 0; i < desc->t; ++i)
    if (desc->d_i[i] % mult)
      return fail(TPMLP_ERR_ALIGNMENT, "d_i[%d] = %lld is not a multiple of %lld", i,
                  static_cast<long long>(desc->d_i[i]), static_cast<long long>(mult));
  if (desc->T > kMax32 || desc->d > kMax32 || dff > kMax32)
    return fail(TPMLP_ERR_UNSUPPORTED, "T, d and d_ff must each be below 2^31");
  tpmlp_plan* pl = new (std::nothrow) tpmlp_plan;
  if (!pl) return TPMLP_ERR_INVALID_ARG;
  pl->kind = PLAN_MLP;
  pl->T = desc->T;
  pl->d = desc->d;
  pl->t = desc->t;
  pl->d_i.assign(desc->d_i, desc->d_i + desc->t);
  pl->o_i.resize(desc->t);
  int64_t o = 0;
  for (int i = 0; i < desc->t; ++i) {
    pl->o_i[i] = o;
    o += pl->d_i[i];
  }
  pl->dff = dff;
  pl->act = desc->act;
  pl->dtype = desc->dtype;
  pl->timeout_ns = kDefaultTimeoutNs;
  pl->stall_injection = 0;
  pl->stream_k = TPMLP_STREAM_K_AUTO;
  if (const char* s = std::getenv("TPMLP_WAIT_TIMEOUT_MS")) {
    const long long ms = std::atoll(s);
    if (ms > 0) pl->timeout_ns = static_cast<uint64_t>(ms) * 1000000ull;
  }
  *out = pl;
  return TPMLP_OK;
}

void tpmlp_plan_destroy(tpmlp_plan* plan) { delete plan; }

tpmlp_status tpmlp_plan_set_timeout(tpmlp_plan* plan, uint32_t timeout_ms) {
  g_last_error[0] = 0;
  if (!plan) return fail(TPMLP_ERR_INVALID_ARG, "plan is NULL");
  if (timeout_ms < 1) return fail(TPMLP_ERR_INVALID_ARG, "timeout must be at least 1 ms");
  plan->timeout_ns = static_cast<uint64_t>(timeout_ms) * 1000000ull;
  return TPMLP_OK;
}

tpmlp_status tpmlp_plan_set_stall_injection(tpmlp_plan* plan, int enable) {
  g_last_error[0] = 0;
  if (!plan) return fail(TPMLP_ERR_INVALID_ARG, "plan is NULL");
  plan->stall_injection = enable == 2 ? 2 : (enable ? 1 : 0);
  return TPMLP_OK;
}

size_t tpmlp_workspace_size(const tpmlp_plan* plan) {
  if (!plan) return 0;
  return plan->dtype == TPMLP_BF16 ? kSkWorkspaceBytes : kStatusBytes;
}

tpmlp_status tpmlp_plan_set_stream_k(tpmlp_plan* plan, int mode) {
  g_last_error[0] = 0;
  if (!plan) return fail(TPMLP_ERR_INVALID_ARG, "plan is NULL");
  if (mode != TPMLP_STREAM_K_OFF && mode != TPMLP_STREAM_K_AUTO && mode != TPMLP_STREAM_K_ALWAYS &&
      mode != TPMLP_STREAM_K_BALANCE)
    return fail(TPMLP_ERR_INVALID_ARG, "stream-K mode %d is not one of 0, 1, 2, 3", mode);
  plan->stream_k = mode;
  return TPMLP_OK;
}

// Optional bias arrays: NULL, or t pointers each non-NULL and 16-byte aligned.
tpmlp_status check_bias(const char* name, const void* const* b, int t) {
  return b ? check_array(name, b, t, false) : TPMLP_OK;
}

tpmlp_status tpmlp_forward_column(const tpmlp_plan* plan, const void* X, const void* const* W1,
                                  const void* const* W3, const void* const* b1, const void* const* b3,
                                  void* const* saved, void* const* H, void* workspace, tpmlp_stream_t stream) {
  g_last_launches = 0;
  DeviceInfo di;
  TPMLP_TRY(common_checks(plan, workspace, &di));
  const bool tz = plan->T == 0;
  TPMLP_TRY(check_ptr("X", X, tz));
  TPMLP_TRY(check_array("W1", W1, plan->t, false));
  if (swiglu(plan)) TPMLP_TRY(check_array("W3", W3, plan->t, false));
  TPMLP_TRY(check_array("saved", saved, nsaved(plan), tz));
  TPMLP_TRY(check_array("H", H, plan->t, tz));
  TPMLP_TRY(check_bias("b1", b1, plan->t));
  if (swiglu(plan)) TPMLP_TRY(check_bias("b3", b3, plan->t));
  return fwd_column(plan, di, X, W1, W3, b1, swiglu(plan) ? b3 : nullptr, saved, H, workspace,
                    reinterpret_cast<cudaStream_t>(stream));
}

tpmlp_status tpmlp_forward_row(const tpmlp_plan* plan, const void* const* W2, const void* b2, void* const* H,
                               void* Y, void* workspace, tpmlp_stream_t stream) {
  g_last_launches = 0;
  DeviceInfo di;
  TPMLP_TRY(common_checks(plan, workspace, &di));
  const bool tz = plan->T == 0;
  TPMLP_TRY(check_array("W2", W2, plan->t, false));
  TPMLP_TRY(check_array("H", H, plan->t, tz));
  TPMLP_TRY(check_ptr("Y", Y, tz));
  TPMLP_TRY(check_ptr("b2", b2, true));
  return fwd_row(plan, di, W2, b2, Y, H, workspace, reinterpret_cast<cudaStream_t>(stream));
}

tpmlp_status tpmlp_forward_row_noalloc(const tpmlp_plan* plan, const void* const* W2, void* const* H, void* Y,
                                       tpmlp_stream_t stream) {
  g_last_launches = 0;
  g_last_error[0] = 0;
  if (!plan) return fail(TPMLP_ERR_INVALID_ARG, "plan is NULL");
  TPMLP_TRY(check_kind(plan, PLAN_MLP));
  DeviceInfo di;
  TPMLP_TRY(device_info(&di));  // also makes the device's primary context current
  const size_t need = kStatusBytes;  // the status word only: no stream-K tail here
  if (need > kStaticScratchBytes)
    return fail(TPMLP_ERR_UNSUPPORTED, "this plan needs %zu bytes of scratch; the static scratch holds %zu", need,
                kStaticScratchBytes);
  const bool tz = plan->T == 0;
  TPMLP_TRY(check_array("W2", W2, plan->t, false));
  TPMLP_TRY(check_array("H", H, plan->t, tz));
  TPMLP_TRY(check_ptr("Y", Y, tz));
  int32_t* scratch = nullptr;
  TPMLP_TRY(static_scratch(&scratch));
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  // The status word must start at zero; the array keeps the last call's contents.
  cudaError_t e = cudaMemsetAsync(scratch, 0, need, st);
  if (e != cudaSuccess) return cuda_fail(e);
  TPMLP_TRY(fwd_row(plan, di, W2, nullptr, Y, H, scratch, st, nullptr, /*sk_workspace=*/false));
  int32_t word = 0;
  e = cudaMemcpyAsync(&word, scratch, sizeof(word), cudaMemcpyDeviceToHost, st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) return cuda_fail(e);
  if (word != kDevOk) return fail(TPMLP_ERR_DEVICE_TIMEOUT, "device wait timed out (code %d)", word);
  return TPMLP_OK;
}

tpmlp_status tpmlp_forward(const tpmlp_plan* plan, const void* X, const void* const* W1, const void* const* W3,
                           const void* const* W2, const void* const* b1, const void* const* b3, const void* b2,
                           void* Y, void* const* saved, void* const* H, void* workspace, tpmlp_stream_t stream) {
  g_last_launches = 0;
  DeviceInfo di;
  TPMLP_TRY(common_checks(plan, workspace, &di));
  const bool tz = plan->T == 0;
  TPMLP_TRY(check_ptr("X", X, tz)); TPMLP_TRY(check_ptr("Y", Y, tz));
  TPMLP_TRY(check_array("W1", W1, plan->t, false));
  if (swiglu(plan)) TPMLP_TRY(check_array("W3", W3, plan->t, false));
  TPMLP_TRY(check_array("W2", W2, plan->t, false));
  TPMLP_TRY(check_array("saved", saved, nsaved(plan), tz));
  TPMLP_TRY(check_array("H", H, plan->t, tz));
  TPMLP_TRY(check_bias("b1", b1, plan->t));
  if (swiglu(plan)) TPMLP_TRY(check_bias("b3", b3, plan->t));
  TPMLP_TRY(check_ptr("b2", b2, true));
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  TPMLP_TRY(fwd_column(plan, di, X, W1, W3, b1, swiglu(plan) ? b3 : nullptr, saved, H, workspace, st));
  return fwd_row(plan, di, W2, b2, Y, H, workspace, st);
}

tpmlp_status tpmlp_backward_dgrad(const tpmlp_plan* plan, const void* const* W2, const void* const* saved,
                                  const void* const* H, const void* dY, void* const* dact, void* const* dW2,
                                  void* db2, void* workspace, tpmlp_stream_t stream) {
  g_last_launches = 0;
  DeviceInfo di;
  TPMLP_TRY(common_checks(plan, workspace, &di));
  const bool tz = plan->T == 0;
  TPMLP_TRY(check_array("W2", W2, plan->t, false));
  TPMLP_TRY(check_array("saved", saved, nsaved(plan), tz));
  TPMLP_TRY(check_array("H", H, plan->t, tz));
  TPMLP_TRY(check_ptr("dY", dY, tz));
  TPMLP_TRY(check_array("dact", dact, nsaved(plan), tz));
  TPMLP_TRY(check_array("dW2", dW2, plan->t, false));
  TPMLP_TRY(check_ptr("db2", db2, true));
  return bwd_dgrad(plan, di, W2, saved, H, dY, dact, dW2, db2, workspace, reinterpret_cast<cudaStream_t>(stream));
}

tpmlp_status tpmlp_backward_fsum(const tpmlp_plan* plan, const void* X, const void* const* W1,
                                 const void* const* W3, const void* const* dact, void* dX, void* const* dW1,
                                 void* const* dW3, void* const* db1, void* const* db3, void* workspace,
                                 tpmlp_stream_t stream) {
  g_last_launches = 0;
  DeviceInfo di;
  TPMLP_TRY(common_checks(plan, workspace, &di));
  const bool tz = plan->T == 0;
  TPMLP_TRY(check_ptr("X", X, tz)); TPMLP_TRY(check_ptr("dX", dX, tz));
  TPMLP_TRY(check_array("W1", W1, plan->t, false));
  if (swiglu(plan)) {
    TPMLP_TRY(check_array("W3", W3, plan->t, false));
    TPMLP_TRY(check_array("dW3", dW3, plan->t, false));
  }
  TPMLP_TRY(check_array("dact", dact, nsaved(plan), tz));
  TPMLP_TRY(check_array("dW1", dW1, plan->t, false));
  TPMLP_TRY(check_bias("db1", db1, plan->t));
  if (swiglu(plan)) TPMLP_TRY(check_bias("db3", db3, plan->t));
  return bwd_fsum(plan, di, X, W1, W3, dact, dX, dW1, dW3, db1, swiglu(plan) ? db3 : nullptr, workspace,
                  reinterpret_cast<cudaStream_t>(stream));
}

tpmlp_status tpmlp_backward(const tpmlp_plan* plan, const void* X, const void* const* W1, const void* const* W3,
                            const void* const* W2, const void* const* saved, const void* const* H, const void* dY,
                            void* const* dact, void* dX, void* const* dW1, void* const* dW3, void* const* dW2,
                            void* const* db1, void* const* db3, void* db2, void* workspace, tpmlp_stream_t stream) {
  g_last_launches = 0;
  DeviceInfo di;
  TPMLP_TRY(common_checks(plan, workspace, &di));
  const bool tz = plan->T == 0;
  TPMLP_TRY(check_ptr("X", X, tz)); TPMLP_TRY(check_ptr("dY", dY, tz)); TPMLP_TRY(check_ptr("dX", dX, tz));
  TPMLP_TRY(check_array("W1", W1, plan->t, false));
  TPMLP_TRY(check_array("W2", W2, plan->t, false));
  if (swiglu(plan)) {
    TPMLP_TRY(check_array("W3", W3, plan->t, false));
    TPMLP_TRY(check_array("dW3", dW3, plan->t, false));
  }
  TPMLP_TRY(check_array("saved", saved, nsaved(plan), tz));
  TPMLP_TRY(check_array("H", H, plan->t, tz));
  TPMLP_TRY(check_array("dact", dact, nsaved(plan), tz));
  TPMLP_TRY(check_array("dW1", dW1, plan->t, false));
  TPMLP_TRY(check_array("dW2", dW2, plan->t, false));
  TPMLP_TRY(check_bias("db1", db1, plan->t));
  if (swiglu(plan)) TPMLP_TRY(check_bias("db3", db3, plan->t));
  TPMLP_TRY(check_ptr("db2", db2, true));
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  TPMLP_TRY(bwd_dgrad(plan, di, W2, saved, H, dY, dact, dW2, db2, workspace, st));
  return bwd_fsum(plan, di, X, W1, W3, dact, dX, dW1, dW3, db1, swiglu(plan) ? db3 : nullptr, workspace, st);
}

tpmlp_status tpmlp_backward_recompute(const tpmlp_plan* plan, const void* X, const void* const* W1,
                                      const void* const* W3, const void* const* W2, const void* const* saved,
                                      void* const* H, const void* dY, void* const* dact, void* dX,
                                      void* const* dW1, void* const* dW3, void* const* dW2, void* const* db1,
                                      void* const* db3, void* db2, void* workspace, tpmlp_stream_t stream) {
  g_last_launches = 0;
  DeviceInfo di;
  TPMLP_TRY(common_checks(plan, workspace, &di));
  const bool tz = plan->T == 0;
  TPMLP_TRY(check_ptr("X", X, tz)); TPMLP_TRY(check_ptr("dY", dY, tz)); TPMLP_TRY(check_ptr("dX", dX, tz));
  TPMLP_TRY(check_array("W1", W1, plan->t, false));
  TPMLP_TRY(check_array("W2", W2, plan->t, false));
  if (swiglu(plan)) {
    TPMLP_TRY(check_array("W3", W3, plan->t, false));
    TPMLP_TRY(check_array("dW3", dW3, plan->t, false));
  }
  TPMLP_TRY(check_array("saved", saved, nsaved(plan), tz));
  TPMLP_TRY(check_array("H", H, plan->t, tz));
  TPMLP_TRY(check_array("dact", dact, nsaved(plan), tz));
  TPMLP_TRY(check_array("dW1", dW1, plan->t, false));
  TPMLP_TRY(check_array("dW2", dW2, plan->t, false));
  TPMLP_TRY(check_bias("db1", db1, plan->t));
  if (swiglu(plan)) TPMLP_TRY(check_bias("db3", db3, plan->t));
  TPMLP_TRY(check_ptr("db2", db2, true));
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (tz) {  // nothing to recompute; zero-filled gradients as in tpmlp_backward
    TPMLP_TRY(bwd_dgrad(plan, di, W2, saved, H, dY, dact, dW2, db2, workspace, st));
    return bwd_fsum(plan, di, X, W1, W3, dact, dX, dW1, dW3, db1, swiglu(plan) ? db3 : nullptr, workspace, st);
  }
  TPMLP_TRY(bwd_dgrad(plan, di, W2, saved, H, dY, dact, dW2, db2, workspace, st, /*recompute=*/true));
  return bwd_fsum(plan, di, X, W1, W3, dact, dX, dW1, dW3, db1, swiglu(plan) ? db3 : nullptr, workspace, st, H,
                  dY, dW2);
}

tpmlp_status tpmlp_attn_plan_create(const tpmlp_attn_desc* desc, tpmlp_plan** out) {
  g_last_error[0] = 0;
  if (!out) return fail(TPMLP_ERR_INVALID_ARG, "out is NULL");
  *out = nullptr;
  if (!desc || !desc->dq_i || !desc->dkv_i) return fail(TPMLP_ERR_INVALID_ARG, "desc, dq_i or dkv_i is NULL");
  if (desc->dtype != TPMLP_BF16 && desc->dtype != TPMLP_FP32)
    return fail(TPMLP_ERR_INVALID_ARG, "unknown dtype %d", static_cast<int>(desc->dtype));
  if (desc->T < 0 || desc->d < 1 || desc->t < 1 || desc->t > TPMLP_MAX_SHARDS)
    return fail(TPMLP_ERR_SHAPE, "need T >= 0, d >= 1, 1 <= t <= %d (got T=%lld d=%lld t=%d)", TPMLP_MAX_SHARDS,
                static_cast<long long>(desc->T), static_cast<long long>(desc->d), desc->t);
  const int64_t mult = desc->dtype == TPMLP_BF16 ? 8 : 4;
  const int64_t kMax32 = (int64_t(1) << 31) - 1;
  int64_t total = 0;
  for (int i = 0; i < desc->t; ++i) {
    if (desc->dq_i[i] < 1 || desc->dkv_i[i] < 1)
      return fail(TPMLP_ERR_SHAPE, "shard %d: dq_i = %lld and dkv_i = %lld must be >= 1", i,
                  static_cast<long long>(desc->dq_i[i]), static_cast<long long>(desc->dkv_i[i]));
    total += desc->dq_i[i] + 2 * desc->dkv_i[i];
  }
  if (desc->d % mult)
    return fail(TPMLP_ERR_ALIGNMENT, "d = %lld is not a multiple of %lld", static_cast<long long>(desc->d),
                static_cast<long long>(mult));
  for (int i = 0; i < desc->t; ++i)
    if (desc->dq_i[i] % mult || desc->dkv_i[i] % mult)
      return fail(TPMLP_ERR_ALIGNMENT, "shard %d: dq_i = %lld and dkv_i = %lld must be multiples of %lld", i,
                  static_cast<long long>(desc->dq_i[i]), static_cast<long long>(desc->dkv_i[i]),
                  static_cast<long long>(mult));
  if (desc->T > kMax32 || desc->d > kMax32 || total > kMax32)
    return fail(TPMLP_ERR_UNSUPPORTED, "T, d and the total QKV width must each be below 2^31");
  tpmlp_plan* pl = new (std::nothrow) tpmlp_plan;
  if (!pl) return TPMLP_ERR_INVALID_ARG;
  pl->kind = PLAN_ATTN;
  pl->T = desc->T;
  pl->d = desc->d;
  pl->t = desc->t;
  pl->dq_i.assign(desc->dq_i, desc->dq_i + desc->t);
  pl->dkv_i.assign(desc->dkv_i, desc->dkv_i + desc->t);
  pl->d_i.resize(desc->t);
  pl->o_i.resize(desc->t);
  int64_t o = 0;
  for (int i = 0; i < desc->t; ++i) {
    pl->d_i[i] = pl->dq_i[i] + 2 * pl->dkv_i[i];
    pl->o_i[i] = o;
    o += pl->d_i[i];
  }
  pl->dff = o;
  pl->act = TPMLP_ACT_GELU;  // unused by the attention entry points
  pl->dtype = desc->dtype;
  pl->timeout_ns = kDefaultTimeoutNs;
  pl->stall_injection = 0;
  pl->stream_k = TPMLP_STREAM_K_AUTO;
  if (const char* s = std::getenv("TPMLP_WAIT_TIMEOUT_MS")) {
    const long long ms = std::atoll(s);
    if (ms > 0) pl->timeout_ns = static_cast<uint64_t>(ms) * 1000000ull;
  }
  *out = pl;
  return TPMLP_OK;
}

tpmlp_status tpmlp_attn_qkv_forward(const tpmlp_plan* plan, const void* X, const void* const* Wqkv,
                                    void* const* QKV, void* workspace, tpmlp_stream_t stream) {
  g_last_launches = 0;
  DeviceInfo di;
  TPMLP_TRY(common_checks(plan, workspace, &di, PLAN_ATTN));
  const bool tz = plan->T == 0;
  TPMLP_TRY(check_ptr("X", X, tz));
  TPMLP_TRY(check_array("Wqkv", Wqkv, plan->t, false));
  TPMLP_TRY(check_array("QKV", QKV, plan->t, tz));
  return attn_qkv_fwd(plan, di, X, Wqkv, QKV, workspace, reinterpret_cast<cudaStream_t>(stream));
}

tpmlp_status tpmlp_attn_out_forward(const tpmlp_plan* plan, const void* const* WO, const void* const* O, void* Z,
                                    void* workspace, tpmlp_stream_t stream) {
  g_last_launches = 0;
  DeviceInfo di;
  TPMLP_TRY(common_checks(plan, workspace, &di, PLAN_ATTN));
  const bool tz = plan->T == 0;
  TPMLP_TRY(check_array("WO", WO, plan->t, false));
  TPMLP_TRY(check_array("O", O, plan->t, tz));
  TPMLP_TRY(check_ptr("Z", Z, tz));
  return attn_out_fwd(plan, di, WO, O, Z, workspace, reinterpret_cast<cudaStream_t>(stream));
}

tpmlp_status tpmlp_attn_out_backward(const tpmlp_plan* plan, const void* const* WO, const void* const* O,
                                     const void* dZ, void* const* dO, void* const* dWO, void* workspace,
                                     tpmlp_stream_t stream) {
  g_last_launches = 0;
  DeviceInfo di;
  TPMLP_TRY(common_checks(plan, workspace, &di, PLAN_ATTN));
  const bool tz = plan->T == 0;
  TPMLP_TRY(check_array("WO", WO, plan->t, false));
  TPMLP_TRY(check_array("O", O, plan->t, tz));
  TPMLP_TRY(check_ptr("dZ", dZ, tz));
  TPMLP_TRY(check_array("dO", dO, plan->t, tz));
  TPMLP_TRY(check_array("dWO", dWO, plan->t, false));
  return attn_out_bwd(plan, di, WO, O, dZ, dO, dWO, workspace, reinterpret_cast<cudaStream_t>(stream));
}

tpmlp_status tpmlp_attn_qkv_backward(const tpmlp_plan* plan, const void* X, const void* const* Wqkv,
                                     const void* const* dQKV, void* dX, void* const* dWqkv, void* workspace,
                                     tpmlp_stream_t stream) {
  g_last_launches = 0;
  DeviceInfo di;
  TPMLP_TRY(common_checks(plan, workspace, &di, PLAN_ATTN));
  const bool tz = plan->T == 0;
  TPMLP_TRY(check_ptr("X", X, tz));
  TPMLP_TRY(check_ptr("dX", dX, tz));
  TPMLP_TRY(check_array("Wqkv", Wqkv, plan->t, false));
  TPMLP_TRY(check_array("dQKV", dQKV, plan->t, tz));
  TPMLP_TRY(check_array("dWqkv", dWqkv, plan->t, false));
  return attn_qkv_bwd(plan, di, X, Wqkv, dQKV, dX, dWqkv, workspace, reinterpret_cast<cudaStream_t>(stream));
}

tpmlp_status tpmlp_plan_set_sequence_stripes(tpmlp_plan* plan, int32_t nstripes, const int64_t* stripe_rows) {
  g_last_error[0] = 0;
  if (!plan) return fail(TPMLP_ERR_INVALID_ARG, "plan is NULL");
  if (plan->kind != PLAN_MLP) return fail(TPMLP_ERR_INVALID_ARG, "sequence stripes apply to MLP plans");
  if (!stripe_rows) return fail(TPMLP_ERR_INVALID_ARG, "stripe_rows is NULL");
  if (nstripes < 1 || nstripes > TPMLP_MAX_SHARDS)
    return fail(TPMLP_ERR_SHAPE, "need 1 <= nstripes <= %d (got %d)", TPMLP_MAX_SHARDS, nstripes);
  int64_t r = 0;
  for (int j = 0; j < nstripes; ++j) {
    if (stripe_rows[j] < 0) return fail(TPMLP_ERR_SHAPE, "stripe %d has %lld rows", j, (long long)stripe_rows[j]);
    if (j > 0 && r % 128)
      return fail(TPMLP_ERR_ALIGNMENT, "stripe %d starts at row %lld, not a multiple of 128", j, (long long)r);
    r += stripe_rows[j];
  }
  if (r != plan->T)
    return fail(TPMLP_ERR_SHAPE, "the stripes hold %lld rows, the plan %lld tokens", (long long)r, (long long)plan->T);
  plan->stripe_rows.assign(stripe_rows, stripe_rows + nstripes);
  return TPMLP_OK;
}

// Stripe pointer arrays: one entry per stripe; entries of non-empty stripes
// non-NULL and 16-byte aligned (empty stripes may be NULL).
tpmlp_status check_stripes(const char* name, const void* const* arr, const tpmlp_plan* pl) {
  if (pl->stripe_rows.empty())
    return fail(TPMLP_ERR_INVALID_ARG, "no sequence stripes set (tpmlp_plan_set_sequence_stripes)");
  if (!arr) return fail(TPMLP_ERR_INVALID_ARG, "stripe array %s is NULL", name);
  for (size_t j = 0; j < pl->stripe_rows.size(); ++j) {
    if (pl->stripe_rows[j] == 0) continue;
    if (!arr[j]) return fail(TPMLP_ERR_INVALID_ARG, "%s[%zu] is NULL", name, j);
    if (!aligned16(arr[j])) return fail(TPMLP_ERR_ALIGNMENT, "%s[%zu] (%p) is not 16-byte aligned", name, j, arr[j]);
  }
  return TPMLP_OK;
}

tpmlp_status tpmlp_forward_sp(const tpmlp_plan* plan, const void* const* X_stripes, const void* const* W1,
                              const void* const* W3, const void* const* W2, const void* const* b1,
                              const void* const* b3, const void* b2, void* const* Y_stripes, void* const* saved,
                              void* const* H, void* workspace, tpmlp_stream_t stream) {
  g_last_launches = 0;
  DeviceInfo di;
  TPMLP_TRY(common_checks(plan, workspace, &di));
  const bool tz = plan->T == 0;
  TPMLP_TRY(check_stripes("X_stripes", X_stripes, plan));
  TPMLP_TRY(check_stripes("Y_stripes", Y_stripes, plan));
  TPMLP_TRY(check_array("W1", W1, plan->t, false));
  if (swiglu(plan)) TPMLP_TRY(check_array("W3", W3, plan->t, false));
  TPMLP_TRY(check_array("W2", W2, plan->t, false));
  TPMLP_TRY(check_array("saved", saved, nsaved(plan), tz));
  TPMLP_TRY(check_array("H", H, plan->t, tz));
  TPMLP_TRY(check_bias("b1", b1, plan->t));
  if (swiglu(plan)) TPMLP_TRY(check_bias("b3", b3, plan->t));
  TPMLP_TRY(check_ptr("b2", b2, true));
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  TPMLP_TRY(fwd_column(plan, di, nullptr, W1, W3, b1, swiglu(plan) ? b3 : nullptr, saved, H, workspace, st,
                       X_stripes));
  return fwd_row(plan, di, W2, b2, nullptr, H, workspace, st, Y_stripes);
}

tpmlp_status tpmlp_backward_sp(const tpmlp_plan* plan, const void* const* X_stripes, const void* const* W1,
                               const void* const* W3, const void* const* W2, const void* const* saved,
                               const void* const* H, const void* const* dY_stripes, void* const* dact,
                               void* const* dX_stripes, void* const* dW1, void* const* dW3, void* const* dW2,
                               void* const* db1, void* const* db3, void* db2, void* workspace,
                               tpmlp_stream_t stream) {
  g_last_launches = 0;
  DeviceInfo di;
  TPMLP_TRY(common_checks(plan, workspace, &di));
  const bool tz = plan->T == 0;
  TPMLP_TRY(check_stripes("X_stripes", X_stripes, plan));
  TPMLP_TRY(check_stripes("dY_stripes", dY_stripes, plan));
  TPMLP_TRY(check_stripes("dX_stripes", dX_stripes, plan));
  TPMLP_TRY(check_array("W1", W1, plan->t, false));
  TPMLP_TRY(check_array("W2", W2, plan->t, false));
  if (swiglu(plan)) {
    TPMLP_TRY(check_array("W3", W3, plan->t, false));
    TPMLP_TRY(check_array("dW3", dW3, plan->t, false));
  }
  TPMLP_TRY(check_array("saved", saved, nsaved(plan), tz));
  TPMLP_TRY(check_array("H", H, plan->t, tz));
  TPMLP_TRY(check_array("dact", dact, nsaved(plan), tz));
  TPMLP_TRY(check_array("dW1", dW1, plan->t, false));
  TPMLP_TRY(check_array("dW2", dW2, plan->t, false));
  TPMLP_TRY(check_bias("db1", db1, plan->t));
  if (swiglu(plan)) TPMLP_TRY(check_bias("db3", db3, plan->t));
  TPMLP_TRY(check_ptr("db2", db2, true));
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  TPMLP_TRY(bwd_dgrad(plan, di, W2, saved, H, nullptr, dact, dW2, db2, workspace, st, false, dY_stripes));
  return bwd_fsum(plan, di, nullptr, W1, W3, dact, nullptr, dW1, dW3, db1, swiglu(plan) ? db3 : nullptr, workspace,
                  st, nullptr, nullptr, nullptr, X_stripes, dX_stripes);
}

tpmlp_status tpmlp_check(const tpmlp_plan* plan, void* workspace, tpmlp_stream_t stream) {
  if (!plan || !workspace) return TPMLP_ERR_INVALID_ARG;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) return cuda_fail(e);
  int32_t word = 0;
  e = cudaMemcpy(&word, workspace, sizeof(word), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_fail(e);
  if (word != kDevOk) {
    // Clear the status word and, for bf16 plans, the stream-K ticket counters
    // that an aborted launch may have left behind.
    const size_t n = plan->dtype == TPMLP_BF16 ? kSkSlotsOffset : sizeof(word);
    e = cudaMemset(workspace, 0, n);
    if (e != cudaSuccess) return cuda_fail(e);
    return TPMLP_ERR_DEVICE_TIMEOUT;
  }
  return TPMLP_OK;
}

const char* tpmlp_status_string(tpmlp_status s) {
  switch (s) {
    case TPMLP_OK: return "TPMLP_OK";
    case TPMLP_ERR_INVALID_ARG: return "TPMLP_ERR_INVALID_ARG";
    case TPMLP_ERR_SHAPE: return "TPMLP_ERR_SHAPE";
    case TPMLP_ERR_ALIGNMENT: return "TPMLP_ERR_ALIGNMENT";
    case TPMLP_ERR_UNSUPPORTED: return "TPMLP_ERR_UNSUPPORTED";
    case TPMLP_ERR_CUDA: return "TPMLP_ERR_CUDA";
    case TPMLP_ERR_DEVICE_TIMEOUT: return "TPMLP_ERR_DEVICE_TIMEOUT";
    case TPMLP_ERR_NOT_IMPLEMENTED: return "TPMLP_ERR_NOT_IMPLEMENTED";
  }
  return "TPMLP_ERR_UNKNOWN";
}

int tpmlp_last_cuda_error(void) { return g_last_cuda_error; }
const char* tpmlp_last_error(void) { return g_last_error; }
int tpmlp_version(void) { return 105; }
int tpmlp_last_launch_count(void) { return g_last_launches; }

tpmlp_status tpmlp_eval_activation(int fn, const float* x, const float* y, const float* dh, float* out0,
                                   float* out1, float* out2, int64_t n, tpmlp_stream_t stream) {
  g_last_launches = 0;
  g_last_error[0] = 0;
  if (fn < TPMLP_ACT_EVAL_GELU || fn > TPMLP_ACT_EVAL_FP32_SWIGLU)
    return fail(TPMLP_ERR_INVALID_ARG, "unknown activation form %d", fn);
  if (n < 0) return fail(TPMLP_ERR_INVALID_ARG, "n = %lld < 0", static_cast<long long>(n));
  const bool sw = fn == TPMLP_ACT_EVAL_SWIGLU || fn == TPMLP_ACT_EVAL_SWIGLU_BWD ||
                  fn == TPMLP_ACT_EVAL_SWIGLU_BWD_H || fn == TPMLP_ACT_EVAL_FP32_SWIGLU;
  const bool bwd = fn != TPMLP_ACT_EVAL_GELU && fn != TPMLP_ACT_EVAL_SWIGLU;
  const int nout = fn == TPMLP_ACT_EVAL_GELU || fn == TPMLP_ACT_EVAL_GELU_BWD || fn == TPMLP_ACT_EVAL_SWIGLU
                       ? 1
                       : (fn == TPMLP_ACT_EVAL_GELU_BWD_H || fn == TPMLP_ACT_EVAL_SWIGLU_BWD ||
                                  fn == TPMLP_ACT_EVAL_FP32_GELU
                              ? 2
                              : 3);
  const void* need[6] = {x, sw ? y : x, bwd ? dh : x, out0, nout > 1 ? out1 : out0, nout > 2 ? out2 : out0};
  const char* names[6] = {"x", "y", "dh", "out0", "out1", "out2"};
  for (int i = 0; i < 6; ++i) {
    if (n > 0 && !need[i]) return fail(TPMLP_ERR_INVALID_ARG, "%s is NULL", names[i]);
    if (reinterpret_cast<uintptr_t>(need[i]) & 3u)
      return fail(TPMLP_ERR_ALIGNMENT, "%s (%p) is not 4-byte aligned", names[i], need[i]);
  }
  DeviceInfo di;
  TPMLP_TRY(device_info(&di));
  cudaError_t e = launch_act_eval(fn, x, sw ? y : nullptr, bwd ? dh : nullptr, out0, nout > 1 ? out1 : nullptr,
                                  nout > 2 ? out2 : nullptr, n, reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e);
  if (n > 0) ++g_last_launches;
  return TPMLP_OK;
}

int tpmlp_last_split_tiles(int launch_kind, int64_t* tiles, int cap) {
  if (launch_kind < 0 || launch_kind >= kNumKernelTags) return -1;
  const std::vector<int64_t>& v = g_last_split[launch_kind];
  const int n = static_cast<int>(v.size() / 4);
  if (tiles)
    for (int i = 0; i < std::min(n, cap) * 4; ++i) tiles[i] = v[i];
  return n;
}

}  // extern "C"
