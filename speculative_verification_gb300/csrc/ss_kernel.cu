// ss_kernel.cu -- sm_103a kernels and C ABI of libss (see include/ss.h).
//
// Execution model (fixed shape; one launch per call, or two concurrent
// launches for a sampling call whose rows split into heavy and light):
//   * one thread-block cluster of C CTAs per task; a task is one logits row
//     (ss_process_sample), one target position (request i, draft j) of
//     ss_spec_verify, or one node of a draft tree (ss_tree_verify).  The
//     row's vocabulary is cut into C slices of `slice_len` tokens; each CTA
//     stages its slice in shared memory with 1-D bulk (TMA) copies, once, and
//     every later pass runs on shared memory.
//   * launches of many tasks are ordered: cluster i takes the i-th task in
//     decreasing cost, so the longest rows start in the first wave; a sampling
//     call gives its heavy rows (top-p without top-k) a concurrent launch with
//     2C CTAs per row.
//   * penalised / biased tokens live in a per-CTA hash table ("patches") and
//     are excluded from the raw slice; their processed values are computed
//     from the global row and visited alongside the slice.
//   * stage 1, overlapped with the copies, stores for every 16-byte vector of
//     the slice an upper bound of its largest processed logit (a tile max, as
//     on the FlashSampling page: per-tile maxima, then a cross-tile
//     reduction).  Every later pass skips whole vectors the bound rules out.
//   * cuts (SonicSampler abstract: hierarchical two-stage top-k, top-p): a
//     histogram of the tile maxima bounds the cut from below; tokens above the
//     bound are bucketed by d = y_max - y into 64 buckets of a power-of-two
//     width; the bucket holding a cut is refined into 64 sub-buckets (64x the
//     scale, so levels nest exactly) until it holds at most kListCap tokens,
//     which are gathered into every CTA, sorted by (y desc, index asc) and
//     resolved exactly.  Counts are integers and probability masses 40-bit
//     fixed point, so no result depends on the order in which threads add.
//     Rows the buckets cannot resolve use an exact radix selection instead.
//   * the draw is Gumbel-max over the kept set, per thread, then across the
//     cluster (the argmax decomposes over partitions).  Tokens whose logit
//     plus the largest possible noise cannot beat the running best skip the
//     RNG, whole vectors at a time.  A position that tests drafts sums the
//     mass of the kept set instead and draws only from a residual.
//   * CTAs exchange partial results by writing them into every CTA of the
//     cluster (distributed shared memory) before a cluster barrier, so each
//     exchange costs one barrier and every CTA derives identical decisions.
//   * code size matters as much as instruction count: a row executes its
//     passes once, so every pass is one out-of-line function that all call
//     sites share, and the per-CTA state lives in shared memory (`g`).
#include <cooperative_groups.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>
#include <algorithm>
#include <string.h>

#include <mutex>

#include "ss.h"
#include "ss_nvtx.h"
#include "ss_hist.h"
#include "ss_philox.cuh"
#include "ss_ptx.cuh"

namespace cg = cooperative_groups;

namespace ss {

constexpr int kThreads = 512;  // 2 CTAs per SM with up to 64 registers per thread
constexpr int kWarps = kThreads / 32;
constexpr int kHashCap = SS_MAX_PATCHED;
constexpr int kHashShift = 32 - 10;  // log2(kHashCap) = 10
static_assert(kHashCap == 1024, "hash shift assumes 1024 slots");
static_assert(kHashCap % kThreads == 0, "patch-table loops run the same trip count in every thread");
static_assert(kThreads >= 256, "histogram folding uses 4 threads per bucket");
constexpr uint32_t kChunkBytes = 8192;
constexpr int kMaxChunks = 20;
constexpr uint32_t kTargetSliceBytes = 66000u;
constexpr uint32_t kMaxSliceBytes = kMaxChunks * kChunkBytes;
constexpr int kMaxCluster = 8;
// Largest max_draft a verification call takes (tree calls: SS_TREE_MAX_NODES).
constexpr uint32_t kWaitPolls = 1u << 22;
constexpr float kFixedScale = 1099511627776.0f;  // 2^40
// A token's fixed-point mass (<= 2^40) is histogrammed as two 32-bit halves,
// mass >> 20 and mass & (2^20 - 1).  Each copy of a bucket counter receives
// the tokens of 16 threads, at most 16 * (ceil(kMaxSliceTokens / 8 / 256) * 8
// + 1024 / 256) = 3904 of them, so neither half can wrap.
constexpr int kMassSplit = 20;
constexpr int kMaxSliceTokens = 61440;
constexpr double kFixedInv = 1.0 / 1099511627776.0;
constexpr int kBiasFlag = 1 << 30;
constexpr int kNoCut = 0x7fffffff;
constexpr int kBuckets = 64;
constexpr int kCopies = 16;    // lane-private histogram copies
constexpr int kListCap = 512;  // tokens gathered for an exact resolution
constexpr int kMaxLevels = 3;  // bucket refinement depth
constexpr int kRecs = kMaxLevels + 2;  // level 1, k-chain, scratch, tile level
constexpr float kMassCutoff = 28.5f;  // exp(-28.5) * 2^40 < 1: zero in fixed point
constexpr int kHistRows = 65;  // 64 buckets and a spill row
constexpr uint32_t kWorkBytes = 3 * kHistRows * kCopies * 4;  // histograms / gathered lists / fallback buffers
constexpr int kPartSlots = 4;  // stage 1, draw, residual, normaliser
constexpr int kRedBytes = 2048;

enum TaskMode { kModeSample = 0, kModeVerify = 1, kModeTree = 2 };
// Tree verification: nodes per request, and where the setup keeps the tree
// (parents, tokens, the node's path) in the work region, past the raw logits
// of the patched tokens.
constexpr int kTreeMaxNodes = SS_TREE_MAX_NODES;
constexpr uint32_t kTreeOff = 8192;

__device__ __forceinline__ float neg_inf() { return __int_as_float(0xff800000); }
__device__ __forceinline__ float pos_inf() { return __int_as_float(0x7f800000); }

// Order-preserving key: larger y -> larger key.  -0 is folded into +0 first
// so that the two compare equal, as floats do (equal logits order by index).
__device__ __forceinline__ uint32_t order_key(float y) {
  const uint32_t b = __float_as_uint(y + 0.0f);
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}
__device__ __forceinline__ float key_value(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7fffffffu) : ~k);
}
// Sort key: ascending order = (y descending, token index ascending).
__device__ __forceinline__ unsigned long long sort_key(float y, int32_t t) {
  return (static_cast<unsigned long long>(~order_key(y)) << 32) | static_cast<uint32_t>(t);
}
__device__ __forceinline__ uint32_t sort_key_order(unsigned long long e) { return ~static_cast<uint32_t>(e >> 32); }
__device__ __forceinline__ int32_t sort_key_token(unsigned long long e) {
  return static_cast<int32_t>(static_cast<uint32_t>(e));
}

// Largest of a and b, NaN if either is NaN.
__device__ __forceinline__ float max_nan(float a, float b) {
  float r;
  asm("max.NaN.f32 %0, %1, %2;" : "=f"(r) : "f"(a), "f"(b));
  return r;
}

// Floor of x for 0 <= x < 2^22, as an integer: adding 1.5 * 2^23 with
// round-down leaves floor(x) in the low mantissa bits (the sum's unit in the
// last place is 1).  sm_103 issues float rounding and float <-> integer
// conversion instructions at a small fraction of the add rate, so the hot
// loops use this instead.  For larger x (and +inf) the result is at least
// 2^22, for x < 0 it is negative.
__device__ __forceinline__ int floor_small(float x) { return __float_as_int(__fadd_rd(x, 12582912.0f)) - 0x4B400000; }

// The fixed-point mass trunc(exp(y - m) * 2^40) of a token (y <= m) as a high
// half trunc(e * 2^20) <= 2^20 and a low half < 2^20, e = exp(y - m): both
// scalings by 2^20 and the subtraction of the high half are exact, so
// hi * 2^20 + lo is exactly the truncated product.
__device__ __forceinline__ void fixed_mass_parts(float y, float m, uint32_t& hi, uint32_t& lo) {
  const float t = __fmul_rn(fminf(__expf(y - m), 1.0f), 1048576.0f);
  const float th = __fadd_rd(t, 12582912.0f);
  hi = __float_as_uint(th) - 0x4B400000u;
  const float fr = __fmul_rn(__fsub_rn(t, __fsub_rn(th, 12582912.0f)), 1048576.0f);
  lo = __float_as_uint(__fadd_rd(fr, 12582912.0f)) - 0x4B400000u;
}

__device__ __forceinline__ unsigned long long fixed_mass(float y, float m) {
  uint32_t hi, lo;
  fixed_mass_parts(y, m, hi, lo);
  return (static_cast<unsigned long long>(hi) << kMassSplit) + lo;
}

// Absolute bucket floor((m - y) * scale) of y at a refinement scale (a power
// of two), given ms = m * scale (exact): the fused multiply-add rounds
// m * scale - y * scale once, which equals the rounded m - y times scale.
// y = -inf gives a huge index, outside every bucket range in use (absolute
// buckets stay below 64^3 + 64).
__device__ __forceinline__ int bucket_index(float y, float scale, float ms) {
  return floor_small(__fmaf_rn(-y, scale, ms));
}

// Integer value of an integral float in [0, 2^22], without a conversion
// instruction.
__device__ __forceinline__ int small_int(float b) { return __float_as_int(__fadd_rn(b, 12582912.0f)) - 0x4B400000; }

// Smallest y a token of bucket `abs` at `scale` can have (rounded down).
__device__ __forceinline__ float bucket_floor(float m, float abs, float scale) {
  return m - (abs + 1.0f) / scale - fabsf(m) * 1e-6f - 1e-30f;
}

// Fixed-point mass target ceil(p * S): cum >= target  <=>  cum >= p * S.
__device__ __forceinline__ unsigned long long mass_target(float p, unsigned long long S) {
  return static_cast<unsigned long long>(ceil(static_cast<double>(p) * static_cast<double>(S)));
}

// ----------------------------------------------------------------- layout --

struct Layout {
  int32_t slice_len;   // tokens per CTA, multiple of 32
  int32_t data_bytes;  // raw slice bytes (multiple of 16)
  int32_t vmax_off;    // per-vector bound of the largest processed logit (bf16, rounded up)
  int32_t xm_off;      // exclusion bitmap, slice_len / 32 words
  int32_t hk_off;      // patch table: token ids
  int32_t hc_off;      // patch table: counts | kBiasFlag
  int32_t hv_off;      // patch table: bias value, then processed value
  int32_t work_off;    // kWorkBytes: histograms / gathered lists / fallback buffers
  int32_t rh_off;      // 2 x C x 64 pushed bucket masses (u64) and counts (u32)
  int32_t rec_off;     // kRecs merged histograms
  int32_t red_off;     // per-warp reduction scratch
  int32_t part_off;    // kPartSlots x C pushed partials
  int32_t mbar_off;    // kMaxChunks mbarriers
  int32_t total;
};

// Per-CTA partials exchanged through distributed shared memory.
struct alignas(16) Part {
  float best;
  int32_t arg;
  int32_t count;
  int32_t status;
  unsigned long long mass;
  float ymin;     // smallest allowed processed logit
  float xy;       // processed logit of the draft token (its CTA only)
  int32_t xhere;  // this CTA holds the draft token
  float smax;     // online softmax: running max and
  float ssum;     //   sum of exp(y - smax)
  int32_t pad[3];
};

// Merged histogram of one refinement level.
struct alignas(16) LevelRec {
  float scale;  // bucket(y) = floor((m - y) * scale) - base
  float base;   // 64 * absolute index of the parent bucket (0 at level 1)
  int32_t pad[2];
  uint32_t cnt[kBuckets];
  unsigned long long mass[kBuckets];
};

// Result of one histogram pass of the fallback selection.
struct SelPass {
  uint32_t digit, cnt_before, cnt_bin, reached;
  unsigned long long mass_before, mass_bin, total, target;
};

struct Loc {  // where a count / mass target falls in a LevelRec
  int32_t bucket, found;
  uint32_t cnt_before, pad;
  unsigned long long mass_before;
};

struct KArgs {
  int32_t mode;
  int32_t num_tasks;
  int32_t vocab, max_draft, dtype;
  int64_t row_stride;
  const void* logits;
  const int32_t* draft_offsets;
  const int32_t* draft_tokens;
  const float* draft_probs;
  int64_t draft_stride;
  ss_params p;
  int32_t* out_token;  // sample: [n]; verify: [R, max_draft + 1]
  int32_t* out_num_accepted;
  int32_t* out_status;
  int32_t* out_kept;
  float* debug_processed;
  int4* ws_results;
  int32_t* ws_counters;
  // vocabulary shard: tokens [shard_off, shard_off + shard_len) of the rows;
  // the whole vocabulary (0, vocab) outside the sharded entry point
  int32_t shard_off, shard_len;
  const int32_t* tree_parents;  // tree verification: local parent of every node
  int32_t* out_path;            // tree verification: accepted nodes [R, max_nodes], or NULL
  uint8_t* shard_rec;  // sharded entry point: per-row records, else NULL
  int32_t shard_cap;   // list entries per record
  // 0: every task in launch order; 1 / 2: only the light / heavy rows (see
  // row_is_heavy), the others are left to a concurrent launch of the other
  // class; 3: every task, costliest first (see ordered_task)
  int32_t row_class;
  int32_t overlap;  // trees: launched to overlap the call before it (writes wait for it)
  // trees: the caller's count of tasks (nodes, a request with a bad node
  // count as one; 0: none), checked against the offsets; clusters launched
  // (0: num_tasks; an ordered launch may stop at the stated count)
  int32_t stated_tasks, grid_tasks;
  Layout L;
};

// Rows with a top-p cut and no top-k need the probability mass of the whole
// row (the online softmax sum, then a histogram descent over the flat part of
// the distribution) and draw over a kept set of thousands of tokens: several
// times the work of any other row.  The sampling call gives them twice the
// CTAs of the others (a second, concurrent launch) so that the launch does not
// wait on them.  A pure function of the row's parameters: every row is handled
// by exactly one of the two launches.
__device__ __forceinline__ bool row_is_heavy(float T, int32_t top_k, float top_p) {
  return T > 0.0f && top_k <= 0 && top_p < 1.0f;
}

// Relative cost of a light row, 3 (most) to 0: a large top-k keeps and sorts
// up to a thousand tokens, a row without top-k draws over most of the
// vocabulary, a small top-k over a few tokens, and a greedy row only needs
// the maximum.
constexpr int32_t kLightTopK = 128;
__device__ __forceinline__ int light_cost(float T, int32_t top_k) {
  if (T == 0.0f) return 0;
  if (top_k > kLightTopK) return 3;
  return top_k <= 0 ? 2 : 1;
}

constexpr int kCostLevels = 5;
// Every CTA of an ordered launch reads the parameters of all its tasks: the
// launches order at most this many (beyond, the launch order is kept).
constexpr int kMaxOrderedTasks = 4096;
constexpr int kLevelCacheOff = 32;  // ints: past the counters and warp sums
constexpr int kLevelCache = kRedBytes - kLevelCacheOff * 4;
static_assert(2 + kCostLevels + kWarps <= kLevelCacheOff, "ordering scratch overlaps its level cache");

// Ordered launches.  With row_class 1 or 2 a sampling launch serves one class
// of rows (light or heavy, see row_is_heavy); with 3 a launch serves every
// task, costliest first.  Cluster i takes the i-th task of its launch in that
// order (cost level descending, task index ascending within a level), so the
// longest tasks start in the first wave and the clusters left over (past the
// launch's tasks, they return at once) come last.  A verification position
// past its request's drafts has no work and is left out; one of a request with
// a bad draft count only reports the status (cheapest level).  Every thread of
// the CTA calls it; every CTA of the cluster gets the same answer.  Returns the
// task, or -1, and in *total the number of tasks with work.  sm: kRedBytes of
// shared memory.
__device__ int ordered_task(const KArgs& a, int i, int32_t* sm, int* total) {
  const ss_params& p = a.p;
  const int n = a.num_tasks;
  auto level = [&](int task) -> int {
    int req = task;
    if (a.mode != kModeSample) {
      const int width = a.max_draft + 1;
      req = task / width;
      const int j = task % width;
      // drafts of a linear request, non-root nodes of a tree
      const int32_t k = a.draft_offsets[req + 1] - a.draft_offsets[req] - (a.mode == kModeTree ? 1 : 0);
      if (k < 0 || k > a.max_draft) return j == 0 ? 0 : -1;
      if (j > k) return -1;
    }
    const float T = p.temperature[req];
    const int32_t tk = p.top_k ? p.top_k[req] : 0;
    const bool heavy = row_is_heavy(T, tk, p.top_p ? p.top_p[req] : 1.0f);
    if (a.row_class == 3) return heavy ? 4 : light_cost(T, tk);
    if (1 + static_cast<int>(heavy) != a.row_class) return -1;
    return heavy ? 0 : light_cost(T, tk);
  };
  int32_t* cnt = sm + 2;
  int32_t* wsum = cnt + kCostLevels;
  // the first pass keeps each task's level (+1) for the second, up to kLevelCache tasks
  uint8_t* lev = reinterpret_cast<uint8_t*>(sm + kLevelCacheOff);
  if (threadIdx.x < kCostLevels) cnt[threadIdx.x] = 0;
  if (threadIdx.x == 0) sm[0] = -1;
  __syncthreads();
  for (int r = threadIdx.x; r < n; r += kThreads) {
    const int l = level(r);
    if (r < kLevelCache) lev[r] = static_cast<uint8_t>(l + 1);
    if (l >= 0) atomicAdd(&cnt[l], 1);
  }
  __syncthreads();
  int all = 0;
  for (int l = 0; l < kCostLevels; ++l) all += cnt[l];
  *total = all;
  int lv = kCostLevels - 1, t = i;
  while (lv >= 0 && t >= cnt[lv]) t -= cnt[lv--];
  if (lv < 0) return -1;
  // the t-th task of level lv, in task order
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  int base = 0;
  for (int r0 = 0; r0 < n; r0 += kThreads) {
    const int r = r0 + static_cast<int>(threadIdx.x);
    const bool f = r < n && (r < kLevelCache ? static_cast<int>(lev[r]) - 1 : level(r)) == lv;
    const unsigned b = __ballot_sync(0xffffffffu, f);
    if (lane == 0) wsum[warp] = __popc(b);
    __syncthreads();
    int before = base + __popc(b & ((1u << lane) - 1u)), total = 0;
    for (int w = 0; w < kWarps; ++w) {
      if (w < warp) before += wsum[w];
      total += wsum[w];
    }
    if (f && before == t) sm[0] = r;
    __syncthreads();
    base += total;
    if (base > t) break;  // the same for every thread
  }
  return sm[0];
}

// Tree calls with a stated node count, launches without the ordering: the
// number of tasks with work (a request's nodes, or one for a request with a
// node count outside [1, max_nodes]), summed over the block.  sm[1] is
// scratch.  Every thread calls it.
__device__ int tree_task_count(const KArgs& a, int32_t* sm) {
  const int width = a.max_draft + 1;
  const int R = a.num_tasks / width;
  if (threadIdx.x == 0) sm[1] = 0;
  __syncthreads();
  int s = 0;
  for (int i = threadIdx.x; i < R; i += kThreads) {
    const int32_t k = a.draft_offsets[i + 1] - a.draft_offsets[i] - 1;
    s += (k < 0 || k > a.max_draft) ? 1 : k + 1;
  }
  if (s) atomicAdd(sm + 1, s);
  __syncthreads();
  const int total = sm[1];
  __syncthreads();
  return total;
}

// A stated node count that is not the offsets' sum: every request reports
// SS_ROW_BAD_PARAM (tokens and path -1, none accepted).  The first cluster's
// rank 0 alone, every thread; nothing else of the call runs.
__device__ void report_bad_tree_count(const KArgs& a) {
  asm volatile("griddepcontrol.wait;" ::: "memory");  // the previous call has finished
  const int width = a.max_draft + 1;
  const int R = a.num_tasks / width;
  for (int64_t e = threadIdx.x; e < static_cast<int64_t>(R) * width; e += kThreads) {
    a.out_token[e] = -1;
    if (a.out_path) a.out_path[e] = -1;
  }
  for (int i = threadIdx.x; i < R; i += kThreads) {
    a.out_num_accepted[i] = 0;
    a.out_status[i] = SS_ROW_BAD_PARAM;
  }
}

// Head of a row's shard record (followed by shard_cap (y, token) entries).
struct ShardHead {
  int32_t status;  // the shard's row status (EMPTY_SET: no allowed token here)
  int32_t kind;    // 0 greedy (m, arg), 1 draw (best, best_token), 2 list
  int32_t count;   // allowed tokens in the shard
  int32_t n;       // list entries written
  float m;         // largest processed logit (greedy: logit)
  int32_t arg;     // its lowest token id
  float best;      // draw: largest y + g of the shard
  int32_t best_token;
};
static_assert(sizeof(ShardHead) == 32, "shard record head is 32 bytes");
constexpr int kShardGreedy = 0, kShardDraw = 1, kShardList = 2;

// Per-CTA state in (static) shared memory, visible to every device function.
struct Ctx {
  // regions of the dynamic shared memory
  uint8_t* data;
  __nv_bfloat16* vmax;
  uint32_t* xm;
  int32_t* hkey;
  int32_t* hcnt;
  float* hval;
  uint8_t* work;
  uint32_t* rh_cnt[2];  // [rank][bucket], by step parity
  unsigned long long* rh_mass[2];
  LevelRec* rec;
  uint8_t* red;
  Part* part;  // [slot][rank]
  uint64_t* mbar;
  int32_t ncta, rank;
  // task
  int32_t row, req, j, k, d0, drow, x;
  int32_t bad_k;  // request's draft count outside [0, max_draft]
  int32_t greedy, top_k, use_mask, want_s;
  float temperature, inv_t, top_p, min_p, rep, freq, pres;
  uint32_t seed_lo, seed_hi, pos;
  uint32_t rowid;  // Philox counter word 2
  int32_t h0, h1, b0, b1;
  int32_t lo, n;  // slice start token, tokens in this slice
  int32_t status;
  // after stage 1
  float m, ymin, s_all;
  int32_t arg, count;
  // broadcast slots
  Part fold;
  SelPass sel;
  Loc loc;
  int32_t pick;
  uint32_t cursor[2];      // gather slot cursors (used in rank 0), by step parity
  uint32_t vcount;         // vectors found by for_vectors_above
  int32_t vlist_cap;       // entries of its index list (the exclusion-bitmap region)
  float kabs[kMaxLevels];  // absolute bucket of the top-k cut at each level
  int32_t cut_on, cut_idx, cut_len;
  uint32_t cut_key;
  // tree verification: the node's depth, the request's node count, the
  // node's children (local index, token) in index order
  int32_t depth, nn, nkids;
  int32_t kid_node[kTreeMaxNodes];
  int32_t kid_tok[kTreeMaxNodes];
};

extern __shared__ __align__(128) uint8_t smem_raw[];
__shared__ Ctx g;

__device__ __forceinline__ float vec_bound(int v) {
  return __uint_as_float(static_cast<uint32_t>(__bfloat16_as_ushort(g.vmax[v])) << 16);
}

// fp32 -> bf16 rounded toward +inf, by integer arithmetic on the bits
// (NaN stays NaN, +inf and -inf stay put).
__device__ __forceinline__ __nv_bfloat16 bf16_round_up(float x) {
  const uint32_t b = __float_as_uint(x);
  uint32_t h = (b & 0x80000000u) ? (b >> 16) : ((b + 0xffffu) >> 16);
  if (x != x) h = 0x7fc0u;
  return __ushort_as_bfloat16(static_cast<unsigned short>(h));
}

// ------------------------------------------------------------- dtype glue --

template <int DT>
struct Vec;

template <>
struct Vec<SS_DTYPE_F32> {
  static constexpr int kPer = 4;
  static constexpr int kBytes = 4;
  __device__ static __forceinline__ void unpack(const uint4 v, float (&z)[4]) {
    z[0] = __uint_as_float(v.x);
    z[1] = __uint_as_float(v.y);
    z[2] = __uint_as_float(v.z);
    z[3] = __uint_as_float(v.w);
  }
  // Replace lanes whose bit is set in `bits` by -inf.
  __device__ static __forceinline__ uint4 exclude(uint4 v, uint32_t bits) {
    if (bits & 1u) v.x = 0xff800000u;
    if (bits & 2u) v.y = 0xff800000u;
    if (bits & 4u) v.z = 0xff800000u;
    if (bits & 8u) v.w = 0xff800000u;
    return v;
  }
  __device__ static __forceinline__ float load_global(const void* row, int64_t t) {
    return reinterpret_cast<const float*>(row)[t];
  }
  __device__ static __forceinline__ float load_smem(const uint8_t* data, int e) {
    return reinterpret_cast<const float*>(data)[e];
  }
};

template <>
struct Vec<SS_DTYPE_BF16> {
  static constexpr int kPer = 8;
  static constexpr int kBytes = 2;
  __device__ static __forceinline__ void unpack(const uint4 v, float (&z)[8]) {
    z[0] = __uint_as_float(v.x << 16);
    z[1] = __uint_as_float(v.x & 0xffff0000u);
    z[2] = __uint_as_float(v.y << 16);
    z[3] = __uint_as_float(v.y & 0xffff0000u);
    z[4] = __uint_as_float(v.z << 16);
    z[5] = __uint_as_float(v.z & 0xffff0000u);
    z[6] = __uint_as_float(v.w << 16);
    z[7] = __uint_as_float(v.w & 0xffff0000u);
  }
  __device__ static __forceinline__ uint32_t excl_pair(uint32_t w, uint32_t two) {
    if (two & 1u) w = (w & 0xffff0000u) | 0x0000ff80u;
    if (two & 2u) w = (w & 0x0000ffffu) | 0xff800000u;
    return w;
  }
  __device__ static __forceinline__ uint4 exclude(uint4 v, uint32_t bits) {
    v.x = excl_pair(v.x, bits);
    v.y = excl_pair(v.y, bits >> 2);
    v.z = excl_pair(v.z, bits >> 4);
    v.w = excl_pair(v.w, bits >> 6);
    return v;
  }
  __device__ static __forceinline__ float load_global(const void* row, int64_t t) {
    const uint16_t h = reinterpret_cast<const uint16_t*>(row)[t];
    return __uint_as_float(static_cast<uint32_t>(h) << 16);
  }
  __device__ static __forceinline__ float load_smem(const uint8_t* data, int e) {
    return __uint_as_float(static_cast<uint32_t>(reinterpret_cast<const uint16_t*>(data)[e]) << 16);
  }
};

// --------------------------------------------------------- reductions --

__device__ __forceinline__ bool beats(float v, int32_t i, float bv, int32_t bi) {
  return v > bv || (v == bv && i < bi);
}

// Merge of two online-softmax pairs (sum of exp(y - smax)).
__device__ __forceinline__ void softmax_merge(float& m1, float& s1, float m2, float s2) {
  if (m2 == neg_inf()) return;
  if (m1 == neg_inf()) {
    m1 = m2;
    s1 = s2;
    return;
  }
  const float M = fmaxf(m1, m2);
  s1 = __fadd_rn(__fmul_rn(s1, __expf(m1 - M)), __fmul_rn(s2, __expf(m2 - M)));
  m1 = M;
}

__device__ __forceinline__ Part empty_part() {
  Part p{};
  p.best = neg_inf();
  p.arg = kNoCut;
  p.ymin = pos_inf();
  p.xy = neg_inf();
  p.smax = neg_inf();
  return p;
}

// Combines the partials of the 32 lanes; every lane ends with the total.
// Integer fields use the warp reduction instructions (order-free); floats are
// compared through their order-preserving keys (-0 folded into +0 so that it
// ties with +0, as in a float comparison); the softmax sums are rescaled to the
// common max and added in an xor butterfly, which gives every lane the same
// bits.  Deterministic for a given assignment of partials to lanes.
__device__ __forceinline__ void warp_part_reduce(Part& p) {
  constexpr uint32_t kAll = 0xffffffffu;
  const uint32_t kb = order_key(p.best + 0.0f);
  const uint32_t kmax = __reduce_max_sync(kAll, kb);
  p.arg = static_cast<int32_t>(__reduce_min_sync(kAll, kb == kmax ? static_cast<uint32_t>(p.arg) : 0xffffffffu));
  p.best = key_value(kmax);
  p.count = static_cast<int32_t>(__reduce_add_sync(kAll, static_cast<uint32_t>(p.count)));
  p.status = static_cast<int32_t>(__reduce_max_sync(kAll, static_cast<uint32_t>(p.status)));
  p.ymin = key_value(__reduce_min_sync(kAll, order_key(p.ymin + 0.0f)));
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) p.mass += __shfl_xor_sync(kAll, p.mass, off);
  const float M = key_value(__reduce_max_sync(kAll, order_key(p.smax + 0.0f)));
  float sum = (p.smax == neg_inf()) ? 0.0f : __fmul_rn(p.ssum, __expf(p.smax - M));
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) sum = __fadd_rn(sum, __shfl_xor_sync(kAll, sum, off));
  p.smax = M;
  p.ssum = sum;
  const uint32_t holders = __ballot_sync(kAll, p.xhere != 0);
  if (holders) {
    p.xy = __shfl_sync(kAll, p.xy, __ffs(holders) - 1);
    p.xhere = 1;
  }
}

// Reduces every thread's partial over the block and then over the cluster:
// warp totals go to shared memory, warp 0 combines them, its lanes write the
// CTA total into slot `slot` of every CTA, one cluster barrier, and warp 0
// combines the C totals.  The result lands in g.fold (identical in every CTA).
// Called by all threads.
__device__ __noinline__ void reduce_fold(int slot, float best, int32_t arg, int32_t count, int32_t status,
                                         unsigned long long mass, float ymin, float smax, float ssum, float xy,
                                         int32_t xhere) {
  Part p;
  p.best = best;
  p.arg = arg;
  p.count = count;
  p.status = status;
  p.mass = mass;
  p.ymin = ymin;
  p.xy = xy;
  p.xhere = xhere;
  p.smax = smax;
  p.ssum = ssum;
  warp_part_reduce(p);
  Part* w = reinterpret_cast<Part*>(g.red);
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  __syncthreads();  // the previous user of g.red is done
  if (lane == 0) w[wid] = p;
  __syncthreads();
  cg::cluster_group cl = cg::this_cluster();
  const int n = g.ncta;
  if (wid == 0) {
    Part t = (lane < kWarps) ? w[lane] : empty_part();
    warp_part_reduce(t);
    if (lane < n) *cl.map_shared_rank(g.part + slot * n + g.rank, lane) = t;
  }
  cl.sync();
  if (wid == 0) {
    Part t = (lane < n) ? g.part[slot * n + lane] : empty_part();
    warp_part_reduce(t);
    if (lane == 0) g.fold = t;
  }
  __syncthreads();
}
static_assert((kWarps + 1) * sizeof(Part) <= kRedBytes, "reduction scratch too small");
static_assert(kWarps * sizeof(unsigned long long) <= kRedBytes, "scan scratch too small");
static_assert(kListCap % kThreads == 0, "list runs");

// ------------------------------------------------- bucket refinement --

// Folds the lane-private histogram copies in the work region, writes the
// CTA's totals into every CTA (buffer of this step's parity), one cluster
// barrier, and merges the C totals in rank order into `out`.
__device__ __forceinline__ void push_merge(LevelRec* out, float scale, float base, int step) {
  cg::cluster_group cl = cg::this_cluster();
  const uint32_t* hc = reinterpret_cast<const uint32_t*>(g.work);
  const uint32_t* hmh = hc + kHistRows * kCopies;
  const uint32_t* hml = hmh + kHistRows * kCopies;
  const int tid = threadIdx.x;
  const int par = step & 1;
  __syncthreads();
  if (tid < kBuckets * 4) {  // 4 threads per bucket, each folds 4 copies
    const int b = tid >> 2, q = tid & 3;
    uint32_t cnt = 0;
    unsigned long long mass = 0;
#pragma unroll
    for (int i = 0; i < kCopies / 4; ++i) {
      const int k = b * kCopies + q * (kCopies / 4) + i;
      cnt += hc[k];
      mass += (static_cast<unsigned long long>(hmh[k]) << kMassSplit) + hml[k];
    }
    cnt += __shfl_xor_sync(0xffffffffu, cnt, 1);
    cnt += __shfl_xor_sync(0xffffffffu, cnt, 2);
    mass += __shfl_xor_sync(0xffffffffu, mass, 1);
    mass += __shfl_xor_sync(0xffffffffu, mass, 2);
    // the 4 threads of a bucket hold its total: each writes it into every
    // fourth CTA of the cluster
    for (int r = q; r < g.ncta; r += 4) {
      *cl.map_shared_rank(g.rh_cnt[par] + g.rank * kBuckets + b, r) = cnt;
      *cl.map_shared_rank(g.rh_mass[par] + g.rank * kBuckets + b, r) = mass;
    }
  }
  cl.sync();
  if (tid < kBuckets) {
    uint32_t cnt = 0;
    unsigned long long mass = 0;
    for (int r = 0; r < g.ncta; ++r) {
      cnt += g.rh_cnt[par][r * kBuckets + tid];
      mass += g.rh_mass[par][r * kBuckets + tid];
    }
    out->cnt[tid] = cnt;
    out->mass[tid] = mass;
  }
  if (tid == 0) {
    out->scale = scale;
    out->base = base;
  }
  __syncthreads();
}

// Visits the vectors whose bound reaches `lo` (v < nvec), densely: one scan
// of the bounds records each thread's passing vectors in a bit mask (vector
// tid + j * kThreads is bit j); when they fit, their indices are compacted
// into the exclusion-bitmap region (free once stage 1 is done) so that every
// lane of a warp has a vector, rather than the few whose vector passes while
// the rest idle through the same instructions; when more pass, the slice is
// walked with the masks.  Every thread calls f(v) the same number of times,
// v = -1 for none, so f may use warp-collective operations.  Called by all
// threads.
template <int DT, typename F>
__device__ __forceinline__ void for_vectors_above(float lo, F&& f) {
  using V = Vec<DT>;
  static_assert(kMaxSliceTokens / 4 <= 32 * kThreads, "one mask bit per vector and thread");
  const int nvec = (g.n + V::kPer - 1) / V::kPer;
  const int iters = (nvec + kThreads - 1) / kThreads;
  uint16_t* list = reinterpret_cast<uint16_t*>(g.xm);
  const uint32_t cap = static_cast<uint32_t>(g.vlist_cap);
  const int lane = threadIdx.x & 31;
  __syncthreads();  // the previous call's readers are done
  if (threadIdx.x == 0) g.vcount = 0;
  // the bounds as raw bf16 bits: with the pointer hoisted and the loop
  // unrolled, the loads of several iterations are in flight together
  const unsigned short* __restrict__ vb = reinterpret_cast<const unsigned short*>(g.vmax);
  uint32_t bits = 0;
#pragma unroll 8
  for (int j = 0; j < iters; ++j) {
    const int v = j * kThreads + static_cast<int>(threadIdx.x);
    if (v < nvec && __uint_as_float(static_cast<uint32_t>(vb[v]) << 16) >= lo) bits |= 1u << j;
  }
  const uint32_t mine = static_cast<uint32_t>(__popc(bits));
  uint32_t incl = mine;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const uint32_t t = __shfl_up_sync(0xffffffffu, incl, off);
    if (lane >= off) incl += t;
  }
  __syncthreads();  // vcount reset is visible
  uint32_t at = 0;
  if (lane == 31 && incl) at = atomicAdd(&g.vcount, incl);
  at = __shfl_sync(0xffffffffu, at, 31) + incl - mine;
  __syncthreads();
  const uint32_t total = g.vcount;
  if (total <= cap) {
    for (uint32_t r = bits; r; r &= r - 1u) list[at++] = static_cast<uint16_t>((__ffs(r) - 1) * kThreads + threadIdx.x);
    __syncthreads();
    for (uint32_t b = 0; b < total; b += kThreads) {
      const uint32_t i = b + threadIdx.x;
      f(i < total ? static_cast<int>(list[i]) : -1);
    }
  } else {
    for (int j = 0; j < iters; ++j) f(((bits >> j) & 1u) ? j * kThreads + static_cast<int>(threadIdx.x) : -1);
  }
}

// Histogram entry of y: counter row of its bucket when that lies in
// [base, base + 64), else the spill row kBuckets, so that every entry issues
// the same instructions (a per-entry branch around the atomics costs far more
// than the spilled atomics).  y = -inf lands in the spill row.
__device__ __forceinline__ int hist_slot(float y, float scale, float ms, int base, int copy) {
  const int b = bucket_index(y, scale, ms) - base;
  return (static_cast<uint32_t>(b) < static_cast<uint32_t>(kBuckets) ? b : kBuckets) * kCopies + copy;
}

// Counts, and with kMass the fixed-point masses split into a high and a low
// half (32-bit shared atomics; the 64-bit ones are several times slower).
template <bool kMass>
__device__ __forceinline__ void hist_add(uint32_t* hc, float m, float y, float scale, float ms, int base, int copy) {
  const int k = hist_slot(y, scale, ms, base, copy);
  atomicAdd(hc + k, 1u);
  if (kMass) {
    uint32_t hi, lo;
    fixed_mass_parts(y, m, hi, lo);  // 0 for y = -inf
    atomicAdd(hc + kHistRows * kCopies + k, hi);
    atomicAdd(hc + 2 * kHistRows * kCopies + k, lo);
  }
}

// Token level: every token of the vectors whose bound reaches lo_y, and the
// patched tokens at or above lo_y.
template <int DT, bool kMass>
__device__ __forceinline__ void hist_tokens(uint32_t* hc, float scale, float base, float lo_y, int copy) {
  using V = Vec<DT>;
  const int nvec = (g.n + V::kPer - 1) / V::kPer;
  const uint4* __restrict__ data = reinterpret_cast<const uint4*>(g.data);
  const float m = g.m, inv_t = g.inv_t, ms = __fmul_rn(g.m, scale);
  const int ib = small_int(base);
  for_vectors_above<DT>(lo_y, [&](int v) {
    if (v < 0) return;
    float z[V::kPer];
    V::unpack(data[v], z);
#pragma unroll
    for (int e = 0; e < V::kPer; ++e) hist_add<kMass>(hc, m, __fmul_rn(z[e], inv_t), scale, ms, ib, copy);
  });
  for (int s = threadIdx.x; s < kHashCap; s += kThreads) {
    const float y = g.hval[s];
    hist_add<kMass>(hc, m, (g.hkey[s] >= 0 && y >= lo_y) ? y : neg_inf(), scale, ms, ib, copy);
  }
}

// Tile level (base 0): one entry per 16-byte vector valued at a lower bound
// of its largest processed logit, one per patched token; k entries at or
// above a bucket imply k tokens there, and their masses bound the tokens'
// mass from below.
template <bool kMass>
__device__ __forceinline__ void hist_tiles(uint32_t* hc, float scale, int nvec, int copy) {
  const float m = g.m, ms = __fmul_rn(g.m, scale);
  constexpr int kB = 8;  // independent loads first, then the atomics
  for (int v0 = threadIdx.x; v0 < nvec; v0 += kThreads * kB) {
    float ub[kB];
#pragma unroll
    for (int u = 0; u < kB; ++u) {
      const int v = v0 + u * kThreads;
      ub[u] = (v < nvec) ? vec_bound(v) : neg_inf();
    }
    // the stored bound is rounded up to bf16: one bf16 step below is <= the max
#pragma unroll
    for (int u = 0; u < kB; ++u)
      hist_add<kMass>(hc, m, fminf(ub[u] - fabsf(ub[u]) * 0.0078125f - 1e-30f, m), scale, ms, 0, copy);
  }
  for (int s = threadIdx.x; s < kHashCap; s += kThreads)
    hist_add<kMass>(hc, m, g.hkey[s] >= 0 ? g.hval[s] : neg_inf(), scale, ms, 0, copy);
}

// Histogram into `out`: token level (tile = 0) of the buckets
// [base, base + 64) at `scale`, skipping vectors whose bound is below lo_y, or
// tile level (tile = 1).
template <int DT>
__device__ __noinline__ void hist_pass(int tile, float scale, float base, int need_mass, float lo_y, int step,
                                       LevelRec* out) {
  using V = Vec<DT>;
  uint32_t* hc = reinterpret_cast<uint32_t*>(g.work);
  const int tid = threadIdx.x;
  for (int i = tid; i < 3 * kHistRows * kCopies; i += kThreads) hc[i] = 0;
  __syncthreads();
  const int copy = tid & (kCopies - 1);
  if (tile) {
    const int nvec = (g.n + V::kPer - 1) / V::kPer;
    if (need_mass)
      hist_tiles<true>(hc, scale, nvec, copy);
    else
      hist_tiles<false>(hc, scale, nvec, copy);
  } else if (need_mass) {
    hist_tokens<DT, true>(hc, scale, base, lo_y, copy);
  } else {
    hist_tokens<DT, false>(hc, scale, base, lo_y, copy);
  }
  push_merge(out, scale, base, step);
}

// Bucket of `r` where the running count (or mass) from the top first reaches
// `target`; warp 0 computes, the result lands in g.loc.
__device__ __noinline__ void locate(const LevelRec* r, int by_mass, unsigned long long target, uint32_t above_c,
                                    unsigned long long above_m) {
  if (threadIdx.x < 32) {
    const int lane = threadIdx.x;
    const uint32_t c0 = r->cnt[2 * lane], c1 = r->cnt[2 * lane + 1];
    const unsigned long long m0 = r->mass[2 * lane], m1 = r->mass[2 * lane + 1];
    uint32_t ic = c0 + c1;
    unsigned long long im = m0 + m1;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const uint32_t oc = __shfl_up_sync(0xffffffffu, ic, off);
      const unsigned long long om = __shfl_up_sync(0xffffffffu, im, off);
      if (lane >= off) {
        ic += oc;
        im += om;
      }
    }
    const uint32_t ec = ic - c0 - c1;
    const unsigned long long em = im - m0 - m1;
    const bool hit_all = by_mass ? (above_m + im >= target) : (static_cast<unsigned long long>(above_c + ic) >= target);
    const bool hit_one =
        by_mass ? (above_m + em + m0 >= target) : (static_cast<unsigned long long>(above_c + ec + c0) >= target);
    const unsigned ball = __ballot_sync(0xffffffffu, hit_all);
    if (lane == 0 && !ball) g.loc = Loc{0, 0, 0, 0, 0};
    if (ball && lane == __ffs(ball) - 1) {
      Loc l;
      l.found = 1;
      l.pad = 0;
      if (hit_one) {
        l.bucket = 2 * lane;
        l.cnt_before = ec;
        l.mass_before = em;
      } else {
        l.bucket = 2 * lane + 1;
        l.cnt_before = ec + c0;
        l.mass_before = em + m0;
      }
      g.loc = l;
    }
  }
  __syncthreads();
}

// Gathers every token of bucket `abs` at `scale` into every CTA's list (the
// buffer of this step's parity).
// Appends the entries flagged in `hits` (bit e: token t0 + e, logit y[e]) of
// every lane of the warp to the cluster's list: one slot reservation per warp
// at the cursor in rank 0, then each lane writes its entries into every CTA.
// Called by all 32 lanes.
template <int N>
__device__ __forceinline__ void warp_append(uint32_t hits, const float (&y)[N], int32_t t0, uint32_t* cursor,
                                            unsigned long long* list) {
  cg::cluster_group cl = cg::this_cluster();
  const int lane = threadIdx.x & 31;
  const uint32_t nh = static_cast<uint32_t>(__popc(hits));
  uint32_t incl = nh;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const uint32_t t = __shfl_up_sync(0xffffffffu, incl, off);
    if (lane >= off) incl += t;
  }
  const uint32_t total = __shfl_sync(0xffffffffu, incl, 31);
  uint32_t base = 0;
  if (lane == 0) base = atomicAdd(cursor, total);
  uint32_t slot = __shfl_sync(0xffffffffu, base, 0) + incl - nh;
  const int ncta = g.ncta;
#pragma unroll
  for (int e = 0; e < N; ++e) {
    if ((hits >> e) & 1u) {
      if (slot < static_cast<uint32_t>(kListCap)) {
        const unsigned long long k = sort_key(y[e], t0 + e);
        for (int r = 0; r < ncta; ++r) *cl.map_shared_rank(list + slot, r) = k;
      }
      ++slot;
    }
  }
}

// Gathers the tokens of absolute bucket `abs` at `scale` (their logits are at
// least lo_y) into every CTA's list of this step's parity; the count is known
// from the histogram.
template <int DT>
__device__ __noinline__ void gather_pass(float scale, float abs, float lo_y, int step) {
  using V = Vec<DT>;
  cg::cluster_group cl = cg::this_cluster();
  const int par = step & 1;
  unsigned long long* list = reinterpret_cast<unsigned long long*>(g.work) + par * kListCap;
  uint32_t* cursor = cl.map_shared_rank(&g.cursor[par], 0);
  const float inv_t = g.inv_t, ms = __fmul_rn(g.m, scale);
  const int ia = small_int(abs);
  const int nvec = (g.n + V::kPer - 1) / V::kPer;
  const uint4* data = reinterpret_cast<const uint4*>(g.data);
  const int lo = g.lo;
  // every thread makes the same number of calls (warp-collective appends)
  for_vectors_above<DT>(lo_y, [&](int v) {
    float y[V::kPer];
    uint32_t hits = 0;
    if (v >= 0) {
      float z[V::kPer];
      V::unpack(data[v], z);
#pragma unroll
      for (int e = 0; e < V::kPer; ++e) {
        y[e] = __fmul_rn(z[e], inv_t);
        hits |= static_cast<uint32_t>(bucket_index(y[e], scale, ms) == ia) << e;  // -inf: never
      }
    }
    if (__any_sync(0xffffffffu, hits != 0)) warp_append<V::kPer>(hits, y, lo + v * V::kPer, cursor, list);
  });
  for (int sb = 0; sb < kHashCap; sb += kThreads) {
    const int s = sb + static_cast<int>(threadIdx.x);
    const int32_t t = g.hkey[s];
    float y[1] = {g.hval[s]};
    const uint32_t hit = (t >= 0 && y[0] >= lo_y && bucket_index(y[0], scale, ms) == ia) ? 1u : 0u;
    if (__any_sync(0xffffffffu, hit != 0)) warp_append<1>(hit, y, t, cursor, list);
  }
  cl.sync();
  if (g.rank == 0 && threadIdx.x == 0) g.cursor[par] = 0;  // its next use is two steps away
}

// Sorts list[0..n) ascending in place (n <= kListCap) and writes the
// inclusive prefix sums of the fixed-point masses to `pre`.
__device__ __noinline__ void sort_and_scan(unsigned long long* list, int n, unsigned long long* pre) {
  // Rank sort: the keys are distinct (a token is gathered once), so the
  // position of an entry is the number of smaller keys.  One pass of
  // broadcast reads and a single barrier, instead of the log^2 barriers of
  // a sorting network.
  const int tid = threadIdx.x;
  constexpr int kMine = (kListCap + kThreads - 1) / kThreads;
  unsigned long long key[kMine];
  int rank[kMine];
#pragma unroll
  for (int r = 0; r < kMine; ++r) {
    const int i = tid + r * kThreads;
    key[r] = (i < n) ? list[i] : 0ull;
    rank[r] = 0;
  }
  if (tid < n) {
    int j = 0;
    for (; j + 4 <= n; j += 4) {
      const unsigned long long b0 = list[j], b1 = list[j + 1], b2 = list[j + 2], b3 = list[j + 3];
#pragma unroll
      for (int r = 0; r < kMine; ++r)
        rank[r] += static_cast<int>(b0 < key[r]) + static_cast<int>(b1 < key[r]) + static_cast<int>(b2 < key[r]) +
                   static_cast<int>(b3 < key[r]);
    }
    for (; j < n; ++j) {
      const unsigned long long b = list[j];
#pragma unroll
      for (int r = 0; r < kMine; ++r) rank[r] += static_cast<int>(b < key[r]);
    }
  }
  __syncthreads();
#pragma unroll
  for (int r = 0; r < kMine; ++r)
    if (tid + r * kThreads < n) list[rank[r]] = key[r];
  __syncthreads();
  // inclusive scan of masses in sorted order: each thread owns a run
  constexpr int kPer = kListCap / kThreads;
  const float m = g.m;
  unsigned long long run[kPer];
  unsigned long long tot = 0;
#pragma unroll
  for (int r = 0; r < kPer; ++r) {
    const int i = tid * kPer + r;
    run[r] = (i < n) ? fixed_mass(key_value(sort_key_order(list[i])), m) : 0ull;
    tot += run[r];
  }
  const int lane = tid & 31, wid = tid >> 5;
  unsigned long long x = tot;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const unsigned long long y = __shfl_up_sync(0xffffffffu, x, off);
    if (lane >= off) x += y;
  }
  unsigned long long* ws = reinterpret_cast<unsigned long long*>(g.red);
  if (lane == 31) ws[wid] = x;
  __syncthreads();
  if (wid == 0) {
    unsigned long long y = (lane < kWarps) ? ws[lane] : 0ull;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const unsigned long long z = __shfl_up_sync(0xffffffffu, y, off);
      if (lane >= off) y += z;
    }
    if (lane < kWarps) ws[lane] = y;
  }
  __syncthreads();
  unsigned long long acc = x - tot + ((wid > 0) ? ws[wid - 1] : 0ull);  // exclusive prefix of this run
#pragma unroll
  for (int r = 0; r < kPer; ++r) {
    const int i = tid * kPer + r;
    acc += run[r];
    if (i < n) pre[i] = acc;
  }
  __syncthreads();
}

// First position i in [0, limit] where above + pre[i] >= target (limit when
// none), computed by all threads cooperatively.
__device__ __noinline__ int first_reaching(const unsigned long long* pre, int limit, unsigned long long above,
                                           unsigned long long target) {
  const int tid = threadIdx.x;
  if (tid == 0) g.pick = limit;
  __syncthreads();
  for (int i = tid; i <= limit; i += kThreads) {
    const bool here = above + pre[i] >= target;
    const bool before = i > 0 && above + pre[i - 1] >= target;
    if (here && !before) g.pick = i;
  }
  __syncthreads();
  const int p = g.pick;
  __syncthreads();
  return p;
}

// --------------------------------------------------- fallback selection --

// Buffers of the fallback selection inside the work region.
__device__ __forceinline__ uint32_t* fb_cnt(int buf) { return reinterpret_cast<uint32_t*>(g.work) + 256 * buf; }
__device__ __forceinline__ unsigned long long* fb_mass(int buf) {
  return reinterpret_cast<unsigned long long*>(g.work + 2048) + 256 * buf;
}
__device__ __forceinline__ uint32_t* fb_mcnt() { return reinterpret_cast<uint32_t*>(g.work + 6144); }
__device__ __forceinline__ unsigned long long* fb_mmass() { return reinterpret_cast<unsigned long long*>(g.work + 7168); }

// One exact radix selection over the whole slice (4 passes of 8-bit digits
// over a 32-bit key), for rows the bucket refinement cannot resolve; slow.
// Key: order_key(y) (by_index = 0) or ~index (by_index = 1, the tokens of
// key `eq_key` only).  Tokens after the cut (lim_key, lim_idx) are ignored
// when `limited`.  by_mass: where the running fixed-point mass first reaches
// the target (target = ceil(frac * total mass) when frac > 0); otherwise
// where the running count reaches it.  Result in g.sel (digit = final key).
template <int DT>
__device__ __noinline__ uint32_t radix_select(int& pass, int by_index, uint32_t eq_key, int limited, uint32_t lim_key,
                                              int32_t lim_idx, int by_mass, unsigned long long target, float frac,
                                              uint32_t& cnt_gt, uint32_t& cnt_eq, unsigned long long& mass_gt,
                                              unsigned long long& mass_eq, unsigned long long& total,
                                              uint32_t& reached_out) {
  using V = Vec<DT>;
  cg::cluster_group cl = cg::this_cluster();
  const int ncta = g.ncta;
  uint32_t prefix = 0, pmask = 0, base_c = 0, reached_all = 1;
  unsigned long long base_m = 0;
  const float m = g.m;
  for (int level = 0; level < 4; ++level) {
    const int shift = 24 - 8 * level;
    const int buf = pass & 1;
    ++pass;
    uint32_t* hc = fb_cnt(buf);
    unsigned long long* hm = fb_mass(buf);
    for (int b = threadIdx.x; b < 256; b += kThreads) {
      hc[b] = 0;
      hm[b] = 0;
    }
    __syncthreads();
    auto add = [&](int32_t t, float y) {
      const uint32_t ky = order_key(y);
      if (limited && !(ky > lim_key || (ky == lim_key && t <= lim_idx))) return;
      if (by_index && ky != eq_key) return;
      const uint32_t key = by_index ? ~static_cast<uint32_t>(t) : ky;
      if ((key & pmask) != prefix) return;
      const uint32_t d = (key >> shift) & 255u;
      atomicAdd(hc + d, 1u);
      if (by_mass) atomicAdd(hm + d, fixed_mass(y, m));
    };
    const int nvec = (g.n + V::kPer - 1) / V::kPer;
    const uint4* data = reinterpret_cast<const uint4*>(g.data);
    for (int v = threadIdx.x; v < nvec; v += kThreads) {
      float z[V::kPer];
      V::unpack(data[v], z);
#pragma unroll
      for (int e = 0; e < V::kPer; ++e) {
        const float y = __fmul_rn(z[e], g.inv_t);
        if (y != neg_inf()) add(g.lo + v * V::kPer + e, y);
      }
    }
    for (int s = threadIdx.x; s < kHashCap; s += kThreads)
      if (g.hkey[s] >= 0 && g.hval[s] != neg_inf()) add(g.hkey[s], g.hval[s]);
    __syncthreads();
    cl.sync();
    for (int b = threadIdx.x; b < 256; b += kThreads) {
      uint32_t cc = 0;
      unsigned long long mm = 0;
      for (int r = 0; r < ncta; ++r) {
        cc += *cl.map_shared_rank(hc + b, r);
        mm += *cl.map_shared_rank(hm + b, r);
      }
      fb_mcnt()[b] = cc;
      fb_mmass()[b] = mm;
    }
    __syncthreads();
    if (threadIdx.x < 32) {
      const int lane = threadIdx.x;
      uint32_t c8[8];
      unsigned long long m8[8];
      uint32_t cs = 0;
      unsigned long long ms = 0;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int b = 255 - 8 * lane - i;
        c8[i] = fb_mcnt()[b];
        m8[i] = fb_mmass()[b];
        cs += c8[i];
        ms += m8[i];
      }
      uint32_t ic = cs;
      unsigned long long im = ms;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const uint32_t oc = __shfl_up_sync(0xffffffffu, ic, off);
        const unsigned long long om = __shfl_up_sync(0xffffffffu, im, off);
        if (lane >= off) {
          ic += oc;
          im += om;
        }
      }
      const unsigned long long tot_m = __shfl_sync(0xffffffffu, im, 31);
      unsigned long long tgt = target;
      if (level > 0)
        tgt = g.sel.target;
      else if (frac > 0.0f)
        tgt = mass_target(frac, tot_m);
      auto hit = [&](uint32_t cc, unsigned long long mm) {
        return by_mass ? (base_m + mm >= tgt) : (static_cast<unsigned long long>(base_c + cc) >= tgt);
      };
      const unsigned ball = __ballot_sync(0xffffffffu, hit(ic, im));
      const unsigned nz = __ballot_sync(0xffffffffu, cs > 0);
      int L;
      uint32_t reached = 1;
      if (ball) {
        L = __ffs(ball) - 1;
      } else {  // target not reached (rounding): take the last admitted element
        L = nz ? 31 - __clz(nz) : 31;
        reached = 0;
      }
      __syncwarp();
      if (lane == L) {
        uint32_t cc = ic - cs;
        unsigned long long mmv = im - ms;
        int last = 0;
#pragma unroll
        for (int i = 0; i < 8; ++i)
          if (c8[i] > 0) last = i;
        bool done = false;
        int pick = 7;
        uint32_t pc = 0, pcb = 0;
        unsigned long long pm = 0, pmb = 0;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const bool h = reached ? hit(cc + c8[i], mmv + m8[i]) : (i == last);
          if (!done && h) {
            done = true;
            pick = i;
            pc = cc;
            pm = mmv;
            pcb = c8[i];
            pmb = m8[i];
          }
          cc += c8[i];
          mmv += m8[i];
        }
        SelPass sp;
        sp.digit = static_cast<uint32_t>(255 - 8 * L - pick);
        sp.cnt_before = pc;
        sp.cnt_bin = pcb;
        sp.mass_before = pm;
        sp.mass_bin = pmb;
        sp.reached = reached;
        sp.total = tot_m;
        sp.target = tgt;
        g.sel = sp;
      }
    }
    __syncthreads();
    const SelPass sp = g.sel;
    if (level == 0) total = sp.total;  // mass of every admitted element
    prefix |= sp.digit << shift;
    pmask |= 255u << shift;
    base_c += sp.cnt_before;
    base_m += sp.mass_before;
    cnt_eq = sp.cnt_bin;
    mass_eq = sp.mass_bin;
    if (!sp.reached) reached_all = 0;
    __syncthreads();
  }
  cnt_gt = base_c;
  mass_gt = base_m;
  reached_out = reached_all;
  return prefix;
}

// Exact top-k / top-p cut by radix selection over the slice; result in g.cut_*.
template <int DT>
__device__ __noinline__ void fallback_cuts(int k_on, int p_on) {
  int pass = 0;
  uint32_t cnt_gt, cnt_eq, reached;
  unsigned long long mass_gt, mass_eq, total;
  uint32_t k_key = 0;
  int32_t k_idx = kNoCut;
  int on = 0;
  uint32_t cut_key = 0;
  int32_t cut_idx = kNoCut;
  if (k_on) {
    const uint32_t key = radix_select<DT>(pass, 0, 0u, 0, 0u, 0, 0, static_cast<unsigned long long>(g.top_k), 0.0f,
                                          cnt_gt, cnt_eq, mass_gt, mass_eq, total, reached);
    const uint32_t ntie = static_cast<uint32_t>(g.top_k) - cnt_gt;
    int32_t idx = kNoCut;
    if (ntie < cnt_eq) {
      uint32_t a, b, r2;
      unsigned long long c2, d2, e2;
      idx = static_cast<int32_t>(~radix_select<DT>(pass, 1, key, 0, 0u, 0, 0, ntie, 0.0f, a, b, c2, d2, e2, r2));
    }
    k_key = key;
    k_idx = idx;
    on = 1;
    cut_key = key;
    cut_idx = idx;
  }
  if (p_on) {
    const uint32_t key = radix_select<DT>(pass, 0, 0u, k_on, k_key, k_idx, 1, 0ull, g.top_p, cnt_gt, cnt_eq, mass_gt,
                                          mass_eq, total, reached);
    const unsigned long long target = mass_target(g.top_p, total);
    uint32_t ntie = cnt_eq;
    if (reached && cnt_eq > 0) {
      const unsigned long long w = mass_eq / cnt_eq;  // every tie has the same mass
      if (w > 0 && target > mass_gt) {
        const unsigned long long nt = (target - mass_gt + w - 1) / w;
        if (nt < cnt_eq) ntie = static_cast<uint32_t>(nt > 0 ? nt : 1);
      } else if (target <= mass_gt) {
        ntie = 1;
      }
    }
    int32_t idx = kNoCut;
    if (ntie < cnt_eq) {
      uint32_t a, b, r2;
      unsigned long long c2, d2, e2;
      idx = static_cast<int32_t>(~radix_select<DT>(pass, 1, key, k_on, k_key, k_idx, 0, ntie, 0.0f, a, b, c2, d2, e2, r2));
    }
    if (!on || key > cut_key || (key == cut_key && idx < cut_idx)) {
      cut_key = key;
      cut_idx = idx;
    }
    on = 1;
  }
  if (threadIdx.x == 0) {
    g.cut_on = on;
    g.cut_key = cut_key;
    g.cut_idx = cut_idx;
    g.cut_len = -1;
  }
  __syncthreads();
}

// The kept set K = the first `len` tokens of the (y desc, index asc) order,
// ending at (key, idx).
__device__ __forceinline__ void tighten(uint32_t key, int32_t idx, int32_t len) {
  if (threadIdx.x == 0 && (!g.cut_on || key > g.cut_key || (key == g.cut_key && idx < g.cut_idx))) {
    g.cut_key = key;
    g.cut_idx = idx;
    g.cut_len = len;
    g.cut_on = 1;
  }
  __syncthreads();
}

// Refines bucket `abs` at `scale` (refinement level `level`) until it holds at
// most kListCap tokens, following a count or mass target; false if it cannot
// within kMaxLevels.  Updates the bucket description in place.
template <int DT>
__device__ __forceinline__ bool refine(int& step, int& level, float& scale, float& abs, uint32_t& above_c,
                                    unsigned long long& above_m, uint32_t& n, int by_mass, unsigned long long target,
                                    LevelRec* scratch) {
  while (n > static_cast<uint32_t>(kListCap)) {
    if (level >= kMaxLevels) return false;
    const float sub = scale * static_cast<float>(kBuckets);
    hist_pass<DT>(0, sub, abs * static_cast<float>(kBuckets), 1, bucket_floor(g.m, abs, scale), step++, scratch);
    locate(scratch, by_mass, target, above_c, above_m);
    const Loc l = g.loc;
    if (!l.found) return false;
    above_c += l.cnt_before;
    above_m += l.mass_before;
    n = scratch->cnt[l.bucket];
    abs = abs * static_cast<float>(kBuckets) + static_cast<float>(l.bucket);
    scale = sub;
    ++level;
  }
  return true;
}

// Resolves the top-k and top-p cuts of a sampling row into g.cut_*.
template <int DT>
__device__ __noinline__ void resolve_cuts(int k_on, int p_on) {
  const float m = g.m;
  int step = 0;
  bool fallback = false;
  if (threadIdx.x == 0) {
    g.cut_on = 0;
    g.cut_key = 0;
    g.cut_idx = kNoCut;
    g.cut_len = -1;
  }
  // level 1: 64 buckets of a power-of-two width covering [ymin, m]
  const float range = fminf(m - g.ymin, 64.0f);
  float s1 = 1.0f;
  while (s1 < 1048576.0f && s1 * 2.0f * range < 64.0f) s1 *= 2.0f;
  // R[0] level 1, R[1..kMaxLevels-1] the k-chain, R[kRecs-2] scratch, R[kRecs-1] tile level
  LevelRec* R = g.rec;
  LevelRec* RS = R + (kRecs - 2);
  LevelRec* RT = R + (kRecs - 1);

  // Without top-k, top-p needs the row's normaliser: from stage 1, or (top_k
  // asked for but inactive) from an exact pass.
  unsigned long long S_all = 0;
  if (p_on && !k_on) {
    if (g.want_s) {
      S_all = static_cast<unsigned long long>(static_cast<double>(g.s_all) * static_cast<double>(kFixedScale));
    } else {
      using V = Vec<DT>;
      unsigned long long mine = 0;
      const float lo_y = m - kMassCutoff - 1.0f - fabsf(m) * 1e-6f;
      const int nvec = (g.n + V::kPer - 1) / V::kPer;
      const uint4* data = reinterpret_cast<const uint4*>(g.data);
      for_vectors_above<DT>(lo_y, [&](int v) {
        if (v < 0) return;
        float z[V::kPer];
        V::unpack(data[v], z);
#pragma unroll
        for (int e = 0; e < V::kPer; ++e) mine += fixed_mass(__fmul_rn(z[e], g.inv_t), m);  // 0 for -inf
      });
      for (int s = threadIdx.x; s < kHashCap; s += kThreads)
        if (g.hkey[s] >= 0 && g.hval[s] != neg_inf()) mine += fixed_mass(g.hval[s], m);
      reduce_fold(3, neg_inf(), kNoCut, 0, 0, mine, pos_inf(), neg_inf(), 0.0f, neg_inf(), 0);
      S_all = g.fold.mass;
    }
  }
  const unsigned long long T_all = mass_target(g.top_p, S_all);

  // Tile level (two-stage selection): the vector maxima bound the cut from
  // below, so the token histogram only needs the vectors above that bound.
  float lo1 = bucket_floor(m, 63.0f, s1);
  hist_pass<DT>(1, s1, 0.0f, p_on && !k_on, 0.0f, step++, RT);
  locate(RT, !k_on, k_on ? static_cast<unsigned long long>(g.top_k) : T_all, 0, 0);
  if (g.loc.found) {
    lo1 = fmaxf(lo1, bucket_floor(m, static_cast<float>(g.loc.bucket), s1));
    // Every token at or above the cut lies in [lo1, m]: the token level only
    // needs to cover that range, so its 64 buckets can be finer (fewer
    // refinement passes).  (m - lo1) * s1 < 63 keeps lo1 inside bucket 62.
    const float range1 = m - lo1;
    while (s1 < 1048576.0f && s1 * 2.0f * range1 < 63.0f) s1 *= 2.0f;
  }
  hist_pass<DT>(0, s1, 0.0f, p_on, lo1, step++, R);

  // ---- top-k: the k-th token of the order
  unsigned long long S_k = 0;
  int kchain_levels = 0;
  unsigned long long* klist = nullptr;
  unsigned long long* kpre = reinterpret_cast<unsigned long long*>(g.work) + 2 * kListCap;
  int k_pos = -1;
  if (k_on) {
    const unsigned long long target = static_cast<unsigned long long>(g.top_k);
    locate(R, 0, target, 0, 0);
    const Loc l = g.loc;
    if (!l.found) {
      fallback = true;
    } else {
      int level = 1;
      float scale = s1, abs = static_cast<float>(l.bucket);
      uint32_t above_c = l.cnt_before, n_in = R[0].cnt[l.bucket];
      unsigned long long above_m = l.mass_before;
      if (threadIdx.x == 0) g.kabs[0] = abs;
      while (n_in > static_cast<uint32_t>(kListCap)) {
        if (level >= kMaxLevels) {
          fallback = true;
          break;
        }
        const float sub = scale * static_cast<float>(kBuckets);
        hist_pass<DT>(0, sub, abs * static_cast<float>(kBuckets), p_on, bucket_floor(m, abs, scale), step++, R + level);
        locate(R + level, 0, target, above_c, above_m);
        const Loc ll = g.loc;
        if (!ll.found) {
          fallback = true;
          break;
        }
        above_c += ll.cnt_before;
        above_m += ll.mass_before;
        n_in = R[level].cnt[ll.bucket];
        abs = abs * static_cast<float>(kBuckets) + static_cast<float>(ll.bucket);
        scale = sub;
        if (threadIdx.x == 0) g.kabs[level] = abs;
        ++level;
      }
      if (!fallback) {
        kchain_levels = level;
        const int par = step & 1;
        gather_pass<DT>(scale, abs, bucket_floor(m, abs, scale), step++);
        klist = reinterpret_cast<unsigned long long*>(g.work) + par * kListCap;
        sort_and_scan(klist, static_cast<int>(n_in), kpre);
        k_pos = g.top_k - static_cast<int>(above_c) - 1;
        const unsigned long long e = klist[k_pos];
        S_k = above_m + kpre[k_pos];
        tighten(sort_key_order(e), sort_key_token(e), g.top_k);
      }
    }
  }

  // ---- top-p: where the mass of the (top-k) prefix reaches p
  if (p_on && !fallback) {
    const unsigned long long T = k_on ? mass_target(g.top_p, S_k) : T_all;
    int level = 1;
    const LevelRec* rec = R;
    uint32_t above_c = 0;
    unsigned long long above_m = 0;
    float scale = s1, abs = 0.0f;
    while (true) {
      locate(rec, 1, T, above_c, above_m);
      const Loc l = g.loc;
      if (!l.found) {  // the target is not reached within the chain (rounding)
        if (!k_on) fallback = true;
        break;  // with top-k on, K stays the top-k prefix
      }
      abs = rec->base + static_cast<float>(l.bucket);
      above_c += l.cnt_before;
      above_m += l.mass_before;
      if (k_on && level <= kchain_levels && abs == g.kabs[level - 1]) {
        if (level < kchain_levels) {  // follow the k-chain one level down
          rec = R + level;
          scale *= static_cast<float>(kBuckets);
          ++level;
          continue;
        }
        // inside the gathered k bucket: exact, limited to the k-prefix
        const int pos = first_reaching(kpre, k_pos, above_m, T);
        const unsigned long long e = klist[pos];
        tighten(sort_key_order(e), sort_key_token(e), static_cast<int32_t>(above_c) + pos + 1);
        break;
      }
      // a bucket entirely above the k-cut (or no top-k): refine and gather it
      uint32_t n_in = rec->cnt[l.bucket];
      if (!refine<DT>(step, level, scale, abs, above_c, above_m, n_in, 1, T, RS)) {
        fallback = true;
        break;
      }
      const int par = step & 1;
      gather_pass<DT>(scale, abs, bucket_floor(m, abs, scale), step++);
      unsigned long long* plist = reinterpret_cast<unsigned long long*>(g.work) + par * kListCap;
      sort_and_scan(plist, static_cast<int>(n_in), kpre);
      const int pos = first_reaching(kpre, static_cast<int>(n_in) - 1, above_m, T);
      const unsigned long long e = plist[pos];
      tighten(sort_key_order(e), sort_key_token(e), static_cast<int32_t>(above_c) + pos + 1);
      break;
    }
  }
  __syncthreads();
  if (fallback) fallback_cuts<DT>(k_on, p_on);
}

// Processed logit of token t if this CTA holds it (slice or patch table).
template <int DT>
__device__ __forceinline__ bool local_value(int32_t t, float& y) {
  using V = Vec<DT>;
  if (t < g.lo || t >= g.lo + g.n) return false;
  uint32_t h = (static_cast<uint32_t>(t) * 2654435761u) >> kHashShift;
  for (int probe = 0; probe < kHashCap; ++probe) {
    const int32_t k = g.hkey[h];
    if (k == t) {
      y = g.hval[h];
      return true;
    }
    if (k < 0) break;
    h = (h + 1) & (kHashCap - 1);
  }
  const float z = V::load_smem(g.data, t - g.lo);  // -inf when excluded
  y = g.greedy ? z : __fmul_rn(z, g.inv_t);
  return true;
}

__device__ __forceinline__ bool in_kept(int32_t t, float y, float m, int mp_on, float min_p) {
  if (g.cut_on) {
    const uint32_t key = order_key(y);
    if (!(key > g.cut_key || (key == g.cut_key && t <= g.cut_idx))) return false;
  }
  if (mp_on && !(__expf(y - m) >= min_p)) return false;
  return true;
}

// Out-of-line copies of the Gumbel transform and of a single Philox word:
// called from rarely taken branches of hot loops, where an inlined logf pair
// or Philox block per unrolled lane would multiply the code the instruction
// cache has to hold.
__device__ __noinline__ float gumbel_noise(uint32_t num) { return gumbel_from_numerator(num); }
__device__ __noinline__ uint32_t philox_numerator(uint64_t seed, uint32_t row, uint32_t pos, uint32_t token,
                                                  uint32_t stream) {
  return uniform_numerator(philox_word(seed, row, pos, token, stream));
}

// The draw: Gumbel-max over K (stream 0).  Also counts |K| and, for a
// verification position, its fixed-point mass; result in g.fold.
template <int DT, bool kDraw>
__device__ __noinline__ void draw_pass(int mp_on, float k_lo, int prune_best, int spec_pos, int count_k, uint64_t seed) {
  using V = Vec<DT>;
  const float m = g.m, min_p = g.min_p, inv_t = g.inv_t;
  const uint32_t rowid = g.rowid, pos = g.pos;
  const int32_t arg = g.arg;
  // the argmax token is always in K: its score seeds the running best
  const float g0 = kDraw ? gumbel_noise(philox_numerator(seed, rowid, pos, arg, 0)) : 0.0f;
  float bv = __fadd_rn(m, g0);
  int32_t bi = arg;
  int32_t kcount = 0;
  unsigned long long kmass = 0;
  auto element = [&](int32_t t, float y) {
    if (!in_kept(t, y, m, mp_on, min_p)) return;
    ++kcount;
    if (spec_pos) kmass += fixed_mass(y, m);
    if (!kDraw) return;
    const float slack = 1e-3f + fabsf(y) * 1e-6f;
    if (y + kGumbelMax + slack < bv) return;
    const uint32_t num = philox_numerator(seed, rowid, pos, static_cast<uint32_t>(t), 0);
    if (y + gumbel_upper_bound(num) + slack < bv) return;
    const float s = __fadd_rn(y, gumbel_noise(num));
    if (beats(s, t, bv, bi)) {
      bv = s;
      bi = t;
    }
  };
  const int nvec = (g.n + V::kPer - 1) / V::kPer;
  const uint4* data = reinterpret_cast<const uint4*>(g.data);
  const int lo = g.lo;
  const uint32_t key0 = static_cast<uint32_t>(seed), key1 = static_cast<uint32_t>(seed >> 32);
  const bool cut_on = g.cut_on != 0;
  const float yc = key_value(g.cut_key);  // the cut token's logit (when cut_on)
  const int32_t cut_idx = g.cut_idx;
  constexpr int kGroups = V::kPer / 4;  // Philox blocks per vector: 4 tokens share one block
  for_vectors_above<DT>(k_lo, [&](int v) {
    // prune against the best score any lane of the warp has reached (a token
    // below it cannot win); the lane's own best (bv, bi) is what it reports
    const float pb = kDraw ? key_value(__reduce_max_sync(0xffffffffu, order_key(bv))) : 0.0f;
    if (v < 0) return;
    const float ub = vec_bound(v);
    // plain rows need no mass: a vector that cannot beat the best is skipped
    if (prune_best && ub + kGumbelMax + 1e-3f + fabsf(ub) * 1e-6f < pb) return;
    float z[V::kPer];
    V::unpack(data[v], z);
    const int32_t t0 = lo + v * V::kPer;  // a multiple of 4
    // membership in K and candidacy, without a branch per token: y > yc or
    // (y == yc and t <= cut_idx) is the key order of the cut (finite yc, so
    // -inf is never a member); a candidate needs y + G >= pb, tested with a
    // slack that covers every candidate (|y| <= |pb| + 20 for candidates)
    const float cand_lo = pb - kGumbelMax - (1e-3f + (fabsf(pb) + 20.0f) * 1e-6f);
    uint32_t mem = 0, cand = 0;
#pragma unroll
    for (int e = 0; e < V::kPer; ++e) {
      const float y = __fmul_rn(z[e], inv_t);
      z[e] = y;
      bool in = cut_on ? (y > yc || (y == yc && t0 + e <= cut_idx)) : (y != neg_inf());
      if (mp_on) in = in && (__expf(y - m) >= min_p);
      if (count_k) mem |= static_cast<uint32_t>(in) << e;
      cand |= static_cast<uint32_t>(in && y >= cand_lo) << e;
      if (spec_pos) kmass += in ? fixed_mass(y, m) : 0ull;
    }
    kcount += __popc(mem);
    if constexpr (kDraw) {
      if (!cand) return;
      uint32_t w[V::kPer];
#pragma unroll
      for (int q = 0; q < kGroups; ++q) {  // independent blocks: their rounds interleave
        const Philox4 r = philox4x32_10(static_cast<uint32_t>(t0 >> 2) + q, pos, rowid, 0u, key0, key1);
#pragma unroll
        for (int i = 0; i < 4; ++i) w[q * 4 + i] = r.w[i];
      }
      // A candidate can still reach the running best only if its noise
      // g >= pb - y - slack >= d, d taken at the largest candidate logit with a
      // slack that covers every candidate (|y| <= |pb| + 20 for candidates).
      // g increases with u, so that is u >= exp(-exp(-d)): one threshold on
      // the 24-bit numerators per vector, lowered by a margin for the fast
      // exponentials; the exact noise is computed only for the survivors.
      float ymax = neg_inf();
#pragma unroll
      for (int e = 0; e < V::kPer; ++e) ymax = fmaxf(ymax, ((cand >> e) & 1u) ? z[e] : neg_inf());
      const float d = pb - ymax - (1e-3f + (fabsf(pb) + 20.0f) * 1e-6f);
      uint32_t thr = 0;
      if (d > 0.0f) {
        const float u_min = __expf(-__expf(-d));
        thr = __float2uint_rd(fmaxf(u_min * 16777216.0f * (1.0f - 1e-5f) - 4.0f, 0.0f));
      }
      uint32_t live = 0;
#pragma unroll
      for (int e = 0; e < V::kPer; ++e) {
        w[e] = uniform_numerator(w[e]);
        live |= static_cast<uint32_t>(w[e] >= thr) << e;
      }
      live &= cand;
      if (!live) return;
      if (live & (live - 1u)) {
        // several survivors: every lane's noise without branches, so that the
        // independent logf chains overlap
        float sc[V::kPer];
#pragma unroll
        for (int e = 0; e < V::kPer; ++e) sc[e] = __fadd_rn(z[e], gumbel_from_numerator(w[e]));
#pragma unroll
        for (int e = 0; e < V::kPer; ++e)
          if (((live >> e) & 1u) && beats(sc[e], t0 + e, bv, bi)) {
            bv = sc[e];
            bi = t0 + e;
          }
      } else {
        const int e = __ffs(live) - 1;
        float ze = z[0];
        uint32_t we = w[0];
#pragma unroll
        for (int q = 1; q < V::kPer; ++q)
          if (q == e) {
            ze = z[q];
            we = w[q];
          }
        const float sc = __fadd_rn(ze, gumbel_noise(we));
        if (beats(sc, t0 + e, bv, bi)) {
          bv = sc;
          bi = t0 + e;
        }
      }
    }
  });
  for (int s = threadIdx.x; s < kHashCap; s += kThreads) {
    const int32_t t = g.hkey[s];
    const float y = g.hval[s];
    if (t >= 0 && y != neg_inf() && y >= k_lo) element(t, y);
  }
  // the draft token's processed logit, from the CTA that holds it
  float xy = neg_inf();
  int32_t xhere = 0;
  if (spec_pos && threadIdx.x == 0) xhere = local_value<DT>(g.x, xy) ? 1 : 0;
  reduce_fold(1, bv, bi, kcount, 0, kmass, pos_inf(), neg_inf(), 0.0f, xy, xhere);
}

// Sharded top-k row: appends the shard's members of K (the k-cut's prefix,
// or every allowed token when there is no cut) to the row's record as
// (y, token id) pairs; `cursor` counts them (set to 0 at set-up).
template <int DT>
__device__ __noinline__ void emit_members(float2* list, int32_t* cursor, int cap) {
  using V = Vec<DT>;
  const bool cut_on = g.cut_on != 0;
  const float yc = key_value(g.cut_key);
  const int32_t cut_idx = g.cut_idx;
  const float inv_t = g.inv_t;
  const int lo = g.lo;
  const uint4* data = reinterpret_cast<const uint4*>(g.data);
  auto put = [&](int32_t t, float y) {
    const bool in = cut_on ? (y > yc || (y == yc && t <= cut_idx)) : (y != neg_inf());
    if (in) {
      const int i = atomicAdd(cursor, 1);
      if (i < cap) list[i] = make_float2(y, __int_as_float(t));
    }
  };
  for_vectors_above<DT>(cut_on ? yc : neg_inf(), [&](int v) {
    if (v < 0) return;
    float z[V::kPer];
    V::unpack(data[v], z);
#pragma unroll
    for (int e = 0; e < V::kPer; ++e) put(lo + v * V::kPer + e, __fmul_rn(z[e], inv_t));
  });
  for (int s = threadIdx.x; s < kHashCap; s += kThreads) {
    const int32_t t = g.hkey[s];
    if (t >= 0) put(t, g.hval[s]);
  }
  __syncthreads();
}

// Residual max(P - q, 0) at a rejected position: argmax of log r + g over K
// (stream 2); result in g.fold (arg kNoCut when no token has P > q).
template <int DT>
__device__ __noinline__ void residual_pass(int mp_on, float memb_lo, float inv_s, float log_s, const float* qrow,
                                           uint64_t seed, const float* invz, int nz, int slot) {
  using V = Vec<DT>;
  const float m = g.m, min_p = g.min_p, inv_t = g.inv_t;
  const uint32_t rowid = g.rowid, pos = g.pos;
  float bv = neg_inf();
  int32_t bi = kNoCut;
  auto relem = [&](int32_t t, float y) {
    if (!in_kept(t, y, m, mp_on, min_p)) return;
    // log r <= log p_nz <= log P + sum log(1/Z) = y - m - log_s (log_s net of the 1/Z factors)
    if (y - m - log_s + kGumbelMax + 1e-3f + fabsf(y) * 1e-6f < bv) return;
    const float qt = qrow[t];
    float P = __fmul_rn(__expf(y - m), inv_s);
    for (int z = 0; z < nz; ++z) P = __fmul_rn(fmaxf(__fsub_rn(P, qt), 0.0f), invz[z]);
    const float r = __fsub_rn(P, qt);
    if (!(r > 0.0f)) return;
    const uint32_t num = philox_numerator(seed, rowid, pos, static_cast<uint32_t>(t), 2);
    const float s = __fadd_rn(logf(r), gumbel_noise(num));
    if (beats(s, t, bv, bi)) {
      bv = s;
      bi = t;
    }
  };
  const int nvec = (g.n + V::kPer - 1) / V::kPer;
  const uint4* data = reinterpret_cast<const uint4*>(g.data);
  const int lo = g.lo;
  for_vectors_above<DT>(memb_lo, [&](int v) {
    if (v < 0) return;
    const float ub = vec_bound(v);
    if (ub - m - log_s + kGumbelMax + 1e-3f + fabsf(ub) * 1e-6f < bv) return;
    float z[V::kPer];
    V::unpack(data[v], z);
#pragma unroll
    for (int e = 0; e < V::kPer; ++e) {
      const float y = __fmul_rn(z[e], inv_t);
      if (y != neg_inf()) relem(lo + v * V::kPer + e, y);
    }
  });
  for (int s = threadIdx.x; s < kHashCap; s += kThreads) {
    const int32_t t = g.hkey[s];
    const float y = g.hval[s];
    if (t >= 0 && y != neg_inf()) relem(t, y);
  }
  reduce_fold(slot, bv, bi, 0, 0, 0, pos_inf(), neg_inf(), 0.0f, neg_inf(), 0);
}

// Fixed-point sum (2^-40 units) over the kept set of max(p_nz - q, 0), the
// normaliser of the residual after a rejection at a tree node; p_0 = P and
// p_{i+1} = max(p_i - q, 0) / Z_{i+1} (invz holds the 1/Z_i).  The result is
// in g.fold.mass.
template <int DT>
__device__ __noinline__ void tree_mass_pass(int mp_on, float memb_lo, float inv_s, const float* qrow,
                                            const float* invz, int nz, int slot) {
  using V = Vec<DT>;
  const float m = g.m, min_p = g.min_p, inv_t = g.inv_t;
  unsigned long long mass = 0;
  auto melem = [&](int32_t t, float y) {
    if (!in_kept(t, y, m, mp_on, min_p)) return;
    const float qt = qrow[t];
    float P = __fmul_rn(__expf(y - m), inv_s);
    for (int z = 0; z < nz; ++z) P = __fmul_rn(fmaxf(__fsub_rn(P, qt), 0.0f), invz[z]);
    const float r = __fsub_rn(P, qt);
    if (r > 0.0f) mass += static_cast<unsigned long long>(__fmul_rn(fminf(r, 1.0f), 1099511627776.0f));
  };
  const int lo = g.lo;
  const uint4* data = reinterpret_cast<const uint4*>(g.data);
  for_vectors_above<DT>(memb_lo, [&](int v) {
    if (v < 0) return;
    float z[V::kPer];
    V::unpack(data[v], z);
#pragma unroll
    for (int e = 0; e < V::kPer; ++e) {
      const float y = __fmul_rn(z[e], inv_t);
      if (y != neg_inf()) melem(lo + v * V::kPer + e, y);
    }
  });
  for (int s = threadIdx.x; s < kHashCap; s += kThreads) {
    const int32_t t = g.hkey[s];
    const float y = g.hval[s];
    if (t >= 0 && y != neg_inf()) melem(t, y);
  }
  reduce_fold(slot, neg_inf(), kNoCut, 0, 0, mass, pos_inf(), neg_inf(), 0.0f, neg_inf(), 0);
}

// A tree node's children (recursive rejection; "Accelerating Sonar through
// speculation", section "EAGLE", names tree drafts, the rule is a reading):
// child i, drawn from q at this node, is accepted with probability
// min(1, p_i(x)/q(x)), p_0 = P, p_{i+1} = max(p_i - q, 0) / Z_{i+1}; the uniform
// is word i of stream 1 at this node's position.  On the first acceptance
// acc_node is the child's local index; when every child is rejected, token is
// the Gumbel-max draw from max(p_{m-1} - q, 0) (stream 2).  Returns true when
// the token must be the stream-0 draw from P instead (a residual that sums to
// zero, by rounding): the caller draws it.  Every CTA of the cluster takes the
// same decisions (cluster-wide sums).
template <int DT>
__device__ __noinline__ bool tree_children(int mp_on, float memb_lo, float SK, const float* qrow, uint64_t seed,
                                           int32_t& acc_node, int32_t& token) {
  cg::cluster_group cl = cg::this_cluster();
  const int m = g.nkids;
  // the processed logit of every child token, from the CTA whose slice holds
  // it, to every CTA (one writer per entry; the work region is free now)
  float* kid_y = reinterpret_cast<float*>(g.work);
  float* invz = kid_y + kTreeMaxNodes;
  if (threadIdx.x < m) {
    float y;
    if (local_value<DT>(g.kid_tok[threadIdx.x], y))
      for (int r = 0; r < g.ncta; ++r) *cl.map_shared_rank(kid_y + threadIdx.x, r) = y;
  }
  cl.sync();
  const float inv_s = __fdiv_rn(1.0f, SK);
  float log_s = logf(SK);  // net of the 1/Z factors applied so far
  int nz = 0;
  for (int i = 0; i < m; ++i) {
    const int32_t x = g.kid_tok[i];
    const float y = kid_y[i];
    const bool x_in = (y != neg_inf()) && in_kept(x, y, g.m, mp_on, g.min_p);
    const float qx = qrow[x];
    float px = x_in ? __fmul_rn(__expf(y - g.m), inv_s) : 0.0f;
    for (int z = 0; z < nz; ++z) px = __fmul_rn(fmaxf(__fsub_rn(px, qx), 0.0f), invz[z]);
    const float u = uniform_from_numerator(uniform_numerator(philox_word(seed, g.rowid, g.pos, i, 1)));
    if (__fmul_rn(u, qx) < px) {
      acc_node = g.kid_node[i];
      token = x;
      return false;
    }
    // consecutive reductions alternate between two part slots
    const int slot = 2 + (nz & 1);
    if (i == m - 1) {
      residual_pass<DT>(mp_on, memb_lo, inv_s, log_s, qrow, seed, invz, nz, slot);
      const Part rall = g.fold;
      if (rall.arg == kNoCut || !(rall.best > neg_inf())) return true;
      token = rall.arg;
      return false;
    }
    tree_mass_pass<DT>(mp_on, memb_lo, inv_s, qrow, invz, nz, slot);
    const unsigned long long zm = g.fold.mass;
    if (zm == 0) return true;  // nothing left (rounding): the stream-0 draw
    const float Z = static_cast<float>(static_cast<double>(zm) * kFixedInv);
    __syncthreads();  // every thread has read g.fold and invz
    if (threadIdx.x == 0) invz[nz] = __fdiv_rn(1.0f, Z);
    __syncthreads();
    ++nz;
    log_s += logf(Z);
  }
  return false;
}
// A position that tests drafts, after the pass that summed the mass of K
// (mass, in 2^-40 units) and fetched the draft token's processed logit yx:
// a linear position accepts its draft with u * q(x) < P(x) (stream 1, word 0)
// and otherwise draws from the residual max(P - q, 0) (stream 2); a tree node
// tests its children (tree_children).  When the residual is empty (rounding)
// the token is the stream-0 draw from P, drawn here.  Out of line so that the
// sampling path's register allocation does not carry it.
template <int DT>
__device__ __noinline__ void spec_position(int tree, int mp_on, float memb_lo, unsigned long long mass, float yx,
                                           const float* qrow, uint64_t seed, int32_t& accept, int32_t& acc_node,
                                           int32_t& token) {
  const float SK = static_cast<float>(static_cast<double>(mass) * kFixedInv);
  bool fallback = false;
  if (tree) {
    fallback = tree_children<DT>(mp_on, memb_lo, SK, qrow, seed, acc_node, token);
  } else {
    const bool x_in = (yx != neg_inf()) && in_kept(g.x, yx, g.m, mp_on, g.min_p);
    const float inv_s = __fdiv_rn(1.0f, SK);
    const float Px = x_in ? __fmul_rn(__expf(yx - g.m), inv_s) : 0.0f;
    const float q = qrow[g.x];
    const float u = uniform_from_numerator(uniform_numerator(philox_word(seed, g.rowid, g.pos, 0, 1)));
    accept = (__fmul_rn(u, q) < Px) ? 1 : 0;
    if (accept) {
      token = g.x;
    } else {
      residual_pass<DT>(mp_on, memb_lo, inv_s, logf(SK), qrow, seed, nullptr, 0, 2);
      const Part rall = g.fold;
      if (rall.arg != kNoCut && rall.best > neg_inf())
        token = rall.arg;
      else
        fallback = true;
    }
  }
  if (fallback) {
    draw_pass<DT, true>(mp_on, memb_lo, 1, 0, 0, seed);
    token = g.fold.arg;
  }
}

// ------------------------------------------------------------- kernel --

template <int DT>
__global__ void __launch_bounds__(kThreads, 2) ss_row_kernel(const KArgs a) {
  using V = Vec<DT>;
  cg::cluster_group cl = cg::this_cluster();
  const int rank = static_cast<int>(cl.block_rank());
  const int ncta = static_cast<int>(cl.num_blocks());
  const Layout& L = a.L;
  // Programmatic dependent launch (tree calls with SS_TREE_OVERLAP_PREVIOUS):
  // a next call may start its CTAs once every CTA of this one has started;
  // this call's own global writes wait for the grid before it (no-ops in a
  // launch without the attribute).  Debug rows are written throughout, so a
  // call that writes them waits at once.
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  if (a.debug_processed) asm volatile("griddepcontrol.wait;" ::: "memory");
  int task = static_cast<int>(blockIdx.x) / ncta;
  int with_work = -1;
  if (a.row_class != 0) {
    task = ordered_task(a, task, reinterpret_cast<int32_t*>(smem_raw + L.red_off), &with_work);
  } else if (a.stated_tasks > 0) {
    with_work = tree_task_count(a, reinterpret_cast<int32_t*>(smem_raw + L.red_off));
  }
  if (a.stated_tasks > 0 && with_work != a.stated_tasks) {
    // the same in every CTA: the call verifies nothing
    if (blockIdx.x < static_cast<unsigned>(ncta) && rank == 0) report_bad_tree_count(a);
    return;
  }
  if (task < 0) return;  // the whole cluster: no task left for it
  Ctx& c = g;
  const int tid = threadIdx.x;
  const int V_ = a.vocab;

  // ---------------------------------------------------------------- setup
  if (tid == 0) {
    uint8_t* base = smem_raw;
    c.data = base;
    c.vmax = reinterpret_cast<__nv_bfloat16*>(base + L.vmax_off);
    c.xm = reinterpret_cast<uint32_t*>(base + L.xm_off);
    c.vlist_cap = L.slice_len / 32 * 2;  // 16-bit entries in the bitmap's words
    c.hkey = reinterpret_cast<int32_t*>(base + L.hk_off);
    c.hcnt = reinterpret_cast<int32_t*>(base + L.hc_off);
    c.hval = reinterpret_cast<float*>(base + L.hv_off);
    c.work = base + L.work_off;
    const int per = ncta * kBuckets;
    c.rh_mass[0] = reinterpret_cast<unsigned long long*>(base + L.rh_off);
    c.rh_mass[1] = c.rh_mass[0] + per;
    c.rh_cnt[0] = reinterpret_cast<uint32_t*>(base + L.rh_off + 2 * per * 8);
    c.rh_cnt[1] = c.rh_cnt[0] + per;
    c.rec = reinterpret_cast<LevelRec*>(base + L.rec_off);
    c.red = base + L.red_off;
    c.part = reinterpret_cast<Part*>(base + L.part_off);
    c.mbar = reinterpret_cast<uint64_t*>(base + L.mbar_off);
    c.ncta = ncta;
    c.rank = rank;
    int32_t status = SS_ROW_OK;
    int32_t req = task, j = 0, k = 0, d0 = 0, row = task, x = -1, drow = -1;
    bool live = true;
    int32_t bad_k = 0;
    if (a.mode == kModeVerify) {
      const int width = a.max_draft + 1;
      req = task / width;
      j = task % width;
      d0 = a.draft_offsets[req];
      k = a.draft_offsets[req + 1] - d0;
      if (k < 0 || k > a.max_draft) {
        status = SS_ROW_BAD_PARAM;
        live = (j == 0);
        k = 0;
        bad_k = 1;
      } else if (j > k) {
        live = false;
      }
      row = d0 + req + j;
      if (j < k) {
        drow = d0 + j;
        x = a.draft_tokens[drow];
      }
    } else if (a.mode == kModeTree) {
      // node j of request req; k = its non-root node count (the position
      // range check below covers the deepest possible node)
      const int width = a.max_draft + 1;
      req = task / width;
      j = task % width;
      d0 = a.draft_offsets[req];
      const int32_t nn = a.draft_offsets[req + 1] - d0;
      k = nn - 1;
      if (nn < 1 || nn > width) {
        status = SS_ROW_BAD_PARAM;
        live = (j == 0);
        k = 0;
        bad_k = 1;
      } else if (j >= nn) {
        live = false;
      }
      row = d0 + j;
      drow = d0 + j;
      c.nn = bad_k ? 1 : nn;
      c.depth = 0;
      c.nkids = 0;
    }
    c.row = live ? row : -1;
    c.bad_k = bad_k;
    c.req = req;
    // Every per-request parameter in one batch of independent read-only
    // loads (global, so none can alias the shared-memory stores below).
    const ss_params& p = a.p;
    const uint32_t rid = p.row_id ? __ldg(p.row_id + req) : static_cast<uint32_t>(req);
    const float T = __ldg(p.temperature + req);
    const int32_t top_k = p.top_k ? __ldg(p.top_k + req) : 0;
    const float top_p = p.top_p ? __ldg(p.top_p + req) : 1.0f;
    const float min_p = p.min_p ? __ldg(p.min_p + req) : 0.0f;
    const float rep = p.repetition ? __ldg(p.repetition + req) : 1.0f;
    const float freq = p.frequency ? __ldg(p.frequency + req) : 0.0f;
    const float pres = p.presence ? __ldg(p.presence + req) : 0.0f;
    const int32_t h0 = p.hist_offsets ? __ldg(p.hist_offsets + req) : 0;
    const int32_t h1 = p.hist_offsets ? __ldg(p.hist_offsets + req + 1) : 0;
    const int32_t b0 = p.bias_offsets ? __ldg(p.bias_offsets + req) : 0;
    const int32_t b1 = p.bias_offsets ? __ldg(p.bias_offsets + req + 1) : 0;
    const bool use_mask = (p.bitmask != nullptr) && (p.use_bitmask == nullptr || __ldg(p.use_bitmask + req) != 0);
    const uint64_t seed = __ldg(reinterpret_cast<const unsigned long long*>(p.seed) + req);
    const int64_t pos = __ldg(reinterpret_cast<const long long*>(p.position) + req);
    c.rowid = rid;
    c.j = j;
    c.k = k;
    c.d0 = d0;
    c.drow = drow;
    c.x = x;
    c.temperature = T;
    c.greedy = (T == 0.0f);
    c.inv_t = __fdiv_rn(1.0f, T);
    c.top_k = top_k;
    c.top_p = top_p;
    c.min_p = min_p;
    c.rep = rep;
    c.freq = freq;
    c.pres = pres;
    c.h0 = h0;
    c.h1 = h1;
    c.b0 = b0;
    c.b1 = b1;
    c.use_mask = use_mask;
    c.seed_lo = static_cast<uint32_t>(seed);
    c.seed_hi = static_cast<uint32_t>(seed >> 32);
    c.pos = static_cast<uint32_t>(pos) + static_cast<uint32_t>(j);
    // parameter validation (identical in every CTA of the cluster)
    if (!(T >= 0.0f) || isinf(T) || top_k < 0 || !(top_p > 0.0f) || !(min_p >= 0.0f && min_p <= 1.0f) ||
        !(rep > 0.0f) || isinf(rep) || !isfinite(freq) || !isfinite(pres) || h1 < h0 || b1 < b0 || pos < 0 ||
        pos + k > 0xffffffffll)
      status = SS_ROW_BAD_PARAM;
    if (a.shard_rec && status == SS_ROW_OK) {
      // a shard can list at most shard_cap candidates, and top-p / min-p
      // without top-k need the whole distribution: not decidable by shards
      if (c.top_k > a.shard_cap || (c.top_k == 0 && !c.greedy && (c.top_p < 1.0f || c.min_p > 0.0f)))
        status = SS_ROW_UNSUPPORTED;
      c.top_p = 1.0f;  // applied by the merge, over the merged top-k list
      c.min_p = 0.0f;
    }
    c.status = status;
    c.lo = a.shard_off + rank * L.slice_len;
    // A row with invalid parameters (including a bad draft count, which makes
    // its row index meaningless) touches no logits: it only reports its status.
    c.n = (status == SS_ROW_BAD_PARAM || status == SS_ROW_UNSUPPORTED)
              ? 0
              : max(0, min(a.shard_off + a.shard_len - c.lo, L.slice_len));
    if (a.shard_rec && rank == 0)
      reinterpret_cast<ShardHead*>(a.shard_rec + static_cast<int64_t>(task) * (32 + 8 * a.shard_cap))->n = 0;
    c.cursor[0] = 0;
    c.cursor[1] = 0;
    c.want_s = (T > 0.0f && c.top_p < 1.0f && c.top_k <= 0) ? 1 : 0;
  }
  __syncthreads();
  if (c.row < 0) return;  // whole cluster: no such target position

  if (a.mode == kModeTree && !c.bad_k) {
    // The request's tree, into shared memory: parents, tokens; then the
    // node's depth (its Philox position), its path (its history additions)
    // and its children.  Every node of the request checks every parent, so
    // all of them agree on a malformed tree.
    int32_t* tpar = reinterpret_cast<int32_t*>(c.work + kTreeOff);
    int32_t* ttok = tpar + kTreeMaxNodes;
    int32_t* tpath = ttok + kTreeMaxNodes;
    const int nn = c.nn;
    if (tid < nn) {
      tpar[tid] = a.tree_parents[c.d0 + tid];
      ttok[tid] = a.draft_tokens[c.d0 + tid];
    }
    __syncthreads();
    if (tid == 0) {
      bool ok = true;
      for (int v = 1; v < nn; ++v) ok = ok && tpar[v] >= 0 && tpar[v] < v;
      int dep = 0, m = 0;
      if (ok) {
        for (int v = c.j; v > 0; v = tpar[v]) tpath[dep++] = ttok[v];
        for (int v = c.j + 1; v < nn; ++v)
          if (tpar[v] == c.j) {
            c.kid_node[m] = v;
            c.kid_tok[m] = ttok[v];
            ++m;
          }
      } else if (c.status == SS_ROW_OK) {
        c.status = SS_ROW_BAD_PARAM;  // touches no logits
        c.n = 0;
      }
      c.depth = dep;
      c.nkids = m;
      c.pos = static_cast<uint32_t>(a.p.position[c.req]) + static_cast<uint32_t>(dep);
    }
    __syncthreads();
  }

  const int lo = c.lo, n = c.n;
  // addressed by token id: element t of the row is row_ptr[t] (a shard's
  // buffer starts at token shard_off)
  const char* row_ptr = reinterpret_cast<const char*>(a.logits) +
                        (static_cast<int64_t>(c.row) * a.row_stride - a.shard_off) * V::kBytes;
  const uint32_t slice_bytes = static_cast<uint32_t>(n) * V::kBytes;
  // Bulk (TMA) copies need a 16-byte aligned source; a row whose byte stride
  // is not a multiple of 16 (an odd vocabulary size) is staged with plain,
  // coalesced element loads instead.
  const bool bulk_ok = ((reinterpret_cast<uintptr_t>(row_ptr) + static_cast<uintptr_t>(lo) * V::kBytes) & 15u) == 0;
  const uint32_t bulk_bytes = bulk_ok ? (slice_bytes & ~15u) : 0u;
  const int nchunks = static_cast<int>((bulk_bytes + kChunkBytes - 1) / kChunkBytes);

  // Issue the slice's bulk copies first so that HBM traffic starts at once.
  if (tid == 0) {
    for (int ch = 0; ch < nchunks; ++ch) mbar_init(c.mbar + ch, 1);
    fence_barrier_init();
    const char* src = row_ptr + static_cast<int64_t>(lo) * V::kBytes;
    for (int ch = 0; ch < nchunks; ++ch) {
      const uint32_t off = static_cast<uint32_t>(ch) * kChunkBytes;
      const uint32_t bytes = min(kChunkBytes, bulk_bytes - off);
      mbar_arrive_expect_tx(c.mbar + ch, bytes);
      bulk_load(c.data + off, src + off, bytes, c.mbar + ch);
    }
  }
  // The rest (a ragged tail < 16 bytes, or the whole slice when unaligned)
  // with plain loads.
  for (int e = static_cast<int>(bulk_bytes / V::kBytes) + tid; e < n; e += kThreads) {
    if (V::kBytes == 4)
      reinterpret_cast<uint32_t*>(c.data)[e] = reinterpret_cast<const uint32_t*>(row_ptr)[lo + e];
    else
      reinterpret_cast<uint16_t*>(c.data)[e] = reinterpret_cast<const uint16_t*>(row_ptr)[lo + e];
  }

  // Exclusion bitmap: grammar mask (inverted) and the tail beyond the slice.
  const int words = L.slice_len / 32;
  for (int w = tid; w < words; w += kThreads) {
    const int first = w * 32;
    uint32_t ex = 0xffffffffu;  // words past the row's end: all excluded
    if (first < n) {            // (lo + first) / 32 < ceil(V / 32): inside the mask row
      ex = 0;
      if (c.use_mask)
        ex = ~static_cast<uint32_t>(a.p.bitmask[static_cast<int64_t>(c.req) * a.p.bitmask_stride + (lo >> 5) + w]);
      if (first + 32 > n) ex |= 0xffffffffu << (n - first);
    }
    c.xm[w] = ex;
  }
  for (int s = tid; s < kHashCap; s += kThreads) {
    c.hkey[s] = -1;
    c.hcnt[s] = 0;
    c.hval[s] = 0.0f;
  }
  // Raw logits of the patched tokens, by slot, until stage 1: the work region
  // is not in use before the first histogram.
  float* hraw = reinterpret_cast<float*>(c.work);
  static_assert(kHashCap * sizeof(float) <= kTreeOff, "raw patched logits stay below the tree");
  static_assert(kTreeOff + 3 * kTreeMaxNodes * sizeof(int32_t) <= kWorkBytes, "the tree fits the work region");
  static_assert(2 * kTreeMaxNodes * sizeof(float) <= kTreeOff, "child logits and 1/Z fit below the tree");

  // The logit of a patched token, -inf when the grammar mask disallows it
  // (the mask is applied after penalties and bias, which keep -inf at -inf).
  auto raw_logit = [&](int32_t t) -> float {
    float z = V::load_global(row_ptr, t);
    if (c.use_mask) {
      const uint32_t word = static_cast<uint32_t>(a.p.bitmask[static_cast<int64_t>(c.req) * a.p.bitmask_stride + (t >> 5)]);
      if (((word >> (t & 31)) & 1u) == 0u) z = neg_inf();
    }
    return z;
  };
  // Prefetch, before the table is ready: this thread's first history entry,
  // draft and bias entry, with their logits, so that the global round trips
  // overlap the initialisation above.
  const bool row_ok = (c.status == SS_ROW_OK);
  const int eh = c.h0 + tid, eb = c.b0 + tid;
  const int32_t th = (row_ok && eh < c.h1) ? a.p.hist_ids[eh] : -1;
  const int32_t tb = (row_ok && eb < c.b1) ? a.p.bias_ids[eb] : -1;
  const float bb = (row_ok && eb < c.b1) ? a.p.bias_vals[eb] : 0.0f;
  const int32_t td = (row_ok && a.mode == kModeVerify && tid < c.k) ? a.draft_tokens[c.d0 + tid] : -1;
  auto in_slice = [&](int32_t t) { return t >= lo && t < lo + n; };
  const float zh = in_slice(th) ? raw_logit(th) : 0.0f;
  const float zb = in_slice(tb) ? raw_logit(tb) : 0.0f;
  const float zd = in_slice(td) ? raw_logit(td) : 0.0f;
  __syncthreads();

  // Patch table: history (+ drafts before this position) and bias entries.
  int32_t st_local = SS_ROW_OK;
  auto insert = [&](int32_t t) -> int {
    uint32_t h = (static_cast<uint32_t>(t) * 2654435761u) >> kHashShift;
    for (int probe = 0; probe < kHashCap; ++probe) {
      const int32_t prev = atomicCAS(c.hkey + h, -1, t);
      if (prev == -1 || prev == t) return static_cast<int>(h);
      h = (h + 1) & (kHashCap - 1);
    }
    return -1;
  };
  // one counted occurrence of t (its raw logit z): duplicates write the same z
  auto count = [&](int32_t t, float z) {
    if (t < 0 || t >= V_) {
      st_local = max(st_local, SS_ROW_BAD_INDEX);
      return;
    }
    if (!in_slice(t)) return;
    const int s = insert(t);
    if (s < 0) {
      st_local = max(st_local, SS_ROW_LIMIT);
      return;
    }
    atomicAdd(c.hcnt + s, 1);
    hraw[s] = z;
  };
  if (row_ok) {
    if (eh < c.h1) count(th, zh);
    for (int e = eh + kThreads; e < c.h1; e += kThreads) {  // histories longer than the block
      const int32_t t = a.p.hist_ids[e];
      count(t, in_slice(t) ? raw_logit(t) : 0.0f);
    }
    if (a.mode == kModeVerify) {
      // every draft must be a token id; the history of position j holds the drafts before j
      if (tid < c.k) {
        if (td < 0 || td >= V_)
          st_local = max(st_local, SS_ROW_BAD_INDEX);
        else if (tid < c.j)
          count(td, zd);
      }
      for (int e = tid + kThreads; e < c.k; e += kThreads) {
        const int32_t t = a.draft_tokens[c.d0 + e];
        if (t < 0 || t >= V_)
          st_local = max(st_local, SS_ROW_BAD_INDEX);
        else if (e < c.j)
          count(t, in_slice(t) ? raw_logit(t) : 0.0f);
      }
    }
    if (a.mode == kModeTree) {
      // the tokens on the node's path; every node token must be a token id
      const int32_t* ttok = reinterpret_cast<const int32_t*>(c.work + kTreeOff) + kTreeMaxNodes;
      const int32_t* tpath = ttok + kTreeMaxNodes;
      if (tid < c.depth) {
        const int32_t t = tpath[tid];
        count(t, in_slice(t) ? raw_logit(t) : 0.0f);
      }
      if (tid >= 1 && tid < c.nn && (ttok[tid] < 0 || ttok[tid] >= V_)) st_local = max(st_local, SS_ROW_BAD_INDEX);
    }
    for (int e = eb; e < c.b1; e += kThreads) {
      const int32_t t = (e == eb) ? tb : a.p.bias_ids[e];
      const float b = (e == eb) ? bb : a.p.bias_vals[e];
      if (!isfinite(b)) st_local = max(st_local, SS_ROW_BAD_PARAM);
      if (t < 0 || t >= V_) {
        st_local = max(st_local, SS_ROW_BAD_INDEX);
        continue;
      }
      if (!in_slice(t)) continue;
      const int s = insert(t);
      if (s < 0) {
        st_local = max(st_local, SS_ROW_LIMIT);
        continue;
      }
      if (atomicOr(c.hcnt + s, kBiasFlag) & kBiasFlag) st_local = max(st_local, SS_ROW_BAD_INDEX);  // duplicate
      c.hval[s] = b;
      hraw[s] = (e == eb) ? zb : raw_logit(t);
    }
  }
  __syncthreads();
  // Processed values of patched tokens.
  for (int s = tid; s < kHashCap; s += kThreads) {
    const int32_t t = c.hkey[s];
    if (t < 0) continue;
    atomicOr(c.xm + ((t - lo) >> 5), 1u << ((t - lo) & 31));
    float z = hraw[s];
    const int32_t hc = c.hcnt[s];
    const int32_t cnt = hc & ~kBiasFlag;
    if (cnt > 0) {
      z = (z > 0.0f) ? __fdiv_rn(z, c.rep) : __fmul_rn(z, c.rep);
      z = __fsub_rn(z, __fmul_rn(c.freq, static_cast<float>(cnt)));
      z = __fsub_rn(z, c.pres);
    }
    if (hc & kBiasFlag) z = __fadd_rn(z, c.hval[s]);
    c.hval[s] = c.greedy ? z : __fmul_rn(z, c.inv_t);
  }

  // --------------------------------------------------------------- stage 1
  // Wait for each chunk, write -inf over excluded lanes, store each vector's
  // bound, and accumulate the row max (lowest index on ties), the smallest
  // allowed value, the allowed count and non-finite flags.
  float a_best = neg_inf(), a_ymin = pos_inf(), a_smax = neg_inf(), a_ssum = 0.0f;
  int32_t a_arg = kNoCut, a_count = 0, a_status = st_local;
  bool timed_out = false;
  __syncthreads();  // exclusion bits of patched tokens are in place
  {
    const int nvec = (n + V::kPer - 1) / V::kPer;
    const int vec_per_chunk = static_cast<int>(kChunkBytes / 16);
    uint4* data = reinterpret_cast<uint4*>(c.data);
    float* dbg = (a.debug_processed && !c.bad_k) ? a.debug_processed + static_cast<int64_t>(c.row) * V_ : nullptr;
    const bool greedy = c.greedy != 0;
    const float inv_t = c.inv_t;
    int waited = -1;
    float best_v = neg_inf();
    int best_vec = -1;
    const bool want_s = c.want_s != 0;
    // Two vectors per iteration: both loads are issued before any arithmetic.
    constexpr int kB = 2;
    for (int v0 = tid; v0 < nvec; v0 += kB * kThreads) {
      const int vlast = min(v0 + (kB - 1) * kThreads, nvec - 1);
      const int ch = min(vlast / vec_per_chunk, nchunks - 1);
      if (nchunks > 0 && ch > waited) {
        for (int w = waited + 1; w <= ch; ++w)
          if (!mbar_wait_bounded(c.mbar + w, 0, kWaitPolls)) timed_out = true;
        waited = ch;
      }
      uint4 raw[kB];
      uint32_t bits[kB];
#pragma unroll
      for (int u = 0; u < kB; ++u) {
        const int v = v0 + u * kThreads;
        const int e0 = v * V::kPer;
        if (v < nvec) {
          raw[u] = data[v];
          bits[u] = (c.xm[e0 >> 5] >> (e0 & 31)) & ((1u << V::kPer) - 1u);
        } else {
          raw[u] = V::exclude(make_uint4(0u, 0u, 0u, 0u), 0xffu);
          bits[u] = 0;
        }
      }
#pragma unroll
      for (int u = 0; u < kB; ++u) {
        const int v = v0 + u * kThreads;
        raw[u] = V::exclude(raw[u], bits[u]);  // selects: no branch per vector
        float z[V::kPer];
        V::unpack(raw[u], z);
        float vmax = neg_inf(), vmin = pos_inf();
        int allowed = 0;
#pragma unroll
        for (int e = 0; e < V::kPer; ++e) {
          z[e] = greedy ? z[e] : __fmul_rn(z[e], inv_t);
          vmax = max_nan(vmax, z[e]);
          const bool ok = (z[e] != neg_inf());
          allowed += ok ? 1 : 0;
          vmin = fminf(vmin, ok ? z[e] : pos_inf());
        }
        if (want_s) {  // online softmax normaliser of the row
          if (vmax > a_smax) {  // a new running max (rare after the first vectors)
            a_ssum = (a_smax == neg_inf()) ? 0.0f : __fmul_rn(a_ssum, __expf(a_smax - vmax));
            a_smax = vmax;
          }
          const float ms = (a_smax == neg_inf()) ? 0.0f : a_smax;  // exp(-inf - ms) = 0
          float part = 0.0f;
#pragma unroll
          for (int e = 0; e < V::kPer; ++e) part = __fadd_rn(part, __expf(z[e] - ms));
          a_ssum = __fadd_rn(a_ssum, part);
        }
        a_count += allowed;
        a_ymin = fminf(a_ymin, vmin);
        if (vmax != vmax || vmax == pos_inf()) a_status = max(a_status, SS_ROW_NONFINITE);
        if (vmax > best_v) {
          best_v = vmax;
          best_vec = v;
        }
        if (v < nvec) {
          data[v] = raw[u];
          c.vmax[v] = bf16_round_up(vmax);
        }
      }
    }
    // chunks no thread of this CTA touched still need their completion
    if (tid == 0)
      for (int w = waited + 1; w < nchunks; ++w)
        if (!mbar_wait_bounded(c.mbar + w, 0, kWaitPolls)) timed_out = true;
    if (timed_out) a_status = max(a_status, SS_ROW_TIMEOUT);
    if (best_vec >= 0) {  // lowest index of the maximum inside the best vector
      float z[V::kPer];
      V::unpack(data[best_vec], z);
#pragma unroll
      for (int e = V::kPer - 1; e >= 0; --e) {
        const float y = greedy ? z[e] : __fmul_rn(z[e], inv_t);
        if (y == best_v) {
          a_best = best_v;
          a_arg = lo + best_vec * V::kPer + e;
        }
      }
    }
    if (dbg) {
      __syncthreads();
      for (int v = tid; v < nvec; v += kThreads) {
        float z[V::kPer];
        V::unpack(data[v], z);
#pragma unroll
        for (int e = 0; e < V::kPer; ++e)
          if (v * V::kPer + e < n) dbg[lo + v * V::kPer + e] = greedy ? z[e] : __fmul_rn(z[e], inv_t);
      }
    }
    __syncthreads();  // debug writes of the raw slice precede the patched ones
    for (int s = tid; s < kHashCap; s += kThreads) {
      const int32_t t = c.hkey[s];
      if (t < 0) continue;
      const float y = c.hval[s];
      if (dbg) dbg[t] = y;
      if (y == neg_inf()) continue;
      a_count += 1;
      a_ymin = fminf(a_ymin, y);
      if (!(y < pos_inf())) a_status = max(a_status, SS_ROW_NONFINITE);
      if (beats(y, t, a_best, a_arg)) {
        a_best = y;
        a_arg = t;
      }
      if (want_s) softmax_merge(a_smax, a_ssum, y, 1.0f);
    }
  }
  reduce_fold(0, a_best, a_arg, a_count, max(a_status, c.status), 0, a_ymin, a_smax, a_ssum, neg_inf(), 0);
  const Part all = g.fold;
  int32_t status = all.status;
  if (status == SS_ROW_OK && all.count == 0) status = SS_ROW_EMPTY_SET;
  const float m = all.best;
  const int32_t argmax_tok = all.arg;
  if (tid == 0) {
    c.m = m;
    c.ymin = all.ymin;
    c.arg = argmax_tok;
    c.count = all.count;
    c.s_all = (all.smax == neg_inf()) ? 0.0f : __fmul_rn(all.ssum, __expf(all.smax - m));
  }
  __syncthreads();

  int32_t token = -1, kept = 0, accept = 0, acc_node = -1;
  if (status == SS_ROW_OK) {
    // a position that tests drafts: a linear one before the last, a tree node with children
    const bool spec_pos = (a.mode == kModeVerify) ? (c.j < c.k) : (a.mode == kModeTree && c.nkids > 0);
    const uint64_t seed = (static_cast<uint64_t>(c.seed_hi) << 32) | c.seed_lo;
    const uint32_t rowid = c.rowid;
    if (c.greedy) {
      kept = 1;
      token = argmax_tok;
      if (spec_pos && a.mode == kModeTree) {
        // greedy: the first child carrying the argmax is accepted
        for (int i = 0; i < c.nkids; ++i)
          if (c.kid_tok[i] == argmax_tok) {
            acc_node = c.kid_node[i];
            break;
          }
      } else if (spec_pos) {
        const float q = a.draft_probs[static_cast<int64_t>(c.drow) * a.draft_stride + c.x];
        const float u = uniform_from_numerator(uniform_numerator(philox_word(seed, rowid, c.pos, 0, 1)));
        const float P = (c.x == argmax_tok) ? 1.0f : 0.0f;
        accept = (__fmul_rn(u, q) < P) ? 1 : 0;
        token = accept ? c.x : argmax_tok;
      }
    } else {
      // ------------------------------------------------------ the cuts
      const bool k_on = c.top_k > 0 && c.top_k < c.count;
      const bool p_on = c.top_p < 1.0f;
      const bool mp_on = c.min_p > 0.0f;
      if (k_on || p_on) {
        resolve_cuts<DT>(k_on, p_on);
      } else if (tid == 0) {
        c.cut_on = 0;
        c.cut_key = 0;
        c.cut_idx = kNoCut;
        c.cut_len = -1;
      }
      __syncthreads();
      const bool cut_on = c.cut_on != 0;
      const int32_t cut_len = c.cut_len;

      // ------------------------------------------------------ the draw
      const float min_p = c.min_p;
      // |K| is known unless min-p or the fallback selection decided it
      const bool need_count = mp_on || (cut_on && cut_len < 0);
      // lowest logit a member can have: vectors below it hold no member
      float k_lo = cut_on ? key_value(c.cut_key) : neg_inf();
      if (mp_on) k_lo = fmaxf(k_lo, m + logf(min_p) - 1e-3f * (1.0f + fabsf(m)));
      const float memb_lo = k_lo;
      // the mass S_K needed by a verification position ignores tokens whose
      // fixed-point mass is zero
      if (spec_pos && !need_count) k_lo = fmaxf(k_lo, m - kMassCutoff - 1.0f - fabsf(m) * 1e-6f);
      if (a.shard_rec && c.top_k > 0) {
        // sharded top-k row: the shard's top-k (all its allowed tokens when
        // it has no more than k) go to the record; the merge selects and draws
        emit_members<DT>(reinterpret_cast<float2*>(a.shard_rec + static_cast<int64_t>(task) * (32 + 8 * a.shard_cap) + 32),
                         &reinterpret_cast<ShardHead*>(a.shard_rec + static_cast<int64_t>(task) * (32 + 8 * a.shard_cap))->n,
                         a.shard_cap);
        kept = cut_on ? cut_len : c.count;
        token = -1;
      } else {
      // a position that tests a draft needs the mass of K, not the stream-0
      // draw: that is only the fallback of an empty residual (drawn then)
      if (spec_pos)
        draw_pass<DT, false>(mp_on, k_lo, 0, 1, need_count, seed);
      else
        draw_pass<DT, true>(mp_on, k_lo, !need_count, 0, need_count, seed);
      const Part dall = g.fold;
      kept = need_count ? dall.count : (cut_on ? cut_len : c.count);
      token = dall.arg;
      if (a.shard_rec && rank == 0 && tid == 0) {
        ShardHead* h = reinterpret_cast<ShardHead*>(a.shard_rec + static_cast<int64_t>(task) * (32 + 8 * a.shard_cap));
        h->best = dall.best;
        h->best_token = dall.arg;
      }
      if (spec_pos)
        spec_position<DT>(a.mode == kModeTree, mp_on, memb_lo, dall.mass, dall.xhere ? dall.xy : neg_inf(),
                          a.draft_probs + static_cast<int64_t>(c.drow) * a.draft_stride, seed, accept, acc_node,
                          token);
      }
    }
  }

  // ------------------------------------------------------------- outputs
  if (rank == 0 && tid == 0) {
    asm volatile("griddepcontrol.wait;" ::: "memory");  // the previous call has finished
    if (status != SS_ROW_OK) {
      token = -1;
      kept = 0;
      accept = 0;
    }
    if (a.shard_rec) {
      ShardHead* h = reinterpret_cast<ShardHead*>(a.shard_rec + static_cast<int64_t>(task) * (32 + 8 * a.shard_cap));
      h->status = status;
      h->kind = c.greedy ? kShardGreedy : (c.top_k > 0 ? kShardList : kShardDraw);
      h->count = (status == SS_ROW_OK) ? c.count : 0;
      h->m = m;
      h->arg = argmax_tok;
    } else if (a.out_kept && !c.bad_k) {
      a.out_kept[c.row] = kept;
    }
    if (a.shard_rec) {
      // the record is the output
    } else if (a.mode == kModeSample) {
      a.out_token[c.row] = token;
      a.out_status[c.row] = status;
    } else if (a.mode == kModeTree) {
      const int width = a.max_draft + 1;
      const int i = c.req;
      int32_t* out = a.out_token + static_cast<int64_t>(i) * width;
      int32_t* path = a.out_path ? a.out_path + static_cast<int64_t>(i) * width : nullptr;
      if (c.bad_k) {
        // invalid node count: only node 0 exists and reports it
        for (int w = 0; w < width; ++w) {
          out[w] = -1;
          if (path) path[w] = -1;
        }
        a.out_num_accepted[i] = 0;
        a.out_status[i] = status;
      } else {
        int4* res = a.ws_results + static_cast<int64_t>(i) * width;
        res[c.j] = make_int4(status, acc_node, token, kept);
        __threadfence();
        const int prev = atomicAdd(a.ws_counters + i, 1);
        if (prev == c.nn - 1) {  // last node of this request to finish: walk the tree
          __threadfence();
          int32_t st = SS_ROW_OK;
          for (int w = 0; w < c.nn; ++w) st = max(st, __ldcg(&res[w].x));
          int nacc = 0;
          for (int w = 0; w < width; ++w) {
            out[w] = -1;
            if (path) path[w] = -1;
          }
          if (st == SS_ROW_OK) {
            int u = 0;
            for (int step = 0; step < c.nn; ++step) {  // accepted children have larger indices
              const int4 r = __ldcg(res + u);
              out[nacc] = r.z;
              if (r.y <= u || r.y >= c.nn) break;
              if (path) path[nacc] = r.y;
              ++nacc;
              u = r.y;
            }
          }
          a.out_num_accepted[i] = nacc;
          a.out_status[i] = st;
          a.ws_counters[i] = 0;  // ready for the next call
        }
      }
    } else {
      const int width = a.max_draft + 1;
      const int i = c.req;
      if (c.bad_k) {
        // invalid draft count: only position 0 exists and reports it
        for (int w = 0; w < width; ++w) a.out_token[static_cast<int64_t>(i) * width + w] = -1;
        a.out_num_accepted[i] = 0;
        a.out_status[i] = status;
      } else {
        int4* res = a.ws_results + static_cast<int64_t>(i) * width;
        res[c.j] = make_int4(status, accept, token, kept);
        __threadfence();
        const int prev = atomicAdd(a.ws_counters + i, 1);
        if (prev == c.k) {  // last position of this request to finish
          __threadfence();
          int32_t st = SS_ROW_OK;
          for (int w = 0; w <= c.k; ++w) st = max(st, __ldcg(&res[w].x));
          int32_t* out = a.out_token + static_cast<int64_t>(i) * width;
          int nacc = 0;
          if (st == SS_ROW_OK) {
            int w = 0;
            for (; w < c.k; ++w) {
              const int4 r = __ldcg(res + w);
              out[w] = r.z;
              if (!r.y) break;
              ++nacc;
            }
            if (w == c.k) out[w] = __ldcg(&res[w].z);
            for (int f = nacc + 1; f < width; ++f) out[f] = -1;
          } else {
            for (int f = 0; f < width; ++f) out[f] = -1;
          }
          a.out_num_accepted[i] = nacc;
          a.out_status[i] = st;
          a.ws_counters[i] = 0;  // ready for the next call
        }
      }
    }
  }
  // The fallback selection reads other CTAs' shared memory; no CTA may leave
  // while that can still happen.
  cl.sync();
}

// ------------------------------------------------ accepted-token commit --

// One thread per request: append the emitted tokens, advance the length and
// the position, set the next input token (see ss_commit_accepted).
__global__ void ss_commit_kernel(int32_t num_requests, int32_t width, const int32_t* __restrict__ out_tokens,
                                 const int32_t* __restrict__ num_accepted, const int32_t* __restrict__ status,
                                 int32_t* __restrict__ tokens, int32_t capacity, int32_t* __restrict__ seq_len,
                                 int64_t* __restrict__ position, int32_t* __restrict__ next_token,
                                 int32_t* __restrict__ commit_status) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= num_requests) return;
  if (status[i] != SS_ROW_OK) {
    commit_status[i] = status[i];
    return;
  }
  const int32_t count = num_accepted[i] + 1;
  const int32_t len = seq_len[i];
  if (count < 1 || count > width || len < 0 || static_cast<int64_t>(len) + count > capacity) {
    commit_status[i] = SS_ROW_LIMIT;
    return;
  }
  const int32_t* emitted = out_tokens + static_cast<int64_t>(i) * width;
  int32_t* dst = tokens + static_cast<int64_t>(i) * capacity + len;
  int32_t last = -1;
  for (int j = 0; j < count; ++j) {
    last = emitted[j];
    dst[j] = last;
  }
  seq_len[i] = len + count;
  position[i] += count;
  next_token[i] = last;
  commit_status[i] = SS_ROW_OK;
}

// ------------------------------------------------ vocabulary shards --

constexpr int kMaxShards = 8;

struct MergeArgs {
  int32_t num_rows, num_shards, cap;
  const uint8_t* rec[kMaxShards];
  ss_params p;
  int32_t* out_token;
  int32_t* out_status;
  int32_t* out_kept;
};

// Inclusive block-wide scan of one 64-bit value per thread.
__device__ __forceinline__ unsigned long long block_scan_u64(unsigned long long x, unsigned long long* ws) {
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const unsigned long long y = __shfl_up_sync(0xffffffffu, x, off);
    if (lane >= off) x += y;
  }
  __syncthreads();
  if (lane == 31) ws[wid] = x;
  __syncthreads();
  if (wid == 0) {
    unsigned long long y = (lane < kWarps) ? ws[lane] : 0ull;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const unsigned long long z = __shfl_up_sync(0xffffffffu, y, off);
      if (lane >= off) y += z;
    }
    if (lane < kWarps) ws[lane] = y;
  }
  __syncthreads();
  return x + ((wid > 0) ? ws[wid - 1] : 0ull);
}

// Merge of the shards' records of one row (one CTA per row).  Greedy rows:
// the largest logit over the shards (lowest id on ties); draw rows: the
// largest y + g (Gumbel-max decomposes over any partition of the
// vocabulary); top-k rows: the top-k of the union of the shards' top-k lists
// (two-stage top-k), then top-p over its renormalised fixed-point masses and
// min-p, exactly as the unsharded kernel takes them, then the draw over the
// kept prefix with the same counter-based noise.
__global__ void __launch_bounds__(kThreads) ss_merge_kernel(const MergeArgs a) {
  extern __shared__ __align__(16) unsigned long long mkeys[];
  __shared__ unsigned long long ws[kWarps];
  __shared__ int32_t s_status, s_kind, s_token, s_kept, s_total, s_lim;
  __shared__ unsigned long long s_sum;
  __shared__ int32_t s_n[kMaxShards];
  const int r = blockIdx.x, tid = threadIdx.x;
  const int64_t rec_bytes = 32 + 8 * static_cast<int64_t>(a.cap);
  if (tid == 0) {
    int32_t st = SS_ROW_OK, kind = kShardDraw, token = -1, kept = 0, total = 0;
    bool any = false;
    float bv = neg_inf();
    int32_t bi = kNoCut;
    for (int s = 0; s < a.num_shards; ++s) {
      const ShardHead* h = reinterpret_cast<const ShardHead*>(a.rec[s] + r * rec_bytes);
      kind = h->kind;
      s_n[s] = 0;
      if (h->status == SS_ROW_EMPTY_SET) continue;
      if (h->status != SS_ROW_OK) {
        st = max(st, h->status);
        continue;
      }
      any = true;
      kept += h->count;
      const float v = (kind == kShardGreedy) ? h->m : h->best;
      const int32_t t = (kind == kShardGreedy) ? h->arg : h->best_token;
      if (kind != kShardList && beats(v, t, bv, bi)) {
        bv = v;
        bi = t;
      }
      s_n[s] = min(h->n, a.cap);
      total += s_n[s];
    }
    if (st == SS_ROW_OK && !any) st = SS_ROW_EMPTY_SET;
    if (kind == kShardGreedy) kept = 1;
    token = bi;
    s_status = st;
    s_kind = kind;
    s_token = token;
    s_kept = kept;
    s_total = total;
  }
  __syncthreads();
  if (s_status == SS_ROW_OK && s_kind == kShardList) {
    // the union of the lists as sort keys (y descending, id ascending)
    const int total = s_total;
    int np2 = 1;
    while (np2 < total) np2 <<= 1;
    int at = 0;
    for (int s = 0; s < a.num_shards; ++s) {
      const float2* list = reinterpret_cast<const float2*>(a.rec[s] + r * rec_bytes + 32);
      for (int i = tid; i < s_n[s]; i += kThreads) {
        const float2 e = list[i];
        mkeys[at + i] = sort_key(e.x, __float_as_int(e.y));
      }
      at += s_n[s];
    }
    for (int i = total + tid; i < np2; i += kThreads) mkeys[i] = ~0ull;
    __syncthreads();
    for (int k = 2; k <= np2; k <<= 1)
      for (int j = k >> 1; j > 0; j >>= 1) {
        for (int q = tid; q < (np2 >> 1); q += kThreads) {
          const int i = ((q & ~(j - 1)) << 1) | (q & (j - 1));
          const unsigned long long x = mkeys[i], y = mkeys[i + j];
          if ((x > y) == ((i & k) == 0)) {
            mkeys[i] = y;
            mkeys[i + j] = x;
          }
        }
        __syncthreads();
      }
    const int32_t top_k = a.p.top_k ? a.p.top_k[r] : 0;
    const float top_p = a.p.top_p ? a.p.top_p[r] : 1.0f;
    const float min_p = a.p.min_p ? a.p.min_p[r] : 0.0f;
    const int kk = min(top_k, total);  // the exact top-k (all when k >= allowed)
    const float m = key_value(sort_key_order(mkeys[0]));
    if (tid == 0) s_lim = kk;
    __syncthreads();
    if (top_p < 1.0f) {
      // S = the top-k's fixed-point mass; the cut is the first prefix whose
      // mass reaches ceil(p * S)
      unsigned long long part = 0;
      for (int i = tid; i < kk; i += kThreads) part += fixed_mass(key_value(sort_key_order(mkeys[i])), m);
      unsigned long long incl = block_scan_u64(part, ws);
      if (tid == kThreads - 1) s_sum = incl;
      __syncthreads();
      const unsigned long long T = mass_target(top_p, s_sum);
      unsigned long long before = 0;
      for (int base = 0; base < kk; base += kThreads) {
        const int i = base + tid;
        const unsigned long long f = (i < kk) ? fixed_mass(key_value(sort_key_order(mkeys[i])), m) : 0ull;
        incl = block_scan_u64(f, ws) + before;
        if (i < kk && incl >= T && incl - f < T) s_lim = i + 1;  // the one crossing entry
        if (tid == kThreads - 1) s_sum = incl;
        __syncthreads();
        before = s_sum;
        __syncthreads();
        if (s_lim < kk || before >= T) break;
      }
    }
    if (min_p > 0.0f) {
      for (int i = tid; i < kk; i += kThreads)
        if (!(__expf(key_value(sort_key_order(mkeys[i])) - m) >= min_p)) atomicMin(&s_lim, i);
      __syncthreads();
    }
    const int L = s_lim;
    // the draw over the kept prefix
    const uint64_t seed = a.p.seed[r];
    const uint32_t rowid = a.p.row_id ? a.p.row_id[r] : static_cast<uint32_t>(r);
    const uint32_t pos = static_cast<uint32_t>(a.p.position[r]);
    float bv = neg_inf();
    int32_t bi = kNoCut;
    for (int i = tid; i < L; i += kThreads) {
      const unsigned long long e = mkeys[i];
      const int32_t t = sort_key_token(e);
      const float sc = __fadd_rn(key_value(sort_key_order(e)), gumbel_noise(philox_numerator(seed, rowid, pos, t, 0)));
      if (beats(sc, t, bv, bi)) {
        bv = sc;
        bi = t;
      }
    }
    Part pp = empty_part();
    pp.best = bv;
    pp.arg = bi;
    warp_part_reduce(pp);
    Part* wp = reinterpret_cast<Part*>(mkeys);  // the keys are no longer needed
    __syncthreads();
    if ((tid & 31) == 0) wp[tid >> 5] = pp;
    __syncthreads();
    if (tid < 32) {
      Part t = (tid < kWarps) ? wp[tid] : empty_part();
      warp_part_reduce(t);
      if (tid == 0) {
        s_token = t.arg;
        s_kept = L;
      }
    }
    __syncthreads();
  }
  if (tid == 0) {
    const bool ok = (s_status == SS_ROW_OK);
    a.out_token[r] = ok ? s_token : -1;
    a.out_status[r] = s_status;
    if (a.out_kept) a.out_kept[r] = ok ? s_kept : 0;
  }
}

// ------------------------------------------------------------------ host --

static thread_local int32_t g_last_cuda_error = 0;
void set_last_cuda_error(int32_t e) { g_last_cuda_error = e; }

static Layout make_layout(int32_t vocab, int32_t es, int cs) {
  Layout L{};
  L.slice_len = static_cast<int32_t>(((static_cast<int64_t>(vocab) + cs - 1) / cs + 31) / 32 * 32);
  int64_t off = (static_cast<int64_t>(L.slice_len) * es + 15) / 16 * 16;
  L.data_bytes = static_cast<int32_t>(off);
  auto take = [&](int64_t bytes, int64_t align) {
    off = (off + align - 1) / align * align;
    const int32_t at = static_cast<int32_t>(off);
    off += bytes;
    return at;
  };
  const int64_t nvec = L.slice_len / (16 / es);
  L.vmax_off = take(nvec * 2, 16);
  L.xm_off = take(L.slice_len / 32 * 4, 16);
  L.hk_off = take(kHashCap * 4, 16);
  L.hc_off = take(kHashCap * 4, 16);
  L.hv_off = take(kHashCap * 4, 16);
  L.work_off = take(kWorkBytes, 16);
  L.rh_off = take(2 * static_cast<int64_t>(cs) * kBuckets * 12, 16);
  L.rec_off = take(kRecs * sizeof(LevelRec), 16);
  L.red_off = take(kRedBytes, 16);
  L.part_off = take(kPartSlots * static_cast<int64_t>(cs) * sizeof(Part), 16);
  L.mbar_off = take(kMaxChunks * 8, 16);
  L.total = static_cast<int32_t>((off + 127) / 128 * 128);
  return L;
}

// Largest shared memory one CTA may hold on this GPU family (227 KiB, dynamic
// and static together).
constexpr int64_t kSmemPerCta = 232448;

static bool layout_fits(int32_t vocab, int32_t es, int cs) {
  // the kernel's static context, and a margin for what the compiler adds
  return make_layout(vocab, es, cs).total + static_cast<int64_t>(sizeof(Ctx)) + 256 <= kSmemPerCta;
}

static int choose_cluster(int32_t vocab, int32_t es) {
  for (int cs = 1; cs <= kMaxCluster; cs <<= 1) {
    const int64_t slice = ((static_cast<int64_t>(vocab) + cs - 1) / cs + 31) / 32 * 32;
    if (slice * es <= kTargetSliceBytes) return cs;
  }
  const int64_t slice = ((static_cast<int64_t>(vocab) + kMaxCluster - 1) / kMaxCluster + 31) / 32 * 32;
  if (slice * es <= kMaxSliceBytes && slice <= kMaxSliceTokens && layout_fits(vocab, es, kMaxCluster))
    return kMaxCluster;
  return 0;
}


template <int DT>
static cudaError_t launch(const KArgs& ka, int cs, cudaStream_t stream) {
  const void* fn = reinterpret_cast<const void*>(&ss_row_kernel<DT>);
  cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, ka.L.total);
  if (e != cudaSuccess) return e;
  // The largest shared-memory carve-out for every launch, whatever its
  // cluster size: an SM switches carve-outs only when idle, so launches that
  // asked for different ones could not share SMs.
  e = cudaFuncSetAttribute(fn, cudaFuncAttributePreferredSharedMemoryCarveout, cudaSharedmemCarveoutMaxShared);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(static_cast<unsigned>(ka.grid_tasks > 0 ? ka.grid_tasks : ka.num_tasks) * cs, 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = ka.L.total;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = cs;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = ka.overlap ? 2 : 1;
  return cudaLaunchKernelEx(&cfg, ss_row_kernel<DT>, ka);
}

static bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

static ss_status check_params(const ss_params& p) {
  if (!p.temperature || !p.seed || !p.position) return SS_ERR_INVALID_ARG;
  if ((p.hist_offsets == nullptr) != (p.hist_ids == nullptr)) return SS_ERR_INVALID_ARG;
  if (p.bias_offsets && (!p.bias_ids || !p.bias_vals)) return SS_ERR_INVALID_ARG;
  return SS_OK;
}

static ss_status run(const KArgs& ka, int32_t dtype, cudaStream_t stream, int cs_override = 0) {
  const int es = (dtype == SS_DTYPE_BF16) ? 2 : 4;
  KArgs k = ka;
  if (!k.shard_rec) {  // the whole vocabulary
    k.shard_off = 0;
    k.shard_len = k.vocab;
  }
  const int cs = cs_override ? cs_override : choose_cluster(k.shard_len, es);
  if (cs == 0) return SS_ERR_UNSUPPORTED;
  k.L = make_layout(k.shard_len, es, cs);
  const cudaError_t e = (dtype == SS_DTYPE_BF16) ? launch<SS_DTYPE_BF16>(k, cs, stream)
                                                 : launch<SS_DTYPE_F32>(k, cs, stream);
  if (e != cudaSuccess) {
    g_last_cuda_error = static_cast<int32_t>(e);
    return SS_ERR_CUDA;
  }
  return SS_OK;
}

// A second stream and fork / join events per host thread and device, for the
// concurrent heavy-row launch.  Created by the thread's first split call on
// the device, outside stream capture; they live as long as the thread.
struct SideStream {
  cudaStream_t stream = nullptr;
  cudaEvent_t fork = nullptr, join = nullptr;
};

static SideStream* side_stream(cudaStream_t main) {
  static thread_local SideStream side[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  SideStream& s = side[dev];
  if (!s.stream) {
    cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(main, &cap) != cudaSuccess || cap != cudaStreamCaptureStatusNone) return nullptr;
    // relaxed capture mode for this thread while creating them, so that a
    // graph another thread may be capturing is not disturbed
    cudaStreamCaptureMode mode = cudaStreamCaptureModeRelaxed;
    if (cudaThreadExchangeStreamCaptureMode(&mode) != cudaSuccess) return nullptr;
    cudaStream_t st = nullptr;
    cudaEvent_t f = nullptr, j = nullptr;
    const bool ok = cudaStreamCreateWithFlags(&st, cudaStreamNonBlocking) == cudaSuccess &&
                    cudaEventCreateWithFlags(&f, cudaEventDisableTiming) == cudaSuccess &&
                    cudaEventCreateWithFlags(&j, cudaEventDisableTiming) == cudaSuccess;
    cudaThreadExchangeStreamCaptureMode(&mode);  // restore the thread's mode
    if (!ok) {
      if (j) cudaEventDestroy(j);
      if (f) cudaEventDestroy(f);
      if (st) cudaStreamDestroy(st);
      return nullptr;
    }
    s.stream = st;
    s.fork = f;
    s.join = j;
  }
  return &s;
}

// Sampling launch: when the rows are many and the cluster can double, the
// heavy rows run on a second stream with twice the CTAs per row while the
// light rows run on the caller's stream; the caller's stream waits for both.
static ss_status run_sample(const KArgs& ka, int32_t dtype, cudaStream_t stream) {
  const int es = (dtype == SS_DTYPE_BF16) ? 2 : 4;
  const int cs = choose_cluster(ka.vocab, es);
  SideStream* side = nullptr;
  if (ka.num_tasks >= 16 && ka.num_tasks <= kMaxOrderedTasks && cs >= 2 && 2 * cs <= kMaxCluster &&
      !ka.debug_processed)
    side = side_stream(stream);
  if (!side) return run(ka, dtype, stream);
  KArgs heavy = ka, light = ka;
  heavy.row_class = 2;
  light.row_class = 1;
  cudaError_t e = cudaEventRecord(side->fork, stream);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(side->stream, side->fork, 0);
  if (e != cudaSuccess) {
    g_last_cuda_error = static_cast<int32_t>(e);
    return SS_ERR_CUDA;
  }
  const ss_status sh = run(heavy, dtype, side->stream, 2 * cs);
  const ss_status sl = run(light, dtype, stream, cs);
  e = cudaEventRecord(side->join, side->stream);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(stream, side->join, 0);
  if (e != cudaSuccess) {
    g_last_cuda_error = static_cast<int32_t>(e);
    return SS_ERR_CUDA;
  }
  return sh != SS_OK ? sh : sl;
}

// Host-side checks of a verification call (everything but the workspace).
static ss_status check_verify(const ss_verify_args* args) {
  if (!args) return SS_ERR_INVALID_ARG;
  const ss_verify_args& A = *args;
  if (A.num_requests < 0 || A.vocab < 1 || A.max_draft < 0 || A.max_draft > kMaxDraft) return SS_ERR_INVALID_ARG;
  if (A.dtype != SS_DTYPE_F32 && A.dtype != SS_DTYPE_BF16) return SS_ERR_INVALID_ARG;
  if (A.flags & ~SS_VERIFY_OVERLAP_PREVIOUS) return SS_ERR_INVALID_ARG;
  if (A.num_target_rows != 0 &&
      (A.num_target_rows < A.num_requests ||
       A.num_target_rows > static_cast<int64_t>(A.num_requests) * (static_cast<int64_t>(A.max_draft) + 1)))
    return SS_ERR_INVALID_ARG;
  if (A.num_requests == 0) return SS_OK;
  const int es = (A.dtype == SS_DTYPE_BF16) ? 2 : 4;
  if (!A.target_logits || (reinterpret_cast<uintptr_t>(A.target_logits) % es) != 0 || !A.draft_offsets)
    return SS_ERR_INVALID_ARG;
  if (A.max_draft > 0 && (!A.draft_tokens || !A.draft_probs)) return SS_ERR_INVALID_ARG;
  if (A.row_stride < A.vocab) return SS_ERR_INVALID_ARG;
  if (A.max_draft > 0 && A.draft_stride < A.vocab) return SS_ERR_INVALID_ARG;
  if (!A.out_tokens || !A.out_num_accepted || !A.out_status) return SS_ERR_INVALID_ARG;
  if (check_params(A.params) != SS_OK) return SS_ERR_INVALID_ARG;
  if (A.params.bitmask && A.params.bitmask_stride < (static_cast<int64_t>(A.vocab) + 31) / 32) return SS_ERR_INVALID_ARG;
  const int64_t tasks = static_cast<int64_t>(A.num_requests) * (static_cast<int64_t>(A.max_draft) + 1);
  if (tasks > 0x7fffffff / kMaxCluster) return SS_ERR_UNSUPPORTED;
  return SS_OK;
}

// The per-request words (arrival counters, then rejection words) sit at the
// end of the workspace and the per-position results at its start.  A workspace sized for (R, max_draft)
// then never holds a counter of one call where another call of a different
// shape put its results, so the counters stay at zero between calls (each
// call leaves its counters at zero) whatever the calls' shapes.
static int32_t* counters_at_end(void* workspace, size_t bytes, int32_t num_requests) {
  const uintptr_t end = reinterpret_cast<uintptr_t>(workspace) + bytes;
  return reinterpret_cast<int32_t*>((end - 8u * static_cast<uintptr_t>(num_requests)) & ~static_cast<uintptr_t>(15));
}

// One verification launch on a checked call and a large enough workspace.
static ss_status verify_launch(const ss_verify_args& A, void* workspace, size_t workspace_bytes,
                               cudaStream_t stream) {
  const int64_t tasks = static_cast<int64_t>(A.num_requests) * (static_cast<int64_t>(A.max_draft) + 1);
  int4* results = reinterpret_cast<int4*>(workspace);
  int32_t* counters = counters_at_end(workspace, workspace_bytes, A.num_requests);
  if (hist_cluster_size(A.vocab, A.dtype) > 0) {
    // bf16 logits: the histogram kernel
    const ss_status s = hist_verify(A, results, counters, stream);
    if (s == SS_ERR_CUDA) g_last_cuda_error = hist_last_error();
    return s;
  }
  KArgs k{};
  k.mode = kModeVerify;
  k.num_tasks = static_cast<int32_t>(tasks);
  k.vocab = A.vocab;
  k.max_draft = A.max_draft;
  k.dtype = A.dtype;
  k.row_stride = A.row_stride;
  k.logits = A.target_logits;
  k.draft_offsets = A.draft_offsets;
  k.draft_tokens = A.draft_tokens;
  k.draft_probs = A.draft_probs;
  k.draft_stride = A.draft_stride;
  k.p = A.params;
  k.out_token = A.out_tokens;
  k.out_num_accepted = A.out_num_accepted;
  k.out_status = A.out_status;
  k.out_kept = A.out_kept;
  k.debug_processed = A.debug_processed;
  k.ws_results = results;
  k.ws_counters = counters;
  // many positions run in several waves: start the costliest first
  if (tasks >= 16 && tasks <= kMaxOrderedTasks) k.row_class = 3;
  return run(k, A.dtype, stream);
}

}  // namespace ss

extern "C" {

size_t ss_workspace_size(int32_t max_requests, int32_t max_draft) {
  if (max_requests < 0 || max_draft < 0 || max_draft > ss::kMaxDraft) return 0;
  const size_t results = static_cast<size_t>(max_requests) * (static_cast<size_t>(max_draft) + 1) * sizeof(int4);
  return results + 2 * static_cast<size_t>(max_requests) * sizeof(int32_t) + 256;
}

ss_status ss_workspace_init(void* workspace, size_t workspace_bytes, ss_stream_t stream) {
  SS_NVTX_RANGE("ss_workspace_init");
  if (!workspace) return SS_ERR_WORKSPACE;
  const cudaError_t e = cudaMemsetAsync(workspace, 0, workspace_bytes, reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) {
    ss::g_last_cuda_error = static_cast<int32_t>(e);
    return SS_ERR_CUDA;
  }
  return SS_OK;
}

// Checks of a sampling call (everything the launch needs).
static ss_status check_sample(const ss_sample_args* args) {
  using namespace ss;
  if (!args) return SS_ERR_INVALID_ARG;
  const ss_sample_args& A = *args;
  if (A.num_rows < 0 || A.vocab < 1) return SS_ERR_INVALID_ARG;
  if (A.dtype != SS_DTYPE_F32 && A.dtype != SS_DTYPE_BF16) return SS_ERR_INVALID_ARG;
  if (A.flags & ~SS_SAMPLE_OVERLAP_PREVIOUS) return SS_ERR_INVALID_ARG;
  if (A.num_rows == 0) return SS_OK;
  const int es = (A.dtype == SS_DTYPE_BF16) ? 2 : 4;
  if (!A.logits || (reinterpret_cast<uintptr_t>(A.logits) % es) != 0 || !A.out_token || !A.out_status)
    return SS_ERR_INVALID_ARG;
  if (A.row_stride != 0 && A.row_stride < A.vocab) return SS_ERR_INVALID_ARG;
  if (check_params(A.params) != SS_OK) return SS_ERR_INVALID_ARG;
  if (A.params.bitmask && A.params.bitmask_stride < (static_cast<int64_t>(A.vocab) + 31) / 32) return SS_ERR_INVALID_ARG;
  return SS_OK;
}

ss_status ss_selftest_wait_timeout(const ss_sample_args* args, uint32_t polls, ss_stream_t stream) {
  SS_NVTX_RANGE("ss_selftest_wait_timeout");
  using namespace ss;
  const ss_status chk = check_sample(args);
  if (chk != SS_OK || args->num_rows == 0) return chk;
  if (polls == 0 || hist_cluster_size(args->vocab, args->dtype) <= 0) return SS_ERR_UNSUPPORTED;
  const ss_status s = hist_sample(*args, reinterpret_cast<cudaStream_t>(stream), polls);
  if (s == SS_ERR_CUDA) g_last_cuda_error = hist_last_error();
  return s;
}

ss_status ss_process_sample(const ss_sample_args* args, ss_stream_t stream) {
  SS_NVTX_RANGE("ss_process_sample");
  using namespace ss;
  const ss_status chk = check_sample(args);
  if (chk != SS_OK || args->num_rows == 0) return chk;
  const ss_sample_args& A = *args;
  KArgs k{};
  k.mode = kModeSample;
  k.num_tasks = A.num_rows;
  k.vocab = A.vocab;
  k.max_draft = 0;
  k.dtype = A.dtype;
  k.row_stride = A.row_stride;
  k.logits = A.logits;
  k.p = A.params;
  k.out_token = A.out_token;
  k.out_status = A.out_status;
  k.out_kept = A.out_kept;
  k.debug_processed = A.debug_processed;
  if (hist_cluster_size(A.vocab, A.dtype) > 0) {
    // bf16 logits: the histogram kernel
    const ss_status s = hist_sample(A, reinterpret_cast<cudaStream_t>(stream));
    if (s == SS_ERR_CUDA) g_last_cuda_error = hist_last_error();
    return s;
  }
  return run_sample(k, A.dtype, reinterpret_cast<cudaStream_t>(stream));
}

ss_status ss_commit_accepted(int32_t num_requests, int32_t max_draft, const int32_t* out_tokens,
                             const int32_t* num_accepted, const int32_t* status, int32_t* tokens, int32_t capacity,
                             int32_t* seq_len, int64_t* position, int32_t* next_token, int32_t* commit_status,
                             ss_stream_t stream) {
  SS_NVTX_RANGE("ss_commit_accepted");
  using namespace ss;
  if (num_requests < 0 || max_draft < 0 || capacity < 1) return SS_ERR_INVALID_ARG;
  if (num_requests == 0) return SS_OK;
  if (!out_tokens || !num_accepted || !status || !tokens || !seq_len || !position || !next_token || !commit_status)
    return SS_ERR_INVALID_ARG;
  const int threads = 256;
  ss_commit_kernel<<<(num_requests + threads - 1) / threads, threads, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
      num_requests, max_draft + 1, out_tokens, num_accepted, status, tokens, capacity, seq_len, position, next_token,
      commit_status);
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) {
    g_last_cuda_error = static_cast<int32_t>(e);
    return SS_ERR_CUDA;
  }
  return SS_OK;
}

size_t ss_shard_record_bytes(int32_t list_cap) {
  if (list_cap < 1 || list_cap > SS_SHARD_MAX_LIST) return 0;
  return 32 + 8 * static_cast<size_t>(list_cap);
}

ss_status ss_sample_shard(const ss_sample_args* args, int32_t vocab_offset, int32_t shard_len, int32_t list_cap,
                          void* records, ss_stream_t stream) {
  SS_NVTX_RANGE("ss_sample_shard");
  using namespace ss;
  if (!args) return SS_ERR_INVALID_ARG;
  const ss_sample_args& A = *args;
  if (A.num_rows < 0 || A.vocab < 1) return SS_ERR_INVALID_ARG;
  if (A.dtype != SS_DTYPE_F32 && A.dtype != SS_DTYPE_BF16) return SS_ERR_INVALID_ARG;
  if (vocab_offset < 0 || (vocab_offset & 31) != 0 || shard_len < 1 ||
      static_cast<int64_t>(vocab_offset) + shard_len > A.vocab)
    return SS_ERR_INVALID_ARG;
  if (ss_shard_record_bytes(list_cap) == 0 || !records || (reinterpret_cast<uintptr_t>(records) & 7u) != 0)
    return SS_ERR_INVALID_ARG;
  if (A.debug_processed) return SS_ERR_INVALID_ARG;
  if (A.num_rows == 0) return SS_OK;
  const int es = (A.dtype == SS_DTYPE_BF16) ? 2 : 4;
  if (!A.logits || (reinterpret_cast<uintptr_t>(A.logits) % es) != 0) return SS_ERR_INVALID_ARG;
  if (A.row_stride != 0 && A.row_stride < shard_len) return SS_ERR_INVALID_ARG;
  if (check_params(A.params) != SS_OK) return SS_ERR_INVALID_ARG;
  if (A.params.bitmask && A.params.bitmask_stride < (static_cast<int64_t>(A.vocab) + 31) / 32) return SS_ERR_INVALID_ARG;
  KArgs k{};
  k.mode = kModeSample;
  k.num_tasks = A.num_rows;
  k.vocab = A.vocab;
  k.dtype = A.dtype;
  k.row_stride = A.row_stride;
  k.logits = A.logits;
  k.p = A.params;
  k.shard_off = vocab_offset;
  k.shard_len = shard_len;
  k.shard_rec = static_cast<uint8_t*>(records);
  k.shard_cap = list_cap;
  return run(k, A.dtype, reinterpret_cast<cudaStream_t>(stream));
}

ss_status ss_merge_shards(const ss_sample_args* args, int32_t num_shards, void* const* records, int32_t list_cap,
                          ss_stream_t stream) {
  SS_NVTX_RANGE("ss_merge_shards");
  using namespace ss;
  if (!args || !records) return SS_ERR_INVALID_ARG;
  const ss_sample_args& A = *args;
  if (A.num_rows < 0 || A.vocab < 1 || num_shards < 1 || num_shards > kMaxShards) return SS_ERR_INVALID_ARG;
  if (ss_shard_record_bytes(list_cap) == 0) return SS_ERR_INVALID_ARG;
  if (A.num_rows == 0) return SS_OK;
  if (!A.out_token || !A.out_status || check_params(A.params) != SS_OK) return SS_ERR_INVALID_ARG;
  MergeArgs m{};
  m.num_rows = A.num_rows;
  m.num_shards = num_shards;
  m.cap = list_cap;
  for (int s = 0; s < num_shards; ++s) {
    if (!records[s] || (reinterpret_cast<uintptr_t>(records[s]) & 7u) != 0) return SS_ERR_INVALID_ARG;
    m.rec[s] = static_cast<const uint8_t*>(records[s]);
  }
  m.p = A.params;
  m.out_token = A.out_token;
  m.out_status = A.out_status;
  m.out_kept = A.out_kept;
  // the merged keys, reused for the warp partials of the final argmax
  const size_t smem = std::max(static_cast<size_t>(num_shards) * list_cap * sizeof(unsigned long long),
                               static_cast<size_t>(kWarps) * sizeof(Part));
  const void* fn = reinterpret_cast<const void*>(&ss_merge_kernel);
  cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (e == cudaSuccess) {
    ss_merge_kernel<<<A.num_rows, kThreads, smem, reinterpret_cast<cudaStream_t>(stream)>>>(m);
    e = cudaGetLastError();
  }
  if (e != cudaSuccess) {
    g_last_cuda_error = static_cast<int32_t>(e);
    return SS_ERR_CUDA;
  }
  return SS_OK;
}

ss_status ss_spec_verify(const ss_verify_args* args, void* workspace, size_t workspace_bytes, ss_stream_t stream) {
  SS_NVTX_RANGE("ss_spec_verify");
  using namespace ss;
  const ss_status chk = check_verify(args);
  if (chk != SS_OK || args->num_requests == 0) return chk;
  if (!workspace || !aligned16(workspace) || workspace_bytes < ss_workspace_size(args->num_requests, args->max_draft))
    return SS_ERR_WORKSPACE;
  return verify_launch(*args, workspace, workspace_bytes, reinterpret_cast<cudaStream_t>(stream));
}

ss_status ss_tree_verify(const ss_tree_args* args, void* workspace, size_t workspace_bytes, ss_stream_t stream) {
  SS_NVTX_RANGE("ss_tree_verify");
  using namespace ss;
  if (!args) return SS_ERR_INVALID_ARG;
  const ss_tree_args& A = *args;
  if (A.num_requests < 0 || A.vocab < 1 || A.max_nodes < 1 || A.max_nodes > SS_TREE_MAX_NODES)
    return SS_ERR_INVALID_ARG;
  if (A.dtype != SS_DTYPE_F32 && A.dtype != SS_DTYPE_BF16) return SS_ERR_INVALID_ARG;
  if (A.flags & ~SS_TREE_OVERLAP_PREVIOUS) return SS_ERR_INVALID_ARG;
  if (A.num_nodes_total != 0 &&
      (A.num_nodes_total < A.num_requests ||
       A.num_nodes_total > static_cast<int64_t>(A.num_requests) * A.max_nodes))
    return SS_ERR_INVALID_ARG;
  if (A.num_requests == 0) return SS_OK;
  const int es = (A.dtype == SS_DTYPE_BF16) ? 2 : 4;
  if (!A.target_logits || (reinterpret_cast<uintptr_t>(A.target_logits) % es) != 0 || !A.node_offsets ||
      !A.parents || !A.node_tokens)
    return SS_ERR_INVALID_ARG;
  if (A.max_nodes > 1 && !A.draft_probs) return SS_ERR_INVALID_ARG;
  if (A.row_stride < A.vocab) return SS_ERR_INVALID_ARG;
  if (A.max_nodes > 1 && A.draft_stride < A.vocab) return SS_ERR_INVALID_ARG;
  if (!A.out_tokens || !A.out_num_accepted || !A.out_status) return SS_ERR_INVALID_ARG;
  if (check_params(A.params) != SS_OK) return SS_ERR_INVALID_ARG;
  if (A.params.bitmask && A.params.bitmask_stride < (static_cast<int64_t>(A.vocab) + 31) / 32) return SS_ERR_INVALID_ARG;
  const int64_t tasks = static_cast<int64_t>(A.num_requests) * A.max_nodes;
  if (tasks > 0x7fffffff / kMaxCluster) return SS_ERR_UNSUPPORTED;
  if (!workspace || !aligned16(workspace) || workspace_bytes < ss_workspace_size(A.num_requests, A.max_nodes - 1))
    return SS_ERR_WORKSPACE;
  KArgs k{};
  k.mode = kModeTree;
  k.num_tasks = static_cast<int32_t>(tasks);
  k.vocab = A.vocab;
  k.max_draft = A.max_nodes - 1;
  k.dtype = A.dtype;
  k.row_stride = A.row_stride;
  k.logits = A.target_logits;
  k.draft_offsets = A.node_offsets;
  k.draft_tokens = A.node_tokens;
  k.tree_parents = A.parents;
  k.draft_probs = A.draft_probs;
  k.draft_stride = A.draft_stride;
  k.p = A.params;
  k.out_token = A.out_tokens;
  k.out_path = A.out_path;
  k.out_num_accepted = A.out_num_accepted;
  k.out_status = A.out_status;
  k.out_kept = A.out_kept;
  k.debug_processed = A.debug_processed;
  k.ws_results = reinterpret_cast<int4*>(workspace);
  k.ws_counters = counters_at_end(workspace, workspace_bytes, A.num_requests);
  k.overlap = (A.flags & SS_TREE_OVERLAP_PREVIOUS) ? 1 : 0;
  k.stated_tasks = A.num_nodes_total;
  if (tasks >= 16 && tasks <= kMaxOrderedTasks) {
    k.row_class = 3;
    // the ordering puts the node slots without work last: stop before them
    if (A.num_nodes_total > 0) k.grid_tasks = A.num_nodes_total;
  }
  return run(k, A.dtype, reinterpret_cast<cudaStream_t>(stream));
}

// ----------------------------------------------------- allocation-free --
// Scratch for ss_spec_verify_noalloc: one file-scope device array, loaded with
// the library and kept by every GPU that uses it until the process exits.
static __device__ __align__(256) unsigned char g_noalloc_scratch[SS_NOALLOC_SCRATCH_BYTES];

namespace {
std::mutex g_noalloc_mutex;
void* g_noalloc_ptr[64] = {};  // device address of g_noalloc_scratch, per device
}  // namespace

ss_status ss_spec_verify_noalloc(const ss_verify_args* args, ss_stream_t stream) {
  SS_NVTX_RANGE("ss_spec_verify_noalloc");
  using namespace ss;
  // every argument is checked before the shared scratch is touched: first
  // the batch against the scratch's size, then the rest
  if (!args) return SS_ERR_INVALID_ARG;
  if (args->num_requests < 0 || args->max_draft < 0 || args->max_draft > kMaxDraft) return SS_ERR_INVALID_ARG;
  const size_t need = ss_workspace_size(args->num_requests, args->max_draft);
  if (need > SS_NOALLOC_SCRATCH_BYTES) return SS_ERR_SCRATCH_LIMIT;
  const ss_status chk = check_verify(args);
  if (chk != SS_OK) return chk;
  if (args->num_requests == 0) return SS_OK;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess || dev < 0 || dev >= 64) {
    g_last_cuda_error = static_cast<int32_t>(e);
    return SS_ERR_CUDA;
  }
  void* scratch = nullptr;
  {
    // First call on this device: look the array's device address up with the
    // device current (host code only sees a stand-in for the symbol).
    std::lock_guard<std::mutex> lock(g_noalloc_mutex);
    if (!g_noalloc_ptr[dev]) {
      e = cudaGetSymbolAddress(&g_noalloc_ptr[dev], g_noalloc_scratch);
      if (e != cudaSuccess) {
        g_noalloc_ptr[dev] = nullptr;
        g_last_cuda_error = static_cast<int32_t>(e);
        return SS_ERR_CUDA;
      }
    }
    scratch = g_noalloc_ptr[dev];
  }
  // The per-request arrival counters (at the end of the scratch) must start
  // at zero; the array keeps whatever the previous call left, so clear them
  // on every call.
  int32_t* counters = counters_at_end(scratch, SS_NOALLOC_SCRATCH_BYTES, args->num_requests);
  const size_t clear = static_cast<size_t>(static_cast<char*>(scratch) + SS_NOALLOC_SCRATCH_BYTES -
                                           reinterpret_cast<char*>(counters));
  e = cudaMemsetAsync(counters, 0, clear, reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) {
    g_last_cuda_error = static_cast<int32_t>(e);
    return SS_ERR_CUDA;
  }
  // (no overlap with the call before: the scratch is cleared in between)
  ss_verify_args A = *args;
  A.flags = 0;
  return verify_launch(A, scratch, SS_NOALLOC_SCRATCH_BYTES, reinterpret_cast<cudaStream_t>(stream));
}

int32_t ss_cluster_size(int32_t vocab, int32_t dtype) {
  if (vocab < 1 || (dtype != SS_DTYPE_F32 && dtype != SS_DTYPE_BF16)) return 0;
  const int h = ss::hist_cluster_size(vocab, dtype);
  if (h > 0) return h;
  return ss::choose_cluster(vocab, dtype == SS_DTYPE_BF16 ? 2 : 4);
}

int32_t ss_last_cuda_error(void) { return ss::g_last_cuda_error; }

const char* ss_status_string(ss_status status) {
  switch (status) {
    case SS_OK: return "ok";
    case SS_ERR_INVALID_ARG: return "invalid argument";
    case SS_ERR_UNSUPPORTED: return "unsupported size";
    case SS_ERR_CUDA: return "CUDA runtime error";
    case SS_ERR_WORKSPACE: return "workspace missing or too small";
    case SS_ERR_SCRATCH_LIMIT: return "batch exceeds the allocation-free entry point's static scratch";
  }
  return "unknown status";
}

const char* ss_version(void) { return "ss 0.4.0 (sm_103a)"; }

}  // extern "C"
