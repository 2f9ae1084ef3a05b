// ss_hist.cu -- sm_103a kernel for bf16 logits: batched sampling and linear
// speculative verification (ss_process_sample / ss_spec_verify, see
// include/ss.h), built on an exact histogram of the row's distinct values.
//
// Why a histogram of values works exactly here: a bf16 logit has at most
// 65,536 values, and every later quantity of a token -- its processed logit
// y = z * fp32(1/T), its place in the (y desc, index asc) order, its
// fixed-point probability mass trunc(exp(y - m) * 2^40) -- is a function of
// its value alone.  So a count per distinct value gives, with integer
// arithmetic and no sort, the exact top-k cut (counts from the top), the
// exact mass of every prefix and hence the exact top-p cut (SonicSampler
// abstract: top-k / top-p over large vocabularies), and the min-p cut; only
// tokens tied at the cut value need their indices, and only the kept set needs
// noise for the draw (FlashSampling news page: argmax of logit plus Gumbel
// noise, per-tile maxima then a cross-tile reduction).
//
// Execution model, per task (a logits row, or one target position of a
// verification request): one thread-block cluster of C CTAs, CTA r owning
// tokens [r * slice, (r + 1) * slice) of the row.
//   1. set-up: bulk (TMA) copies of the slice into shared memory in 16 KB
//      chunks; meanwhile the row's parameters, its penalised / biased tokens
//      ("patched") in a table and the grammar mask's allow bits.
//   2. staging pass, chunk by chunk as the copies land: the patched tokens'
//      raw logits go to the table, excluded tokens (mask, patched) are
//      overwritten with -inf in place, tiny non-zero values are moved to the
//      exact entries, each 16-token pair of vectors' maximum is stored.  Then
//      the patched tokens are processed in fp32 into exact entries.
//   3. cluster exchange 1 (distributed shared memory, one cluster barrier):
//      slice maxima, statuses, the draft token's value, greedy arguments, and
//      for top-k rows each CTA's count of 16-token pairs per binade below its
//      maximum.  Summed over the cluster, those counts certify a value tau
//      with at least k tokens at or above it: only tokens >= tau can be in
//      the top-k.
//   4. rows with a top-k or top-p cut: one pass counts the candidate tokens
//      per slot (slot = distinct value, counted from the row maximum down);
//      every CTA sums its counts and masses into 64 coarse groups and pushes
//      them to every CTA (exchange 2).  Every CTA then locates the cuts
//      identically: coarse groups first, then the slots of one group read
//      from all CTAs, merged with the group's entries gathered from all CTAs.
//      Ties at the cut value are resolved by index in the CTA where the cut
//      falls.
//   5. the draw over the kept set with Philox noise keyed by token, pruned by
//      the largest possible noise and by a cheap bound before any logarithm;
//      the best (score, token) of each CTA is reduced over the cluster.
//   6. verification positions accept with u * q(x) < P(x), else draw from the
//      residual max(P - q, 0); the last position of a request to finish
//      writes the request's tokens.
#include <cooperative_groups.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include <algorithm>
#include <type_traits>

#include "ss.h"
#include "ss_hist.h"
#include "ss_philox.cuh"
#include "ss_ptx.cuh"

namespace cg = cooperative_groups;

namespace ss {
namespace hist {

constexpr int kThreads = 512;
constexpr int kWarps = kThreads / 32;
constexpr int kSlots = 6144;      // distinct values counted, from the row maximum down
constexpr int kGroups = 64;       // coarse groups of slots (plus a tail group of entries)
constexpr int kGatherCap = 512;   // entries of one coarse group, over the cluster
constexpr int kFineMax = 256;     // slots one coarse group may span (runs of equal y extend a group)
constexpr int kEntCap = 1024;     // exact entries per CTA (patched tokens and tiny values)
constexpr int kHashCap = 1024;    // patch table slots
constexpr int kCertBins = 64;     // bins below the maximum counted for the top-k certificate
constexpr int kCertShift = 3;     // certificate bin = 16-bit order key >> 3 (16 bins per binade)
constexpr int kTieEnt = 64;       // entries tied at a cut value, per CTA
constexpr int kFastK = 1024;      // short path: top-k rows up to this k
constexpr int kFastCap = 2048;    // short path: candidates of a row, merged into rank 0
constexpr int kRankSortMax = 768; // short path: a CTA's run by rank sort up to this many, else bitonic
constexpr int kChunkTokens = 8192;
constexpr int kMaxChunks = 8;
constexpr int kMaxCluster = 8;
constexpr int kSliceTarget = 32768;  // tokens per CTA that keep two CTAs per SM
constexpr int kSliceMax = 49152;
constexpr uint32_t kWaitPolls = 1u << 22;
constexpr int kBiasFlag = 1 << 30;
constexpr uint32_t kNegInfPair = 0xff80ff80u;
constexpr uint32_t kTinyA = 0x3780u;
// A rejection at draft position j is recorded as kRejBase - j in the
// request's rejection word (atomic maximum): the word exceeds kRejBase - j
// exactly when a position before j has rejected.
constexpr int32_t kRejBase = kMaxDraft + 2;  // |z| below 2^-16: tiny (exact entries unless zero)
// Fixed-point masses of tokens more than this far below the maximum are 0.
constexpr float kMassRange = 28.2f;

static_assert(kSlots % kGroups == 0, "groups tile the slots");
// the entries' group offsets and order sit behind the slot counts, in the
// part of the region the patch table no longer needs
static_assert(kSlots * 2 + (kGroups + 2) * 4 + kEntCap * 2 <= kHashCap * 16, "entry order fits the region");
static_assert(kEntCap % kThreads == 0, "entries per thread");
static_assert(kHashCap * 16 >= kFastCap * 8, "the histogram region holds the short path's candidates");
static_assert((kSliceMax + kChunkTokens - 1) / kChunkTokens < kMaxChunks, "a barrier slot stays free for the self-test");

// Phase timestamps for tracing (built only with -DSS_HIST_STAMPS): the
// global timer at the end of each phase, per CTA, read back with
// ss_hist_stamps_copy.
#ifdef SS_HIST_STAMPS
constexpr int kStampCtas = 16384, kStampPhases = 48;
__device__ unsigned long long g_stamps[kStampCtas][kStampPhases];
#define SS_STAMP(k)                                                                \
  do {                                                                             \
    if (threadIdx.x == 0 && blockIdx.x < kStampCtas) {                             \
      if ((k) == 0) {                                                              \
        unsigned long long t_;                                                     \
        asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t_));                     \
        g_stamps[blockIdx.x][kStampPhases - 1] = t_;                               \
      }                                                                            \
      g_stamps[blockIdx.x][k] = static_cast<unsigned long long>(clock64());        \
    }                                                                              \
  } while (0)
#define SS_TRACE(k, v)                                                             \
  do {                                                                             \
    if (threadIdx.x == 0 && blockIdx.x < kStampCtas) g_stamps[blockIdx.x][k] = (v); \
  } while (0)
#else
#define SS_STAMP(k) \
  do {            \
  } while (0)
#define SS_TRACE(k, v) \
  do {               \
  } while (0)
#endif

// ---------------------------------------------------------------- helpers --

// Programmatic dependent launch (no-ops in a launch without it).
__device__ __forceinline__ void grid_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void grid_dependency_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

__device__ __forceinline__ float ninf() { return __int_as_float(0xff800000); }
__device__ __forceinline__ float pinf() { return __int_as_float(0x7f800000); }
__device__ __forceinline__ float bf16_to_f(uint32_t h) { return __uint_as_float((h & 0xffffu) << 16); }

// Order-preserving key of a float (larger value, larger key); -0 folds to +0.
__device__ __forceinline__ uint32_t okey(float y) {
  const uint32_t b = __float_as_uint(y + 0.0f);
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}
__device__ __forceinline__ float okey_value(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7fffffffu) : ~k);
}
// Entry key: ascending order = (y descending, token ascending).
__device__ __forceinline__ unsigned long long ekey(float y, int32_t t) {
  return (static_cast<unsigned long long>(~okey(y)) << 32) | static_cast<uint32_t>(t);
}
__device__ __forceinline__ float ekey_y(unsigned long long e) { return okey_value(~static_cast<uint32_t>(e >> 32)); }
__device__ __forceinline__ int32_t ekey_t(unsigned long long e) { return static_cast<int32_t>(static_cast<uint32_t>(e)); }

// Fixed-point mass trunc(exp(y - m) * 2^40) (0 for y = -inf); a function of
// y alone for a given row, so every CTA computes the same integers.
// The truncation of e * 2^40 (e in [0, 1]) is taken from e's bits with
// integer shifts: the same integer as the float -> 64-bit conversion, which
// sm_103 issues at a fraction of the integer rate.
__device__ __forceinline__ unsigned long long fmass(float y, float m) {
  const float e = fminf(__expf(__fsub_rn(y, m)), 1.0f);
  const uint32_t b = __float_as_uint(e);
  const int sh = static_cast<int>(b >> 23) - 127 + 40 - 23;  // e * 2^40 = (1.f as an integer) * 2^sh
  const unsigned long long mant = (b & 0x7fffffu) | 0x800000u;
  if (sh >= 0) return mant << sh;  // sh <= 17
  return (sh > -24) ? (mant >> (-sh)) : 0ull;  // zero and subnormal e give 0
}
__device__ __forceinline__ unsigned long long mass_target(float p, unsigned long long S) {
  return static_cast<unsigned long long>(ceil(static_cast<double>(p) * static_cast<double>(S)));
}

__device__ __forceinline__ uint32_t bmax2(uint32_t a, uint32_t b) {  // bf16x2 maximum, NaN propagating
  uint32_t r;
  asm("max.NaN.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}
__device__ __forceinline__ float fmax_nan(float a, float b) {
  float r;
  asm("max.NaN.f32 %0, %1, %2;" : "=f"(r) : "f"(a), "f"(b));
  return r;
}

// Replace the tokens whose allow bit is 0 by -inf.  A = 8 allow bits of the
// vector; each bit is moved to the sign of a byte, and a sign-replicating
// byte permute widens it to the 16-bit lane mask.
__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t sel) {
  uint32_t r;
  asm("prmt.b32 %0, %1, 0, %2;" : "=r"(r) : "r"(a), "r"(sel));
  return r;
}

__device__ __forceinline__ uint4 apply_allow(uint4 d, uint32_t A) {
  const uint32_t s_lo = ((A & 0xfu) * 0x10204080u) & 0x80808080u;
  const uint32_t s_hi = ((A >> 4) * 0x10204080u) & 0x80808080u;
  const uint32_t m0 = prmt(s_lo, 0x9988u), m1 = prmt(s_lo, 0xBBAAu);
  const uint32_t m2 = prmt(s_hi, 0x9988u), m3 = prmt(s_hi, 0xBBAAu);
  d.x = (d.x & m0) | (kNegInfPair & ~m0);
  d.y = (d.y & m1) | (kNegInfPair & ~m1);
  d.z = (d.z & m2) | (kNegInfPair & ~m2);
  d.w = (d.w & m3) | (kNegInfPair & ~m3);
  return d;
}

// Bit 15 / 31 set for the halves that hold a tiny non-zero value
// (0 < |z| < 2^-16).
__device__ __forceinline__ uint32_t tiny_pair(uint32_t w) {
  const uint32_t t = w & 0x7fff7fffu;
  const uint32_t small = ~((t | 0x80008000u) - (kTinyA | (kTinyA << 16))) & 0x80008000u;
  const uint32_t nz = (t + 0x7fff7fffu) & 0x80008000u;
  return small & nz;
}

// The smallest magnitude (16-bit pattern without the sign) among the eight
// bf16 values of a vector: three 16x2 minima and one of the two halves.
__device__ __forceinline__ uint32_t min_mag8(uint4 d) {
  uint32_t a, b, r;
  asm("min.u16x2 %0, %1, %2;" : "=r"(a) : "r"(d.x & 0x7fff7fffu), "r"(d.y & 0x7fff7fffu));
  asm("min.u16x2 %0, %1, %2;" : "=r"(b) : "r"(d.z & 0x7fff7fffu), "r"(d.w & 0x7fff7fffu));
  asm("min.u16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return min(r & 0xffffu, r >> 16);
}

__device__ __forceinline__ bool beats(float s, int32_t t, float bs, int32_t bt) {
  return s > bs || (s == bs && t < bt);
}

// --------------------------------------------------------- slot mapping --
// Slots enumerate distinct bf16 values from the row maximum down: positive
// values by falling magnitude, then one slot for +-0, then negative values by
// rising magnitude.  Tiny non-zero values never reach a slot (they are exact
// entries).  slot(h) = sign ? nb + a' : pb - a', a' = max(|h|, 0x3AFF).
struct SlotMap {
  int32_t pb, nb;
  int32_t zero;  // slot of +-0, or -1 when the maximum is negative
  int32_t ns;    // slots in use (<= kSlots); -inf and below map past it
};

__device__ __forceinline__ int32_t slot_of(const SlotMap& M, uint32_t h) {
  const int32_t a = max(static_cast<int32_t>(h & 0x7fffu), static_cast<int32_t>(kTinyA - 1));
  return (h & 0x8000u) ? M.nb + a : M.pb - a;
}
__device__ __forceinline__ float slot_z(const SlotMap& M, int32_t s) {
  if (M.zero >= 0) {
    if (s < M.zero) return bf16_to_f(static_cast<uint32_t>(M.pb - s));
    if (s == M.zero) return 0.0f;
  }
  return bf16_to_f(0x8000u | static_cast<uint32_t>(s - M.nb));
}

__device__ SlotMap make_slot_map(float zmax) {
  SlotMap M;
  const uint32_t hb = __float_as_uint(zmax) >> 16;  // zmax is a bf16 value
  const int32_t a = static_cast<int32_t>(hb & 0x7fffu);
  if (zmax == ninf()) {
    M.pb = 0;
    M.nb = 0;
    M.zero = -1;
    M.ns = 0;
    return M;
  }
  if (!(hb & 0x8000u) || a == 0) {  // maximum >= 0 (it is 0 or at least 2^-9: tiny values are entries)
    M.pb = max(a, static_cast<int32_t>(kTinyA - 1));
    M.zero = M.pb - static_cast<int32_t>(kTinyA - 1);
    M.nb = M.zero + 1 - static_cast<int32_t>(kTinyA);
  } else {
    M.pb = -(1 << 20);
    M.zero = -1;
    M.nb = -a;
  }
  M.ns = min(kSlots, M.nb + 0x7f80);  // -inf and everything below the window land past ns
  return M;
}

// ------------------------------------------------------------------ args --

struct HArgs {
  int32_t mode;  // 0 sampling, 1 verification
  int32_t num_tasks;
  int32_t vocab, max_draft;
  // verification: the number of requests; the caller's count of target rows
  // (0: none; checked against the offsets when given); compact: the launch
  // has one cluster per target row (num_tasks = target_rows), else one per
  // (request, position up to max_draft)
  int32_t nreq, target_rows, compact;
  int64_t row_stride;
  const uint16_t* logits;
  const int32_t* draft_offsets;
  const int32_t* draft_tokens;
  const float* draft_probs;
  int64_t draft_stride;
  ss_params p;
  int32_t* out_token;  // sampling [n]; verification [R, max_draft + 1]
  int32_t* out_num_accepted;
  int32_t* out_status;
  int32_t* out_kept;
  float* debug;
  int4* ws_results;
  int32_t* ws_counters;
  int32_t ncta, slice, bulk;
  int32_t o_vb, o_hist, o_el, o_xm, o_mg, o_mbar, total;
  uint32_t stall_polls;  // self-test: a bounded wait on a barrier nothing completes
  int32_t overlap;       // sampling: launched to overlap the sampling call before it
};

// Per-CTA partial of exchange 1.
struct alignas(16) Part1 {
  float zmax;     // largest staged logit (bf16 value, NaN if any)
  float emax;     // largest entry y (z for greedy rows)
  int32_t arg;    // greedy: lowest index of the CTA's largest item
  int32_t status;
  int32_t nent;
  float xy;       // processed value of the draft token (its CTA)
  int32_t xhere;
  int32_t zbin;   // certificate bin of zmax (16-bit order key >> kCertShift)
  int32_t rej;    // verification: the request's rejection word as this CTA read it
  int32_t pad[3];
  uint32_t cert[kCertBins / 2];  // 16-token pairs whose maximum lies d bins below zbin (16-bit halves)
};

// Per-CTA partial of a draw / mass exchange.
struct alignas(16) PartD {
  float best;
  int32_t arg;
  int32_t count;
  int32_t pad;
  unsigned long long mass;
  unsigned long long pad2;
};

struct Ctx {
  // task
  int32_t valid, row, req, j, k, bad_k, d0, x, drow, nreq;
  int32_t skip_draw;  // verification: a position before this one has rejected
  int64_t row_off;
  int32_t lo, n, nvec, nch, n8;
  // parameters
  float T, inv_t, top_p, min_p, rep, freq, pres, lmp;
  int32_t greedy, top_k, k_on, p_on, mp_on, need_hist, use_mask, has_excl;
  uint32_t seed_lo, seed_hi, pos, rowid;
  int32_t h0, h1, b0, b1;
  int32_t status;   // local, then cluster-wide
  int32_t pstatus;  // what the parameters alone give
  int32_t nent;     // local entries appended
  int32_t ne;       // local entries kept
  int32_t n_g;      // entries gathered for one coarse group
  int32_t npatch;
  // after exchange 1
  float m, zmax;
  int32_t arg;
  float xy;
  int32_t xhere;
  uint32_t tau_key;  // top-k candidates: tokens whose 16-bit order key is >= this
  unsigned long long tau_pairs;  // pairs at or above tau (summed over the cluster)
  SlotMap M;
  // cut: K = {y > cut_v} U {y == cut_v, token <= cut_t}
  float cut_v;
  int32_t cut_t;
  unsigned long long kcount, kmass;  // |K| and its fixed-point mass
  // locate results
  int32_t w_found, w_slot, w_grp;
  float w_v;
  unsigned long long w_take, w_cc, w_cm;
  int32_t tie_rank, tie_local;
  // this CTA's largest staged pair (index) and largest entry: the draw's seeds
  int32_t seed_pair, seed_et;
  float seed_ey;
  unsigned long long below;
  unsigned long long ntot, stot;  // count and mass of every counted item
  // scratch
  int32_t pick;
  int32_t tcut_in;  // tie cutoff, written by the CTA that resolves it
  int32_t xpar;     // buffer of the next draw / mass exchange
  uint32_t fail_key;  // the largest entry key failing min-p (cluster), and this CTA's
  uint32_t fail_loc;
};

__shared__ Ctx g;
__shared__ Part1 g_p1[kMaxCluster];
__shared__ Part1 g_mine;
__shared__ PartD g_pd[2][kMaxCluster];
__shared__ __align__(16) unsigned char g_red[(kWarps + 1) * 8];
__shared__ unsigned long long g_scan[2 * (kWarps + 1)];
__shared__ __align__(16) unsigned char g_red2[(kWarps + 1) * 16];
__shared__ int32_t g_gb[kGroups + 2];                // coarse group bounds (slots)
__shared__ uint32_t g_gcnt[kGroups + 1];
__shared__ unsigned long long g_gmass[kGroups + 1];
__shared__ uint32_t g_ecnt[kGroups + 1];             // this CTA's entries per group
__shared__ unsigned long long g_emass[kGroups + 1];
__shared__ uint32_t g_fc[kFineMax];                  // one group's slot counts (all CTAs)
__shared__ int16_t g_epos[kEntCap];                  // slot position of each local entry
__shared__ int32_t g_goff[kMaxCluster + 1];
__shared__ int32_t g_gr0[kMaxCluster];       // one group's entry range in every CTA
__shared__ int32_t g_grc[kMaxCluster + 1];
__shared__ uint32_t g_rtie[kMaxCluster];
__shared__ uint32_t g_cert[kCertBins / 2];  // two 16-bit bin counts per word
__shared__ int32_t g_tietok[kTieEnt];
__shared__ uint32_t g_prm[32];           // the request's parameter words
__shared__ int32_t g_loc[3];             // compact verification: request, position, count matches
__shared__ uint32_t g_dscore;            // the draw's best score so far (order key; 0: none)
__shared__ int32_t g_dtok;               // the lowest token holding it
__shared__ int32_t g_fpos[3];            // short path: first failing positions (top-p, min-p), draft position
__shared__ int32_t g_runs[kMaxCluster][2];  // short path: every CTA's run (region flag, length)

extern __shared__ __align__(128) uint8_t g_dyn[];

__device__ __forceinline__ uint32_t key16(uint32_t h) { return (h & 0x8000u) ? (~h & 0xffffu) : (h | 0x8000u); }
__device__ __forceinline__ uint32_t key16_bits(uint32_t k) { return (k & 0x8000u) ? (k & 0x7fffu) : (~k & 0xffffu); }

// ------------------------------------------------------ block reductions --
// Warp partials go through shared memory; 32-bit partials are read back by
// every thread as four 16-byte loads, wider ones are combined by warp 0 and
// broadcast.  Either way the combine over the 16 warps is not a 16-step loop
// in every thread.

__device__ __forceinline__ void warp_best(float& s, int32_t& t, int width) {
  for (int o = width >> 1; o; o >>= 1) {
    const float os = __shfl_xor_sync(0xffffffffu, s, o);
    const int32_t ot = __shfl_xor_sync(0xffffffffu, t, o);
    if (beats(os, ot, s, t)) {
      s = os;
      t = ot;
    }
  }
}

// (score desc, token asc) arg-reduction over the block; every thread gets it.
__device__ __forceinline__ void block_best(float& s, int32_t& t) {
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  warp_best(s, t, 32);
  float* rs = reinterpret_cast<float*>(g_red);
  int32_t* rt = reinterpret_cast<int32_t*>(g_red) + (kWarps + 1);
  __syncthreads();
  if (lane == 0) {
    rs[wid] = s;
    rt[wid] = t;
  }
  __syncthreads();
  if (wid == 0) {
    float x = (lane < kWarps) ? rs[lane] : ninf();
    int32_t y = (lane < kWarps) ? rt[lane] : 0x7fffffff;
    warp_best(x, y, kWarps);
    if (lane == 0) {
      rs[kWarps] = x;
      rt[kWarps] = y;
    }
  }
  __syncthreads();
  s = rs[kWarps];
  t = rt[kWarps];
}

// Two (score desc, token asc) arg-reductions over the block in one pass.
__device__ __forceinline__ void block_best2(float& s1, int32_t& t1, float& s2, int32_t& t2) {
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  warp_best(s1, t1, 32);
  warp_best(s2, t2, 32);
  float* rs1 = reinterpret_cast<float*>(g_red2);
  int32_t* rt1 = reinterpret_cast<int32_t*>(rs1 + (kWarps + 1));
  float* rs2 = reinterpret_cast<float*>(rt1 + (kWarps + 1));
  int32_t* rt2 = reinterpret_cast<int32_t*>(rs2 + (kWarps + 1));
  __syncthreads();
  if (lane == 0) {
    rs1[wid] = s1;
    rt1[wid] = t1;
    rs2[wid] = s2;
    rt2[wid] = t2;
  }
  __syncthreads();
  if (wid == 0) {
    float x1 = (lane < kWarps) ? rs1[lane] : ninf(), x2 = (lane < kWarps) ? rs2[lane] : ninf();
    int32_t y1 = (lane < kWarps) ? rt1[lane] : 0x7fffffff, y2 = (lane < kWarps) ? rt2[lane] : 0x7fffffff;
    warp_best(x1, y1, kWarps);
    warp_best(x2, y2, kWarps);
    if (lane == 0) {
      rs1[kWarps] = x1;
      rt1[kWarps] = y1;
      rs2[kWarps] = x2;
      rt2[kWarps] = y2;
    }
  }
  __syncthreads();
  s1 = rs1[kWarps];
  t1 = rt1[kWarps];
  s2 = rs2[kWarps];
  t2 = rt2[kWarps];
}

template <typename T>
__device__ __forceinline__ T block_sum(T v) {
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
#pragma unroll
  for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  T* r = reinterpret_cast<T*>(g_red);
  __syncthreads();
  if (lane == 0) r[wid] = v;
  __syncthreads();
  if constexpr (sizeof(T) == 4) {
    const uint4* r4 = reinterpret_cast<const uint4*>(r);
    T acc = 0;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint4 q = r4[i];
      acc += (static_cast<T>(q.x) + static_cast<T>(q.y)) + (static_cast<T>(q.z) + static_cast<T>(q.w));
    }
    return acc;
  } else {
    if (wid == 0) {
      T x = (lane < kWarps) ? r[lane] : T(0);
#pragma unroll
      for (int o = kWarps >> 1; o; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
      if (lane == 0) r[kWarps] = x;
    }
    __syncthreads();
    return r[kWarps];
  }
}

// Exclusive prefix over the block (thread order); *total gets the sum.
__device__ __forceinline__ int32_t block_excl_scan(int32_t v, int32_t* total) {
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  int32_t x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int32_t y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  int32_t* r = reinterpret_cast<int32_t*>(g_red);
  __syncthreads();
  if (lane == 31) r[wid] = x;
  __syncthreads();
  if (wid == 0) {  // exclusive prefix of the warp totals, and the total
    const int32_t w = (lane < kWarps) ? r[lane] : 0;
    int32_t inc = w;
#pragma unroll
    for (int o = 1; o < kWarps; o <<= 1) {
      const int32_t y = __shfl_up_sync(0xffffffffu, inc, o);
      if (lane >= o) inc += y;
    }
    __syncwarp();
    if (lane < kWarps) r[lane] = inc - w;
    if (lane == kWarps - 1) r[kWarps] = inc;
  }
  __syncthreads();
  *total = r[kWarps];
  return r[wid] + x - v;
}

// Inclusive prefix over the block of a (count, mass) pair (thread order);
// the totals land in *tc / *tm.  Called by all threads.
__device__ __forceinline__ void block_scan2(unsigned long long& c, unsigned long long& m, unsigned long long* tc,
                                            unsigned long long* tm) {
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const unsigned long long yc = __shfl_up_sync(0xffffffffu, c, o);
    const unsigned long long ym = __shfl_up_sync(0xffffffffu, m, o);
    if (lane >= o) {
      c += yc;
      m += ym;
    }
  }
  unsigned long long* r = reinterpret_cast<unsigned long long*>(g_scan);
  __syncthreads();
  if (lane == 31) {
    r[wid] = c;
    r[(kWarps + 1) + wid] = m;
  }
  __syncthreads();
  if (wid == 0) {
    const unsigned long long wc = (lane < kWarps) ? r[lane] : 0, wm = (lane < kWarps) ? r[(kWarps + 1) + lane] : 0;
    unsigned long long ic = wc, im = wm;
#pragma unroll
    for (int o = 1; o < kWarps; o <<= 1) {
      const unsigned long long yc = __shfl_up_sync(0xffffffffu, ic, o);
      const unsigned long long ym = __shfl_up_sync(0xffffffffu, im, o);
      if (lane >= o) {
        ic += yc;
        im += ym;
      }
    }
    __syncwarp();
    if (lane < kWarps) {
      r[lane] = ic - wc;
      r[(kWarps + 1) + lane] = im - wm;
    }
    if (lane == kWarps - 1) {
      r[kWarps] = ic;
      r[(kWarps + 1) + kWarps] = im;
    }
  }
  __syncthreads();
  c += r[wid];
  m += r[(kWarps + 1) + wid];
  *tc = r[kWarps];
  *tm = r[(kWarps + 1) + kWarps];
}

// The coarse group where the running count (by_mass = 0) or mass (1) first
// reaches `target`, and the count / mass before it; one warp.  Returns the
// group (-1 if none) in g.pick and the sums in g.w_cc / g.w_cm.
__device__ void coarse_locate(int by_mass, unsigned long long target) {
  Ctx& c = g;
  if (threadIdx.x < 32) {
    const int lane = threadIdx.x;
    constexpr int kPer = (kGroups + 1 + 31) / 32;  // groups per lane, in order
    unsigned long long cc = 0, cm = 0;
    for (int i = 0; i < kPer; ++i) {
      const int q = lane * kPer + i;
      if (q <= kGroups) {
        cc += g_gcnt[q];
        cm += g_gmass[q];
      }
    }
    unsigned long long ic = cc, im = cm;  // inclusive over lanes
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const unsigned long long yc = __shfl_up_sync(0xffffffffu, ic, o);
      const unsigned long long ym = __shfl_up_sync(0xffffffffu, im, o);
      if (lane >= o) {
        ic += yc;
        im += ym;
      }
    }
    unsigned long long bc = ic - cc, bm = im - cm;  // before this lane's groups
    int found = -1;
    unsigned long long fc = 0, fm = 0;
    for (int i = 0; i < kPer; ++i) {
      const int q = lane * kPer + i;
      if (q > kGroups) break;
      const unsigned long long add = by_mass ? g_gmass[q] : g_gcnt[q];
      if (found < 0 && add > 0 && (by_mass ? bm : bc) + add >= target) {
        found = q;
        fc = bc;
        fm = bm;
      }
      bc += g_gcnt[q];
      bm += g_gmass[q];
    }
    const unsigned ball = __ballot_sync(0xffffffffu, found >= 0);
    if (ball == 0) {
      if (lane == 0) c.pick = -1;
    } else if (lane == __ffs(ball) - 1) {
      c.pick = found;
      c.w_cc = fc;
      c.w_cm = fm;
    }
  }
  __syncthreads();
}

// ------------------------------------------------------------- the task --

// Thread 0: the task's row, its slice, and the bulk copies (issued first, so
// that they overlap everything else of the set-up); then the parameters.
__device__ void decode_and_copy(const HArgs& a, int req, int j, int rank) {
  Ctx& c = g;
  c.valid = 1;
  c.bad_k = 0;
  c.status = SS_ROW_OK;
  c.nent = 0;
  c.npatch = 0;
  c.xpar = 0;
  c.kcount = 0;
  c.kmass = 0;
  c.nreq = 0;
  c.skip_draw = 0;
  c.x = -1;
  c.drow = -1;
  c.d0 = 0;
  int k = 0;
  int64_t row = req;
  if (a.mode == 1) {
    c.nreq = a.nreq;
    c.d0 = a.draft_offsets[req];
    k = a.draft_offsets[req + 1] - c.d0;
    if (k < 0 || k > a.max_draft) {
      c.bad_k = 1;
      c.status = SS_ROW_BAD_PARAM;
      if (j != 0) c.valid = 0;
      row = -1;
    } else {
      if (j > k) c.valid = 0;
      row = static_cast<int64_t>(c.d0) + req + j;
    }
  }
  c.req = req;
  c.j = j;
  c.k = k;
  c.row = static_cast<int32_t>(row);
  c.lo = rank * a.slice;
  c.n = max(0, min(a.slice, a.vocab - c.lo));
  c.nvec = a.slice / 8;
  c.n8 = c.n & ~7;
  c.nch = 0;
  if (!c.valid || c.bad_k) return;
  c.row_off = row * a.row_stride;
  if (a.bulk && c.n8 > 0) {
    uint64_t* mbar = reinterpret_cast<uint64_t*>(g_dyn + a.o_mbar);
    const int nch = (c.n8 + kChunkTokens - 1) / kChunkTokens;
    for (int ch = 0; ch < nch; ++ch) mbar_init(mbar + ch, 1);
    fence_barrier_init();
    const uint16_t* src = a.logits + c.row_off + c.lo;
    for (int ch = 0; ch < nch; ++ch) {
      const int t0 = ch * kChunkTokens;
      const uint32_t bytes = static_cast<uint32_t>(min(kChunkTokens, c.n8 - t0)) * 2u;
      mbar_arrive_expect_tx(mbar + ch, bytes);
      bulk_load(g_dyn + t0 * 2, src + t0, bytes, mbar + ch);
    }
    c.nch = nch;
  }
  if (a.mode == 1 && j < k) {
    c.x = a.draft_tokens[c.d0 + j];
    c.drow = c.d0 + j;
  }
}

__device__ void read_params(const HArgs& a, int j);

// Warp 1: the request's parameter words, one global load per lane (all in
// flight at once), into g_prm; then its lane 0 checks them (read_params),
// while thread 0 issues the bulk copies.
__device__ void load_params(const HArgs& a, int req, int j) {
  const ss_params& p = a.p;
  const int lane = threadIdx.x & 31;
  const int i = req;
  uint32_t v = 0;
  switch (lane) {
    case 0: v = __float_as_uint(p.temperature[i]); break;
    case 1: v = p.top_k ? static_cast<uint32_t>(p.top_k[i]) : 0u; break;
    case 2: v = __float_as_uint(p.top_p ? p.top_p[i] : 1.0f); break;
    case 3: v = __float_as_uint(p.min_p ? p.min_p[i] : 0.0f); break;
    case 4: v = __float_as_uint(p.repetition ? p.repetition[i] : 1.0f); break;
    case 5: v = __float_as_uint(p.frequency ? p.frequency[i] : 0.0f); break;
    case 6: v = __float_as_uint(p.presence ? p.presence[i] : 0.0f); break;
    case 7: v = static_cast<uint32_t>(p.seed[i]); break;
    case 8: v = static_cast<uint32_t>(p.seed[i] >> 32); break;
    case 9: v = p.row_id ? p.row_id[i] : static_cast<uint32_t>(i); break;
    case 10: v = static_cast<uint32_t>(p.position[i]); break;
    case 11: v = static_cast<uint32_t>(static_cast<uint64_t>(p.position[i]) >> 32); break;
    case 12: v = p.hist_offsets ? static_cast<uint32_t>(p.hist_offsets[i]) : 0u; break;
    case 13: v = p.hist_offsets ? static_cast<uint32_t>(p.hist_offsets[i + 1]) : 0u; break;
    case 14: v = p.bias_offsets ? static_cast<uint32_t>(p.bias_offsets[i]) : 0u; break;
    case 15: v = p.bias_offsets ? static_cast<uint32_t>(p.bias_offsets[i + 1]) : 0u; break;
    case 16: v = (p.bitmask && (!p.use_bitmask || p.use_bitmask[i])) ? 1u : 0u; break;
    case 17: v = (a.mode == 1) ? static_cast<uint32_t>(a.draft_offsets[i]) : 0u; break;
    case 18: v = (a.mode == 1) ? static_cast<uint32_t>(a.draft_offsets[i + 1]) : 0u; break;
    default: break;
  }
  // the loads are issued: let thread 0 queue the bulk copies behind them
  asm volatile("bar.arrive 1, 64;" ::: "memory");
  if (lane < 19) g_prm[lane] = v;
  __syncwarp();
  if (lane == 0) read_params(a, j);
}

// Compact verification launches (the caller gave the number of target
// rows): one cluster per target row, in the order of the full launch --
// position-major, every request's position 0 first, then position 1 of the
// requests that have one, and so on.  A request's draft count k_i counts as 0
// when it lies outside [0, max_draft] (such a request has position 0 only,
// which reports it).
__device__ __forceinline__ int drafts_of(const HArgs& a, int i) {
  const int32_t k = __ldg(a.draft_offsets + i + 1) - __ldg(a.draft_offsets + i);
  return (k < 0 || k > a.max_draft) ? 0 : k;
}

// Warp-wide: the sum over requests of min(k_i, cap), in every lane.
__device__ long long sum_min_drafts(const HArgs& a, int cap) {
  const int lane = threadIdx.x & 31;
  long long s = 0;
  for (int i = lane; i < a.nreq; i += 32) s += min(drafts_of(a, i), cap);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
  return s;
}

// Warp 0 of the CTAs with launch index nreq + t: the task's request and
// position (g_loc[0], g_loc[1]) and whether the caller's count equals the
// offsets' sum (g_loc[2]; on a mismatch the request is -1).
__device__ void locate_position(const HArgs& a, long long t) {
  const int lane = threadIdx.x & 31;
  const long long past0 = sum_min_drafts(a, a.max_draft);
  const bool ok = a.nreq + past0 == a.target_rows;
  int req = -1, j = 0;
  if (ok && t < past0) {
    // the smallest position j with more than t tasks at positions 1..j
    int lo = 1, hi = a.max_draft;
    while (lo < hi) {
      const int mid = lo + (hi - lo) / 2;
      if (sum_min_drafts(a, mid) > t)
        hi = mid;
      else
        lo = mid + 1;
    }
    j = lo;
    long long idx = (j == 1) ? t : t - sum_min_drafts(a, j - 1);
    // the idx-th request, in request order, with at least j drafts
    for (int base = 0; base < a.nreq; base += 32) {
      const int i = base + lane;
      const bool has = i < a.nreq && drafts_of(a, i) >= j;
      const unsigned m = __ballot_sync(0xffffffffu, has);
      const int n = __popc(m);
      if (idx < n) {
        const int before = __popc(m & ((1u << lane) - 1u));
        const unsigned pick = __ballot_sync(0xffffffffu, has && before == idx);
        req = base + __ffs(pick) - 1;
        break;
      }
      idx -= n;
    }
  }
  if (lane == 0) {
    g_loc[0] = req;
    g_loc[1] = j;
    g_loc[2] = ok ? 1 : 0;
  }
}

// Warp 2 of the other CTAs of a launch with a count, beside the parameter
// loads: whether the caller's count equals the offsets' sum (g_loc[2]).
__device__ void check_row_count(const HArgs& a) {
  const long long past0 = sum_min_drafts(a, a.max_draft);
  if ((threadIdx.x & 31) == 0) g_loc[2] = (a.nreq + past0 == a.target_rows) ? 1 : 0;
}

// Lane 0 of warp 1, after load_params: the parameters, checked (the status
// they give goes to c.pstatus; decode_and_copy runs meanwhile).
__device__ void read_params(const HArgs& a, int j) {
  Ctx& c = g;
  int st = SS_ROW_OK;
  int32_t k = 0;
  if (a.mode == 1) k = static_cast<int32_t>(g_prm[18]) - static_cast<int32_t>(g_prm[17]);
  const float T = __uint_as_float(g_prm[0]);
  c.T = T;
  c.top_k = static_cast<int32_t>(g_prm[1]);
  c.top_p = __uint_as_float(g_prm[2]);
  c.min_p = __uint_as_float(g_prm[3]);
  c.rep = __uint_as_float(g_prm[4]);
  c.freq = __uint_as_float(g_prm[5]);
  c.pres = __uint_as_float(g_prm[6]);
  c.seed_lo = g_prm[7];
  c.seed_hi = g_prm[8];
  c.rowid = g_prm[9];
  const int64_t pos64 = static_cast<int64_t>((static_cast<uint64_t>(g_prm[11]) << 32) | g_prm[10]);
  const int64_t last = pos64 + k;
  if (pos64 < 0 || last > 0xFFFFFFFFLL) st = max(st, SS_ROW_BAD_PARAM);
  c.pos = static_cast<uint32_t>(pos64) + static_cast<uint32_t>(j);
  c.h0 = static_cast<int32_t>(g_prm[12]);
  c.h1 = static_cast<int32_t>(g_prm[13]);
  c.b0 = static_cast<int32_t>(g_prm[14]);
  c.b1 = static_cast<int32_t>(g_prm[15]);
  if (!(T >= 0.0f) || isinf(T)) st = max(st, SS_ROW_BAD_PARAM);
  if (c.top_k < 0) st = max(st, SS_ROW_BAD_PARAM);
  if (!(c.top_p > 0.0f)) st = max(st, SS_ROW_BAD_PARAM);
  if (!(c.min_p >= 0.0f && c.min_p <= 1.0f)) st = max(st, SS_ROW_BAD_PARAM);
  if (!(c.rep > 0.0f) || isinf(c.rep)) st = max(st, SS_ROW_BAD_PARAM);
  if (!isfinite(c.freq) || !isfinite(c.pres)) st = max(st, SS_ROW_BAD_PARAM);
  if (c.h1 < c.h0 || c.b1 < c.b0) {
    st = max(st, SS_ROW_BAD_PARAM);
    c.h1 = c.h0;
    c.b1 = c.b0;
  }
  c.pstatus = st;
  c.greedy = (T == 0.0f);
  c.inv_t = (c.greedy || !(T > 0.0f)) ? 1.0f : __frcp_rn(T);
  c.k_on = (!c.greedy && c.top_k > 0 && c.top_k < a.vocab);
  c.p_on = (!c.greedy && c.top_p < 1.0f);
  c.mp_on = (!c.greedy && c.min_p > 0.0f);
  c.lmp = c.mp_on ? logf(c.min_p) : 0.0f;
  c.need_hist = c.k_on || c.p_on;
  c.use_mask = g_prm[16] != 0;
}

// ----------------------------------------------------------- patch table --

__device__ __forceinline__ int hash_slot(int32_t t) { return static_cast<int>((static_cast<uint32_t>(t) * 2654435761u) >> 22); }

// The patch table (in the histogram region during set-up): token ids with
// their occurrence count | kBiasFlag, bias value (later the processed value)
// and raw logit | allowed flag.  Returns the slot, or -1 when the table is
// full.
__device__ __forceinline__ int patch_insert(int32_t* keys, int32_t t) {
  int h = hash_slot(t);
  for (int probe = 0; probe < kHashCap; ++probe) {
    const int32_t prev = atomicCAS(keys + h, -1, t);
    if (prev == -1 || prev == t) return h;
    h = (h + 1) & (kHashCap - 1);
  }
  return -1;
}
__device__ __forceinline__ int patch_find(const int32_t* keys, int32_t t) {
  int h = hash_slot(t);
  for (int probe = 0; probe < kHashCap; ++probe) {
    const int32_t k = keys[h];
    if (k == t) return h;
    if (k == -1) return -1;
    h = (h + 1) & (kHashCap - 1);
  }
  return -1;
}

__device__ __forceinline__ void add_entry(unsigned long long* el, float y, int32_t t) {
  const int i = atomicAdd(&g.nent, 1);
  if (i < kEntCap)
    el[i] = ekey(y, t);
  else
    atomicMax(&g.status, SS_ROW_LIMIT);
}

// Membership of an item of processed value y and token t in K.
__device__ __forceinline__ bool in_cut(float y, int32_t t, float cv, int32_t ct) {
  return y > cv || (y == cv && t <= ct);
}

// ------------------------------------------------------------- exchanges --

// Writes this CTA's PartD into every CTA, cluster barrier, and
// combines the C partials in rank order (identical in every CTA): best
// (score desc, token asc), and with SUMS the counts and masses summed.
// Called by all threads.
// With REDUCED the caller's (best, arg) is already the CTA's (the same in
// every thread).
// With SUMS and REDUCED both, the counts are summed (not the masses) and the
// bests combined.
template <bool SUMS, bool REDUCED>
__device__ PartD exchange_d(float best, int32_t arg, int32_t count, unsigned long long mass) {
  cg::cluster_group cl = cg::this_cluster();
  if (SUMS) {
    count = block_sum<int32_t>(count);
    if (!REDUCED) mass = block_sum<unsigned long long>(mass);
  } else if (REDUCED) {
    __syncthreads();
  } else {
    block_best(best, arg);
  }
  SS_STAMP(37);
  // (a block barrier above: g.xpar is current) consecutive exchanges
  // alternate between two buffers, so a CTA still reading the previous result
  // is never overwritten
  const int par = g.xpar;
  const int C = static_cast<int>(cl.num_blocks());
  if (threadIdx.x < C) {
    PartD d;
    d.best = best;
    d.arg = arg;
    d.count = count;
    d.pad = 0;
    d.mass = mass;
    d.pad2 = 0;
    *cl.map_shared_rank(&g_pd[par][cl.block_rank()], threadIdx.x) = d;
  }
  cl.sync();
  if (threadIdx.x == 0) g.xpar = par ^ 1;
  PartD r = g_pd[par][0];
  for (int q = 1; q < C; ++q) {
    const PartD& o = g_pd[par][q];
    if (SUMS) {
      r.count += o.count;
      r.mass += o.mass;
    }
    if ((!SUMS || REDUCED) && beats(o.best, o.arg, r.best, r.arg)) {
      r.best = o.best;
      r.arg = o.arg;
    }
  }
  return r;
}

// ---------------------------------------------------------------- passes --

// The score of a token that passed the cheap noise bound: base + Gumbel
// noise, base = y (the draw over K) or log(P - q) (the residual); -inf when
// the residual is empty there or the token cannot beat `bs`.  Out of line:
// most tokens never get here.
template <bool RES>
__device__ __noinline__ float draw_score(float y, int32_t t, uint32_t num, float ub, float m, float inv_s,
                                         const float* qrow, float bs) {
  float base = y;
  if (RES) {
    const float P = __fmul_rn(__expf(__fsub_rn(y, m)), inv_s);
    const float r = __fsub_rn(P, qrow[t]);
    if (!(r > 0.0f)) return ninf();
    base = logf(r);
    if (base + ub < bs) return ninf();
  }
  return __fadd_rn(base, gumbel_from_numerator(num));
}

// The draw over K (stream 0) or, with RES, over the residual
// max(P - q, 0) (stream 2, log r + g); P(t) = exp(y - m) / S.  The CTA's
// best score so far lives in g_dscore as a 32-bit order key (a native shared
// atomic maximum: a 64-bit (score, token) key would need a compare-and-swap
// loop, and every thread's first candidate lands at once); every thread
// prunes against it, so a token whose score bound is below the best of the
// whole CTA costs no logarithm.  Each thread keeps its own best (score,
// lowest token); after the pass the threads holding the CTA's best score
// take the lowest token among them.  draw_reset() before the pass (then a
// block barrier); cta_best() reads the result.  Entries are visited by the
// CTA that owns their token.
__device__ __forceinline__ void draw_reset() {
  g_dscore = 0;
  g_dtok = 0x7fffffff;
}

__device__ __forceinline__ void cta_best(float& bs, int32_t& bt) {
  __syncthreads();
  const uint32_t k = g_dscore;
  bs = k ? okey_value(k) : ninf();
  bt = g_dtok;
}

// With COUNT the pass also counts this thread's members of K (rows whose K
// is a plain predicate: the count needs no pass of its own).
template <bool RES, bool COUNT = false>
__device__ void draw_pass(const HArgs& a, float cv, int32_t ct, bool mp_on, float inv_s, float log_s,
                          const float* qrow, const unsigned long long* ents, int n_ents, int32_t* count = nullptr) {
  const Ctx& c = g;
  const uint4* data = reinterpret_cast<const uint4*>(g_dyn);
  const uint16_t* vb = reinterpret_cast<const uint16_t*>(g_dyn + a.o_vb);
  const float inv_t = c.inv_t, m = c.m, lmp = c.lmp;
  const uint32_t k0 = c.seed_lo, k1 = c.seed_hi, pos = c.pos, rid = c.rowid;
  const uint32_t stream = RES ? 2u : 0u;
  float bs = ninf();                 // a lower bound of the CTA's best score
  float ms = ninf();                 // this thread's best (score, token)
  int32_t mt = 0x7fffffff;
  auto refresh = [&]() {
    const uint32_t k = *reinterpret_cast<volatile uint32_t*>(&g_dscore);
    if (k) bs = fmaxf(bs, okey_value(k));
  };
  auto reach = [&](float y) -> float {
    return RES ? (y - m - log_s + kGumbelMax + 1e-3f + fabsf(y) * 1e-6f) : (y + kGumbelMax);
  };
  auto member = [&](float y, int32_t t) -> bool {
    return y != ninf() && in_cut(y, t, cv, ct) && (!mp_on || __fsub_rn(y, m) >= lmp);
  };
#ifdef SS_HIST_STAMPS
  int n_score = 0, n_philox = 0, n_vec = 0;
#endif
  auto consider = [&](float y, int32_t t, uint32_t word) {
    const uint32_t num = uniform_numerator(word);
    const float ub = gumbel_upper_bound(num);
    // an upper bound of the base (for the residual log r <= log P), before
    // any logarithm or read of the draft's q
    const float base_ub = RES ? (y - m - log_s + 1e-3f + fabsf(y) * 1e-6f) : y;
    if (base_ub + ub < bs || !member(y, t)) return;
#ifdef SS_HIST_STAMPS
    ++n_score;
#endif
    const float s = draw_score<RES>(y, t, num, ub, m, inv_s, qrow, bs);
    if (s > ninf() && beats(s, t, ms, mt)) {
      ms = s;
      mt = t;
      // only a score at or above the CTA's best so far can still win (bs
      // is always a score already published)
      if (s >= bs) {
        atomicMax(&g_dscore, okey(s));
        bs = s;
      }
    }
  };
  // Seeds (sampling calls): thread 0 scores the CTA's largest staged token
  // and its largest entry when they are drawn from, so that every thread
  // prunes from its first vector on.  Only the score is published: the pass
  // visits both tokens again, and the lowest token holding the best is taken
  // at its end.  (Measured: a gain for sampling calls, a loss for the
  // verification launches of many waves, which skip it.)
  const bool seeded = !RES && a.mode == 0;
  if (seeded && threadIdx.x == 0) {
    float best = ninf();
    auto seed = [&](float y, int32_t t) {
      if (!member(y, t)) return;
      const Philox4 r = philox4x32_10(static_cast<uint32_t>(t) >> 2, pos, rid, stream, k0, k1);
      best = fmaxf(best, __fadd_rn(y, gumbel_from_numerator(uniform_numerator(r.w[t & 3]))));
    };
    const int sp = c.seed_pair;
    if (sp >= 0 && sp < c.nvec / 2) {
      const uint16_t* d16 = reinterpret_cast<const uint16_t*>(g_dyn) + sp * 16;
      int eb = -1;
      for (int e = 0; e < 16; ++e)
        if (d16[e] != 0xff80u && (eb < 0 || bf16_to_f(d16[e]) > bf16_to_f(d16[eb]))) eb = e;
      if (eb >= 0) seed(__fmul_rn(bf16_to_f(d16[eb]), inv_t), c.lo + sp * 16 + eb);
    }
    if (c.seed_et >= c.lo && c.seed_et < c.lo + c.n) seed(c.seed_ey, c.seed_et);
    if (best > ninf()) g_dscore = okey(best);
  }
  if (seeded) __syncthreads();
  const int nvec = c.nvec;
  int32_t cnt = 0;
  for (int v = threadIdx.x; v < nvec; v += kThreads) {
    const float vy = __fmul_rn(bf16_to_f(vb[v >> 1]), inv_t);
    refresh();
    if (vy < cv || vy == ninf() || (!COUNT && reach(vy) < bs)) continue;
    if (mp_on && !(__fsub_rn(vy, m) >= lmp)) continue;
#ifdef SS_HIST_STAMPS
    ++n_vec;
#endif
    const uint4 d = data[v];
    const uint32_t w[4] = {d.x, d.y, d.z, d.w};
    const int32_t t0 = c.lo + v * 8;
    if (COUNT) {
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const uint32_t word = w[e >> 1];
        const float y = __fmul_rn((e & 1) ? __uint_as_float(word & 0xffff0000u) : __uint_as_float(word << 16), inv_t);
        cnt += member(y, t0 + e) ? 1 : 0;
      }
      if (reach(vy) < bs) continue;
    }
    auto y_of = [&](int e) {
      const uint32_t word = w[e >> 1];
      return __fmul_rn((e & 1) ? __uint_as_float(word & 0xffff0000u) : __uint_as_float(word << 16), inv_t);
    };
    const uint32_t q0 = static_cast<uint32_t>(t0) >> 2;
    if (RES) {
      float y[8];
      bool any = false;
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        y[e] = y_of(e);
        const bool ok = member(y[e], t0 + e) && reach(y[e]) >= bs;
        if (!ok) y[e] = ninf();
        any |= ok;
      }
      if (!any) continue;
      const Philox4 r0 = philox4x32_10(q0, pos, rid, stream, k0, k1);
      const Philox4 r1 = philox4x32_10(q0 + 1u, pos, rid, stream, k0, k1);
#pragma unroll
      for (int e = 0; e < 8; ++e)
        if (y[e] != ninf()) consider(y[e], t0 + e, (e < 4) ? r0.w[e] : r1.w[e - 4]);
    } else {
      // One noise threshold for the vector, from its largest y: a token can
      // win only if its noise bound ln2 * (clz(2^24 - n) - 7) reaches
      // D = bs - vy (less a slack far above the fp32 rounding), i.e. only if
      // clz(2^24 - n) >= c = ceil(7 + D / ln2), i.e. 2^24 - n < 2^(32 - c);
      // with n = 2 * (x >> 9) + 1 that is one comparison of the raw Philox
      // word x.  Tokens past it get the exact tests (their own y, K).
      uint32_t x_thr = 0;
      if (bs > ninf()) {
        const float D = bs - vy - 1e-3f * fmaxf(1.0f, fabsf(bs));
        if (D > 0.0f) {
          const float cf = ceilf(7.0f + D * 1.44269504f);
          if (cf >= 32.0f) continue;  // no token of the vector can win
          const int cc = static_cast<int>(cf);  // 8 .. 31
          if (cc > 8) {
            const uint32_t mthr = 1u << (32 - cc);  // <= 2^23
            x_thr = (((1u << 24) - mthr - 1u) / 2u + 1u) << 9;
          }
        }
      }
#ifdef SS_HIST_STAMPS
      n_philox += 2;
#endif
      // both halves' noise words at once: two independent Philox chains
      const Philox4 r0 = philox4x32_10(q0, pos, rid, stream, k0, k1);
      const Philox4 r1 = philox4x32_10(q0 + 1u, pos, rid, stream, k0, k1);
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const uint32_t x = (e < 4) ? r0.w[e] : r1.w[e - 4];
        if (x >= x_thr) consider(y_of(e), t0 + e, x);
      }
    }
  }
  for (int i = threadIdx.x; i < n_ents; i += kThreads) {
    const unsigned long long e = ents[i];
    const int32_t t = ekey_t(e);
    if (t < c.lo || t >= c.lo + c.n) continue;
    const float y = ekey_y(e);
    if (COUNT) cnt += member(y, t) ? 1 : 0;
    if (!member(y, t) || reach(y) < bs) continue;
    const Philox4 r = philox4x32_10(static_cast<uint32_t>(t) >> 2, pos, rid, stream, k0, k1);
    consider(y, t, r.w[t & 3]);
  }
  if (COUNT) *count = cnt;
  // the lowest token among the threads holding the CTA's best score
  __syncthreads();
  const uint32_t best = g_dscore;
  if (best && mt != 0x7fffffff && okey(ms) == best) atomicMin(&g_dtok, mt);
}

// |K| and its fixed-point mass for rows whose K is a plain predicate (no
// histogram): every allowed token, with the min-p test when it is on.
__device__ void count_pass(const HArgs& a, bool want_mass, const unsigned long long* ents, int n_ents,
                           int32_t& cnt, unsigned long long& mass) {
  const Ctx& c = g;
  const uint4* data = reinterpret_cast<const uint4*>(g_dyn);
  const uint16_t* vb = reinterpret_cast<const uint16_t*>(g_dyn + a.o_vb);
  const float inv_t = c.inv_t, m = c.m, lmp = c.lmp;
  const bool mp_on = c.mp_on != 0;
  for (int v = threadIdx.x; v < c.nvec; v += kThreads) {
    const float vy = __fmul_rn(bf16_to_f(vb[v >> 1]), inv_t);
    if (vy == ninf() || (mp_on && !(__fsub_rn(vy, m) >= lmp))) continue;
    const uint4 d = data[v];
    const uint32_t w[4] = {d.x, d.y, d.z, d.w};
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      const uint32_t word = w[e >> 1];
      const float y = __fmul_rn((e & 1) ? __uint_as_float(word & 0xffff0000u) : __uint_as_float(word << 16), inv_t);
      const bool in = y != ninf() && (!mp_on || __fsub_rn(y, m) >= lmp);
      cnt += in ? 1 : 0;
      if (want_mass && in) mass += fmass(y, m);
    }
  }
  for (int i = threadIdx.x; i < n_ents; i += kThreads) {
    const float y = ekey_y(ents[i]);
    const bool in = y != ninf() && (!mp_on || __fsub_rn(y, m) >= lmp);
    cnt += in ? 1 : 0;
    if (want_mass && in) mass += fmass(y, m);
  }
}

// ----------------------------------------------------------- the locator --
// Items are the staged tokens (counted per slot, in every CTA) and the exact
// entries (each CTA's list).  Entry e sits at slot position epos[e] = the
// first slot whose value is <= its y: before that slot's tokens when its y is
// larger, tied with them when equal.  Coarse group q holds the slots
// [gb[q], gb[q + 1]) and the entries positioned there; the tail group kGroups
// holds the entries past the last slot.

__device__ __forceinline__ float slot_y(int32_t s) {
  const float z = slot_z(g.M, s);
  return __fmul_rn(z, g.inv_t);
}

// The first slot whose y is <= v (ns if none), from an estimate: the slot of
// v's value before the temperature (bf16, truncated), then a walk to the
// exact answer (slot_y falls with the slot, so the walk is short and always
// ends right).
__device__ int32_t first_slot_le_near(float v) {
  const SlotMap& M = g.M;
  const float z = __fmul_rn(v, g.T);
  int32_t s = slot_of(M, __float_as_uint(z) >> 16);
  s = min(max(s, 0), M.ns);
  if (s < M.ns && slot_y(s) <= v) {
    while (s > 0 && slot_y(s - 1) <= v) --s;
  } else {
    while (s < M.ns && slot_y(s) > v) ++s;
  }
  return s;
}

// A 64-bit shared-memory sum built from two 32-bit atomics (the low word's
// carry goes to the high word): much cheaper than a 64-bit shared atomic.
__device__ __forceinline__ void atomic_add_u64_split(unsigned long long* addr, unsigned long long v) {
  uint32_t* w = reinterpret_cast<uint32_t*>(addr);
  const uint32_t lo = static_cast<uint32_t>(v);
  const uint32_t old = atomicAdd(w, lo);
  const uint32_t hi = static_cast<uint32_t>(v >> 32) + ((old + lo < old) ? 1u : 0u);
  if (hi) atomicAdd(w + 1, hi);
}

// The last group q with gb[q] <= p: group q starts at slot q * (kSlots /
// kGroups) or later (a run of equal values pushes it on), so start there and
// walk.
__device__ __forceinline__ int group_of(int32_t p) {
  if (p >= g.M.ns) return kGroups;
  int q = min(p / (kSlots / kGroups), kGroups - 1);
  while (q > 0 && g_gb[q] > p) --q;
  while (q + 1 < kGroups && g_gb[q + 1] <= p) ++q;
  return q;
}

// First entry of a sorted list whose y is < v (the number of entries >= v).
__device__ __forceinline__ int first_entry_lt(const unsigned long long* el, int n, float v) {
  int lo = 0, hi = n;
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    if (ekey_y(el[mid]) < v)
      hi = mid;
    else
      lo = mid + 1;
  }
  return lo;
}

// The range of coarse group `grp` in every CTA's group-ordered entry list:
// g_gr0[r] its start, g_grc[r] the entries of the group in CTAs before r
// (g_grc[C] the total).  Called by all threads; warp 0 does the work and,
// with BARRIER, every thread waits for it (else the caller's next block
// barrier publishes it).
template <bool BARRIER = true>
__device__ void group_ranges(const HArgs& a, int grp) {
  cg::cluster_group cl = cg::this_cluster();
  const int C = static_cast<int>(cl.num_blocks());
  const int32_t* eoff = reinterpret_cast<const int32_t*>(g_dyn + a.o_hist + kSlots * 2);
  if (threadIdx.x < 32) {
    const int r = threadIdx.x;
    int32_t lo = 0, n = 0;
    if (r < C) {
      const int32_t* ro = cl.map_shared_rank(eoff, r);
      lo = ro[grp];
      n = ro[grp + 1] - lo;
    }
    int32_t inc = n;
#pragma unroll
    for (int o = 1; o < kMaxCluster; o <<= 1) {
      const int32_t y = __shfl_up_sync(0xffffffffu, inc, o);
      if (r >= o) inc += y;
    }
    if (r < C) {
      g_gr0[r] = lo;
      g_grc[r] = inc - n;
    }
    if (r == C - 1) g_grc[C] = inc;
  }
  if (BARRIER) __syncthreads();
}

// Reads the slot counts of coarse group `grp` from every CTA into g_fc, and
// gathers the group's entries from every CTA's list into (gk, gp), sorted
// (y desc, token asc) by rank; g.n_g is their number (-1 if more than
// kGatherCap).  The entries are gathered unsorted into the merge region and
// ranked into the exchange-2 region (free once the coarse sums are read).
// Called by all threads; ends with a block barrier.
__device__ void load_group(const HArgs& a, int grp) {
  cg::cluster_group cl = cg::this_cluster();
  const int C = static_cast<int>(cl.num_blocks());
  const int s0 = g_gb[grp], s1 = g_gb[grp + 1];
  const uint32_t* hist = reinterpret_cast<const uint32_t*>(g_dyn + a.o_hist);
  const unsigned long long* el = reinterpret_cast<const unsigned long long*>(g_dyn + a.o_el);
  const int16_t* eord = reinterpret_cast<const int16_t*>(g_dyn + a.o_hist + kSlots * 2 + (kGroups + 2) * 4);
  unsigned long long* gk = reinterpret_cast<unsigned long long*>(g_dyn + a.o_xm);
  int16_t* gp = reinterpret_cast<int16_t*>(gk + kGatherCap);
  unsigned long long* uk = reinterpret_cast<unsigned long long*>(g_dyn + a.o_mg);
  int16_t* up = reinterpret_cast<int16_t*>(uk + kGatherCap);
  __syncthreads();  // the previous readers of g_fc and of the buffers are done
  // the entry ranges (warp 0) and the slot counts (every thread) are
  // independent remote reads: both in flight before one barrier
  group_ranges<false>(a, grp);
  for (int i = threadIdx.x; i < s1 - s0; i += kThreads) {
    uint32_t cnt = 0;
    const int q = s0 + i;
#pragma unroll
    for (int r = 0; r < kMaxCluster; ++r)
      if (r < C) cnt += (*cl.map_shared_rank(hist + (q >> 1), r) >> ((q & 1) << 4)) & 0xffffu;
    g_fc[i] = cnt;
  }
  __syncthreads();
  const int n = g_grc[C];
  if (n > kGatherCap) {
    __syncthreads();
    if (threadIdx.x == 0) g.n_g = -1;
    __syncthreads();
    return;
  }
  for (int i = threadIdx.x; i < n; i += kThreads) {
    int r = 0;
    while (i >= g_grc[r + 1]) ++r;
    const int e = *cl.map_shared_rank(eord + g_gr0[r] + (i - g_grc[r]), r);
    uk[i] = *cl.map_shared_rank(el + e, r);
    up[i] = *cl.map_shared_rank(g_epos + e, r);
  }
  __syncthreads();
  // rank sort: the keys are distinct (one entry per token)
  for (int i = threadIdx.x; i < n; i += kThreads) {
    const unsigned long long k = uk[i];
    int rk = 0;
    for (int j = 0; j < n; ++j) rk += (uk[j] < k) ? 1 : 0;
    gk[rk] = k;
    gp[rk] = up[i];
  }
  if (threadIdx.x == 0) g.n_g = n;
  __syncthreads();
}

// Where the running count (by_mass = 0) or mass (1) of the items first
// reaches `target`: the cut value g.w_v, the number of items of that value to
// take g.w_take, and the count / mass of the items above it (g.w_cc,
// g.w_cm).  g.w_found = 0 when the items do not reach the target, -1 when the
// cut would fall among tokens below the counted slots or cannot be resolved.
// Within the group, slots and entries are merged by value (each keeps its
// list's order; an entry goes before the slots its value is not above), the
// merged items are prefix-summed by the block, and the first item reaching
// the target names the cut's value.  Called by all threads.
__device__ void locate(const HArgs& a, int by_mass, unsigned long long target) {
  Ctx& c = g;
  coarse_locate(by_mass, target);
  if (threadIdx.x == 0) {
    const int grp = c.pick;
    c.w_found = (grp < 0) ? 0 : 1;
    if (grp == kGroups && c.below) c.w_found = -1;
    if (grp >= 0 && grp < kGroups && g_gb[grp + 1] - g_gb[grp] > kFineMax) c.w_found = -1;
  }
  __syncthreads();
  if (c.w_found != 1) return;
  const int grp = c.pick;
  load_group(a, grp);
  SS_STAMP(28);
  if (c.n_g < 0) {
    if (threadIdx.x == 0) c.w_found = -1;
    __syncthreads();
    return;
  }
  if (threadIdx.x == 0) c.w_grp = grp;
  const unsigned long long* gk = reinterpret_cast<const unsigned long long*>(g_dyn + a.o_xm);
  const int16_t* gp = reinterpret_cast<const int16_t*>(gk + kGatherCap);
  const int s0 = g_gb[grp], ns = g_gb[grp + 1] - s0, ng = c.n_g;
  const int m = ns + ng;  // <= kFineMax + kGatherCap
  float* g_mv = reinterpret_cast<float*>(g_dyn + a.o_mg);  // the group's items merged by value
  uint32_t* g_mc = reinterpret_cast<uint32_t*>(g_mv + kFineMax + kGatherCap);
  // merged position of every slot and entry (a merge of two lists sorted by
  // value, an entry before a slot of equal value, so every position is
  // taken exactly once); value and count by position
  for (int i = threadIdx.x; i < m; i += kThreads) {
    float v;
    unsigned long long cnt;
    int at;
    if (i < ns) {
      v = slot_y(s0 + i);
      cnt = g_fc[i];
      at = i + first_entry_lt(gk, ng, v);  // the entries not below slot i come first
    } else {
      const int e = i - ns;
      v = ekey_y(gk[e]);
      cnt = 1;
      at = e + (gp[e] - s0);  // the slots above it: those before its position
    }
    g_mv[at] = v;
    g_mc[at] = static_cast<uint32_t>(cnt);
  }
  __syncthreads();
  SS_STAMP(29);
  const unsigned long long before_c = c.w_cc, before_m = c.w_cm;
  // block prefix: kItemsPer merged items per thread, in order
  constexpr int kItemsPer = (kFineMax + kGatherCap + kThreads - 1) / kThreads;
  unsigned long long tc = 0, tm = 0;
  const int i0 = threadIdx.x * kItemsPer;
  for (int k = 0; k < kItemsPer; ++k) {
    const int i = i0 + k;
    if (i < m && g_mc[i]) {
      tc += g_mc[i];
      tm += static_cast<unsigned long long>(g_mc[i]) * fmass(g_mv[i], c.m);
    }
  }
  unsigned long long ic = tc, im = tm, totc, totm;
  block_scan2(ic, im, &totc, &totm);
  SS_STAMP(30);
  // the first item whose running total reaches the target
  unsigned long long rc = before_c + ic - tc, rm = before_m + im - tm;
  if (threadIdx.x == 0) c.pick = 0x7fffffff;
  __syncthreads();
  for (int k = 0; k < kItemsPer; ++k) {
    const int i = i0 + k;
    if (i >= m || !g_mc[i]) continue;
    const unsigned long long n = g_mc[i], w = fmass(g_mv[i], c.m);
    const unsigned long long step = by_mass ? n * w : n;
    if (step > 0 && (by_mass ? rm : rc) + step >= target) {
      atomicMin(&c.pick, i);
      break;
    }
    rc += n;
    rm += n * w;
  }
  __syncthreads();
  // the value group of the hit starts a few items earlier at most (equal
  // values are adjacent)
  if (threadIdx.x == 0) {
    const int hit = c.pick;
    if (hit == 0x7fffffff) {
      c.w_found = 0;
    } else {
      int f = hit;
      while (f > 0 && g_mv[f - 1] == g_mv[hit]) --f;
      c.w_slot = f;
    }
  }
  __syncthreads();
  if (c.w_found == 1) {
    // the thread that owns the group's first item has the sums before it
    const int f = c.w_slot;
    if (f / kItemsPer == static_cast<int>(threadIdx.x)) {
      unsigned long long cc = before_c + ic - tc, cm = before_m + im - tm;
      for (int i = i0; i < f; ++i) {
        cc += g_mc[i];
        cm += static_cast<unsigned long long>(g_mc[i]) * fmass(g_mv[i], c.m);
      }
      const float v = g_mv[f];
      const unsigned long long w = fmass(v, c.m);
      c.w_v = v;
      c.w_take = by_mass ? (target - cm + w - 1) / w : target - cc;
      c.w_cc = cc;
      c.w_cm = cm;
    }
  }
  __syncthreads();
}

// Count and mass of the items whose y is strictly above v.  Called by all
// threads; result in g.w_cc / g.w_cm (g.w_found = -1 if unknown).
__device__ void above_value(const HArgs& a, float v) {
  Ctx& c = g;
  if (threadIdx.x == 0) {
    // the group holding the first slot <= v
    const int grp = group_of(first_slot_le_near(v));
    unsigned long long cc = 0, cm = 0;
    for (int q = 0; q < grp; ++q) {
      cc += g_gcnt[q];
      cm += g_gmass[q];
    }
    c.pick = grp;
    c.w_cc = cc;
    c.w_cm = cm;
    c.w_found = 1;
    // uncounted tokens below the slots may lie above v
    if (grp == kGroups && c.below) c.w_found = -1;
    if (grp < kGroups && g_gb[grp + 1] - g_gb[grp] > kFineMax) c.w_found = -1;
  }
  __syncthreads();
  if (c.w_found != 1) return;
  const int grp = c.pick;
  load_group(a, grp);
  if (c.n_g < 0) {
    if (threadIdx.x == 0) c.w_found = -1;
    __syncthreads();
    return;
  }
  const unsigned long long* gk = reinterpret_cast<const unsigned long long*>(g_dyn + a.o_xm);
  const int s0 = g_gb[grp], ns = g_gb[grp + 1] - s0;
  unsigned long long cc = 0, cm = 0;
  for (int i = threadIdx.x; i < ns + c.n_g; i += kThreads) {
    const float y = (i < ns) ? slot_y(s0 + i) : ekey_y(gk[i - ns]);
    const unsigned long long n = (i < ns) ? g_fc[i] : 1;
    if (y > v && n) {
      cc += n;
      cm += n * fmass(y, c.m);
    }
  }
  cc = block_sum<unsigned long long>(cc);
  cm = block_sum<unsigned long long>(cm);
  if (threadIdx.x == 0) {
    c.w_cc += cc;
    c.w_cm += cm;
  }
  __syncthreads();
}

// Sorts kFastCap (2048) keys ascending: a bitonic network with four keys per
// thread in registers; strides 1 and 2 stay in the thread, strides 4 to 64 go
// through warp shuffles, and only strides of 128 and more through shared
// memory (10 of the network's 66 stages, two block barriers each).  Called by
// all threads; ends with a block barrier.
__device__ __noinline__ void sort_fast_cap(unsigned long long* key) {
  static_assert(kFastCap == 4 * kThreads, "four keys per thread");
  const int tid = threadIdx.x;
  const int e0 = 4 * tid;  // this thread's first element
  unsigned long long v0 = key[e0], v1 = key[e0 + 1], v2 = key[e0 + 2], v3 = key[e0 + 3];
  auto cas = [](unsigned long long& lo, unsigned long long& hi, bool asc) {
    if ((lo > hi) == asc) {
      const unsigned long long t = lo;
      lo = hi;
      hi = t;
    }
  };
  auto merge = [](unsigned long long mine, unsigned long long other, bool keep_min) {
    return keep_min ? (mine < other ? mine : other) : (mine > other ? mine : other);
  };
  for (int k = 2; k <= kFastCap; k <<= 1) {
    const bool asc = (e0 & k) == 0;  // k >= 4: the same for the thread's four elements
    for (int j = k >> 1; j > 0; j >>= 1) {
      if (j >= 128) {
        __syncthreads();  // the previous stage's reads are done
        key[e0] = v0;
        key[e0 + 1] = v1;
        key[e0 + 2] = v2;
        key[e0 + 3] = v3;
        __syncthreads();
        const bool keep_min = ((e0 & j) == 0) == asc;  // the lower of the pair keeps the minimum when ascending
        v0 = merge(v0, key[e0 ^ j], keep_min);
        v1 = merge(v1, key[(e0 + 1) ^ j], keep_min);
        v2 = merge(v2, key[(e0 + 2) ^ j], keep_min);
        v3 = merge(v3, key[(e0 + 3) ^ j], keep_min);
      } else if (j >= 4) {
        const int lj = j >> 2;
        const bool keep_min = ((e0 & j) == 0) == asc;
        v0 = merge(v0, __shfl_xor_sync(0xffffffffu, v0, lj), keep_min);
        v1 = merge(v1, __shfl_xor_sync(0xffffffffu, v1, lj), keep_min);
        v2 = merge(v2, __shfl_xor_sync(0xffffffffu, v2, lj), keep_min);
        v3 = merge(v3, __shfl_xor_sync(0xffffffffu, v3, lj), keep_min);
      } else if (j == 2) {
        const bool a = (k == 2) ? true : asc;
        cas(v0, v2, a);
        cas(v1, v3, a);
      } else {
        // k == 2: pairs (0,1) ascending, (2,3) descending; k >= 4: both by asc
        cas(v0, v1, (k == 2) ? true : asc);
        cas(v2, v3, (k == 2) ? false : asc);
      }
    }
  }
  __syncthreads();
  key[e0] = v0;
  key[e0 + 1] = v1;
  key[e0 + 2] = v2;
  key[e0 + 3] = v3;
  __syncthreads();
}

// One step of the short path's merge, in every CTA of a cluster of C: each
// item of this CTA's sorted run goes to its place in the cluster-wide order,
// its index in its own run plus, for every other run, the number of that
// run's items below it (keys are distinct: one per token), found by binary
// searches in the other CTAs' runs, all runs' steps interleaved so that the
// remote loads overlap.  Runs live in the candidate region (flag 1 in g_runs)
// or the run region of their CTA.
template <int C>
__device__ void place_run(const unsigned long long* srun, int nr, int rank, const unsigned long long* cand,
                          const unsigned long long* run, unsigned long long* dst) {
  cg::cluster_group cl = cg::this_cluster();
  const unsigned long long* rq[C];
  int nq[C];
#pragma unroll
  for (int q = 0; q < C; ++q) {
    rq[q] = cl.map_shared_rank(g_runs[q][0] ? cand : run, q);
    nq[q] = (q == rank) ? 0 : g_runs[q][1];
  }
  for (int i = threadIdx.x; i < nr; i += kThreads) {
    const unsigned long long k = srun[i];
    int lo[C], hi[C];
#pragma unroll
    for (int q = 0; q < C; ++q) {
      lo[q] = 0;
      hi[q] = nq[q];
    }
    for (bool more = true; more;) {
      more = false;
#pragma unroll
      for (int q = 0; q < C; ++q)
        if (lo[q] < hi[q]) {
          const int mid = (lo[q] + hi[q]) >> 1;
          if (rq[q][mid] < k)
            lo[q] = mid + 1;
          else
            hi[q] = mid;
          more |= lo[q] < hi[q];
        }
    }
    int place = i;
#pragma unroll
    for (int q = 0; q < C; ++q) place += lo[q];
    dst[place] = k;
  }
}

// ------------------------------------------------------------ short path --
// Rows with 0 < top_k <= kFastK and a top-k certificate: every item of K has
// y >= y(tau) (at least k staged tokens are >= tau), so the candidates --
// staged tokens at or above tau and entries at or above y(tau) -- hold K.
// Every CTA sorts its candidates by (y desc, token asc); when they fit, the
// CTAs merge their runs into rank 0 (each places its own items), and rank 0
// takes every cut (top-k, top-p over the top-k's fixed-point masses, min-p)
// and the draw itself: the items of K are then the first L of that order,
// ties included.  Returns false (in every CTA
// alike) when the candidates do not fit and the row takes the histogram path.
// Called by all threads of every CTA; ends with rank 0's decisions in
// token / accept / kept.
__device__ bool short_path(const HArgs& a, bool tests_draft, const float* qrow, int32_t& token, int32_t& accept,
                           unsigned long long& kept) {
  Ctx& c = g;
  cg::cluster_group cl = cg::this_cluster();
  const int rank = static_cast<int>(cl.block_rank());
  const int tid = threadIdx.x, lane = tid & 31;
  const uint4* data = reinterpret_cast<const uint4*>(g_dyn);
  const uint16_t* vb = reinterpret_cast<const uint16_t*>(g_dyn + a.o_vb);
  const unsigned long long* el = reinterpret_cast<const unsigned long long*>(g_dyn + a.o_el);
  // candidates, in this CTA's histogram region
  unsigned long long* cand = reinterpret_cast<unsigned long long*>(g_dyn + a.o_hist);
  const uint32_t tau = c.tau_key;
  const float inv_t = c.inv_t;
  const float ytau = __fmul_rn(bf16_to_f(key16_bits(tau)), inv_t);
  if (tid == 0) g.n_g = 0;
  __syncthreads();
  // append: one reservation per warp and round
  auto append = [&](int n_mine, auto&& item) {
    int inc = n_mine;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, inc, o);
      if (lane >= o) inc += y;
    }
    const int tot = __shfl_sync(0xffffffffu, inc, 31);
    int base = 0;
    if (lane == 31 && tot) base = atomicAdd(&g.n_g, tot);
    base = __shfl_sync(0xffffffffu, base, 31) + inc - n_mine;
    for (int i = 0; i < n_mine; ++i)
      if (base + i < kFastCap) cand[base + i] = item(i);
  };
  for (int p0 = 0; p0 < c.nvec / 2; p0 += kThreads) {
    const int p = p0 + tid;
    uint32_t hit = 0;  // bit e: token e of the pair is a candidate
    uint4 d0 = make_uint4(0, 0, 0, 0), d1 = d0;
    if (p < c.nvec / 2 && vb[p] != 0xff80u && key16(vb[p]) >= tau) {
      d0 = data[2 * p];
      d1 = data[2 * p + 1];
      const uint32_t w[8] = {d0.x, d0.y, d0.z, d0.w, d1.x, d1.y, d1.z, d1.w};
#pragma unroll
      for (int e = 0; e < 16; ++e) {
        const uint32_t h = (w[e >> 1] >> ((e & 1) ? 16 : 0)) & 0xffffu;
        if (h != 0xff80u && key16(h) >= tau) hit |= 1u << e;
      }
    }
    const uint32_t wds[8] = {d0.x, d0.y, d0.z, d0.w, d1.x, d1.y, d1.z, d1.w};
    append(__popc(hit), [&](int i) {
      uint32_t m = hit;
      for (int j = 0; j < i; ++j) m &= m - 1;
      const int e = __ffs(m) - 1;
      const uint32_t h = (wds[e >> 1] >> ((e & 1) ? 16 : 0)) & 0xffffu;
      return ekey(__fmul_rn(bf16_to_f(h), inv_t), c.lo + p * 16 + e);
    });
  }
  for (int i0 = 0; i0 < c.ne; i0 += kThreads) {
    const int i = i0 + tid;
    const bool take = i < c.ne && ekey_y(el[i]) >= ytau;
    append(take ? 1 : 0, [&](int) { return el[i]; });
  }
  __syncthreads();
  const int nr = g.n_g;  // this CTA's candidates
  // this CTA's sorted run: a rank sort while small, else the bitonic network
  unsigned long long* run = reinterpret_cast<unsigned long long*>(g_dyn + a.o_xm);  // xm and mg, contiguous
  unsigned long long* srun = run;
  if (nr <= kRankSortMax) {
    for (int i = tid; i < nr; i += kThreads) {
      const unsigned long long k = cand[i];
      int r = 0;
      for (int j = 0; j < nr; ++j) r += (cand[j] < k) ? 1 : 0;
      run[r] = k;
    }
  } else if (nr <= kFastCap) {
    for (int i = nr + tid; i < kFastCap; i += kThreads) cand[i] = ~0ull;
    __syncthreads();
    sort_fast_cap(cand);
    srun = cand;
  }
  // every CTA learns every run's length and region
  const int C = static_cast<int>(cl.num_blocks());
  if (tid < C) {
    *cl.map_shared_rank(&g_runs[rank][0], tid) = (srun == cand) ? 1 : 0;
    *cl.map_shared_rank(&g_runs[rank][1], tid) = nr;
  }
  SS_STAMP(38);
  cl.sync();  // every run is sorted, and rank 0's slice is free
  SS_STAMP(42);
  int n = 0;
  for (int r = 0; r < C; ++r) n += g_runs[r][1];
  SS_TRACE(43, n);
  if (n > kFastCap) return false;
  const unsigned long long* sorted = srun;  // one CTA: its run is the order
  if (C > 1) {
    // the merge, spread over the cluster: every CTA places its own items in
    // rank 0's slice region (a cluster of two or more has slices of 16384
    // tokens or more: the region holds kFastCap keys)
    unsigned long long* dst = cl.map_shared_rank(reinterpret_cast<unsigned long long*>(g_dyn), 0);
    if (C == 2)
      place_run<2>(srun, nr, rank, cand, run, dst);
    else if (C == 4)
      place_run<4>(srun, nr, rank, cand, run, dst);
    else
      place_run<8>(srun, nr, rank, cand, run, dst);
    SS_STAMP(41);
    cl.sync();  // the merged order is complete in rank 0
    if (rank != 0) return true;  // (its run stays put until the kernel's last cluster barrier)
    sorted = reinterpret_cast<const unsigned long long*>(g_dyn);
  }
  SS_STAMP(44);
  SS_STAMP(45);
  if (tid == 0) {
    g_fpos[0] = 0x7fffffff;
    g_fpos[1] = 0x7fffffff;
    g_fpos[2] = -1;
  }
  __syncthreads();
  SS_STAMP(46);

  // ---- the cuts: prefix masses of the top k (two items per thread, in order)
  const int kk = min(c.top_k, n);
  const float m = c.m;
  const int i0 = 2 * tid;
  unsigned long long w0 = 0, w1 = 0;
  if (i0 < kk) w0 = fmass(ekey_y(sorted[i0]), m);
  if (i0 + 1 < kk) w1 = fmass(ekey_y(sorted[i0 + 1]), m);
  unsigned long long ic = 0, im = w0 + w1, tc, tm;
  block_scan2(ic, im, &tc, &tm);
  const unsigned long long before = im - (w0 + w1);
  const unsigned long long Sk = tm;
  const unsigned long long T = c.p_on ? mass_target(c.top_p, Sk) : ~0ull;
  if (c.p_on) {
    if (i0 < kk && before + w0 >= T) atomicMin(&g_fpos[0], i0 + 1);
    else if (i0 + 1 < kk && before + w0 + w1 >= T) atomicMin(&g_fpos[0], i0 + 2);
  }
  if (c.mp_on) {
    for (int i = i0; i < min(i0 + 2, kk); ++i)
      if (!(__fsub_rn(ekey_y(sorted[i]), m) >= c.lmp)) {
        atomicMin(&g_fpos[1], i);
        break;
      }
  }
  __syncthreads();
  const int L = max(1, min(kk, min(g_fpos[0], g_fpos[1])));
  // the kept mass: the prefix through item L - 1
  if (i0 == L - 1) c.kmass = before + w0;
  if (i0 + 1 == L - 1) c.kmass = before + w0 + w1;
  if (tests_draft)
    for (int i = tid; i < L; i += kThreads)
      if (ekey_t(sorted[i]) == c.x) g_fpos[2] = i;
  __syncthreads();
  kept = static_cast<unsigned long long>(L);
  if (tid == 0) c.kcount = kept;
  SS_STAMP(40);

  // ---- the draw, over the first L items
  const uint32_t k0 = c.seed_lo, k1 = c.seed_hi;
  auto draw = [&](bool res, float inv_s) -> int32_t {
    float bs = ninf();
    int32_t bt = 0x7fffffff;
    for (int i = tid; i < L; i += kThreads) {
      const float y = ekey_y(sorted[i]);
      const int32_t t = ekey_t(sorted[i]);
      const uint32_t num = uniform_numerator(
          philox4x32_10(static_cast<uint32_t>(t) >> 2, c.pos, c.rowid, res ? 2u : 0u, k0, k1).w[t & 3]);
      const float sc = res ? draw_score<true>(y, t, num, kGumbelMax, m, inv_s, qrow, ninf())
                           : draw_score<false>(y, t, num, kGumbelMax, m, 0.0f, nullptr, ninf());
      if (sc > ninf() && beats(sc, t, bs, bt)) {
        bs = sc;
        bt = t;
      }
    }
    block_best(bs, bt);
    return bt;
  };
  bool need_draw = !tests_draft;
  if (tests_draft) {
    const float SK = static_cast<float>(static_cast<double>(c.kmass) * (1.0 / 1099511627776.0));
    const float inv_s = __frcp_rn(SK);
    const int xi = g_fpos[2];
    const float Px = (xi >= 0) ? __fmul_rn(__expf(__fsub_rn(ekey_y(sorted[xi]), m)), inv_s) : 0.0f;
    const float q = qrow[c.x];
    const float u = uniform_from_numerator(uniform_numerator(philox4x32_10(0u, c.pos, c.rowid, 1u, k0, k1).w[0]));
    accept = (__fmul_rn(u, q) < Px) ? 1 : 0;
    if (!accept && tid == 0) atomicMax(a.ws_counters + c.nreq + c.req, kRejBase - c.j);
    if (accept) {
      token = c.x;
    } else if (c.skip_draw) {
      token = -1;
    } else {
      const int32_t t = draw(true, inv_s);
      if (t != 0x7fffffff)
        token = t;
      else
        need_draw = true;  // an empty residual (rounding): the stream-0 draw
    }
  }
  if (need_draw) token = c.skip_draw ? -1 : draw(false, 0.0f);
  return true;
}

// Index cutoff for the items of value v when `take` of them (by index) are
// kept.  The CTAs hold increasing index ranges, so the take-th item lies in
// one CTA (tie_rank): CTAs before it keep all their items of value v, CTAs
// after it none, and it finds its own cutoff with one ordered scan of its
// slice.  With `broadcast` every CTA learns that cutoff (one cluster barrier;
// verification needs it for the draft token).  Sets g.cut_t, the cutoff that
// this CTA applies (-1: none of its items of value v, 0x7fffffff: all).
// Called by all threads of every CTA.
__device__ void resolve_ties(const HArgs& a, float v, unsigned long long take, int grp, bool broadcast) {
  Ctx& c = g;
  cg::cluster_group cl = cg::this_cluster();
  const int C = static_cast<int>(cl.num_blocks());
  const int rank = static_cast<int>(cl.block_rank());
  const uint32_t* hist = reinterpret_cast<const uint32_t*>(g_dyn + a.o_hist);
  const unsigned long long* el = reinterpret_cast<const unsigned long long*>(g_dyn + a.o_el);
  const int16_t* eord = reinterpret_cast<const int16_t*>(g_dyn + a.o_hist + kSlots * 2 + (kGroups + 2) * 4);
  if (take == 0) {  // none of them (the same in every CTA)
    __syncthreads();
    if (threadIdx.x == 0) c.cut_t = -1;
    __syncthreads();
    return;
  }
  // per-CTA counts of the items of value v: its run of slots, and its
  // entries of v (all in coarse group grp)
  if (threadIdx.x < C) g_rtie[threadIdx.x] = 0;
  group_ranges(a, grp);
  if (threadIdx.x < C) {
    const int r = threadIdx.x;
    uint32_t n = 0;
    for (int q = first_slot_le_near(v); q < c.M.ns && slot_y(q) == v; ++q)
      n += (*cl.map_shared_rank(hist + (q >> 1), r) >> ((q & 1) << 4)) & 0xffffu;
    atomicAdd(&g_rtie[r], n);
  }
  const int total_e = g_grc[C];
  for (int i = threadIdx.x; i < total_e; i += kThreads) {
    int r = 0;
    while (i >= g_grc[r + 1]) ++r;
    const int e = *cl.map_shared_rank(eord + g_gr0[r] + (i - g_grc[r]), r);
    if (ekey_y(*cl.map_shared_rank(el + e, r)) == v) atomicAdd(&g_rtie[r], 1u);
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    unsigned long long before = 0, total = 0;
    for (int r = 0; r < C; ++r) total += g_rtie[r];
    c.tie_rank = C;  // all of them
    c.tie_local = 0;
    if (take < total) {
      for (int r = 0; r < C; ++r) {
        if (before + g_rtie[r] >= take) {
          c.tie_rank = r;
          c.tie_local = static_cast<int32_t>(take - before);
          break;
        }
        before += g_rtie[r];
      }
    }
    c.cut_t = (rank < c.tie_rank) ? 0x7fffffff : -1;
  }
  __syncthreads();
  const int tr = c.tie_rank;
  if (rank == tr) {
    // this CTA's entries of value v (few): their tokens, sorted
    int32_t* tie_tok = g_tietok;
    if (threadIdx.x == 0) c.n_g = 0;
    __syncthreads();
    for (int e = threadIdx.x; e < c.ne; e += kThreads)
      if (ekey_y(el[e]) == v) {
        const int at = atomicAdd(&c.n_g, 1);
        if (at < kTieEnt) tie_tok[at] = ekey_t(el[e]);
      }
    __syncthreads();
    const bool many = c.n_g > kTieEnt;  // then every entry is checked (slow, rare)
    const int nt = min(c.n_g, kTieEnt);
    if (threadIdx.x == 0)  // a handful of tokens: insertion sort
      for (int i = 1; i < nt; ++i) {
        const int32_t x = tie_tok[i];
        int j = i - 1;
        while (j >= 0 && tie_tok[j] > x) {
          tie_tok[j + 1] = tie_tok[j];
          --j;
        }
        tie_tok[j + 1] = x;
      }
    __syncthreads();
    // each thread takes a contiguous block of vectors, so that one block
    // prefix of the per-thread match counts orders them by index
    const uint4* data = reinterpret_cast<const uint4*>(g_dyn);
    const uint16_t* vb = reinterpret_cast<const uint16_t*>(g_dyn + a.o_vb);
    const int per = (c.nvec + kThreads - 1) / kThreads;
    const int v0 = threadIdx.x * per, v1 = min(v0 + per, c.nvec);
    const int32_t t_lo = c.lo + v0 * 8, t_hi = c.lo + v1 * 8;
    uint32_t mine = 0;
    for (int vv = v0; vv < v1; ++vv) {
      if (__fmul_rn(bf16_to_f(vb[vv >> 1]), c.inv_t) < v) continue;
      const uint4 d = data[vv];
      const uint32_t w[4] = {d.x, d.y, d.z, d.w};
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const uint32_t word = w[e >> 1];
        const float y = __fmul_rn((e & 1) ? __uint_as_float(word & 0xffff0000u) : __uint_as_float(word << 16), c.inv_t);
        mine += (y == v) ? 1u : 0u;
      }
    }
    if (!many) {
      for (int e = 0; e < nt; ++e) mine += (tie_tok[e] >= t_lo && tie_tok[e] < t_hi) ? 1u : 0u;
    } else {
      for (int e = 0; e < c.ne; ++e) {
        const int32_t t = ekey_t(el[e]);
        if (t >= t_lo && t < t_hi && ekey_y(el[e]) == v) ++mine;
      }
    }
    int32_t total = 0;
    const int32_t before = block_excl_scan(static_cast<int32_t>(mine), &total);
    const int want = c.tie_local;
    if (before < want && before + static_cast<int32_t>(mine) >= want) {
      // the crossing thread walks its tokens in index order
      int need = want - before;
      int q = 0;
      while (q < nt && tie_tok[q] < t_lo) ++q;
      for (int vv = v0; vv < v1 && need > 0; ++vv) {
        const uint4 d = data[vv];
        const uint32_t w[4] = {d.x, d.y, d.z, d.w};
        for (int e = 0; e < 8 && need > 0; ++e) {
          const int32_t t = c.lo + vv * 8 + e;
          const uint32_t word = w[e >> 1];
          bool hit = __fmul_rn((e & 1) ? __uint_as_float(word & 0xffff0000u) : __uint_as_float(word << 16),
                               c.inv_t) == v;
          if (!many) {
            while (q < nt && tie_tok[q] < t) ++q;
            if (q < nt && tie_tok[q] == t) hit = true;
          } else if (!hit) {
            for (int e2 = 0; e2 < c.ne; ++e2)
              if (ekey_t(el[e2]) == t && ekey_y(el[e2]) == v) hit = true;
          }
          if (hit && --need == 0) c.cut_t = t;
        }
      }
    }
    __syncthreads();
  }
  if (broadcast) {
    if (rank == tr && threadIdx.x == 0)
      for (int r = 0; r < C; ++r) *cl.map_shared_rank(&g.tcut_in, r) = c.cut_t;
    cl.sync();
    if (threadIdx.x == 0) {
      if (tr < 0)
        c.cut_t = -1;
      else if (tr >= C)
        c.cut_t = 0x7fffffff;
      else
        c.cut_t = c.tcut_in;
    }
    __syncthreads();
  }
}

// ------------------------------------------------------------------ kernel --

__global__ void __launch_bounds__(kThreads, 2) ss_hist_kernel(const HArgs a) {
  cg::cluster_group cl = cg::this_cluster();
  Ctx& c = g;
  const int tid = threadIdx.x;
  const int C = static_cast<int>(cl.num_blocks());
  const int rank = static_cast<int>(cl.block_rank());
  const int launch_task = static_cast<int>(blockIdx.x) / C;
  uint4* data = reinterpret_cast<uint4*>(g_dyn);
  uint16_t* vb = reinterpret_cast<uint16_t*>(g_dyn + a.o_vb);
  uint32_t* hist = reinterpret_cast<uint32_t*>(g_dyn + a.o_hist);
  unsigned long long* el = reinterpret_cast<unsigned long long*>(g_dyn + a.o_el);
  uint32_t* xm = reinterpret_cast<uint32_t*>(g_dyn + a.o_xm);
  uint32_t* pbits = reinterpret_cast<uint32_t*>(g_dyn + a.o_mg);  // patched tokens, until the locator
  uint64_t* mbar = reinterpret_cast<uint64_t*>(g_dyn + a.o_mbar);
  // the patch table shares the histogram region during set-up
  int32_t* hkey = reinterpret_cast<int32_t*>(hist);
  int32_t* hcnt = hkey + kHashCap;
  float* hval = reinterpret_cast<float*>(hcnt + kHashCap);
  uint32_t* hraw = reinterpret_cast<uint32_t*>(hval + kHashCap);  // raw bf16 bits | allowed << 16

  SS_STAMP(0);
  // Programmatic dependent launch: a next call that allows it may start its
  // CTAs as soon as every CTA of this one has started (they take the SM
  // slots this call's finished rows give back).  Such a call reads no output
  // of this one, so only its writes -- outputs, debug rows -- and, for
  // verification, its use of the workspace wait for this grid
  // (griddepcontrol.wait; a no-op in a launch without the attribute).
  grid_launch_dependents();
  // the task's request and position: position-major over (position, request)
  // -- every request's position 0 first, so that later positions tend to
  // start after the earlier ones have decided -- or, in a compact launch,
  // over the target rows that exist
  int req = launch_task, j = 0;
  if (a.mode == 1) {
    if (a.compact && launch_task >= a.nreq) {
      if (tid < 32) locate_position(a, static_cast<long long>(launch_task) - a.nreq);
      __syncthreads();
      req = g_loc[0];
      j = g_loc[1];
    } else {
      j = launch_task / a.nreq;
      req = launch_task - j * a.nreq;
    }
  }
  // the parameter loads go out before the bulk copies (a global load issued
  // after 16 KB copies of every CTA waits behind them)
  if (req >= 0) {
    if (tid < 32) {
      asm volatile("bar.sync 1, 64;" ::: "memory");
      if (tid == 0) decode_and_copy(a, req, j, rank);
    } else if (tid < 64) {
      load_params(a, req, j);
    } else if (tid < 96 && a.target_rows > 0 && !(a.compact && launch_task >= a.nreq)) {
      check_row_count(a);
    }
  }
  __syncthreads();
  SS_STAMP(17);
  if (a.target_rows > 0 && (req < 0 || !g_loc[2])) {
    // the caller's count of target rows is not the offsets' sum: nothing is
    // verified, and the launch's first cluster reports it on every request
    // (a position-0 CTA first waits for the copies it has issued)
    if (req >= 0 && tid == 0)
      for (int q = 0; q < c.nch; ++q) mbar_wait_bounded(mbar + q, 0, kWaitPolls);
    if (launch_task == 0 && rank == 0) {
      grid_dependency_wait();
      const int width = a.max_draft + 1;
      for (int64_t e = tid; e < static_cast<int64_t>(a.nreq) * width; e += kThreads) a.out_token[e] = -1;
      for (int i = tid; i < a.nreq; i += kThreads) {
        a.out_num_accepted[i] = 0;
        a.out_status[i] = SS_ROW_BAD_PARAM;
      }
    }
    __syncthreads();
    return;
  }
  if (!c.valid) return;  // the same for the whole cluster
  if (c.bad_k) {
    // a draft count outside [0, max_draft]: the request's outputs, from its
    // first position only
    grid_dependency_wait();
    if (rank == 0 && tid <= a.max_draft) {
      a.out_token[static_cast<int64_t>(c.req) * (a.max_draft + 1) + tid] = -1;
      if (tid == 0) {
        a.out_num_accepted[c.req] = 0;
        a.out_status[c.req] = SS_ROW_BAD_PARAM;
      }
    }
    return;
  }
  if (tid == 0) c.status = max(c.status, c.pstatus);
  SS_STAMP(19);
  for (int s = tid; s < kHashCap; s += kThreads) {
    hkey[s] = -1;
    hcnt[s] = 0;
    hval[s] = 0.0f;
    hraw[s] = 0;
  }
  if (tid < kCertBins / 2) g_cert[tid] = 0;
  __syncthreads();
  SS_STAMP(20);
  const int32_t V = a.vocab, lo = c.lo, n = c.n;
  const uint16_t* row = a.logits + c.row_off;
  const int words = a.slice / 32;
  {
    const int32_t* mrow = c.use_mask ? a.p.bitmask + static_cast<int64_t>(c.req) * a.p.bitmask_stride + (lo >> 5) : nullptr;
    for (int w = tid; w < words; w += kThreads) {
      const int first = w * 32;
      uint32_t allow = 0;
      if (first < n) {
        allow = mrow ? static_cast<uint32_t>(mrow[w]) : 0xffffffffu;
        if (first + 32 > n) allow &= (1u << (n - first)) - 1u;
      }
      xm[w] = allow;
      pbits[w] = 0;
    }
  }
  SS_STAMP(21);
  // tokens past the bulk copies: plain loads; padding past the row: -inf
  {
    uint16_t* d16 = reinterpret_cast<uint16_t*>(g_dyn);
    const int from = (a.bulk ? c.n8 : 0);
    for (int e = from + tid; e < c.nvec * 8; e += kThreads) d16[e] = (e < n) ? row[lo + e] : 0xff80u;
  }
  __syncthreads();
  SS_STAMP(18);
  // patched tokens: the table, the patched bits, and (from the first insert of
  // each) whether the mask allows it; its staged copy is excluded
  int st = c.status;
  const bool row_ok = st == SS_ROW_OK;
  auto in_slice = [&](int32_t t) { return t >= lo && t < lo + n; };
  auto mark = [&](int32_t t, int s) {
    const uint32_t bit = 1u << ((t - lo) & 31);
    const int w = (t - lo) >> 5;
    if (!(atomicOr(pbits + w, bit) & bit)) {
      c.npatch = 1;  // a flag: some token of the slice is patched
      if (xm[w] & bit) atomicOr(hraw + s, 1u << 16);
    }
  };
  if (row_ok) {
    for (int e = c.h0 + tid; e < c.h1; e += kThreads) {
      const int32_t t = a.p.hist_ids[e];
      if (t < 0 || t >= V) {
        st = max(st, SS_ROW_BAD_INDEX);
      } else if (in_slice(t)) {
        const int s = patch_insert(hkey, t);
        if (s < 0) {
          st = max(st, SS_ROW_LIMIT);
        } else {
          atomicAdd(hcnt + s, 1);
          mark(t, s);
        }
      }
    }
    if (a.mode == 1) {
      // every draft must be a token id (checked at position 0); position j's
      // history holds the drafts before j
      const int lim = (c.j == 0) ? c.k : c.j;
      for (int e = tid; e < lim; e += kThreads) {
        const int32_t t = a.draft_tokens[c.d0 + e];
        if (t < 0 || t >= V) {
          st = max(st, SS_ROW_BAD_INDEX);
        } else if (e < c.j && in_slice(t)) {
          const int s = patch_insert(hkey, t);
          if (s < 0) {
            st = max(st, SS_ROW_LIMIT);
          } else {
            atomicAdd(hcnt + s, 1);
            mark(t, s);
          }
        }
      }
    }
    for (int e = c.b0 + tid; e < c.b1; e += kThreads) {
      const int32_t t = a.p.bias_ids[e];
      const float b = a.p.bias_vals[e];
      if (!isfinite(b)) st = max(st, SS_ROW_BAD_PARAM);
      if (t < 0 || t >= V) {
        st = max(st, SS_ROW_BAD_INDEX);
      } else if (in_slice(t)) {
        const int s = patch_insert(hkey, t);
        if (s < 0) {
          st = max(st, SS_ROW_LIMIT);
        } else {
          if (atomicOr(hcnt + s, kBiasFlag) & kBiasFlag) st = max(st, SS_ROW_BAD_INDEX);  // duplicate id
          hval[s] = b;
          mark(t, s);
        }
      }
    }
  }
  if (st != SS_ROW_OK) atomicMax(&c.status, st);
  __syncthreads();
  if (tid == 0) c.has_excl = c.use_mask;
  __syncthreads();
  SS_STAMP(1);

  // -------------------------------------------------- staging pass
  // Patched tokens stay as staged here; the fix-up after the compaction
  // excludes them and mends their pairs' bounds.
  const bool excl = c.has_excl != 0, tiny = c.need_hist != 0;
  const float inv_t = c.inv_t;
  uint32_t run = kNegInfPair;
  bool timed_out = false;
  {
    const uint8_t* xb = reinterpret_cast<const uint8_t*>(xm);
    const uint8_t* pb = reinterpret_cast<const uint8_t*>(pbits);
    int waited = -1;
    const int nbulk = a.bulk ? c.n8 / 8 : 0;  // vectors landed by bulk copies
    // every thread runs the same number of iterations (the pair exchange
    // below is warp-wide); v past the slice does nothing
    for (int v0 = 0; v0 < c.nvec; v0 += kThreads) {
      const int v = v0 + tid;
      const bool act = v < c.nvec;
      if (act && v < nbulk) {
        const int ch = v / (kChunkTokens / 8);
        if (ch > waited) {
          for (int q = waited + 1; q <= ch; ++q)
            if (!mbar_wait_bounded(mbar + q, 0, kWaitPolls)) timed_out = true;
          waited = ch;
          if (ch == 0) SS_STAMP(22);
          if (ch == 1) SS_STAMP(32);
          if (ch == 2) SS_STAMP(33);
          if (ch == 3) SS_STAMP(34);
        }
      }
      uint4 d = act ? data[v] : make_uint4(kNegInfPair, kNegInfPair, kNegInfPair, kNegInfPair);
      bool dirty = false;
      if (excl && act) {
        const uint32_t A = xb[v];
        if (A != 0xffu) {
          d = apply_allow(d, A);
          dirty = true;
        }
      }
      // (a pre-test first: the smallest magnitude among the eight, zero
      // included, is below the tiny bound -- rare outside exact zeros)
      if (tiny && min_mag8(d) < kTinyA) {
        const uint32_t tm = tiny_pair(d.x) | (tiny_pair(d.y) >> 1) | (tiny_pair(d.z) >> 2) | (tiny_pair(d.w) >> 3);
        if (tm && act) {
          // tiny values move to the entries (patched ones are the fix-up's)
          uint32_t w[4] = {d.x, d.y, d.z, d.w};
          const uint32_t P = pb[v];
          for (int e = 0; e < 8; ++e) {
            const uint32_t sh = (e & 1) ? 16u : 0u;
            const uint32_t h = (w[e >> 1] >> sh) & 0xffffu;
            const uint32_t aa = h & 0x7fffu;
            if (aa != 0 && aa < kTinyA && !((P >> e) & 1u)) {
              add_entry(el, c.greedy ? bf16_to_f(h) : __fmul_rn(bf16_to_f(h), inv_t), lo + v * 8 + e);
              w[e >> 1] = (w[e >> 1] & ~(0xffffu << sh)) | (0xff80u << sh);
            }
          }
          d = make_uint4(w[0], w[1], w[2], w[3]);
          dirty = true;
        }
      }
      if (dirty && act) data[v] = d;
      const uint32_t mx = bmax2(bmax2(d.x, d.y), bmax2(d.z, d.w));
      const uint32_t mh = bmax2(mx, mx >> 16) & 0xffffu;  // max of the two halves in the low half
      // one bound per 16 tokens: vectors v and v ^ 1 sit in lanes tid and
      // tid ^ 1 of the same iteration
      const uint32_t other = __shfl_xor_sync(0xffffffffu, mh, 1);
      if (act && !(v & 1)) vb[v >> 1] = static_cast<uint16_t>(bmax2(mh, other) & 0xffffu);
      run = bmax2(run, mx);
    }
    SS_STAMP(23);
    if (tid == 0)
      for (int q = waited + 1; q < c.nch; ++q)
        if (!mbar_wait_bounded(mbar + q, 0, kWaitPolls)) timed_out = true;
    if (a.stall_polls && tid == 0) {
      // the self-test: the last barrier slot (no chunk uses it) is armed for
      // one arrival that never comes
      uint64_t* bar = mbar + (kMaxChunks - 1);
      mbar_init(bar, 1);
      fence_barrier_init();
      if (!mbar_wait_bounded(bar, 0, a.stall_polls)) timed_out = true;
    }
  }
  if (timed_out) atomicMax(&c.status, SS_ROW_TIMEOUT);
  __syncthreads();
  SS_STAMP(11);
  // processed values of the patched tokens: exact entries (penalties, bias,
  // mask, temperature, each an individually rounded fp32 operation)
  // (every warp runs the loop uniformly: one entry-counter atomic per warp)
  for (int s = tid; s < kHashCap; s += kThreads) {
    const int32_t t = hkey[s];
    float y = ninf();
    if (t >= 0) {
      uint16_t* staged = reinterpret_cast<uint16_t*>(g_dyn) + (t - lo);
      const uint32_t raw = hraw[s] | *staged;
      *staged = 0xff80u;  // the staged copy is excluded: the token is an entry
      float z = bf16_to_f(raw & 0xffffu);
      const int32_t hc = hcnt[s];
      const int32_t cnt = hc & ~kBiasFlag;
      if (cnt > 0) {
        z = (z > 0.0f) ? __fdiv_rn(z, c.rep) : __fmul_rn(z, c.rep);
        z = __fsub_rn(z, __fmul_rn(c.freq, static_cast<float>(cnt)));
        z = __fsub_rn(z, c.pres);
      }
      if (hc & kBiasFlag) z = __fadd_rn(z, hval[s]);
      y = !(raw >> 16) ? ninf() : (c.greedy ? z : __fmul_rn(z, c.inv_t));
      hval[s] = y;  // kept for the draft-token lookup and the debug output
      if (y != y || y == pinf()) {
        atomicMax(&c.status, SS_ROW_NONFINITE);
        y = ninf();
      }
    }
    const bool add = y != ninf();
    const uint32_t ball = __ballot_sync(0xffffffffu, add);
    if (ball) {
      const int lane = tid & 31;
      int base = 0;
      if (lane == __ffs(ball) - 1) base = atomicAdd(&c.nent, __popc(ball));
      base = __shfl_sync(0xffffffffu, base, __ffs(ball) - 1);
      if (add) {
        const int i = base + __popc(ball & ((1u << lane) - 1u));
        if (i < kEntCap)
          el[i] = ekey(y, t);
        else
          atomicMax(&c.status, SS_ROW_LIMIT);
      }
    }
  }
  __syncthreads();
  // fix-up: the bounds of the patched tokens' 16-token pairs are recomputed
  // (their staged copies were excluded above)
  if (c.npatch) {
    for (int s = tid; s < kHashCap; s += kThreads)
      if (hkey[s] >= 0) {
        const int pr = (hkey[s] - lo) >> 4;
        const uint4 d0 = data[2 * pr], d1 = data[2 * pr + 1];
        const uint32_t mx = bmax2(bmax2(bmax2(d0.x, d0.y), bmax2(d0.z, d0.w)), bmax2(bmax2(d1.x, d1.y), bmax2(d1.z, d1.w)));
        vb[pr] = static_cast<uint16_t>(bmax2(mx, mx >> 16) & 0xffffu);
      }
    __syncthreads();
  }
  SS_STAMP(2);

  // -------------------------------------------------- debug output
  if (a.debug) {
    grid_dependency_wait();
    float* out = a.debug + static_cast<int64_t>(c.row) * V;
    const uint16_t* d16 = reinterpret_cast<const uint16_t*>(g_dyn);
    for (int e = tid; e < n; e += kThreads) {
      const float z = bf16_to_f(d16[e]);
      out[lo + e] = c.greedy ? z : __fmul_rn(z, inv_t);
    }
    __syncthreads();
    const int ne = min(c.nent, kEntCap);
    for (int i = tid; i < ne; i += kThreads) out[ekey_t(el[i])] = ekey_y(el[i]);
    __syncthreads();
    // the patched tokens last, from the table: an entry's key folds -0 to +0
    for (int s = tid; s < kHashCap; s += kThreads)
      if (hkey[s] >= 0) out[hkey[s]] = hval[s];
  }

  // -------------------------------------------------- exchange 1
  {
    // one reduction: the CTA's largest staged value with the first pair
    // holding it (a NaN anywhere counts as +inf: the row is non-finite
    // either way), and its largest entry (lowest token among equals)
    float gbest = ninf();
    int gvec = 0x7fffffff;  // the first pair holding it
    for (int p = tid; p < c.nvec / 2; p += kThreads) {
      const float vm = bf16_to_f(vb[p]);
      if (vm > gbest) {
        gbest = vm;
        gvec = p;
      }
    }
    if ((bmax2(run, run >> 16) & 0x7fffu) > 0x7f80u) {
      gbest = pinf();
      gvec = 0;
    }
    float es = ninf();
    int32_t et = 0x7fffffff;
    const int ne = min(c.nent, kEntCap);
    for (int i = tid; i < ne; i += kThreads) {
      const float y = ekey_y(el[i]);
      const int32_t t = ekey_t(el[i]);
      if (beats(y, t, es, et)) {
        es = y;
        et = t;
      }
    }
    block_best2(gbest, gvec, es, et);
    const float zmax = gbest;
    SS_STAMP(12);
    // greedy: lowest index of the CTA's largest staged value
    int32_t garg = 0x7fffffff;
    if (c.greedy && gvec != 0x7fffffff && zmax != pinf() && tid == 0) {
      const uint16_t* d16 = reinterpret_cast<const uint16_t*>(g_dyn) + gvec * 16;
      for (int e = 15; e >= 0; --e)
        if (bf16_to_f(d16[e]) == zmax) garg = lo + gvec * 16 + e;
    }
    // top-k rows: pairs per binade below this CTA's maximum (the certificate)
    const uint32_t zbin = key16(__float_as_uint(zmax) >> 16) >> kCertShift;
    if (c.k_on) {
      const int lane = tid & 31;
      for (int p0 = 0; p0 < c.nvec / 2; p0 += kThreads) {
        const int p = p0 + tid;
        int d = -1;
        if (p < c.nvec / 2) {
          const uint32_t h = vb[p];
          if (h != 0xff80u) d = static_cast<int>(zbin) - static_cast<int>(key16(h) >> kCertShift);
        }
        if (d >= kCertBins) d = -1;
        // warp-aggregated counts: one atomic per distinct bin in the warp
        const uint32_t same = __match_any_sync(0xffffffffu, d);
        if (d >= 0 && lane == __ffs(same) - 1)
          atomicAdd(&g_cert[d >> 1], static_cast<uint32_t>(__popc(same)) << ((d & 1) << 4));
      }
    }
    // the draft token's processed value, in the CTA that owns it
    float xy = ninf();
    int32_t xhere = 0;
    if (c.x >= 0 && in_slice(c.x)) {
      xhere = 1;
      if (tid == 0) {
        const int s = patch_find(hkey, c.x);
        if (s >= 0) {
          xy = hval[s];
        } else {
          const uint16_t h = reinterpret_cast<const uint16_t*>(g_dyn)[c.x - lo];
          xy = c.greedy ? bf16_to_f(h) : __fmul_rn(bf16_to_f(h), inv_t);
          if (h == 0xff80u)  // excluded, or moved to the entries as a tiny value
            for (int i = 0; i < ne; ++i)
              if (ekey_t(el[i]) == c.x) xy = ekey_y(el[i]);
        }
      }
    }
    if (c.k_on) __syncthreads();  // the certificate counts are complete
    if (tid == 0) {
      // verification: the request's rejection word (the workspace is the
      // previous call's until that grid has finished)
      int32_t rej_seen = 0;
      if (a.mode == 1) {
        grid_dependency_wait();
        rej_seen = ld_cg_s32(a.ws_counters + c.nreq + c.req);
      }
      c.seed_pair = gvec;
      c.seed_ey = es;
      c.seed_et = et;
      Part1& p = g_mine;
      p.zmax = zmax;
      p.emax = es;
      // greedy: lowest index among this CTA's items of its largest value
      // (staged tokens and entries, both in z units)
      const float lmax = fmaxf(zmax, es);
      int32_t la = 0x7fffffff;
      if (zmax == lmax) la = garg;
      if (es == lmax) la = min(la, et);
      p.arg = la;
      p.status = c.status;
      p.nent = ne;
      p.xy = xy;
      p.xhere = xhere;
      p.zbin = static_cast<int32_t>(zbin);
      p.rej = rej_seen;
      for (int b = 0; b < kCertBins / 2; ++b) p.cert[b] = c.k_on ? g_cert[b] : 0u;
    }
    __syncthreads();
    SS_STAMP(13);
    if (tid < C) *cl.map_shared_rank(&g_p1[rank], tid) = g_mine;
    cl.sync();
    SS_STAMP(14);
    if (tid == 0) {
      float zm = ninf(), em = ninf();
      int32_t st1 = SS_ROW_OK, zb = -1;
      bool nan = false;
      g_goff[0] = 0;
      for (int r = 0; r < C; ++r) {
        const Part1& p = g_p1[r];
        if (p.zmax != p.zmax) nan = true;
        zm = fmax_nan(zm, p.zmax);
        em = fmaxf(em, p.emax);
        st1 = max(st1, p.status);
        if (p.xhere) c.xy = p.xy;
        if (p.zmax != ninf()) zb = max(zb, p.zbin);
        g_goff[r + 1] = g_goff[r] + p.nent;
      }
      const float ysm = c.greedy ? zm : __fmul_rn(zm, c.inv_t);
      float m = fmax_nan(ysm, em);
      if (nan || m != m || m == pinf()) st1 = max(st1, SS_ROW_NONFINITE);
      else if (m == ninf()) st1 = max(st1, SS_ROW_EMPTY_SET);
      // greedy: the lowest index among the CTAs' items of value m
      int32_t arg = 0x7fffffff;
      if (c.greedy)
        for (int r = 0; r < C; ++r) {
          const Part1& p = g_p1[r];
          if (fmaxf(p.zmax, p.emax) == m && p.arg < arg) arg = p.arg;
        }
      if (a.mode == 1) {
        int32_t rj = 0;
        for (int r = 0; r < C; ++r) rj = max(rj, g_p1[r].rej);
        c.skip_draw = rj > kRejBase - c.j;  // the same in every CTA
      }
      c.tau_key = 0;
      c.tau_pairs = 0;
      c.pick = zb;
      c.arg = arg;
      c.status = st1;
      c.m = m;
      c.zmax = zm;
      c.ne = ne;
      if (c.x < 0) c.xy = ninf();
    }
    __syncthreads();
    // top-k: the highest bin boundary with at least k tokens at or above it
    // (pairs whose maximum is at or above it, summed over the cluster); lane
    // l takes bins 2l and 2l + 1, then a warp prefix
    if (c.k_on && tid < 32) {
      const int zb = c.pick;
      uint32_t cnt[2] = {0, 0};
      for (int h = 0; h < 2; ++h) {
        const int d = 2 * tid + h;
        if (zb >= 0 && d < zb)
          for (int r = 0; r < C; ++r) {
            const Part1& p = g_p1[r];
            const int dd = d - (zb - p.zbin);  // the same bin in rank r's counts
            if (p.zmax != ninf() && dd >= 0 && dd < kCertBins) cnt[h] += (p.cert[dd >> 1] >> ((dd & 1) << 4)) & 0xffffu;
          }
      }
      unsigned long long cum = cnt[0] + cnt[1];
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const unsigned long long y = __shfl_up_sync(0xffffffffu, cum, o);
        if (tid >= o) cum += y;
      }
      const unsigned long long lo = cum - cnt[1];  // through bin 2l
      const unsigned long long k = static_cast<unsigned long long>(c.top_k);
      const unsigned ball = __ballot_sync(0xffffffffu, cum >= k);
      if (ball && tid == __ffs(ball) - 1) {
        const int d = (lo >= k) ? 2 * tid : 2 * tid + 1;
        c.tau_key = static_cast<uint32_t>(zb - d) << kCertShift;
        c.tau_pairs = (lo >= k) ? lo : cum;
      }
    }
    __syncthreads();
  }
  SS_STAMP(3);

  // -------------------------------------------------- decisions
  const int32_t status = c.status;
  int32_t token = -1, accept = 0;
  unsigned long long kept = 0;
  const bool verify = a.mode == 1;
  const bool tests_draft = verify && c.j < c.k;
  const float* qrow = tests_draft ? a.draft_probs + static_cast<int64_t>(c.drow) * a.draft_stride : nullptr;
  const uint32_t k0 = c.seed_lo, k1 = c.seed_hi;
  if (status == SS_ROW_OK) {
    if (c.greedy) {
      // the argmax survives every filter; a tested draft is accepted when it
      // is the argmax (P one-hot), else the argmax is emitted
      kept = 1;
      token = c.arg;
      if (tests_draft) {
        const float q = qrow[c.x];
        const float u = uniform_from_numerator(uniform_numerator(philox4x32_10(0u, c.pos, c.rowid, 1u, k0, k1).w[0]));
        const float P = (c.x == c.arg) ? 1.0f : 0.0f;
        accept = (__fmul_rn(u, q) < P) ? 1 : 0;
        token = accept ? c.x : c.arg;
        if (!accept && rank == 0 && tid == 0) atomicMax(a.ws_counters + c.nreq + c.req, kRejBase - c.j);
      }
    } else if (!(c.k_on && c.tau_key != 0 && c.top_k <= kFastK && c.tau_pairs <= kFastCap &&
                 short_path(a, tests_draft, qrow, token, accept, kept))) {
      float cv = ninf();
      int32_t ct = -1;
      bool mp_on = c.mp_on != 0;
      if (c.need_hist) {
        // ---------------------------------------------- histogram
        if (tid == 0) {
          c.M = make_slot_map(c.zmax);
          c.ntot = 0;
          c.stot = 0;
          c.fail_loc = 0;
        }
        for (int s = tid; s < kSlots / 2; s += kThreads) hist[s] = 0;
        if (tid <= kGroups) {
          g_ecnt[tid] = 0;
          g_emass[tid] = 0;
        }
        __syncthreads();
        const SlotMap M = c.M;
        // group bounds at run boundaries of equal y
        if (tid <= kGroups) {
          int32_t b = min(tid * (kSlots / kGroups), M.ns);
          while (b > 0 && b < M.ns && slot_y(b) == slot_y(b - 1)) ++b;
          g_gb[tid] = (tid == kGroups) ? M.ns : b;
          if (tid == kGroups) g_gb[kGroups + 1] = M.ns;  // the tail group: entries only
        }
        SS_STAMP(27);
        // candidates: top-k rows the tokens at or above the certificate;
        // top-p rows the tokens with a non-zero fixed-point mass
        const uint32_t tau = c.tau_key;
        const float skip = (c.k_on) ? ninf() : __fsub_rn(c.m, kMassRange);
        uint32_t below = 0;
        // (top-p rows have no certificate: their loop skips the key test)
        auto count_pass_b = [&](auto with_tau) {
          for (int v = tid; v < c.nvec; v += kThreads) {
            const uint32_t hb = vb[v >> 1];
            if (hb == 0xff80u || (with_tau.value && key16(hb) < tau) || __fmul_rn(bf16_to_f(hb), inv_t) < skip) continue;
            const uint4 d = data[v];
            const uint32_t w[4] = {d.x, d.y, d.z, d.w};
#pragma unroll
            for (int e = 0; e < 8; ++e) {
              const uint32_t h = (w[e >> 1] >> ((e & 1) ? 16 : 0)) & 0xffffu;
              if (with_tau.value && key16(h) < tau) continue;
              const int32_t s = slot_of(M, h);
              if (static_cast<uint32_t>(s) < static_cast<uint32_t>(M.ns))
                atomicAdd(hist + (s >> 1), 1u << ((s & 1) << 4));
              else if (h != 0xff80u)
                ++below;
            }
          }
        };
        if (tau != 0)
          count_pass_b(std::true_type{});
        else
          count_pass_b(std::false_type{});
        __syncthreads();  // group bounds and histogram complete
        SS_STAMP(4);
        // slot position and group of every local entry, its place within the
        // group (the list is then ordered by group: every CTA reads one
        // group's entries of another CTA as one range), and for min-p the
        // largest entry failing the test
        int32_t* eoff = reinterpret_cast<int32_t*>(g_dyn + a.o_hist + kSlots * 2);
        int16_t* eord = reinterpret_cast<int16_t*>(eoff + (kGroups + 2));
        int eq[kEntCap / kThreads], er[kEntCap / kThreads];
        uint32_t fk = 0;  // min-p: the largest failing entry key of this thread
#pragma unroll
        for (int k = 0; k < kEntCap / kThreads; ++k) {
          const int e = tid + k * kThreads;
          eq[k] = -1;
          if (e < c.ne) {
            const float y = ekey_y(el[e]);
            const int32_t p = first_slot_le_near(y);
            g_epos[e] = static_cast<int16_t>(p);
            const int q = group_of(p);
            eq[k] = q;
            er[k] = static_cast<int>(atomicAdd(&g_ecnt[q], 1u));
            atomic_add_u64_split(&g_emass[q], fmass(y, c.m));
            if (mp_on && !(__fsub_rn(y, c.m) >= c.lmp)) fk = max(fk, okey(y));
          }
        }
        if (mp_on) {  // one atomic per warp
          fk = __reduce_max_sync(0xffffffffu, fk);
          if ((tid & 31) == 0 && fk) atomicMax(&c.fail_loc, fk);
        }
        __syncthreads();
        SS_STAMP(24);
        if (tid < 32) {  // group offsets of the ordered list
          constexpr int kPer = (kGroups + 1 + 31) / 32;
          int32_t loc[kPer], sum = 0;
#pragma unroll
          for (int i = 0; i < kPer; ++i) {
            const int q = tid * kPer + i;
            loc[i] = (q <= kGroups) ? static_cast<int32_t>(g_ecnt[q]) : 0;
            sum += loc[i];
          }
          int32_t inc = sum;
#pragma unroll
          for (int o = 1; o < 32; o <<= 1) {
            const int32_t y = __shfl_up_sync(0xffffffffu, inc, o);
            if (tid >= o) inc += y;
          }
          int32_t run_off = inc - sum;
#pragma unroll
          for (int i = 0; i < kPer; ++i) {
            const int q = tid * kPer + i;
            if (q <= kGroups) eoff[q] = run_off;
            run_off += loc[i];
          }
          if (tid == 31) eoff[kGroups + 1] = inc;
        }
        // coarse counts and masses of this CTA (slots and entries), pushed to
        // every CTA (exchange 2); the tail group also carries the count of
        // uncounted tokens below the slots, and each CTA its min-p fail key
        uint32_t* pc = xm;  // [C][kGroups + 1] counts, then masses, then fail keys
        unsigned long long* pm = reinterpret_cast<unsigned long long*>(xm + ((kMaxCluster * (kGroups + 1) + 1) & ~1));
        uint32_t* pf = reinterpret_cast<uint32_t*>(pm + kMaxCluster * (kGroups + 1));
        {
          const int grp = tid >> 3, sub = tid & 7;  // 8 threads per group
          uint32_t cnt = 0;
          unsigned long long mass = 0;
          const float m = c.m;
          const int s_end = g_gb[grp + 1];
          // no branch on empty slots (their mass term is 0): unrolled, the
          // iterations' loads and exponentials overlap
#pragma unroll 4
          for (int s = g_gb[grp] + sub; s < s_end; s += 8) {
            const uint32_t h = (hist[s >> 1] >> ((s & 1) << 4)) & 0xffffu;
            cnt += h;
            mass += static_cast<unsigned long long>(h) * fmass(slot_y(s), m);
          }
#pragma unroll
          for (int o = 1; o < 8; o <<= 1) {
            cnt += __shfl_xor_sync(0xffffffffu, cnt, o);
            mass += __shfl_xor_sync(0xffffffffu, mass, o);
          }
          cnt += g_ecnt[grp];
          mass += g_emass[grp];
          SS_STAMP(25);
          const uint32_t bsum = block_sum<uint32_t>(below);  // (a block barrier: eoff is complete)
          SS_STAMP(26);
#pragma unroll
          for (int k = 0; k < kEntCap / kThreads; ++k)
            if (eq[k] >= 0) eord[eoff[eq[k]] + er[k]] = static_cast<int16_t>(tid + k * kThreads);
          if (sub < C) {
            *cl.map_shared_rank(pc + rank * (kGroups + 1) + grp, sub) = cnt;
            *cl.map_shared_rank(pm + rank * (kGroups + 1) + grp, sub) = mass;
          }
          if (tid < C) {
            // the tail group's entries, and the uncounted tokens in the top
            // byte of its mass (saturating)
            *cl.map_shared_rank(pc + rank * (kGroups + 1) + kGroups, tid) = g_ecnt[kGroups];
            *cl.map_shared_rank(pm + rank * (kGroups + 1) + kGroups, tid) =
                (g_emass[kGroups] & 0x00ffffffffffffffull) | (static_cast<unsigned long long>(min(bsum, 255u)) << 56);
            *cl.map_shared_rank(pf + rank, tid) = c.fail_loc;
          }
        }
        SS_STAMP(15);
        cl.sync();
        SS_STAMP(16);
        if (tid < 96) {  // the groups, and (warp-reduced) their totals
          uint32_t cnt = 0;
          unsigned long long mass = 0, bel = 0;
          if (tid <= kGroups) {
            for (int r = 0; r < C; ++r) {
              cnt += pc[r * (kGroups + 1) + tid];
              const unsigned long long mm = pm[r * (kGroups + 1) + tid];
              if (tid == kGroups) {
                bel += mm >> 56;
                mass += mm & 0x00ffffffffffffffull;
              } else {
                mass += mm;
              }
            }
            if (tid == kGroups) {
              c.below = bel;  // uncounted tokens below the slots (saturating per CTA)
              uint32_t fk = 0;
              for (int r = 0; r < C; ++r) fk = max(fk, pf[r]);
              c.fail_key = fk;
            }
            g_gcnt[tid] = cnt;
            g_gmass[tid] = mass;
          }
          const uint32_t wc = __reduce_add_sync(0xffffffffu, cnt);
#pragma unroll
          for (int o = 16; o; o >>= 1) mass += __shfl_xor_sync(0xffffffffu, mass, o);
          if ((tid & 31) == 0) {
            atomicAdd(&c.ntot, static_cast<unsigned long long>(wc));
            atomicAdd(&c.stot, mass);
          }
        }
        __syncthreads();
        SS_STAMP(5);

        // ---------------------------------------------- the cuts
        // K = the shortest of the top-k, top-p and min-p prefixes of the
        // (y desc, token asc) order.  A cut is (value v, items of v taken).
        bool unknown = false;
        float bv = ninf();                     // best (shortest) cut so far
        unsigned long long btake = 0, bcc = 0, bcm = 0;
        int bgrp = 0;
        bool have_cut = false;
        unsigned long long Sk = 0;
        if (c.k_on) {
          locate(a, 0, static_cast<unsigned long long>(c.top_k));
          if (c.w_found < 0) unknown = true;
          if (c.w_found > 0) {
            have_cut = true;
            bv = c.w_v;
            btake = c.w_take;
            bcc = c.w_cc;
            bcm = c.w_cm;
            bgrp = c.w_grp;
            Sk = bcm + btake * fmass(bv, c.m);
          }
        }
        if (!have_cut && !unknown) {
          // every item (top-k off or larger than the item count): all must
          // have been counted
          if ((c.below || (c.k_on && c.tau_key)) &&
              (c.k_on || M.ns == 0 || __fmul_rn(slot_z(M, M.ns - 1), inv_t) > skip))
            unknown = true;
          Sk = c.stot;
          if (tid == 0) c.kcount = c.ntot;
        }
        SS_STAMP(6);
        if (c.p_on && !unknown) {
          const unsigned long long T = mass_target(c.top_p, Sk);
          locate(a, 1, T);
          if (c.w_found < 0) unknown = true;
          if (c.w_found > 0 && (!have_cut || c.w_v > bv || (c.w_v == bv && c.w_take < btake))) {
            have_cut = true;
            bv = c.w_v;
            btake = c.w_take;
            bcc = c.w_cc;
            bcm = c.w_cm;
            bgrp = c.w_grp;
          }
        }
        if (c.mp_on && !unknown) {
          // the largest value failing the min-p test: among the slots (they
          // fall monotonically) and every CTA's entries
          if (tid == 0) {
            // the first slot failing it: from the slot of m + log(min_p),
            // a walk to the exact boundary (the test falls with the slot)
            auto fails = [&](int q) { return !(__fsub_rn(slot_y(q), c.m) >= c.lmp); };
            int lo_s = first_slot_le_near(__fadd_rn(c.m, c.lmp));
            if (lo_s < M.ns && fails(lo_s)) {
              while (lo_s > 0 && fails(lo_s - 1)) --lo_s;
            } else {
              while (lo_s < M.ns && !fails(lo_s)) ++lo_s;
            }
            float vf = (lo_s < M.ns) ? slot_y(lo_s) : ninf();
            if (c.fail_key) vf = fmaxf(vf, okey_value(c.fail_key));
            // every counted slot passes, but uncounted tokens below them may
            // not: the min-p cut is unknown unless a shorter cut exists
            c.pick = (lo_s == M.ns && (c.below || c.tau_key) && !have_cut) ? 1 : 0;
            c.w_v = vf;
          }
          __syncthreads();
          const float vf = c.w_v;
          if (c.pick) unknown = true;
          if (!unknown && vf != ninf() && (!have_cut || vf > bv || (vf == bv && btake > 0))) {
            above_value(a, vf);
            if (c.w_found < 0) {
              unknown = true;
            } else {
              have_cut = true;
              bv = vf;
              btake = 0;
              bcc = c.w_cc;
              bcm = c.w_cm;
            }
          }
        }
        SS_STAMP(7);
        if (unknown) {
          if (tid == 0) c.status = SS_ROW_LIMIT;
        } else if (have_cut) {
          if (tid == 0) {
            c.cut_v = bv;
            c.kcount = bcc + btake;
            c.kmass = bcm + btake * fmass(bv, c.m);
          }
          __syncthreads();
          resolve_ties(a, bv, btake, bgrp, tests_draft);
          cv = c.cut_v;
          ct = c.cut_t;
        } else {
          if (tid == 0) c.kmass = Sk;
        }
        __syncthreads();
        mp_on = false;  // min-p is part of the cut
      }
      if (c.status == SS_ROW_OK) {
        const unsigned long long* ents = el;
        const int n_ents = c.ne;
        // |K| (and its mass) for rows without a histogram; a plain draw
        // counts K itself
        const bool fold_count = !c.need_hist && a.out_kept && !tests_draft && !c.skip_draw;
        if (!c.need_hist && (a.out_kept || tests_draft) && !fold_count) {
          int32_t cnt = 0;
          unsigned long long mass = 0;
          count_pass(a, tests_draft, ents, n_ents, cnt, mass);
          const PartD r = exchange_d<true, false>(ninf(), 0x7fffffff, cnt, mass);
          if (tid == 0) {
            c.kcount = static_cast<unsigned long long>(r.count);
            c.kmass = r.mass;
          }
          __syncthreads();
        }
        SS_STAMP(8);
        kept = c.kcount;
        bool need_draw = !tests_draft;
        if (tests_draft) {
          // accept x with u * q(x) < P(x)
          const float SK = static_cast<float>(static_cast<double>(c.kmass) * (1.0 / 1099511627776.0));
          const float inv_s = __frcp_rn(SK);
          const float yx = c.xy;
          const bool xin = yx != ninf() && in_cut(yx, c.x, cv, ct) && (!mp_on || __fsub_rn(yx, c.m) >= c.lmp);
          const float Px = xin ? __fmul_rn(__expf(__fsub_rn(yx, c.m)), inv_s) : 0.0f;
          const float q = qrow[c.x];
          const float u = uniform_from_numerator(uniform_numerator(philox4x32_10(0u, c.pos, c.rowid, 1u, k0, k1).w[0]));
          accept = (__fmul_rn(u, q) < Px) ? 1 : 0;
          if (!accept && rank == 0 && tid == 0) atomicMax(a.ws_counters + c.nreq + c.req, kRejBase - c.j);
          if (accept) {
            token = c.x;
          } else if (c.skip_draw) {
            token = -1;  // an earlier position rejected: this draw is never used
          } else {
            float bs;
            int32_t bt;
            if (tid == 0) draw_reset();
            __syncthreads();
            draw_pass<true>(a, cv, ct, mp_on, inv_s, logf(SK), qrow, ents, n_ents);
            cta_best(bs, bt);
            const PartD r = exchange_d<false, true>(bs, bt, 0, 0);
            if (r.arg != 0x7fffffff && r.best > ninf())
              token = r.arg;
            else
              need_draw = true;  // an empty residual (rounding): the stream-0 draw
          }
        }
        if (need_draw && c.skip_draw) {
          token = -1;
        } else if (need_draw) {
          float bs;
          int32_t bt;
          if (tid == 0) draw_reset();
          __syncthreads();
          if (fold_count) {
            int32_t cnt = 0;
            draw_pass<false, true>(a, cv, ct, mp_on, 0.0f, 0.0f, nullptr, ents, n_ents, &cnt);
            SS_STAMP(36);
            cta_best(bs, bt);
            const PartD r = exchange_d<true, true>(bs, bt, cnt, 0);
            token = r.arg;
            kept = static_cast<unsigned long long>(r.count);
          } else {
            draw_pass<false>(a, cv, ct, mp_on, 0.0f, 0.0f, nullptr, ents, n_ents);
            SS_STAMP(36);
            cta_best(bs, bt);
            const PartD r = exchange_d<false, true>(bs, bt, 0, 0);
            token = r.arg;
          }
        }
      }
    }
  }
  SS_STAMP(9);
  // every CTA of the cluster is done with the others' shared memory
  cl.sync();
  SS_STAMP(10);
  if (rank != 0 || tid != 0) return;
  const int32_t fst = c.status;
  const bool ok = fst == SS_ROW_OK;
  if (!verify) {
    grid_dependency_wait();  // the previous call has written its outputs
    a.out_token[c.row] = ok ? token : -1;
    a.out_status[c.row] = fst;
    if (a.out_kept) a.out_kept[c.row] = ok ? static_cast<int32_t>(kept) : 0;
    return;
  }
  if (a.out_kept) a.out_kept[c.row] = ok ? static_cast<int32_t>(kept) : 0;
  // verification: publish this position; the last one of the request writes
  // the request's outputs
  const int width = a.max_draft + 1;
  int4* res = a.ws_results + static_cast<int64_t>(c.req) * width;
  res[c.j] = make_int4(fst, accept, token, static_cast<int32_t>(kept));
  __threadfence();
  const int prev = atomicAdd(a.ws_counters + c.req, 1);
  if (prev != c.k) return;
  __threadfence();
  int32_t wst = SS_ROW_OK;
  for (int jj = 0; jj <= c.k; ++jj) wst = max(wst, ld_cg_s32(&res[jj].x));
  int32_t* out = a.out_token + static_cast<int64_t>(c.req) * width;
  int nacc = 0;
  if (wst == SS_ROW_OK) {
    int jj = 0;
    for (; jj < c.k; ++jj) {
      const int32_t acc = ld_cg_s32(&res[jj].y);
      if (acc) {
        out[jj] = a.draft_tokens[c.d0 + jj];
        ++nacc;
      } else {
        out[jj] = ld_cg_s32(&res[jj].z);
        break;
      }
    }
    if (jj == c.k) out[c.k] = ld_cg_s32(&res[c.k].z);
    for (int q = nacc + 1; q < width; ++q) out[q] = -1;
  } else {
    for (int q = 0; q < width; ++q) out[q] = -1;
  }
  a.out_num_accepted[c.req] = nacc;
  a.out_status[c.req] = wst;
  a.ws_counters[c.req] = 0;  // ready for the next call
  a.ws_counters[c.nreq + c.req] = 0;
}

// ------------------------------------------------------------------ host --

static int cluster_for(int32_t vocab) {
  for (int cs = 1; cs <= kMaxCluster; cs <<= 1) {
    const int64_t slice = ((static_cast<int64_t>(vocab) + cs - 1) / cs + 63) / 64 * 64;
    if (slice <= kSliceTarget) return cs;
  }
  const int64_t slice = ((static_cast<int64_t>(vocab) + kMaxCluster - 1) / kMaxCluster + 63) / 64 * 64;
  return slice <= kSliceMax ? kMaxCluster : 0;
}

static void layout(HArgs& a) {
  int64_t off = static_cast<int64_t>(a.slice) * 2;
  auto take = [&](int64_t bytes, int64_t align) {
    off = (off + align - 1) / align * align;
    const int32_t at = static_cast<int32_t>(off);
    off += bytes;
    return at;
  };
  a.o_vb = take(static_cast<int64_t>(a.slice / 16) * 2, 16);
  // slot counts as 16-bit halves of 32-bit words (a slot holds at most
  // kSliceMax tokens); the patch table shares the region during set-up
  a.o_hist = take(std::max<int64_t>(kSlots * 2, kHashCap * 16), 16);
  a.o_el = take(kEntCap * 8, 16);
  // one region, in turn: the allow bits, the exchange-2 push, a group's
  // gathered entries
  const int64_t xm_bytes = a.slice / 8;
  const int64_t push_bytes =
      ((kMaxCluster * (kGroups + 1) + 1) & ~1) * 4 + kMaxCluster * (kGroups + 1) * 8 + kMaxCluster * 4;
  const int64_t gather_bytes = kGatherCap * 10;
  a.o_xm = take(std::max(xm_bytes, std::max(push_bytes, gather_bytes)), 16);
  // the patched-token bits during set-up, then a group's items merged by value
  a.o_mg = take(std::max<int64_t>((kFineMax + kGatherCap) * 8, a.slice / 8), 16);
  a.o_mbar = take(kMaxChunks * 8, 16);
  a.total = static_cast<int32_t>((off + 127) / 128 * 128);
}

static thread_local int32_t t_err = 0;

static ss_status launch(HArgs& a, cudaStream_t stream) {
  const int cs = a.ncta;
  layout(a);
  static int set_bytes[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64) dev = 0;
  cudaError_t e = cudaSuccess;
  if (set_bytes[dev] < a.total) {
    e = cudaFuncSetAttribute(ss_hist_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, a.total);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(ss_hist_kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                               cudaSharedmemCarveoutMaxShared);
    if (e == cudaSuccess) set_bytes[dev] = a.total;
  }
  if (e == cudaSuccess) {
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(static_cast<unsigned>(a.num_tasks) * cs, 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = static_cast<size_t>(a.total);
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = cs;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    // with SS_SAMPLE_OVERLAP_PREVIOUS / SS_VERIFY_OVERLAP_PREVIOUS: this
    // launch may begin while the kernel before it on the stream finishes (the
    // kernel orders its writes and its workspace use after that grid)
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = a.overlap ? 2 : 1;
    e = cudaLaunchKernelEx(&cfg, ss_hist_kernel, a);
  }
  if (e != cudaSuccess) {
    t_err = static_cast<int32_t>(e);
    return SS_ERR_CUDA;
  }
  return SS_OK;
}

}  // namespace hist

int hist_cluster_size(int32_t vocab, int32_t dtype) {
  if (dtype != SS_DTYPE_BF16 || vocab < 1) return 0;
  return hist::cluster_for(vocab);
}

int32_t hist_last_error() { return hist::t_err; }

}  // namespace ss

#ifdef SS_HIST_STAMPS
extern "C" int ss_hist_stamps_copy(void* host, size_t bytes) {
  return static_cast<int>(cudaMemcpyFromSymbol(host, ss::hist::g_stamps, bytes));
}
extern "C" int ss_hist_stamps_set(const void* host, size_t bytes) {
  return static_cast<int>(cudaMemcpyToSymbol(ss::hist::g_stamps, host, bytes));
}
#endif

namespace ss {

ss_status hist_sample(const ss_sample_args& A, cudaStream_t stream, uint32_t stall_polls) {
  hist::HArgs a{};
  a.stall_polls = stall_polls;
  a.mode = 0;
  a.num_tasks = A.num_rows;
  a.vocab = A.vocab;
  a.max_draft = 0;
  a.row_stride = A.row_stride;
  a.logits = static_cast<const uint16_t*>(A.logits);
  a.p = A.params;
  a.out_token = A.out_token;
  a.out_status = A.out_status;
  a.out_kept = A.out_kept;
  a.debug = A.debug_processed;
  a.overlap = (A.flags & SS_SAMPLE_OVERLAP_PREVIOUS) ? 1 : 0;
  a.ncta = hist::cluster_for(A.vocab);
  const int64_t slice = ((static_cast<int64_t>(A.vocab) + a.ncta - 1) / a.ncta + 63) / 64 * 64;
  a.slice = static_cast<int32_t>(slice);
  a.bulk = ((reinterpret_cast<uintptr_t>(A.logits) & 15u) == 0 && ((A.row_stride * 2) & 15) == 0) ? 1 : 0;
  return hist::launch(a, stream);
}

ss_status hist_verify(const ss_verify_args& A, int4* results, int32_t* counters, cudaStream_t stream) {
  hist::HArgs a{};
  a.mode = 1;
  a.nreq = A.num_requests;
  a.target_rows = A.num_target_rows;
  // one cluster per target row when the idle clusters of the full launch
  // (positions past a request's drafts) would outnumber the rows past
  // position 0, whose clusters then search the offsets for their position
  const int64_t full = static_cast<int64_t>(A.num_requests) * (A.max_draft + 1);
  const int64_t rows = A.num_target_rows;
  a.compact = (rows > 0 && full - rows > rows - A.num_requests) ? 1 : 0;
  a.num_tasks = a.compact ? A.num_target_rows : static_cast<int32_t>(full);
  a.vocab = A.vocab;
  a.max_draft = A.max_draft;
  a.row_stride = A.row_stride;
  a.logits = static_cast<const uint16_t*>(A.target_logits);
  a.draft_offsets = A.draft_offsets;
  a.draft_tokens = A.draft_tokens;
  a.draft_probs = A.draft_probs;
  a.draft_stride = A.draft_stride;
  a.p = A.params;
  a.out_token = A.out_tokens;
  a.out_num_accepted = A.out_num_accepted;
  a.out_status = A.out_status;
  a.out_kept = A.out_kept;
  a.debug = A.debug_processed;
  a.overlap = (A.flags & SS_VERIFY_OVERLAP_PREVIOUS) ? 1 : 0;
  a.ws_results = results;
  a.ws_counters = counters;
  a.ncta = hist::cluster_for(A.vocab);
  const int64_t slice = ((static_cast<int64_t>(A.vocab) + a.ncta - 1) / a.ncta + 63) / 64 * 64;
  a.slice = static_cast<int32_t>(slice);
  a.bulk = ((reinterpret_cast<uintptr_t>(A.target_logits) & 15u) == 0 && ((A.row_stride * 2) & 15) == 0) ? 1 : 0;
  return hist::launch(a, stream);
}

}  // namespace ss
