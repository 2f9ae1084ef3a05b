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
constexpr int kCertBins = 32;     // binades below the maximum counted for the top-k certificate
constexpr int kTieEnt = 64;       // entries tied at a cut value, per CTA
constexpr int kChunkTokens = 8192;
constexpr int kMaxChunks = 8;
constexpr int kMaxCluster = 8;
constexpr int kSliceTarget = 32768;  // tokens per CTA that keep two CTAs per SM
constexpr int kSliceMax = 49152;
constexpr uint32_t kWaitPolls = 1u << 22;
constexpr int kBiasFlag = 1 << 30;
constexpr uint32_t kNegInfPair = 0xff80ff80u;
constexpr uint32_t kTinyA = 0x3780u;  // |z| below 2^-16: tiny (exact entries unless zero)
// Fixed-point masses of tokens more than this far below the maximum are 0.
constexpr float kMassRange = 28.2f;

static_assert(kSlots % kGroups == 0, "groups tile the slots");

// Phase timestamps for tracing (built only with -DSS_HIST_STAMPS): the
// global timer at the end of each phase, per CTA, read back with
// ss_hist_stamps_copy.
#ifdef SS_HIST_STAMPS
constexpr int kStampCtas = 16384, kStampPhases = 24;
__device__ unsigned long long g_stamps[kStampCtas][kStampPhases];
#define SS_STAMP(k)                                                                \
  do {                                                                             \
    if (threadIdx.x == 0 && blockIdx.x < kStampCtas) {                             \
      unsigned long long t_;                                                       \
      asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t_));                       \
      g_stamps[blockIdx.x][k] = t_;                                                \
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
__device__ __forceinline__ unsigned long long fmass(float y, float m) {
  const float e = fminf(__expf(__fsub_rn(y, m)), 1.0f);
  return static_cast<unsigned long long>(__fmul_rn(e, 1099511627776.0f));
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
  int32_t zbin;   // binade of zmax (16-bit order key >> 7)
  uint32_t cert[kCertBins];  // 16-token pairs whose maximum lies d binades below zbin
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
  int32_t valid, row, req, j, k, bad_k, d0, x, drow;
  int64_t row_off;
  int32_t lo, n, nvec, nch, n8;
  // parameters
  float T, inv_t, top_p, min_p, rep, freq, pres, lmp;
  int32_t greedy, top_k, k_on, p_on, mp_on, need_hist, use_mask, has_excl;
  uint32_t seed_lo, seed_hi, pos, rowid;
  int32_t h0, h1, b0, b1;
  int32_t status;   // local, then cluster-wide
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
  SlotMap M;
  // cut: K = {y > cut_v} U {y == cut_v, token <= cut_t}
  float cut_v;
  int32_t cut_t;
  unsigned long long kcount, kmass;  // |K| and its fixed-point mass
  // locate results
  int32_t w_found, w_slot;
  float w_v;
  unsigned long long w_take, w_cc, w_cm;
  int32_t tie_rank, tie_local;
  unsigned long long below;
  // scratch
  int32_t pick;
  int32_t tcut_in;  // tie cutoff, written by the CTA that resolves it
  int32_t xpar;     // buffer of the next draw / mass exchange
  uint32_t fail_key;
};

__shared__ Ctx g;
__shared__ Part1 g_p1[kMaxCluster];
__shared__ Part1 g_mine;
__shared__ PartD g_pd[2][kMaxCluster];
__shared__ unsigned char g_red[kWarps * 16];
__shared__ unsigned long long g_scan[2 * kWarps];
__shared__ int32_t g_gb[kGroups + 2];                // coarse group bounds (slots)
__shared__ uint32_t g_gcnt[kGroups + 1];
__shared__ unsigned long long g_gmass[kGroups + 1];
__shared__ uint32_t g_ecnt[kGroups + 1];             // this CTA's entries per group
__shared__ unsigned long long g_emass[kGroups + 1];
__shared__ uint32_t g_fc[kFineMax];                  // one group's slot counts (all CTAs)
__shared__ int16_t g_epos[kEntCap];                  // slot position of each local entry
__shared__ int32_t g_goff[kMaxCluster + 1];
__shared__ uint32_t g_rtie[kMaxCluster];
__shared__ uint32_t g_cert[kCertBins];
__shared__ int32_t g_tietok[kTieEnt];

extern __shared__ __align__(128) uint8_t g_dyn[];

__device__ __forceinline__ uint32_t key16(uint32_t h) { return (h & 0x8000u) ? (~h & 0xffffu) : (h | 0x8000u); }
__device__ __forceinline__ uint32_t key16_bits(uint32_t k) { return (k & 0x8000u) ? (k & 0x7fffu) : (~k & 0xffffu); }

// ------------------------------------------------------ block reductions --

__device__ __forceinline__ float block_max_nan(float v) {
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
#pragma unroll
  for (int o = 16; o; o >>= 1) v = fmax_nan(v, __shfl_xor_sync(0xffffffffu, v, o));
  float* r = reinterpret_cast<float*>(g_red);
  __syncthreads();
  if (lane == 0) r[wid] = v;
  __syncthreads();
  v = r[0];
  for (int w = 1; w < kWarps; ++w) v = fmax_nan(v, r[w]);
  return v;
}

// (score desc, token asc) arg-reduction over the block; every thread gets it.
__device__ __forceinline__ void block_best(float& s, int32_t& t) {
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
#pragma unroll
  for (int o = 16; o; o >>= 1) {
    const float os = __shfl_xor_sync(0xffffffffu, s, o);
    const int32_t ot = __shfl_xor_sync(0xffffffffu, t, o);
    if (beats(os, ot, s, t)) {
      s = os;
      t = ot;
    }
  }
  float* rs = reinterpret_cast<float*>(g_red);
  int32_t* rt = reinterpret_cast<int32_t*>(g_red) + kWarps;
  __syncthreads();
  if (lane == 0) {
    rs[wid] = s;
    rt[wid] = t;
  }
  __syncthreads();
  s = rs[0];
  t = rt[0];
  for (int w = 1; w < kWarps; ++w)
    if (beats(rs[w], rt[w], s, t)) {
      s = rs[w];
      t = rt[w];
    }
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
  v = r[0];
  for (int w = 1; w < kWarps; ++w) v += r[w];
  return v;
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
  int32_t before = 0, tot = 0;
  for (int w = 0; w < kWarps; ++w) {
    if (w < wid) before += r[w];
    tot += r[w];
  }
  *total = tot;
  return before + x - v;
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
    r[kWarps + wid] = m;
  }
  __syncthreads();
  unsigned long long bc = 0, bm = 0, sc = 0, sm = 0;
  for (int w = 0; w < kWarps; ++w) {
    if (w < wid) {
      bc += r[w];
      bm += r[kWarps + w];
    }
    sc += r[w];
    sm += r[kWarps + w];
  }
  c += bc;
  m += bm;
  *tc = sc;
  *tm = sm;
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
__device__ void decode_and_copy(const HArgs& a, int task, int rank) {
  Ctx& c = g;
  c.valid = 1;
  c.bad_k = 0;
  c.status = SS_ROW_OK;
  c.nent = 0;
  c.npatch = 0;
  c.xpar = 0;
  c.kcount = 0;
  c.kmass = 0;
  c.x = -1;
  c.drow = -1;
  c.d0 = 0;
  int req = task, j = 0, k = 0;
  int64_t row = task;
  if (a.mode == 1) {
    const int width = a.max_draft + 1;
    req = task / width;
    j = task - req * width;
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

__device__ void read_params(const HArgs& a) {
  Ctx& c = g;
  const ss_params& p = a.p;
  const int i = c.req;
  int st = c.status;
  const float T = p.temperature[i];
  c.T = T;
  c.top_k = p.top_k ? p.top_k[i] : 0;
  c.top_p = p.top_p ? p.top_p[i] : 1.0f;
  c.min_p = p.min_p ? p.min_p[i] : 0.0f;
  c.rep = p.repetition ? p.repetition[i] : 1.0f;
  c.freq = p.frequency ? p.frequency[i] : 0.0f;
  c.pres = p.presence ? p.presence[i] : 0.0f;
  const uint64_t seed = p.seed[i];
  c.seed_lo = static_cast<uint32_t>(seed);
  c.seed_hi = static_cast<uint32_t>(seed >> 32);
  c.rowid = p.row_id ? p.row_id[i] : static_cast<uint32_t>(i);
  const int64_t pos64 = p.position[i];
  const int64_t last = pos64 + (a.mode == 1 ? c.k : 0);
  if (pos64 < 0 || last > 0xFFFFFFFFLL) st = max(st, SS_ROW_BAD_PARAM);
  c.pos = static_cast<uint32_t>(pos64) + static_cast<uint32_t>(c.j);
  c.h0 = c.h1 = c.b0 = c.b1 = 0;
  if (p.hist_offsets) {
    c.h0 = p.hist_offsets[i];
    c.h1 = p.hist_offsets[i + 1];
  }
  if (p.bias_offsets) {
    c.b0 = p.bias_offsets[i];
    c.b1 = p.bias_offsets[i + 1];
  }
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
  c.status = st;
  c.greedy = (T == 0.0f);
  c.inv_t = (c.greedy || !(T > 0.0f)) ? 1.0f : __frcp_rn(T);
  c.k_on = (!c.greedy && c.top_k > 0 && c.top_k < a.vocab);
  c.p_on = (!c.greedy && c.top_p < 1.0f);
  c.mp_on = (!c.greedy && c.min_p > 0.0f);
  c.lmp = c.mp_on ? logf(c.min_p) : 0.0f;
  c.need_hist = c.k_on || c.p_on;
  c.use_mask = p.bitmask && (!p.use_bitmask || p.use_bitmask[i]);
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
// (score desc, token asc), count and mass summed.  Called by all threads.
__device__ PartD exchange_d(float best, int32_t arg, int32_t count, unsigned long long mass) {
  cg::cluster_group cl = cg::this_cluster();
  block_best(best, arg);  // (a block barrier: g.xpar below is current)
  // consecutive exchanges alternate between two buffers: a CTA still reading
  // the previous result is never overwritten
  const int par = g.xpar;
  count = block_sum<int32_t>(count);
  mass = block_sum<unsigned long long>(mass);
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
    if (beats(o.best, o.arg, r.best, r.arg)) {
      r.best = o.best;
      r.arg = o.arg;
    }
    r.count += o.count;
    r.mass += o.mass;
  }
  return r;
}

// ---------------------------------------------------------------- passes --

// The draw over K (stream 0) or, with RES, over the residual
// max(P - q, 0) (stream 2, log r + g); P(t) = exp(y - m) / S.  Returns this
// thread's best (score, token); entries are visited by the CTA that owns
// their token.
template <bool RES>
__device__ void draw_pass(const HArgs& a, float cv, int32_t ct, bool mp_on, float inv_s, float log_s,
                          const float* qrow, const unsigned long long* ents, int n_ents, float& bs, int32_t& bt) {
  const Ctx& c = g;
  const uint4* data = reinterpret_cast<const uint4*>(g_dyn);
  const uint16_t* vb = reinterpret_cast<const uint16_t*>(g_dyn + a.o_vb);
  const float inv_t = c.inv_t, m = c.m, lmp = c.lmp;
  const uint32_t k0 = c.seed_lo, k1 = c.seed_hi, pos = c.pos, rid = c.rowid;
  const uint32_t stream = RES ? 2u : 0u;
  // the largest score a token of processed value y can reach
  auto reach = [&](float y) -> float {
    return RES ? (y - m - log_s + kGumbelMax + 1e-3f + fabsf(y) * 1e-6f) : (y + kGumbelMax);
  };
  auto member = [&](float y, int32_t t) -> bool {
    return y != ninf() && in_cut(y, t, cv, ct) && (!mp_on || __fsub_rn(y, m) >= lmp);
  };
  auto consider = [&](float y, int32_t t, uint32_t word) {
    const uint32_t num = uniform_numerator(word);
    float base = y;
    if (RES) {
      const float P = __fmul_rn(__expf(__fsub_rn(y, m)), inv_s);
      const float r = __fsub_rn(P, qrow[t]);
      if (!(r > 0.0f)) return;
      base = logf(r);
    }
    if (base + gumbel_upper_bound(num) < bs) return;
    const float s = __fadd_rn(base, gumbel_from_numerator(num));
    if (beats(s, t, bs, bt)) {
      bs = s;
      bt = t;
    }
  };
  const int nvec = c.nvec;
  for (int v = threadIdx.x; v < nvec; v += kThreads) {
    const float vy = __fmul_rn(bf16_to_f(vb[v >> 1]), inv_t);
    if (vy < cv || vy == ninf() || reach(vy) < bs) continue;
    if (mp_on && !(__fsub_rn(vy, m) >= lmp)) continue;
    const uint4 d = data[v];
    const uint32_t w[4] = {d.x, d.y, d.z, d.w};
    const int32_t t0 = c.lo + v * 8;
#pragma unroll
    for (int half = 0; half < 2; ++half) {
      float y[4];
      bool any = false;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const uint32_t word = w[half * 2 + (e >> 1)];
        y[e] = __fmul_rn((e & 1) ? __uint_as_float(word & 0xffff0000u) : __uint_as_float(word << 16), inv_t);
        const int32_t t = t0 + half * 4 + e;
        const bool ok = member(y[e], t) && reach(y[e]) >= bs;
        if (!ok) y[e] = ninf();
        any |= ok;
      }
      if (!any) continue;
      const int32_t tq = t0 + half * 4;
      const Philox4 r = philox4x32_10(static_cast<uint32_t>(tq) >> 2, pos, rid, stream, k0, k1);
#pragma unroll
      for (int e = 0; e < 4; ++e)
        if (y[e] != ninf()) consider(y[e], tq + e, r.w[e]);
    }
  }
  for (int i = threadIdx.x; i < n_ents; i += kThreads) {
    const unsigned long long e = ents[i];
    const int32_t t = ekey_t(e);
    if (t < c.lo || t >= c.lo + c.n) continue;
    const float y = ekey_y(e);
    if (!member(y, t) || reach(y) < bs) continue;
    const Philox4 r = philox4x32_10(static_cast<uint32_t>(t) >> 2, pos, rid, stream, k0, k1);
    consider(y, t, r.w[t & 3]);
  }
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

// First slot in [lo, hi) whose y is <= v (hi if none); y falls with s.
__device__ int32_t first_slot_le(float v, int32_t lo, int32_t hi) {
  while (lo < hi) {
    const int32_t mid = (lo + hi) >> 1;
    if (slot_y(mid) <= v)
      hi = mid;
    else
      lo = mid + 1;
  }
  return lo;
}

__device__ __forceinline__ int group_of(int32_t p) {
  if (p >= g.M.ns) return kGroups;
  int lo = 0, hi = kGroups - 1;  // the last q with gb[q] <= p
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (g_gb[mid] <= p)
      lo = mid;
    else
      hi = mid - 1;
  }
  return lo;
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

// Reads the slot counts of coarse group `grp` from every CTA into g_fc, and
// gathers the group's entries from every CTA's list into (gk, gp), sorted
// (y desc, token asc); g.n_g is their number (-1 if more than kGatherCap).
// The gather buffer is the exchange-2 region, free once the coarse sums are
// read.  Called by all threads; ends with a block barrier.
__device__ void load_group(const HArgs& a, int grp) {
  cg::cluster_group cl = cg::this_cluster();
  const int C = static_cast<int>(cl.num_blocks());
  const int s0 = g_gb[grp], s1 = g_gb[grp + 1];
  const uint32_t* hist = reinterpret_cast<const uint32_t*>(g_dyn + a.o_hist);
  const unsigned long long* el = reinterpret_cast<const unsigned long long*>(g_dyn + a.o_el);
  unsigned long long* gk = reinterpret_cast<unsigned long long*>(g_dyn + a.o_xm);
  int16_t* gp = reinterpret_cast<int16_t*>(gk + kGatherCap);
  __syncthreads();  // the previous readers of g_fc and of the buffer are done
  if (threadIdx.x == 0) g.n_g = 0;
  for (int i = threadIdx.x; i < s1 - s0; i += kThreads) {
    uint32_t cnt = 0;
    const int q = s0 + i;
    for (int r = 0; r < C; ++r) cnt += (*cl.map_shared_rank(hist + (q >> 1), r) >> ((q & 1) << 4)) & 0xffffu;
    g_fc[i] = cnt;
  }
  __syncthreads();
  // every (CTA, entry) pair: the entries of this group, appended
  const int total = g_goff[C];
  for (int i = threadIdx.x; i < total; i += kThreads) {
    int r = 0;
    while (i >= g_goff[r + 1]) ++r;
    const int e = i - g_goff[r];
    const int16_t p = *cl.map_shared_rank(g_epos + e, r);
    if (group_of(p) != grp) continue;
    const int at = atomicAdd(&g.n_g, 1);
    if (at < kGatherCap) {
      gk[at] = *cl.map_shared_rank(el + e, r);
      gp[at] = p;
    }
  }
  __syncthreads();
  const int n = g.n_g;
  __syncthreads();
  if (n > kGatherCap) {
    if (threadIdx.x == 0) g.n_g = -1;
    __syncthreads();
    return;
  }
  if (n > 1) {
    int np2 = 1;
    while (np2 < n) np2 <<= 1;
    for (int i = n + threadIdx.x; i < np2; i += kThreads) {
      gk[i] = ~0ull;
      gp[i] = 0x7fff;
    }
    __syncthreads();
    for (int k = 2; k <= np2; k <<= 1)
      for (int j = k >> 1; j > 0; j >>= 1) {
        for (int q = threadIdx.x; q < (np2 >> 1); q += kThreads) {
          const int i = ((q & ~(j - 1)) << 1) | (q & (j - 1));
          const unsigned long long x = gk[i], y = gk[i + j];
          if ((x > y) == ((i & k) == 0)) {
            gk[i] = y;
            gk[i + j] = x;
            const int16_t t = gp[i];
            gp[i] = gp[i + j];
            gp[i + j] = t;
          }
        }
        __syncthreads();
      }
  }
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
  if (c.n_g < 0) {
    if (threadIdx.x == 0) c.w_found = -1;
    __syncthreads();
    return;
  }
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
    const int grp = group_of(first_slot_le(v, 0, c.M.ns));
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

// Index cutoff for the items of value v when `take` of them (by index) are
// kept.  The CTAs hold increasing index ranges, so the take-th item lies in
// one CTA (tie_rank): CTAs before it keep all their items of value v, CTAs
// after it none, and it finds its own cutoff with one ordered scan of its
// slice.  With `broadcast` every CTA learns that cutoff (one cluster barrier;
// verification needs it for the draft token).  Sets g.cut_t, the cutoff that
// this CTA applies (-1: none of its items of value v, 0x7fffffff: all).
// Called by all threads of every CTA.
__device__ void resolve_ties(const HArgs& a, float v, unsigned long long take, bool broadcast) {
  Ctx& c = g;
  cg::cluster_group cl = cg::this_cluster();
  const int C = static_cast<int>(cl.num_blocks());
  const int rank = static_cast<int>(cl.block_rank());
  const uint32_t* hist = reinterpret_cast<const uint32_t*>(g_dyn + a.o_hist);
  const unsigned long long* el = reinterpret_cast<const unsigned long long*>(g_dyn + a.o_el);
  // per-CTA counts of the items of value v: its run of slots and its entries
  if (threadIdx.x < C) g_rtie[threadIdx.x] = 0;
  __syncthreads();
  if (threadIdx.x < C) {
    const int r = threadIdx.x;
    uint32_t n = 0;
    for (int q = first_slot_le(v, 0, c.M.ns); q < c.M.ns && slot_y(q) == v; ++q)
      n += (*cl.map_shared_rank(hist + (q >> 1), r) >> ((q & 1) << 4)) & 0xffffu;
    atomicAdd(&g_rtie[r], n);
  }
  const int total_e = g_goff[C];
  for (int i = threadIdx.x; i < total_e; i += kThreads) {
    int r = 0;
    while (i >= g_goff[r + 1]) ++r;
    if (ekey_y(*cl.map_shared_rank(el + (i - g_goff[r]), r)) == v) atomicAdd(&g_rtie[r], 1u);
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    unsigned long long before = 0, total = 0;
    for (int r = 0; r < C; ++r) total += g_rtie[r];
    c.tie_rank = C;  // all of them
    c.tie_local = 0;
    if (take == 0) {
      c.tie_rank = -1;
    } else if (take < total) {
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
  const int task = static_cast<int>(blockIdx.x) / C;
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
  if (tid == 0) decode_and_copy(a, task, rank);
  __syncthreads();
  if (!c.valid) return;  // the same for the whole cluster
  if (c.bad_k) {
    // a draft count outside [0, max_draft]: the request's outputs, from its
    // first position only
    if (rank == 0 && tid <= a.max_draft) {
      a.out_token[static_cast<int64_t>(c.req) * (a.max_draft + 1) + tid] = -1;
      if (tid == 0) {
        a.out_num_accepted[c.req] = 0;
        a.out_status[c.req] = SS_ROW_BAD_PARAM;
      }
    }
    return;
  }
  if (tid == 0) read_params(a);
  for (int s = tid; s < kHashCap; s += kThreads) {
    hkey[s] = -1;
    hcnt[s] = 0;
    hval[s] = 0.0f;
    hraw[s] = 0;
  }
  __syncthreads();
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
  // tokens past the bulk copies: plain loads; padding past the row: -inf
  {
    uint16_t* d16 = reinterpret_cast<uint16_t*>(g_dyn);
    const int from = (a.bulk ? c.n8 : 0);
    for (int e = from + tid; e < c.nvec * 8; e += kThreads) d16[e] = (e < n) ? row[lo + e] : 0xff80u;
  }
  __syncthreads();
  // patched tokens: the table, the patched bits, and (from the first insert of
  // each) whether the mask allows it; its staged copy is excluded
  int st = c.status;
  const bool row_ok = st == SS_ROW_OK;
  auto in_slice = [&](int32_t t) { return t >= lo && t < lo + n; };
  auto mark = [&](int32_t t, int s) {
    const uint32_t bit = 1u << ((t - lo) & 31);
    const int w = (t - lo) >> 5;
    if (!(atomicOr(pbits + w, bit) & bit)) {
      atomicAdd(&c.npatch, 1);
      if (atomicAnd(xm + w, ~bit) & bit) atomicOr(hraw + s, 1u << 16);
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
  if (tid == 0) c.has_excl = c.use_mask || c.npatch > 0;
  __syncthreads();
  SS_STAMP(1);

  // -------------------------------------------------- staging pass
  const bool excl = c.has_excl != 0, tiny = c.need_hist != 0;
  const float inv_t = c.inv_t;
  uint32_t run = kNegInfPair;
  float gbest = ninf();  // greedy: this thread's largest vector maximum and its first vector
  int gvec = 0x7fffffff;
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
        }
      }
      uint4 d = act ? data[v] : make_uint4(kNegInfPair, kNegInfPair, kNegInfPair, kNegInfPair);
      bool dirty = false;
      if (excl && act) {
        const uint32_t P = pb[v];
        if (P) {  // the raw logits of the patched tokens, into the table
          const uint32_t w[4] = {d.x, d.y, d.z, d.w};
          for (int e = 0; e < 8; ++e)
            if ((P >> e) & 1u) {
              const int s = patch_find(hkey, lo + v * 8 + e);
              if (s >= 0) hraw[s] |= (w[e >> 1] >> ((e & 1) ? 16 : 0)) & 0xffffu;
            }
        }
        const uint32_t A = xb[v];
        if (A != 0xffu) {
          d = apply_allow(d, A);
          dirty = true;
        }
      }
      if (tiny) {
        const uint32_t tm = tiny_pair(d.x) | (tiny_pair(d.y) >> 1) | (tiny_pair(d.z) >> 2) | (tiny_pair(d.w) >> 3);
        if (tm && act) {
          uint32_t w[4] = {d.x, d.y, d.z, d.w};
          for (int e = 0; e < 8; ++e) {
            const uint32_t sh = (e & 1) ? 16u : 0u;
            const uint32_t h = (w[e >> 1] >> sh) & 0xffffu;
            const uint32_t aa = h & 0x7fffu;
            if (aa != 0 && aa < kTinyA) {
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
      const float vm = bf16_to_f(mh);
      if (act && vm > gbest) {
        gbest = vm;
        gvec = v;
      }
    }
    if (tid == 0)
      for (int q = waited + 1; q < c.nch; ++q)
        if (!mbar_wait_bounded(mbar + q, 0, kWaitPolls)) timed_out = true;
  }
  if (timed_out) atomicMax(&c.status, SS_ROW_TIMEOUT);
  __syncthreads();
  SS_STAMP(11);
  // processed values of the patched tokens: exact entries (penalties, bias,
  // mask, temperature, each an individually rounded fp32 operation)
  for (int s = tid; s < kHashCap; s += kThreads) {
    const int32_t t = hkey[s];
    if (t < 0) continue;
    const uint32_t raw = hraw[s];
    float z = bf16_to_f(raw & 0xffffu);
    const int32_t hc = hcnt[s];
    const int32_t cnt = hc & ~kBiasFlag;
    if (cnt > 0) {
      z = (z > 0.0f) ? __fdiv_rn(z, c.rep) : __fmul_rn(z, c.rep);
      z = __fsub_rn(z, __fmul_rn(c.freq, static_cast<float>(cnt)));
      z = __fsub_rn(z, c.pres);
    }
    if (hc & kBiasFlag) z = __fadd_rn(z, hval[s]);
    const float y = !(raw >> 16) ? ninf() : (c.greedy ? z : __fmul_rn(z, c.inv_t));
    hval[s] = y;  // kept for the draft-token lookup and the debug output
    if (y != y || y == pinf()) atomicMax(&c.status, SS_ROW_NONFINITE);
    else if (y != ninf()) add_entry(el, y, t);
  }
  __syncthreads();
  SS_STAMP(2);

  // -------------------------------------------------- debug output
  if (a.debug) {
    float* out = a.debug + static_cast<int64_t>(c.row) * V;
    const uint16_t* d16 = reinterpret_cast<const uint16_t*>(g_dyn);
    for (int e = tid; e < n; e += kThreads) {
      const float z = bf16_to_f(d16[e]);
      out[lo + e] = c.greedy ? z : __fmul_rn(z, inv_t);
    }
    __syncthreads();
    for (int s = tid; s < kHashCap; s += kThreads)
      if (hkey[s] >= 0) out[hkey[s]] = hval[s];
    const int ne = min(c.nent, kEntCap);
    for (int i = tid; i < ne; i += kThreads) out[ekey_t(el[i])] = ekey_y(el[i]);
  }

  // -------------------------------------------------- exchange 1
  {
    const uint32_t rmax = bmax2(run, run >> 16) & 0xffffu;
    const float zmax = block_max_nan(bf16_to_f(rmax));
    SS_STAMP(12);
    // greedy: lowest index of the CTA's largest staged value
    int32_t garg = 0x7fffffff;
    if (c.greedy) {
      float s = (gbest == zmax) ? 0.0f : ninf();
      int32_t t = (gbest == zmax) ? gvec : 0x7fffffff;
      block_best(s, t);  // smallest vector index among those holding the maximum
      if (t != 0x7fffffff && tid == 0) {
        const uint4 d = data[t];
        const uint32_t w[4] = {d.x, d.y, d.z, d.w};
        for (int e = 7; e >= 0; --e) {
          const uint32_t h = (w[e >> 1] >> ((e & 1) ? 16 : 0)) & 0xffffu;
          if (bf16_to_f(h) == zmax) garg = lo + t * 8 + e;
        }
      }
    }
    // top-k rows: pairs per binade below this CTA's maximum (the certificate)
    const uint32_t zbin = key16(__float_as_uint(zmax) >> 16) >> 7;
    if (c.k_on) {
      if (tid < kCertBins) g_cert[tid] = 0;
      __syncthreads();
      const int lane = tid & 31;
      for (int p0 = 0; p0 < c.nvec / 2; p0 += kThreads) {
        const int p = p0 + tid;
        int d = -1;
        if (p < c.nvec / 2) {
          const uint32_t h = vb[p];
          if (h != 0xff80u) d = static_cast<int>(zbin) - static_cast<int>(key16(h) >> 7);
        }
        if (d >= kCertBins) d = -1;
        // warp-aggregated counts: one atomic per distinct binade in the warp
        uint32_t todo = __ballot_sync(0xffffffffu, d >= 0);
        while (todo) {
          const int leader = __ffs(todo) - 1;
          const int dl = __shfl_sync(0xffffffffu, d, leader);
          const uint32_t same = __ballot_sync(0xffffffffu, d == dl);
          if (lane == leader) atomicAdd(&g_cert[dl], static_cast<uint32_t>(__popc(same)));
          todo &= ~same;
        }
      }
    }
    // largest entry (lowest token among equals)
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
    block_best(es, et);
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
    if (tid == 0) {
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
      for (int b = 0; b < kCertBins; ++b) p.cert[b] = c.k_on ? g_cert[b] : 0u;
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
      c.tau_key = 0;
      c.pick = zb;
      c.arg = arg;
      c.status = st1;
      c.m = m;
      c.zmax = zm;
      c.ne = ne;
      if (c.x < 0) c.xy = ninf();
    }
    __syncthreads();
    // top-k: the highest binade boundary with at least k tokens at or above
    // it (pairs whose maximum is at or above it, summed over the cluster);
    // one lane per binade, then a warp prefix
    if (c.k_on && tid < 32) {
      const int zb = c.pick, d = tid;
      uint32_t cnt = 0;
      if (zb >= 0 && d < kCertBins && d < zb)
        for (int r = 0; r < C; ++r) {
          const Part1& p = g_p1[r];
          const int dd = d - (zb - p.zbin);  // the same binade in rank r's counts
          if (p.zmax != ninf() && dd >= 0 && dd < kCertBins) cnt += p.cert[dd];
        }
      unsigned long long cum = cnt;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const unsigned long long y = __shfl_up_sync(0xffffffffu, cum, o);
        if (tid >= o) cum += y;
      }
      const unsigned ball = __ballot_sync(0xffffffffu, cum >= static_cast<unsigned long long>(c.top_k));
      if (ball && tid == __ffs(ball) - 1) c.tau_key = static_cast<uint32_t>(zb - d) << 7;
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
      }
    } else {
      float cv = ninf();
      int32_t ct = -1;
      bool mp_on = c.mp_on != 0;
      if (c.need_hist) {
        // ---------------------------------------------- histogram
        if (tid == 0) c.M = make_slot_map(c.zmax);
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
        // candidates: top-k rows the tokens at or above the certificate;
        // top-p rows the tokens with a non-zero fixed-point mass
        const uint32_t tau = c.tau_key;
        const float skip = (c.k_on) ? ninf() : __fsub_rn(c.m, kMassRange);
        uint32_t below = 0;
        for (int v = tid; v < c.nvec; v += kThreads) {
          const uint32_t hb = vb[v >> 1];
          if (hb == 0xff80u || key16(hb) < tau || __fmul_rn(bf16_to_f(hb), inv_t) < skip) continue;
          const uint4 d = data[v];
          const uint32_t w[4] = {d.x, d.y, d.z, d.w};
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            const uint32_t h = (w[e >> 1] >> ((e & 1) ? 16 : 0)) & 0xffffu;
            if (key16(h) < tau) continue;
            const int32_t s = slot_of(M, h);
            if (static_cast<uint32_t>(s) < static_cast<uint32_t>(M.ns))
              atomicAdd(hist + (s >> 1), 1u << ((s & 1) << 4));
            else if (h != 0xff80u)
              ++below;
          }
        }
        __syncthreads();  // group bounds and histogram complete
        SS_STAMP(4);
        // slot position and group of every local entry
        for (int e = tid; e < c.ne; e += kThreads) {
          const float y = ekey_y(el[e]);
          const int32_t p = first_slot_le(y, 0, M.ns);
          g_epos[e] = static_cast<int16_t>(p);
          const int q = group_of(p);
          atomicAdd(&g_ecnt[q], 1u);
          atomicAdd(&g_emass[q], fmass(y, c.m));
        }
        __syncthreads();
        // coarse counts and masses of this CTA (slots and entries), pushed to
        // every CTA (exchange 2); the tail group also carries the count of
        // uncounted tokens below the slots
        uint32_t* pc = xm;  // [C][kGroups + 1] counts, then masses
        unsigned long long* pm = reinterpret_cast<unsigned long long*>(xm + ((kMaxCluster * (kGroups + 1) + 1) & ~1));
        {
          const int grp = tid >> 3, sub = tid & 7;  // 8 threads per group
          uint32_t cnt = 0;
          unsigned long long mass = 0;
          for (int s = g_gb[grp] + sub; s < g_gb[grp + 1]; s += 8) {
            const uint32_t h = (hist[s >> 1] >> ((s & 1) << 4)) & 0xffffu;
            if (h) {
              cnt += h;
              mass += static_cast<unsigned long long>(h) * fmass(slot_y(s), c.m);
            }
          }
#pragma unroll
          for (int o = 1; o < 8; o <<= 1) {
            cnt += __shfl_xor_sync(0xffffffffu, cnt, o);
            mass += __shfl_xor_sync(0xffffffffu, mass, o);
          }
          cnt += g_ecnt[grp];
          mass += g_emass[grp];
          const uint32_t bsum = block_sum<uint32_t>(below);
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
          }
        }
        SS_STAMP(15);
        cl.sync();
        SS_STAMP(16);
        if (tid <= kGroups) {
          uint32_t cnt = 0;
          unsigned long long mass = 0, bel = 0;
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
          if (tid == kGroups) c.below = bel;  // uncounted tokens below the slots (saturating per CTA)
          g_gcnt[tid] = cnt;
          g_gmass[tid] = mass;
        }
        __syncthreads();
        SS_STAMP(5);

        // ---------------------------------------------- the cuts
        // K = the shortest of the top-k, top-p and min-p prefixes of the
        // (y desc, token asc) order.  A cut is (value v, items of v taken).
        bool unknown = false;
        float bv = ninf();                     // best (shortest) cut so far
        unsigned long long btake = 0, bcc = 0, bcm = 0;
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
            Sk = bcm + btake * fmass(bv, c.m);
          }
          SS_TRACE(19, c.tau_key);
          SS_TRACE(20, __float_as_uint(bv));
          SS_TRACE(21, btake | (bcc << 32));
          SS_TRACE(22, c.pick);
        }
        if (!have_cut && !unknown) {
          // every item (top-k off or larger than the item count): all must
          // have been counted
          if ((c.below || (c.k_on && c.tau_key)) &&
              (c.k_on || M.ns == 0 || __fmul_rn(slot_z(M, M.ns - 1), inv_t) > skip))
            unknown = true;
          Sk = 0;
          for (int q = 0; q <= kGroups; ++q) Sk += g_gmass[q];
          if (tid == 0) {
            unsigned long long cnt = 0;
            for (int q = 0; q <= kGroups; ++q) cnt += g_gcnt[q];
            c.kcount = cnt;
          }
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
          }
        }
        if (c.mp_on && !unknown) {
          // the largest value failing the min-p test: among the slots (they
          // fall monotonically) and every CTA's entries
          if (tid == 0) c.fail_key = 0;
          __syncthreads();
          const int total_e = g_goff[C];
          for (int i = tid; i < total_e; i += kThreads) {
            int r = 0;
            while (i >= g_goff[r + 1]) ++r;
            const float y = ekey_y(*cl.map_shared_rank(el + (i - g_goff[r]), r));
            if (!(__fsub_rn(y, c.m) >= c.lmp)) atomicMax(&c.fail_key, okey(y));
          }
          __syncthreads();
          if (tid == 0) {
            int lo_s = 0, hi_s = M.ns;
            while (lo_s < hi_s) {
              const int mid = (lo_s + hi_s) >> 1;
              if (!(__fsub_rn(slot_y(mid), c.m) >= c.lmp))
                hi_s = mid;
              else
                lo_s = mid + 1;
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
          SS_TRACE(23, __float_as_uint(vf) | (static_cast<unsigned long long>(__float_as_uint(c.m)) << 32));
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
          resolve_ties(a, bv, btake, tests_draft);
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
        // |K| (and its mass) for rows without a histogram
        if (!c.need_hist && (a.out_kept || tests_draft)) {
          int32_t cnt = 0;
          unsigned long long mass = 0;
          count_pass(a, tests_draft, ents, n_ents, cnt, mass);
          const PartD r = exchange_d(ninf(), 0x7fffffff, cnt, mass);
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
          if (accept) {
            token = c.x;
          } else {
            float bs = ninf();
            int32_t bt = 0x7fffffff;
            draw_pass<true>(a, cv, ct, mp_on, inv_s, logf(SK), qrow, ents, n_ents, bs, bt);
            const PartD r = exchange_d(bs, bt, 0, 0);
            if (r.arg != 0x7fffffff && r.best > ninf())
              token = r.arg;
            else
              need_draw = true;  // an empty residual (rounding): the stream-0 draw
          }
        }
        if (need_draw) {
          float bs = ninf();
          int32_t bt = 0x7fffffff;
          draw_pass<false>(a, cv, ct, mp_on, 0.0f, 0.0f, nullptr, ents, n_ents, bs, bt);
          const PartD r = exchange_d(bs, bt, 0, 0);
          token = r.arg;
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
  const int64_t push_bytes = ((kMaxCluster * (kGroups + 1) + 1) & ~1) * 4 + kMaxCluster * (kGroups + 1) * 8;
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
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = cs;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
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
#endif

namespace ss {

ss_status hist_sample(const ss_sample_args& A, cudaStream_t stream) {
  hist::HArgs a{};
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
  a.ncta = hist::cluster_for(A.vocab);
  const int64_t slice = ((static_cast<int64_t>(A.vocab) + a.ncta - 1) / a.ncta + 63) / 64 * 64;
  a.slice = static_cast<int32_t>(slice);
  a.bulk = ((reinterpret_cast<uintptr_t>(A.logits) & 15u) == 0 && ((A.row_stride * 2) & 15) == 0) ? 1 : 0;
  return hist::launch(a, stream);
}

ss_status hist_verify(const ss_verify_args& A, int4* results, int32_t* counters, cudaStream_t stream) {
  hist::HArgs a{};
  a.mode = 1;
  a.num_tasks = A.num_requests * (A.max_draft + 1);
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
  a.ws_results = results;
  a.ws_counters = counters;
  a.ncta = hist::cluster_for(A.vocab);
  const int64_t slice = ((static_cast<int64_t>(A.vocab) + a.ncta - 1) / a.ncta + 63) / 64 * 64;
  a.slice = static_cast<int32_t>(slice);
  a.bulk = ((reinterpret_cast<uintptr_t>(A.target_logits) & 15u) == 0 && ((A.row_stride * 2) & 15) == 0) ? 1 : 0;
  return hist::launch(a, stream);
}

}  // namespace ss
