// ss_kernel.cu -- sm_103a kernels and C ABI of libss (see include/ss.h).
//
// Execution model (one launch per call, fixed shape):
//   * one thread-block cluster of C CTAs per task; a task is one logits row
//     (ss_process_sample) or one target position (request i, draft j) of
//     ss_spec_verify.  The row's vocabulary is cut into C slices of
//     `slice_len` tokens; each CTA stages its slice in shared memory with 1-D
//     bulk (TMA) copies, once, and every later pass runs on shared memory.
//   * penalised / biased tokens live in a per-CTA hash table ("patches") and
//     are excluded from the raw slice; their processed values are computed
//     from the global row and visited alongside the slice.
//   * statistics are reduced warp -> CTA -> cluster (distributed shared
//     memory reads after a cluster barrier); every CTA derives the same
//     decisions from the same reduced values, so control flow stays uniform.
//   * top-k / top-p cuts are exact radix selections over order-preserving
//     32-bit keys of y (descending), with probability masses accumulated in
//     40-bit fixed point so that sums do not depend on thread order; ties at a
//     cut are resolved by a second selection over token indices.
//   * the draw is Gumbel-max over the kept set, per thread, then across the
//     cluster (FlashSampling page: per-tile max, then a cross-tile reduction;
//     the argmax decomposes over partitions).  Tokens whose logit plus the
//     largest possible noise cannot beat the running best skip the RNG.
#include <cooperative_groups.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>
#include <string.h>

#include <mutex>

#include "ss.h"
#include "ss_philox.cuh"
#include "ss_ptx.cuh"

namespace cg = cooperative_groups;

namespace ss {

constexpr int kThreads = 512;
constexpr int kWarps = kThreads / 32;
constexpr int kHashCap = SS_MAX_PATCHED;
constexpr int kHashShift = 32 - 10;  // log2(kHashCap) = 10
static_assert(kHashCap == 1024, "hash shift assumes 1024 slots");
constexpr uint32_t kChunkBytes = 8192;
constexpr int kMaxChunks = 20;
constexpr uint32_t kTargetSliceBytes = 80u * 1024u;
constexpr uint32_t kMaxSliceBytes = kMaxChunks * kChunkBytes;
constexpr int kMaxCluster = 8;
constexpr uint32_t kWaitPolls = 1u << 22;
constexpr float kFixedScale = 1099511627776.0f;  // 2^40
constexpr double kFixedInv = 1.0 / 1099511627776.0;
constexpr int kBiasFlag = 1 << 30;
constexpr int kNoCut = 0x7fffffff;

enum TaskMode { kModeSample = 0, kModeVerify = 1 };

__device__ __forceinline__ float neg_inf() { return __int_as_float(0xff800000); }
__device__ __forceinline__ float pos_inf() { return __int_as_float(0x7f800000); }

// Order-preserving key: larger y -> larger key.
__device__ __forceinline__ uint32_t order_key(float y) {
  const uint32_t b = __float_as_uint(y);
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

// ----------------------------------------------------------------- layout --

struct Layout {
  int32_t slice_len;   // tokens per CTA, multiple of 32
  int32_t data_bytes;  // raw slice bytes (multiple of 16)
  int32_t xm_off;      // exclusion bitmap, slice_len / 32 words
  int32_t hk_off;      // patch table: token ids
  int32_t hc_off;      // patch table: counts | kBiasFlag
  int32_t hv_off;      // patch table: bias value, then processed value
  int32_t hist_off;    // 2 x 256 counts (u32) + 2 x 256 masses (u64)
  int32_t merge_off;   // 256 counts + 256 masses, merged over the cluster
  int32_t red_off;     // per-warp reduction scratch
  int32_t part_off;    // per-CTA partial results read by the other CTAs
  int32_t ctl_off;     // task control block
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
  float xw;       // exp(y_x - m) of the draft token if this CTA holds it, else -1
  int32_t x_in;   // draft token in K (1) / not (0) / not here (-1)
  float score;
  int32_t pad;
};
constexpr int kPartSlots = 6;

// Result of one histogram pass (written by warp 0, read by all threads).
struct SelPass {
  uint32_t digit, cnt_before, cnt_bin, reached;
  unsigned long long mass_before, mass_bin, total;
  double target;
};

struct SelOut {
  uint32_t key, cnt_gt, cnt_eq, reached;
  unsigned long long mass_gt, mass_eq, total;
};

struct Ctl {
  int32_t row, req, j, k, d0, drow, x;
  int32_t bad_k;  // request's draft count outside [0, max_draft]
  int32_t greedy, top_k, use_mask;
  float temperature, inv_t, top_p, min_p, rep, freq, pres;
  uint32_t seed_lo, seed_hi, pos;
  int32_t h0, h1, b0, b1;
  int32_t lo, n;  // slice start token, tokens in this slice
  int32_t status;
  // after stage 1
  float m;
  int32_t arg, count;
  // selection result broadcast
  SelPass sel;
  double sel_target;
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
  Layout L;
};

struct Smem {
  uint8_t* data;
  uint32_t* xm;
  int32_t* hkey;
  int32_t* hcnt;
  float* hval;
  uint32_t* hcnt_buf[2];
  unsigned long long* hmass_buf[2];
  uint32_t* mcnt;
  unsigned long long* mmass;
  uint8_t* red;
  Part* part;
  Ctl* ctl;
  uint64_t* mbar;
};

__device__ __forceinline__ Smem carve(uint8_t* base, const Layout& L) {
  Smem s;
  s.data = base;
  s.xm = reinterpret_cast<uint32_t*>(base + L.xm_off);
  s.hkey = reinterpret_cast<int32_t*>(base + L.hk_off);
  s.hcnt = reinterpret_cast<int32_t*>(base + L.hc_off);
  s.hval = reinterpret_cast<float*>(base + L.hv_off);
  s.hcnt_buf[0] = reinterpret_cast<uint32_t*>(base + L.hist_off);
  s.hcnt_buf[1] = s.hcnt_buf[0] + 256;
  s.hmass_buf[0] = reinterpret_cast<unsigned long long*>(base + L.hist_off + 2048);
  s.hmass_buf[1] = s.hmass_buf[0] + 256;
  s.mcnt = reinterpret_cast<uint32_t*>(base + L.merge_off);
  s.mmass = reinterpret_cast<unsigned long long*>(base + L.merge_off + 1024);
  s.red = base + L.red_off;
  s.part = reinterpret_cast<Part*>(base + L.part_off);
  s.ctl = reinterpret_cast<Ctl*>(base + L.ctl_off);
  s.mbar = reinterpret_cast<uint64_t*>(base + L.mbar_off);
  return s;
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
};

// --------------------------------------------------------- reductions --

struct ArgMax {
  float v;
  int32_t i;
};

__device__ __forceinline__ void argmax_merge(ArgMax& a, float v, int32_t i) {
  if (v > a.v || (v == a.v && i < a.i)) {
    a.v = v;
    a.i = i;
  }
}

__device__ __forceinline__ ArgMax warp_argmax(ArgMax a) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    const float v = __shfl_xor_sync(0xffffffffu, a.v, off);
    const int32_t i = __shfl_xor_sync(0xffffffffu, a.i, off);
    argmax_merge(a, v, i);
  }
  return a;
}

template <typename T>
__device__ __forceinline__ T warp_sum(T v) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
  return v;
}

__device__ __forceinline__ int32_t warp_max_i(int32_t v) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) v = max(v, __shfl_xor_sync(0xffffffffu, v, off));
  return v;
}

// Block reduction of (argmax, count, status max, mass sum); result valid in
// every thread.  Uses the `red` scratch (kWarps * 32 bytes).
struct BlockAcc {
  ArgMax am;
  int32_t count;
  int32_t status;
  unsigned long long mass;
};

__device__ BlockAcc block_reduce(const Smem& sm, BlockAcc a) {
  a.am = warp_argmax(a.am);
  a.count = warp_sum(a.count);
  a.status = warp_max_i(a.status);
  a.mass = warp_sum(a.mass);
  struct alignas(8) W {
    float v;
    int32_t i, c, s;
    unsigned long long m;
  };
  W* w = reinterpret_cast<W*>(sm.red);
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  __syncthreads();
  if (lane == 0) w[wid] = W{a.am.v, a.am.i, a.count, a.status, a.mass};
  __syncthreads();
  BlockAcc r;
  r.am = ArgMax{neg_inf(), kNoCut};
  r.count = 0;
  r.status = 0;
  r.mass = 0;
  for (int k = 0; k < kWarps; ++k) {  // fixed order: deterministic
    argmax_merge(r.am, w[k].v, w[k].i);
    r.count += w[k].c;
    r.status = max(r.status, w[k].s);
    r.mass += w[k].m;
  }
  return r;
}

// Exchange one Part per CTA through the cluster and fold them in rank order.
__device__ Part cluster_fold(const Smem& sm, int slot, const Part& mine) {
  cg::cluster_group cl = cg::this_cluster();
  if (threadIdx.x == 0) sm.part[slot] = mine;
  cl.sync();
  Part r = mine;
  r.best = neg_inf();
  r.arg = kNoCut;
  r.count = 0;
  r.status = 0;
  r.mass = 0;
  r.xw = -1.0f;
  r.x_in = -1;
  r.score = neg_inf();
  const int n = static_cast<int>(cl.num_blocks());
  for (int c = 0; c < n; ++c) {
    const Part* q = cl.map_shared_rank(sm.part + slot, c);
    const Part p = *q;
    if (p.best > r.best || (p.best == r.best && p.arg < r.arg)) {
      r.best = p.best;
      r.arg = p.arg;
      r.score = p.score;
    }
    r.count += p.count;
    r.status = max(r.status, p.status);
    r.mass += p.mass;
    if (p.x_in >= 0) {
      r.x_in = p.x_in;
      r.xw = p.xw;
    }
  }
  return r;
}

// -------------------------------------------------------------- visitor --

// Calls f(t, y) for every allowed token of this CTA's slice (raw slice plus
// patch table); y is the processed logit (z for greedy rows).
template <int DT, typename F>
__device__ __forceinline__ void visit(const Smem& sm, const Ctl& c, F&& f) {
  using V = Vec<DT>;
  const int nvec = (c.n + V::kPer - 1) / V::kPer;
  const uint4* data = reinterpret_cast<const uint4*>(sm.data);
  const bool greedy = c.greedy != 0;
  const float inv_t = c.inv_t;
  for (int v = threadIdx.x; v < nvec; v += kThreads) {
    float z[V::kPer];
    V::unpack(data[v], z);
#pragma unroll
    for (int e = 0; e < V::kPer; ++e) {
      const float y = greedy ? z[e] : __fmul_rn(z[e], inv_t);
      if (y != neg_inf()) f(c.lo + v * V::kPer + e, y);
    }
  }
  for (int s = threadIdx.x; s < kHashCap; s += kThreads) {
    const int32_t t = sm.hkey[s];
    if (t >= 0) {
      const float y = sm.hval[s];
      if (y != neg_inf()) f(t, y);
    }
  }
}

__device__ __forceinline__ unsigned long long fixed_mass(float y, float m) {
  return __float2ull_rz(__expf(y - m) * kFixedScale);
}

// One exact radix selection (4 passes of 8-bit digits over a 32-bit key).
// Elements are those `accept(t, y)` admits; key(t, y) orders them, larger
// first.  by_mass: the selected element is where the running fixed-point mass
// first reaches `target` (or target_frac * total mass when target_frac > 0);
// otherwise where the running count reaches `target`.
template <int DT, bool kMass, typename KeyF, typename AccF>
__device__ SelOut radix_select(const Smem& sm, const Ctl& c, int& pass, bool by_mass, double target,
                               double target_frac, KeyF keyf, AccF accept) {
  cg::cluster_group cl = cg::this_cluster();
  const int ncta = static_cast<int>(cl.num_blocks());
  uint32_t prefix = 0, pmask = 0, base_c = 0;
  unsigned long long base_m = 0, total = 0;
  SelOut out{};
  out.reached = 1;
  const float m = c.m;
  for (int level = 0; level < 4; ++level) {
    const int shift = 24 - 8 * level;
    const int buf = pass & 1;
    ++pass;
    uint32_t* hc = sm.hcnt_buf[buf];
    unsigned long long* hm = sm.hmass_buf[buf];
    for (int b = threadIdx.x; b < 256; b += kThreads) {
      hc[b] = 0;
      if (kMass) hm[b] = 0;
    }
    __syncthreads();
    visit<DT>(sm, c, [&](int32_t t, float y) {
      const uint32_t key = keyf(t, y);
      if ((key & pmask) != prefix) return;
      if (!accept(t, y)) return;
      const uint32_t d = (key >> shift) & 255u;
      atomicAdd(hc + d, 1u);
      if (kMass) atomicAdd(hm + d, fixed_mass(y, m));
    });
    __syncthreads();
    cl.sync();
    for (int b = threadIdx.x; b < 256; b += kThreads) {
      uint32_t cc = 0;
      unsigned long long mm = 0;
      for (int r = 0; r < ncta; ++r) {
        cc += *cl.map_shared_rank(hc + b, r);
        if (kMass) mm += *cl.map_shared_rank(hm + b, r);
      }
      sm.mcnt[b] = cc;
      sm.mmass[b] = mm;
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
        c8[i] = sm.mcnt[b];
        m8[i] = kMass ? sm.mmass[b] : 0ull;
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
      double tgt = target;
      if (level > 0)
        tgt = sm.ctl->sel_target;
      else if (target_frac > 0.0)
        tgt = target_frac * static_cast<double>(tot_m);
      const bool cross = by_mass ? (static_cast<double>(base_m + im) >= tgt)
                                 : (static_cast<double>(base_c + ic) >= tgt);
      const unsigned ball = __ballot_sync(0xffffffffu, cross);
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
        int pick = 7;
        if (reached) {
          for (int i = 0; i < 8; ++i) {
            const bool hit = by_mass ? (static_cast<double>(base_m + mmv + m8[i]) >= tgt)
                                     : (static_cast<double>(base_c + cc + c8[i]) >= tgt);
            if (hit) {
              pick = i;
              break;
            }
            cc += c8[i];
            mmv += m8[i];
          }
        } else {
          int last = 7;
          for (int i = 7; i >= 0; --i)
            if (c8[i] > 0) {
              last = i;
              break;
            }
          for (int i = 0; i < last; ++i) {
            cc += c8[i];
            mmv += m8[i];
          }
          pick = last;
        }
        SelPass sp;
        sp.digit = static_cast<uint32_t>(255 - 8 * L - pick);
        sp.cnt_before = cc;
        sp.cnt_bin = c8[pick];
        sp.mass_before = mmv;
        sp.mass_bin = m8[pick];
        sp.reached = reached;
        sp.total = tot_m;
        sp.target = tgt;
        sm.ctl->sel = sp;
        sm.ctl->sel_target = tgt;
      }
    }
    __syncthreads();
    const SelPass sp = sm.ctl->sel;
    if (level == 0) total = sp.total;  // mass of every admitted element
    prefix |= sp.digit << shift;
    pmask |= 255u << shift;
    base_c += sp.cnt_before;
    base_m += sp.mass_before;
    out.cnt_eq = sp.cnt_bin;
    out.mass_eq = sp.mass_bin;
    if (!sp.reached) out.reached = 0;
    __syncthreads();
  }
  out.key = prefix;
  out.cnt_gt = base_c;
  out.mass_gt = base_m;
  out.total = total;
  return out;
}

// ------------------------------------------------------------- kernel --

template <int DT>
__global__ void __launch_bounds__(kThreads, 2) ss_row_kernel(const KArgs a) {
  using V = Vec<DT>;
  extern __shared__ __align__(128) uint8_t smem_raw[];
  cg::cluster_group cl = cg::this_cluster();
  const int rank = static_cast<int>(cl.block_rank());
  const int ncta = static_cast<int>(cl.num_blocks());
  const int task = static_cast<int>(blockIdx.x) / ncta;
  const Layout& L = a.L;
  Smem sm = carve(smem_raw, L);
  Ctl& c = *sm.ctl;
  const int tid = threadIdx.x;
  const int V_ = a.vocab;

  // ---------------------------------------------------------------- setup
  if (tid == 0) {
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
    }
    c.row = live ? row : -1;
    c.bad_k = bad_k;
    c.req = req;
    c.j = j;
    c.k = k;
    c.d0 = d0;
    c.drow = drow;
    c.x = x;
    const ss_params& p = a.p;
    const float T = p.temperature[req];
    c.temperature = T;
    c.greedy = (T == 0.0f);
    c.inv_t = __fdiv_rn(1.0f, T);
    c.top_k = p.top_k ? p.top_k[req] : 0;
    c.top_p = p.top_p ? p.top_p[req] : 1.0f;
    c.min_p = p.min_p ? p.min_p[req] : 0.0f;
    c.rep = p.repetition ? p.repetition[req] : 1.0f;
    c.freq = p.frequency ? p.frequency[req] : 0.0f;
    c.pres = p.presence ? p.presence[req] : 0.0f;
    c.h0 = p.hist_offsets ? p.hist_offsets[req] : 0;
    c.h1 = p.hist_offsets ? p.hist_offsets[req + 1] : 0;
    c.b0 = p.bias_offsets ? p.bias_offsets[req] : 0;
    c.b1 = p.bias_offsets ? p.bias_offsets[req + 1] : 0;
    c.use_mask = (p.bitmask != nullptr) && (p.use_bitmask == nullptr || p.use_bitmask[req] != 0);
    const uint64_t seed = p.seed[req];
    c.seed_lo = static_cast<uint32_t>(seed);
    c.seed_hi = static_cast<uint32_t>(seed >> 32);
    const int64_t pos = p.position[req];
    c.pos = static_cast<uint32_t>(pos) + static_cast<uint32_t>(j);
    // parameter validation (identical in every CTA of the cluster)
    if (!(T >= 0.0f) || isinf(T) || c.top_k < 0 || !(c.top_p > 0.0f) || !(c.min_p >= 0.0f && c.min_p <= 1.0f) ||
        !(c.rep > 0.0f) || isinf(c.rep) || !isfinite(c.freq) || !isfinite(c.pres) || c.h1 < c.h0 ||
        c.b1 < c.b0 || pos < 0 || pos + k > 0xffffffffll)
      status = SS_ROW_BAD_PARAM;
    c.status = status;
    c.lo = rank * L.slice_len;
    c.n = (status == SS_ROW_BAD_PARAM) ? 0 : max(0, min(V_ - c.lo, L.slice_len));
  }
  __syncthreads();
  if (c.row < 0) return;  // whole cluster: no such target position

  // A row with invalid parameters (including a bad draft count, which makes
  // its row index meaningless) touches no logits: it only reports its status.
  const bool touch = (c.status != SS_ROW_BAD_PARAM);
  const int lo = c.lo, n = touch ? c.n : 0;
  const char* row_ptr = reinterpret_cast<const char*>(a.logits) + static_cast<int64_t>(c.row) * a.row_stride * V::kBytes;
  const uint32_t slice_bytes = static_cast<uint32_t>(n) * V::kBytes;
  // Bulk (TMA) copies need a 16-byte aligned source; a row whose byte stride
  // is not a multiple of 16 (an odd vocabulary size) is staged with plain,
  // coalesced element loads instead.
  const bool bulk_ok = ((reinterpret_cast<uintptr_t>(row_ptr) + static_cast<uintptr_t>(lo) * V::kBytes) & 15u) == 0;
  const uint32_t bulk_bytes = bulk_ok ? (slice_bytes & ~15u) : 0u;
  const int nchunks = static_cast<int>((bulk_bytes + kChunkBytes - 1) / kChunkBytes);

  // Issue the slice's bulk copies first so that HBM traffic starts at once.
  if (tid == 0) {
    for (int ch = 0; ch < nchunks; ++ch) mbar_init(sm.mbar + ch, 1);
    fence_barrier_init();
    const char* src = row_ptr + static_cast<int64_t>(lo) * V::kBytes;
    for (int ch = 0; ch < nchunks; ++ch) {
      const uint32_t off = static_cast<uint32_t>(ch) * kChunkBytes;
      const uint32_t bytes = min(kChunkBytes, bulk_bytes - off);
      mbar_arrive_expect_tx(sm.mbar + ch, bytes);
      bulk_load(sm.data + off, src + off, bytes, sm.mbar + ch);
    }
  }
  // The rest (a ragged tail < 16 bytes, or the whole slice when unaligned)
  // with plain loads.
  for (int e = static_cast<int>(bulk_bytes / V::kBytes) + tid; e < n; e += kThreads) {
    if (V::kBytes == 4)
      reinterpret_cast<uint32_t*>(sm.data)[e] = reinterpret_cast<const uint32_t*>(row_ptr)[lo + e];
    else
      reinterpret_cast<uint16_t*>(sm.data)[e] = reinterpret_cast<const uint16_t*>(row_ptr)[lo + e];
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
    sm.xm[w] = ex;
  }
  for (int s = tid; s < kHashCap; s += kThreads) {
    sm.hkey[s] = -1;
    sm.hcnt[s] = 0;
    sm.hval[s] = 0.0f;
  }
  __syncthreads();

  // Patch table: history (+ drafts before this position) and bias entries.
  int32_t st_local = SS_ROW_OK;
  auto insert = [&](int32_t t) -> int {
    uint32_t h = (static_cast<uint32_t>(t) * 2654435761u) >> kHashShift;
    for (int probe = 0; probe < kHashCap; ++probe) {
      const int32_t prev = atomicCAS(sm.hkey + h, -1, t);
      if (prev == -1 || prev == t) return static_cast<int>(h);
      h = (h + 1) & (kHashCap - 1);
    }
    return -1;
  };
  if (c.status == SS_ROW_OK) {
    for (int e = c.h0 + tid; e < c.h1; e += kThreads) {
      const int32_t t = a.p.hist_ids[e];
      if (t < 0 || t >= V_) {
        st_local = max(st_local, SS_ROW_BAD_INDEX);
        continue;
      }
      if (t < lo || t >= lo + n) continue;
      const int s = insert(t);
      if (s < 0)
        st_local = max(st_local, SS_ROW_LIMIT);
      else
        atomicAdd(sm.hcnt + s, 1);
    }
    if (a.mode == kModeVerify) {
      for (int e = tid; e < c.k; e += kThreads) {  // every draft must be a token id
        const int32_t t = a.draft_tokens[c.d0 + e];
        if (t < 0 || t >= V_) {
          st_local = max(st_local, SS_ROW_BAD_INDEX);
          continue;
        }
        if (e >= c.j || t < lo || t >= lo + n) continue;  // history = drafts before j
        const int s = insert(t);
        if (s < 0)
          st_local = max(st_local, SS_ROW_LIMIT);
        else
          atomicAdd(sm.hcnt + s, 1);
      }
    }
    for (int e = c.b0 + tid; e < c.b1; e += kThreads) {
      const int32_t t = a.p.bias_ids[e];
      const float b = a.p.bias_vals[e];
      if (!isfinite(b)) st_local = max(st_local, SS_ROW_BAD_PARAM);
      if (t < 0 || t >= V_) {
        st_local = max(st_local, SS_ROW_BAD_INDEX);
        continue;
      }
      if (t < lo || t >= lo + n) continue;
      const int s = insert(t);
      if (s < 0) {
        st_local = max(st_local, SS_ROW_LIMIT);
        continue;
      }
      if (atomicOr(sm.hcnt + s, kBiasFlag) & kBiasFlag) st_local = max(st_local, SS_ROW_BAD_INDEX);  // duplicate
      sm.hval[s] = b;
    }
  }
  __syncthreads();
  // Processed values of patched tokens (read straight from the global row).
  for (int s = tid; s < kHashCap; s += kThreads) {
    const int32_t t = sm.hkey[s];
    if (t < 0) continue;
    atomicOr(sm.xm + ((t - lo) >> 5), 1u << ((t - lo) & 31));
    float z = V::load_global(row_ptr, t);
    const int32_t hc = sm.hcnt[s];
    const int32_t cnt = hc & ~kBiasFlag;
    if (cnt > 0) {
      z = (z > 0.0f) ? __fdiv_rn(z, c.rep) : __fmul_rn(z, c.rep);
      z = __fsub_rn(z, __fmul_rn(c.freq, static_cast<float>(cnt)));
      z = __fsub_rn(z, c.pres);
    }
    if (hc & kBiasFlag) z = __fadd_rn(z, sm.hval[s]);
    if (c.use_mask) {
      const uint32_t word = static_cast<uint32_t>(a.p.bitmask[static_cast<int64_t>(c.req) * a.p.bitmask_stride + (t >> 5)]);
      if (((word >> (t & 31)) & 1u) == 0u) z = neg_inf();
    }
    sm.hval[s] = c.greedy ? z : __fmul_rn(z, c.inv_t);
  }

  // --------------------------------------------------------------- stage 1
  // Wait for each chunk, write -inf over excluded lanes, and accumulate the
  // row max (lowest index on ties), the allowed count and non-finite flags.
  BlockAcc acc;
  acc.am = ArgMax{neg_inf(), kNoCut};
  acc.count = 0;
  acc.status = st_local;
  acc.mass = 0;
  bool timed_out = false;
  __syncthreads();  // exclusion bits of patched tokens are in place
  {
    const int nvec = (n + V::kPer - 1) / V::kPer;
    const int vec_per_chunk = static_cast<int>(kChunkBytes / 16);
    uint4* data = reinterpret_cast<uint4*>(sm.data);
    float* dbg = (a.debug_processed && !c.bad_k) ? a.debug_processed + static_cast<int64_t>(c.row) * V_ : nullptr;
    int waited = -1;
    for (int v = tid; v < nvec; v += kThreads) {
      const int ch = min(v / vec_per_chunk, nchunks - 1);
      if (nchunks > 0 && ch > waited) {
        for (int w = waited + 1; w <= ch; ++w)
          if (!mbar_wait_bounded(sm.mbar + w, 0, kWaitPolls)) timed_out = true;
        waited = ch;
      }
      const int e0 = v * V::kPer;
      const uint32_t bits = (sm.xm[e0 >> 5] >> (e0 & 31)) & ((1u << V::kPer) - 1u);
      uint4 raw = data[v];
      if (bits) {
        raw = V::exclude(raw, bits);
        data[v] = raw;
      }
      float z[V::kPer];
      V::unpack(raw, z);
#pragma unroll
      for (int e = 0; e < V::kPer; ++e) {
        const float y = c.greedy ? z[e] : __fmul_rn(z[e], c.inv_t);
        const int32_t t = lo + e0 + e;
        if (dbg && e0 + e < n) dbg[t] = y;
        if (y == neg_inf()) continue;
        acc.count += 1;
        if (!(y < pos_inf())) acc.status = max(acc.status, SS_ROW_NONFINITE);
        argmax_merge(acc.am, y, t);
      }
    }
    // chunks no thread of this CTA touched still need their completion
    if (tid == 0)
      for (int w = waited + 1; w < nchunks; ++w)
        if (!mbar_wait_bounded(sm.mbar + w, 0, kWaitPolls)) timed_out = true;
    if (timed_out) acc.status = max(acc.status, SS_ROW_TIMEOUT);
    __syncthreads();  // debug writes of the raw slice precede the patched ones
    for (int s = tid; s < kHashCap; s += kThreads) {
      const int32_t t = sm.hkey[s];
      if (t < 0) continue;
      const float y = sm.hval[s];
      if (dbg) dbg[t] = y;
      if (y == neg_inf()) continue;
      acc.count += 1;
      if (!(y < pos_inf())) acc.status = max(acc.status, SS_ROW_NONFINITE);
      argmax_merge(acc.am, y, t);
    }
  }
  BlockAcc blk = block_reduce(sm, acc);
  Part mine{};
  mine.best = blk.am.v;
  mine.arg = blk.am.i;
  mine.count = blk.count;
  mine.status = max(blk.status, c.status);
  mine.x_in = -1;
  mine.xw = -1.0f;
  mine.score = neg_inf();
  Part all = cluster_fold(sm, 0, mine);
  int32_t status = all.status;
  if (status == SS_ROW_OK && all.count == 0) status = SS_ROW_EMPTY_SET;
  const float m = all.best;
  const int32_t argmax_tok = all.arg;
  if (tid == 0) {
    c.m = m;
    c.arg = argmax_tok;
    c.count = all.count;
  }
  __syncthreads();

  int32_t token = -1, kept = 0, accept = 0;
  if (status == SS_ROW_OK) {
    const bool spec_pos = (a.mode == kModeVerify) && (c.j < c.k);
    const uint32_t seed_lo = c.seed_lo, seed_hi = c.seed_hi;
    const uint64_t seed = (static_cast<uint64_t>(seed_hi) << 32) | seed_lo;
    const uint32_t rowid = static_cast<uint32_t>(c.req);
    if (c.greedy) {
      kept = 1;
      token = argmax_tok;
      if (spec_pos) {
        const float q = a.draft_probs[static_cast<int64_t>(c.drow) * a.draft_stride + c.x];
        const float u = uniform_from_numerator(uniform_numerator(philox_word(seed, rowid, c.pos, 0, 1)));
        const float P = (c.x == argmax_tok) ? 1.0f : 0.0f;
        accept = (__fmul_rn(u, q) < P) ? 1 : 0;
        token = accept ? c.x : argmax_tok;
      }
    } else {
      // ------------------------------------------------------ the cuts
      int pass = 0;
      const bool k_on = c.top_k > 0 && c.top_k < c.count;
      const bool p_on = c.top_p < 1.0f;
      const bool mp_on = c.min_p > 0.0f;
      bool has_cut = false;
      uint32_t cut_key = 0;
      int32_t cut_idx = kNoCut;
      uint32_t k_key = 0;
      int32_t k_idx = kNoCut;
      auto ykey = [](int32_t, float y) { return order_key(y); };
      auto all_ok = [](int32_t, float) { return true; };
      if (k_on) {
        SelOut s = radix_select<DT, true>(sm, c, pass, false, static_cast<double>(c.top_k), 0.0, ykey, all_ok);
        const uint32_t ntie = static_cast<uint32_t>(c.top_k) - s.cnt_gt;
        int32_t idx = kNoCut;
        if (ntie < s.cnt_eq) {
          const uint32_t kk = s.key;
          SelOut ti = radix_select<DT, false>(
              sm, c, pass, false, static_cast<double>(ntie), 0.0,
              [](int32_t t, float) { return ~static_cast<uint32_t>(t); },
              [kk](int32_t, float y) { return order_key(y) == kk; });
          idx = static_cast<int32_t>(~ti.key);
        }
        k_key = s.key;
        k_idx = idx;
        has_cut = true;
        cut_key = k_key;
        cut_idx = k_idx;
      }
      if (p_on) {
        const uint32_t kk = k_key;
        const int32_t ki = k_idx;
        auto in_topk = [k_on, kk, ki](int32_t t, float y) {
          if (!k_on) return true;
          const uint32_t key = order_key(y);
          return key > kk || (key == kk && t <= ki);
        };
        SelOut s = radix_select<DT, true>(sm, c, pass, true, 0.0, static_cast<double>(c.top_p), ykey, in_topk);
        const double target = static_cast<double>(c.top_p) * static_cast<double>(s.total);
        uint32_t ntie = s.cnt_eq;
        if (s.reached && s.cnt_eq > 0) {
          const unsigned long long w = s.mass_eq / s.cnt_eq;
          if (w > 0) {
            const double need = target - static_cast<double>(s.mass_gt);
            double nt = ceil(need / static_cast<double>(w));
            if (nt < 1.0) nt = 1.0;
            if (nt < static_cast<double>(s.cnt_eq)) ntie = static_cast<uint32_t>(nt);
          }
        }
        int32_t idx = kNoCut;
        if (ntie < s.cnt_eq) {
          const uint32_t pk = s.key;
          SelOut ti = radix_select<DT, false>(
              sm, c, pass, false, static_cast<double>(ntie), 0.0,
              [](int32_t t, float) { return ~static_cast<uint32_t>(t); },
              [pk, in_topk](int32_t t, float y) { return order_key(y) == pk && in_topk(t, y); });
          idx = static_cast<int32_t>(~ti.key);
        }
        if (!has_cut || s.key > cut_key || (s.key == cut_key && idx < cut_idx)) {
          cut_key = s.key;
          cut_idx = idx;
        }
        has_cut = true;
      }

      // ------------------------------------------------------ the draw
      const float min_p = c.min_p;
      auto in_K = [=](int32_t t, float y) {
        if (has_cut) {
          const uint32_t key = order_key(y);
          if (!(key > cut_key || (key == cut_key && t <= cut_idx))) return false;
        }
        if (mp_on && !(__expf(y - m) >= min_p)) return false;
        return true;
      };
      // the argmax token is always in K: its score seeds the running best
      const float g0 = gumbel_from_numerator(uniform_numerator(philox_word(seed, rowid, c.pos, argmax_tok, 0)));
      ArgMax best{__fadd_rn(m, g0), argmax_tok};
      int32_t kcount = 0;
      unsigned long long kmass = 0;
      int32_t x_in = -1;
      float xw = -1.0f;
      const int32_t x = c.x;
      visit<DT>(sm, c, [&](int32_t t, float y) {
        if (t == x) {
          x_in = in_K(t, y) ? 1 : 0;
          xw = __expf(y - m);
        }
        if (!in_K(t, y)) return;
        ++kcount;
        kmass += fixed_mass(y, m);
        const float slack = 1e-3f + fabsf(y) * 1e-6f;
        if (y + kGumbelMax + slack < best.v) return;
        const uint32_t num = uniform_numerator(philox_word(seed, rowid, c.pos, static_cast<uint32_t>(t), 0));
        if (y + gumbel_upper_bound(num) + slack < best.v) return;
        const float s = __fadd_rn(y, gumbel_from_numerator(num));
        argmax_merge(best, s, t);
      });
      BlockAcc d;
      d.am = best;
      d.count = kcount;
      d.status = 0;
      d.mass = kmass;
      // fold x info through the partial: per-block pick any thread holding x
      __shared__ float s_xw;
      __shared__ int s_xin;
      if (tid == 0) {
        s_xw = -1.0f;
        s_xin = -1;
      }
      __syncthreads();
      if (x_in >= 0) {
        s_xw = xw;
        s_xin = x_in;
      }
      BlockAcc db = block_reduce(sm, d);
      Part pd{};
      pd.best = db.am.v;
      pd.arg = db.am.i;
      pd.count = db.count;
      pd.status = 0;
      pd.mass = db.mass;
      pd.xw = s_xw;
      pd.x_in = s_xin;
      pd.score = db.am.v;
      Part dall = cluster_fold(sm, 1, pd);
      kept = dall.count;
      token = dall.arg;
      if (spec_pos) {
        const float SK = static_cast<float>(static_cast<double>(dall.mass) * kFixedInv);
        const float inv_s = __fdiv_rn(1.0f, SK);
        const float Px = (dall.x_in == 1) ? __fmul_rn(dall.xw, inv_s) : 0.0f;
        const float q = a.draft_probs[static_cast<int64_t>(c.drow) * a.draft_stride + x];
        const float u = uniform_from_numerator(uniform_numerator(philox_word(seed, rowid, c.pos, 0, 1)));
        accept = (__fmul_rn(u, q) < Px) ? 1 : 0;
        if (accept) {
          token = x;
        } else {
          // residual max(P - q, 0): argmax of log r + g over K (stream 2)
          const float* qrow = a.draft_probs + static_cast<int64_t>(c.drow) * a.draft_stride;
          ArgMax rb{neg_inf(), kNoCut};
          visit<DT>(sm, c, [&](int32_t t, float y) {
            if (!in_K(t, y)) return;
            const float P = __fmul_rn(__expf(y - m), inv_s);
            const float r = __fsub_rn(P, qrow[t]);
            if (!(r > 0.0f)) return;
            const uint32_t num = uniform_numerator(philox_word(seed, rowid, c.pos, static_cast<uint32_t>(t), 2));
            const float s = __fadd_rn(logf(r), gumbel_from_numerator(num));
            argmax_merge(rb, s, t);
          });
          BlockAcc rbk;
          rbk.am = rb;
          rbk.count = 0;
          rbk.status = 0;
          rbk.mass = 0;
          BlockAcc rr = block_reduce(sm, rbk);
          Part pr{};
          pr.best = rr.am.v;
          pr.arg = rr.am.i;
          pr.x_in = -1;
          pr.xw = -1.0f;
          Part rall = cluster_fold(sm, 2, pr);
          if (rall.arg != kNoCut && rall.best > neg_inf()) token = rall.arg;
          // else: no token with P > q (rounding): keep the stream-0 draw
        }
      }
    }
  }

  // ------------------------------------------------------------- outputs
  if (rank == 0 && tid == 0) {
    if (status != SS_ROW_OK) {
      token = -1;
      kept = 0;
      accept = 0;
    }
    if (a.out_kept && !c.bad_k) a.out_kept[c.row] = kept;
    if (a.mode == kModeSample) {
      a.out_token[c.row] = token;
      a.out_status[c.row] = status;
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
  // No CTA may leave while another can still read its shared memory.
  cl.sync();
}

// ------------------------------------------------------------------ host --

static thread_local int32_t g_last_cuda_error = 0;

static int choose_cluster(int32_t vocab, int32_t es) {
  for (int cs = 1; cs <= kMaxCluster; cs <<= 1) {
    const int64_t slice = ((static_cast<int64_t>(vocab) + cs - 1) / cs + 31) / 32 * 32;
    if (slice * es <= kTargetSliceBytes) return cs;
  }
  const int64_t slice = ((static_cast<int64_t>(vocab) + kMaxCluster - 1) / kMaxCluster + 31) / 32 * 32;
  if (slice * es <= kMaxSliceBytes) return kMaxCluster;
  return 0;
}

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
  L.xm_off = take(L.slice_len / 32 * 4, 16);
  L.hk_off = take(kHashCap * 4, 16);
  L.hc_off = take(kHashCap * 4, 16);
  L.hv_off = take(kHashCap * 4, 16);
  L.hist_off = take(2 * 256 * 4 + 2 * 256 * 8, 16);
  L.merge_off = take(256 * 4 + 256 * 8, 16);
  L.red_off = take(kWarps * 32, 16);
  L.part_off = take(kPartSlots * sizeof(Part), 16);
  L.ctl_off = take(sizeof(Ctl), 16);
  L.mbar_off = take(kMaxChunks * 8, 16);
  L.total = static_cast<int32_t>((off + 127) / 128 * 128);
  return L;
}

template <int DT>
static cudaError_t launch(const KArgs& ka, int cs, cudaStream_t stream) {
  const void* fn = reinterpret_cast<const void*>(&ss_row_kernel<DT>);
  cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, ka.L.total);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(static_cast<unsigned>(ka.num_tasks) * cs, 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = ka.L.total;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = cs;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, ss_row_kernel<DT>, ka);
}

static bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

static ss_status check_params(const ss_params& p) {
  if (!p.temperature || !p.seed || !p.position) return SS_ERR_INVALID_ARG;
  if ((p.hist_offsets == nullptr) != (p.hist_ids == nullptr)) return SS_ERR_INVALID_ARG;
  if (p.bias_offsets && (!p.bias_ids || !p.bias_vals)) return SS_ERR_INVALID_ARG;
  return SS_OK;
}

static ss_status run(const KArgs& ka, int32_t dtype, cudaStream_t stream) {
  const int es = (dtype == SS_DTYPE_BF16) ? 2 : 4;
  const int cs = choose_cluster(ka.vocab, es);
  if (cs == 0) return SS_ERR_UNSUPPORTED;
  KArgs k = ka;
  k.L = make_layout(ka.vocab, es, cs);
  const cudaError_t e = (dtype == SS_DTYPE_BF16) ? launch<SS_DTYPE_BF16>(k, cs, stream)
                                                 : launch<SS_DTYPE_F32>(k, cs, stream);
  if (e != cudaSuccess) {
    g_last_cuda_error = static_cast<int32_t>(e);
    return SS_ERR_CUDA;
  }
  return SS_OK;
}

}  // namespace ss

extern "C" {

size_t ss_workspace_size(int32_t max_requests, int32_t max_draft) {
  if (max_requests < 0 || max_draft < 0) return 0;
  const size_t results = static_cast<size_t>(max_requests) * static_cast<size_t>(max_draft + 1) * sizeof(int4);
  return results + static_cast<size_t>(max_requests) * sizeof(int32_t) + 256;
}

ss_status ss_workspace_init(void* workspace, size_t workspace_bytes, ss_stream_t stream) {
  if (!workspace) return SS_ERR_WORKSPACE;
  const cudaError_t e = cudaMemsetAsync(workspace, 0, workspace_bytes, reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) {
    ss::g_last_cuda_error = static_cast<int32_t>(e);
    return SS_ERR_CUDA;
  }
  return SS_OK;
}

ss_status ss_process_sample(const ss_sample_args* args, ss_stream_t stream) {
  using namespace ss;
  if (!args) return SS_ERR_INVALID_ARG;
  const ss_sample_args& A = *args;
  if (A.num_rows < 0 || A.vocab < 1) return SS_ERR_INVALID_ARG;
  if (A.dtype != SS_DTYPE_F32 && A.dtype != SS_DTYPE_BF16) return SS_ERR_INVALID_ARG;
  if (A.num_rows == 0) return SS_OK;
  const int es = (A.dtype == SS_DTYPE_BF16) ? 2 : 4;
  if (!A.logits || (reinterpret_cast<uintptr_t>(A.logits) % es) != 0 || !A.out_token || !A.out_status)
    return SS_ERR_INVALID_ARG;
  if (A.row_stride != 0 && A.row_stride < A.vocab) return SS_ERR_INVALID_ARG;
  if (check_params(A.params) != SS_OK) return SS_ERR_INVALID_ARG;
  if (A.params.bitmask && A.params.bitmask_stride < (static_cast<int64_t>(A.vocab) + 31) / 32) return SS_ERR_INVALID_ARG;
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
  return run(k, A.dtype, reinterpret_cast<cudaStream_t>(stream));
}

ss_status ss_spec_verify(const ss_verify_args* args, void* workspace, size_t workspace_bytes, ss_stream_t stream) {
  using namespace ss;
  if (!args) return SS_ERR_INVALID_ARG;
  const ss_verify_args& A = *args;
  if (A.num_requests < 0 || A.vocab < 1 || A.max_draft < 0) return SS_ERR_INVALID_ARG;
  if (A.dtype != SS_DTYPE_F32 && A.dtype != SS_DTYPE_BF16) return SS_ERR_INVALID_ARG;
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
  const int64_t tasks = static_cast<int64_t>(A.num_requests) * (A.max_draft + 1);
  if (tasks > 0x7fffffff / kMaxCluster) return SS_ERR_UNSUPPORTED;
  if (!workspace || !aligned16(workspace) || workspace_bytes < ss_workspace_size(A.num_requests, A.max_draft))
    return SS_ERR_WORKSPACE;
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
  k.ws_results = reinterpret_cast<int4*>(workspace);
  k.ws_counters = reinterpret_cast<int32_t*>(reinterpret_cast<char*>(workspace) +
                                             static_cast<size_t>(tasks) * sizeof(int4));
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
  if (!args) return SS_ERR_INVALID_ARG;
  const size_t need = ss_workspace_size(args->num_requests, args->max_draft);
  if (args->num_requests < 0 || args->max_draft < 0) return SS_ERR_INVALID_ARG;
  if (need > SS_NOALLOC_SCRATCH_BYTES) return SS_ERR_SCRATCH_LIMIT;
  if (args->num_requests == 0) return SS_OK;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess || dev < 0 || dev >= 64) {
    ss::g_last_cuda_error = static_cast<int32_t>(e);
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
        ss::g_last_cuda_error = static_cast<int32_t>(e);
        return SS_ERR_CUDA;
      }
    }
    scratch = g_noalloc_ptr[dev];
  }
  // The per-request arrival counters must start at zero; the array keeps
  // whatever the previous call left, so clear them on every call.
  const size_t results = static_cast<size_t>(args->num_requests) * static_cast<size_t>(args->max_draft + 1) * 16u;
  e = cudaMemsetAsync(static_cast<char*>(scratch) + results, 0, static_cast<size_t>(args->num_requests) * 4u,
                      reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) {
    ss::g_last_cuda_error = static_cast<int32_t>(e);
    return SS_ERR_CUDA;
  }
  return ss_spec_verify(args, scratch, SS_NOALLOC_SCRATCH_BYTES, stream);
}

int32_t ss_cluster_size(int32_t vocab, int32_t dtype) {
  if (vocab < 1 || (dtype != SS_DTYPE_F32 && dtype != SS_DTYPE_BF16)) return 0;
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

const char* ss_version(void) { return "ss 0.1.0 (sm_103a)"; }

}  // extern "C"
