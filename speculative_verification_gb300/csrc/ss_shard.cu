// ss_shard.cu -- sampling over vocabulary shards for rows whose kept set
// needs the whole distribution: top-p and / or min-p without top-k (and the
// plain and greedy rows alongside them).  The FlashSampling news page names
// grouped variants for tensor-parallel logits (each GPU holds a slice of the
// vocabulary); Gumbel-max decomposes over the slices (the argmax of the
// parts' maxima), but a top-p cut does not: it needs the row's total mass
// and the order of the tokens around the cut.  So the shards exchange, in
// four rounds, exactly what the cut needs (see include/ss.h):
//   0. each shard's largest processed logit (and its greedy argument, its
//      allowed count, its status)                     -> the row maximum m
//   1. each shard's fixed-point mass sum (trunc(exp(y - m) * 2^40), the
//      histogram kernel's masses) and a histogram of count and mass over
//      1024 buckets of y below m                        -> the total S, the
//      target ceil(p * S) and the bucket holding the cut
//   2. each shard's tokens in that bucket              -> the exact cut item
//      (the first, in (y desc, token asc) order, whose prefix mass reaches
//      the target), or the min-p threshold when that is shorter
//   3. each shard's count of kept tokens and its best y + Gumbel noise (the
//      same Philox keys)                                -> the token, |K|
// Every quantity is the one the single-call kernels compute, so the merged
// result is identical to ss_process_sample's on the whole rows.
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include <algorithm>

#include "ss.h"
#include "ss_nvtx.h"
#include "ss_philox.cuh"

namespace ss {
namespace shard {

constexpr int kThreads = 512;
constexpr int kWarps = kThreads / 32;
constexpr int kBuckets = 1024;
constexpr float kRange = 28.2f;  // masses of tokens further than this below m are 0
constexpr int kList = 1024;      // cut-bucket tokens one shard may list
constexpr int kHash = 1024;      // patched tokens one shard may hold per row
constexpr int kMaxShards = 8;
constexpr int kRounds = 4;
constexpr int kBiasFlag = 1 << 30;

enum { kModeAll = 0, kModeMinP = 1, kModeTopP = 2 };

// Per-row state between rounds (device, 64 bytes).
struct alignas(16) RowState {
  int32_t status, done, mode, bucket;
  float m, cut_v;
  int32_t cut_t, kept;
  unsigned long long S, T, mass_before, count_before;
};
static_assert(sizeof(RowState) == 64, "row state is 64 bytes");

// Per-row record of one shard (device), by round.
struct alignas(16) Rec {
  int32_t status, count, arg, n;     // 0: status, allowed count, greedy argument; 2: listed tokens
  float m, best;                     // 0: largest y (z for greedy rows); 3: best score
  int32_t best_t, pad;
  unsigned long long S;              // 1: the shard's mass sum
  unsigned long long pad2;
  // then, by round: 1: uint32 counts[kBuckets], uint64 masses[kBuckets];
  //                 2: uint64 items[kList] (entry keys: y desc, token asc)
};
constexpr size_t kRecBytes = sizeof(Rec) + kBuckets * 4 + kBuckets * 8;
static_assert(sizeof(Rec) + kList * 8 <= kRecBytes, "a listing fits the record");

struct SArgs {
  int32_t num_rows, vocab, dtype, round;
  int32_t off, len;
  int64_t row_stride;
  const void* logits;
  ss_params p;
  const RowState* state;
  uint8_t* rec;
};

struct MArgs {
  int32_t num_rows, num_shards, round, vocab;
  const uint8_t* rec[kMaxShards];
  ss_params p;
  RowState* state;
  int32_t* out_token;
  int32_t* out_status;
  int32_t* out_kept;
};

__device__ __forceinline__ float ninf() { return __int_as_float(0xff800000); }
__device__ __forceinline__ float pinf() { return __int_as_float(0x7f800000); }

// The histogram kernel's fixed-point mass of y: trunc(exp(y - m) * 2^40), the
// truncation taken from the float's bits (the same integers).
__device__ __forceinline__ unsigned long long fmass(float y, float m) {
  const float e = fminf(__expf(__fsub_rn(y, m)), 1.0f);
  const uint32_t b = __float_as_uint(e);
  const int sh = static_cast<int>(b >> 23) - 127 + 40 - 23;
  const unsigned long long mant = (b & 0x7fffffu) | 0x800000u;
  if (sh >= 0) return mant << sh;
  return (sh > -24) ? (mant >> (-sh)) : 0ull;
}

__device__ __forceinline__ uint32_t okey(float y) {
  const uint32_t b = __float_as_uint(y + 0.0f);
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}
__device__ __forceinline__ float okey_value(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7fffffffu) : ~k);
}
// (y desc, token asc) as an ascending 64-bit key
__device__ __forceinline__ unsigned long long ekey(float y, int32_t t) {
  return (static_cast<unsigned long long>(~okey(y)) << 32) | static_cast<uint32_t>(t);
}
__device__ __forceinline__ float ekey_y(unsigned long long e) { return okey_value(~static_cast<uint32_t>(e >> 32)); }
__device__ __forceinline__ int32_t ekey_t(unsigned long long e) { return static_cast<int32_t>(static_cast<uint32_t>(e)); }

__device__ __forceinline__ bool beats(float s, int32_t t, float bs, int32_t bt) {
  return s > bs || (s == bs && t < bt);
}

__device__ __forceinline__ int bucket_of(float y, float m) {
  const float d = __fsub_rn(m, y);
  if (!(d <= kRange)) return kBuckets;  // (and y = -inf)
  return min(kBuckets - 1, static_cast<int>(__fmul_rn(d, static_cast<float>(kBuckets) / kRange)));
}

__device__ __forceinline__ int hash_slot(int32_t t) { return static_cast<int>((static_cast<uint32_t>(t) * 2654435761u) >> 22); }

// ------------------------------------------------------------ shard round --

struct Row {
  int32_t status, greedy, use_mask;
  float inv_t, rep, freq, pres, top_p, min_p, lmp;
  uint32_t seed_lo, seed_hi, pos, rid;
};

__global__ void __launch_bounds__(kThreads) ss_shard_round_kernel(const SArgs a) {
  __shared__ Row R;
  __shared__ int32_t hkey[kHash], hcnt[kHash];
  __shared__ float hval[kHash];
  __shared__ int32_t s_status, s_count, s_n;
  __shared__ unsigned long long s_S;
  __shared__ float s_red[kWarps];
  __shared__ int32_t s_redt[kWarps];
  extern __shared__ __align__(16) uint8_t dyn[];
  uint32_t* patched = reinterpret_cast<uint32_t*>(dyn);  // one bit per shard token
  const int r = blockIdx.x, tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  const int V = a.vocab, off = a.off, len = a.len;
  Rec* out = reinterpret_cast<Rec*>(a.rec + static_cast<int64_t>(r) * kRecBytes);
  const RowState st = (a.round > 0) ? a.state[r] : RowState{};
  if (a.round > 0 && (st.done || (a.round < 3 && st.mode != kModeTopP))) return;  // nothing for this row

  // parameters (the checks of the single-call kernels)
  if (tid == 0) {
    const ss_params& p = a.p;
    int s = SS_ROW_OK;
    const float T = p.temperature[r];
    const int32_t top_k = p.top_k ? p.top_k[r] : 0;
    R.top_p = p.top_p ? p.top_p[r] : 1.0f;
    R.min_p = p.min_p ? p.min_p[r] : 0.0f;
    R.rep = p.repetition ? p.repetition[r] : 1.0f;
    R.freq = p.frequency ? p.frequency[r] : 0.0f;
    R.pres = p.presence ? p.presence[r] : 0.0f;
    const int64_t pos = p.position[r];
    if (pos < 0 || pos > 0xFFFFFFFFLL) s = SS_ROW_BAD_PARAM;
    if (!(T >= 0.0f) || isinf(T)) s = SS_ROW_BAD_PARAM;
    if (top_k < 0 || !(R.top_p > 0.0f) || !(R.min_p >= 0.0f && R.min_p <= 1.0f)) s = SS_ROW_BAD_PARAM;
    if (!(R.rep > 0.0f) || isinf(R.rep) || !isfinite(R.freq) || !isfinite(R.pres)) s = SS_ROW_BAD_PARAM;
    const int32_t h0 = p.hist_offsets ? p.hist_offsets[r] : 0, h1 = p.hist_offsets ? p.hist_offsets[r + 1] : 0;
    const int32_t b0 = p.bias_offsets ? p.bias_offsets[r] : 0, b1 = p.bias_offsets ? p.bias_offsets[r + 1] : 0;
    if (h1 < h0 || b1 < b0) s = SS_ROW_BAD_PARAM;
    R.greedy = (T == 0.0f);
    // rows with a top-k cut take the list path (ss_sample_shard)
    if (s == SS_ROW_OK && !R.greedy && top_k > 0 && top_k < V) s = SS_ROW_UNSUPPORTED;
    R.inv_t = (R.greedy || !(T > 0.0f)) ? 1.0f : __frcp_rn(T);
    R.lmp = (!R.greedy && R.min_p > 0.0f) ? logf(R.min_p) : 0.0f;
    R.use_mask = p.bitmask && (!p.use_bitmask || p.use_bitmask[r]);
    R.seed_lo = static_cast<uint32_t>(p.seed[r]);
    R.seed_hi = static_cast<uint32_t>(p.seed[r] >> 32);
    R.pos = static_cast<uint32_t>(pos);
    R.rid = p.row_id ? p.row_id[r] : static_cast<uint32_t>(r);
    R.status = s;
    s_status = s;
    s_count = 0;
    s_n = 0;
    s_S = 0;
  }
  for (int i = tid; i < kHash; i += kThreads) {
    hkey[i] = -1;
    hcnt[i] = 0;
    hval[i] = 0.0f;
  }
  for (int w = tid; w < (len + 31) / 32; w += kThreads) patched[w] = 0;
  __syncthreads();
  const ss_params& p = a.p;
  // patched tokens of this shard (ids are global; every shard checks all)
  auto insert = [&](int32_t t) -> int {
    int h = hash_slot(t);
    for (int probe = 0; probe < kHash; ++probe) {
      const int32_t prev = atomicCAS(&hkey[h], -1, t);
      if (prev == -1 || prev == t) return h;
      h = (h + 1) & (kHash - 1);
    }
    return -1;
  };
  if (R.status == SS_ROW_OK) {
    int s = SS_ROW_OK;
    if (p.hist_offsets)
      for (int e = p.hist_offsets[r] + tid; e < p.hist_offsets[r + 1]; e += kThreads) {
        const int32_t t = p.hist_ids[e];
        if (t < 0 || t >= V) {
          s = max(s, SS_ROW_BAD_INDEX);
        } else if (t >= off && t < off + len) {
          const int h = insert(t);
          if (h < 0) {
            s = max(s, SS_ROW_LIMIT);
          } else {
            atomicAdd(&hcnt[h], 1);
            atomicOr(&patched[(t - off) >> 5], 1u << ((t - off) & 31));
          }
        }
      }
    if (p.bias_offsets)
      for (int e = p.bias_offsets[r] + tid; e < p.bias_offsets[r + 1]; e += kThreads) {
        const int32_t t = p.bias_ids[e];
        if (!isfinite(p.bias_vals[e])) s = max(s, SS_ROW_BAD_PARAM);
        if (t < 0 || t >= V) {
          s = max(s, SS_ROW_BAD_INDEX);
        } else if (t >= off && t < off + len) {
          const int h = insert(t);
          if (h < 0) {
            s = max(s, SS_ROW_LIMIT);
          } else {
            if (atomicOr(&hcnt[h], kBiasFlag) & kBiasFlag) s = max(s, SS_ROW_BAD_INDEX);  // a duplicate id
            hval[h] = p.bias_vals[e];
            atomicOr(&patched[(t - off) >> 5], 1u << ((t - off) & 31));
          }
        }
      }
    if (s != SS_ROW_OK) atomicMax(&s_status, s);
  }
  __syncthreads();
  const bool row_ok = s_status == SS_ROW_OK;
  const float inv_t = R.inv_t;
  const bool greedy = R.greedy != 0;
  const int32_t* mrow = R.use_mask ? p.bitmask + static_cast<int64_t>(r) * p.bitmask_stride : nullptr;
  // the processed logit of shard token t (-inf: not allowed)
  auto process = [&](int32_t t) -> float {
    const int64_t at = static_cast<int64_t>(r) * a.row_stride + (t - off);
    float z = (a.dtype == SS_DTYPE_BF16)
                  ? __uint_as_float(static_cast<uint32_t>(static_cast<const uint16_t*>(a.logits)[at]) << 16)
                  : static_cast<const float*>(a.logits)[at];
    if ((patched[(t - off) >> 5] >> ((t - off) & 31)) & 1u) {
      int h = hash_slot(t);
      while (hkey[h] != t) h = (h + 1) & (kHash - 1);
      const int32_t hc = hcnt[h], cnt = hc & ~kBiasFlag;
      if (cnt > 0) {
        z = (z > 0.0f) ? __fdiv_rn(z, R.rep) : __fmul_rn(z, R.rep);
        z = __fsub_rn(z, __fmul_rn(R.freq, static_cast<float>(cnt)));
        z = __fsub_rn(z, R.pres);
      }
      if (hc & kBiasFlag) z = __fadd_rn(z, hval[h]);
    }
    if (mrow && !((static_cast<uint32_t>(mrow[t >> 5]) >> (t & 31)) & 1u)) return ninf();
    return greedy ? z : __fmul_rn(z, inv_t);
  };

  if (a.round == 0) {
    // the shard's largest y (z for greedy rows) and its lowest index, the
    // allowed count, non-finite values
    float best = ninf();
    int32_t arg = 0x7fffffff, cnt = 0;
    bool bad = false;
    if (row_ok)
      for (int t = off + tid; t < off + len; t += kThreads) {
        const float y = process(t);
        if (y == ninf()) continue;
        if (y != y || y == pinf()) bad = true;
        ++cnt;
        if (beats(y, t, best, arg)) {  // larger y, then the lower index
          best = y;
          arg = t;
        }
      }
    if (bad) atomicMax(&s_status, SS_ROW_NONFINITE);
    atomicAdd(&s_count, cnt);
    for (int o = 16; o; o >>= 1) {
      const float ob = __shfl_xor_sync(0xffffffffu, best, o);
      const int32_t oa = __shfl_xor_sync(0xffffffffu, arg, o);
      if (ob > best || (ob == best && oa < arg)) {
        best = ob;
        arg = oa;
      }
    }
    if (lane == 0) {
      s_red[wid] = best;
      s_redt[wid] = arg;
    }
    __syncthreads();
    if (tid == 0) {
      for (int w = 1; w < kWarps; ++w)
        if (s_red[w] > best || (s_red[w] == best && s_redt[w] < arg)) {
          best = s_red[w];
          arg = s_redt[w];
        }
      out->status = s_status;
      out->count = s_count;
      out->m = best;
      out->arg = arg;
    }
    return;
  }
  const float m = st.m;
  if (a.round == 1) {
    // mass sum and the bucket histogram (top-p rows)
    uint32_t* bc = reinterpret_cast<uint32_t*>(reinterpret_cast<uint8_t*>(out) + sizeof(Rec));
    unsigned long long* bm = reinterpret_cast<unsigned long long*>(bc + kBuckets);
    uint32_t* sc = reinterpret_cast<uint32_t*>(dyn + (((len + 31) / 32) * 4 + 15) / 16 * 16);
    unsigned long long* sm = reinterpret_cast<unsigned long long*>(sc + kBuckets);
    for (int b = tid; b < kBuckets; b += kThreads) {
      sc[b] = 0;
      sm[b] = 0;
    }
    __syncthreads();
    unsigned long long S = 0;
    for (int t = off + tid; t < off + len; t += kThreads) {
      const float y = process(t);
      const int b = bucket_of(y, m);
      if (b >= kBuckets) continue;
      const unsigned long long w = fmass(y, m);
      S += w;
      atomicAdd(&sc[b], 1u);
      atomicAdd(&sm[b], w);
    }
    atomicAdd(&s_S, S);
    __syncthreads();
    for (int b = tid; b < kBuckets; b += kThreads) {
      bc[b] = sc[b];
      bm[b] = sm[b];
    }
    if (tid == 0) out->S = s_S;
    return;
  }
  if (a.round == 2) {
    // the tokens of the cut's bucket
    unsigned long long* items = reinterpret_cast<unsigned long long*>(reinterpret_cast<uint8_t*>(out) + sizeof(Rec));
    for (int t = off + tid; t < off + len; t += kThreads) {
      const float y = process(t);
      if (bucket_of(y, m) != st.bucket) continue;
      const int i = atomicAdd(&s_n, 1);
      if (i < kList) items[i] = ekey(y, t);
    }
    __syncthreads();
    if (tid == 0) out->n = s_n;
    return;
  }
  // round 3: the kept count and the draw over this shard's part of K
  float best = ninf();
  int32_t bt = 0x7fffffff, cnt = 0;
  for (int t = off + tid; t < off + len; t += kThreads) {
    const float y = process(t);
    if (y == ninf()) continue;
    bool in = true;
    if (st.mode == kModeMinP) in = __fsub_rn(y, m) >= R.lmp;
    if (st.mode == kModeTopP) in = y > st.cut_v || (y == st.cut_v && t <= st.cut_t);
    if (!in) continue;
    ++cnt;
    const uint32_t num = uniform_numerator(
        philox4x32_10(static_cast<uint32_t>(t) >> 2, R.pos, R.rid, 0u, R.seed_lo, R.seed_hi).w[t & 3]);
    const float sc = __fadd_rn(y, gumbel_from_numerator(num));
    if (beats(sc, t, best, bt)) {
      best = sc;
      bt = t;
    }
  }
  atomicAdd(&s_count, cnt);
  for (int o = 16; o; o >>= 1) {
    const float ob = __shfl_xor_sync(0xffffffffu, best, o);
    const int32_t ot = __shfl_xor_sync(0xffffffffu, bt, o);
    if (beats(ob, ot, best, bt)) {
      best = ob;
      bt = ot;
    }
  }
  if (lane == 0) {
    s_red[wid] = best;
    s_redt[wid] = bt;
  }
  __syncthreads();
  if (tid == 0) {
    for (int w = 1; w < kWarps; ++w)
      if (beats(s_red[w], s_redt[w], best, bt)) {
        best = s_red[w];
        bt = s_redt[w];
      }
    out->count = s_count;
    out->best = best;
    out->best_t = bt;
  }
}

// ------------------------------------------------------------ merge round --

__global__ void __launch_bounds__(256) ss_merge_round_kernel(const MArgs a) {
  extern __shared__ __align__(16) unsigned long long keys[];  // round 2: the listed tokens
  __shared__ int32_t s_total, s_cut;
  __shared__ unsigned long long s_wsum[8], s_wcnt[8];  // rounds 1 and 2: per-warp sums (256 threads)
  const int r = blockIdx.x, tid = threadIdx.x;
  RowState& st = a.state[r];
  auto rec = [&](int s) { return reinterpret_cast<const Rec*>(a.rec[s] + static_cast<int64_t>(r) * kRecBytes); };
  auto finish = [&](int32_t status, int32_t token, int32_t kept) {
    a.out_token[r] = (status == SS_ROW_OK) ? token : -1;
    a.out_status[r] = status;
    if (a.out_kept) a.out_kept[r] = (status == SS_ROW_OK) ? kept : 0;
    st.done = 1;
  };
  if (a.round > 0 && (st.done || (a.round < 3 && st.mode != kModeTopP))) return;
  if (a.round == 0) {
    if (tid != 0) return;
    int32_t status = SS_ROW_OK, count = 0, arg = 0x7fffffff;
    float m = ninf();
    for (int s = 0; s < a.num_shards; ++s) {
      const Rec* h = rec(s);
      status = max(status, h->status);
      count += h->count;
      if (h->count > 0 && (h->m > m || (h->m == m && h->arg < arg))) {
        m = h->m;
        arg = h->arg;
      }
    }
    if (status == SS_ROW_OK && count == 0) status = SS_ROW_EMPTY_SET;
    st = RowState{};
    st.status = status;
    st.m = m;
    const float T = a.p.temperature[r];
    const int32_t top_k = a.p.top_k ? a.p.top_k[r] : 0;
    if (T != 0.0f && top_k > 0 && top_k < a.vocab) {
      st.done = 1;  // a top-k row: ss_merge_shards writes it
      return;
    }
    const float top_p = a.p.top_p ? a.p.top_p[r] : 1.0f;
    const float min_p = a.p.min_p ? a.p.min_p[r] : 0.0f;
    if (status != SS_ROW_OK) {
      finish(status, -1, 0);
    } else if (T == 0.0f) {
      finish(status, arg, 1);  // greedy: the largest logit, lowest index
    } else {
      st.mode = (top_p < 1.0f) ? kModeTopP : (min_p > 0.0f ? kModeMinP : kModeAll);
    }
    return;
  }
  if (a.round == 1) {
    // the target and the bucket holding the cut: each thread sums four
    // buckets over the shards, a block scan of those sums, and the thread
    // whose buckets hold the first one reaching the target records it
    constexpr int kPer = kBuckets / 256;
    static_assert(kBuckets % 256 == 0, "four buckets per thread");
    unsigned long long S = 0;
    for (int s = 0; s < a.num_shards; ++s) S += rec(s)->S;
    const float top_p = a.p.top_p[r];
    const unsigned long long T = static_cast<unsigned long long>(ceil(static_cast<double>(top_p) * static_cast<double>(S)));
    unsigned long long mb[kPer], cb[kPer], cm = 0, cc = 0;
#pragma unroll
    for (int i = 0; i < kPer; ++i) {
      const int b = tid * kPer + i;
      mb[i] = 0;
      cb[i] = 0;
      for (int s = 0; s < a.num_shards; ++s) {
        const uint32_t* bc = reinterpret_cast<const uint32_t*>(reinterpret_cast<const uint8_t*>(rec(s)) + sizeof(Rec));
        const unsigned long long* bm = reinterpret_cast<const unsigned long long*>(bc + kBuckets);
        mb[i] += bm[b];
        cb[i] += bc[b];
      }
      cm += mb[i];
      cc += cb[i];
    }
    const int lane = tid & 31, wid = tid >> 5;
    unsigned long long im = cm, ic = cc;  // inclusive within the warp
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const unsigned long long ym = __shfl_up_sync(0xffffffffu, im, o), yc = __shfl_up_sync(0xffffffffu, ic, o);
      if (lane >= o) {
        im += ym;
        ic += yc;
      }
    }
    if (lane == 31) {
      s_wsum[wid] = im;
      s_wcnt[wid] = ic;
    }
    if (tid == 0) s_cut = 0x7fffffff;
    __syncthreads();
    unsigned long long bm_run = im - cm, bc_run = ic - cc;  // before this thread's buckets
    for (int w = 0; w < wid; ++w) {
      bm_run += s_wsum[w];
      bc_run += s_wcnt[w];
    }
    int found = -1;
    unsigned long long fm = 0, fc = 0;
#pragma unroll
    for (int i = 0; i < kPer; ++i) {
      if (found < 0 && mb[i] > 0 && bm_run + mb[i] >= T) {
        found = tid * kPer + i;
        fm = bm_run;
        fc = bc_run;
      }
      bm_run += mb[i];
      bc_run += cb[i];
    }
    if (found >= 0) atomicMin(&s_cut, found);
    __syncthreads();
    if (found >= 0 && found == s_cut) {
      st.S = S;
      st.T = T;
      st.bucket = found;
      st.mass_before = fm;
      st.count_before = fc;
    }
    return;
  }
  if (a.round == 2) {
    // every shard's tokens of the bucket, sorted (y desc, token asc); the
    // first whose prefix mass reaches the target is the cut
    if (tid == 0) {
      int total = 0;
      for (int s = 0; s < a.num_shards; ++s) {
        const int n = rec(s)->n;
        if (n > kList) total = -1;
        if (total >= 0) total += n;
      }
      s_total = total;
    }
    __syncthreads();
    const int n = s_total;
    if (n <= 0) {  // a listing overflowed (or the bucket is empty: cannot happen)
      if (tid == 0) finish(SS_ROW_LIMIT, -1, 0);
      return;
    }
    int np2 = 1;
    while (np2 < n) np2 <<= 1;
    for (int i = tid; i < np2; i += blockDim.x) keys[i] = ~0ull;
    __syncthreads();
    int base = 0;
    for (int s = 0; s < a.num_shards; ++s) {
      const Rec* h = rec(s);
      const unsigned long long* items = reinterpret_cast<const unsigned long long*>(reinterpret_cast<const uint8_t*>(h) + sizeof(Rec));
      for (int i = tid; i < h->n; i += blockDim.x) keys[base + i] = items[i];
      base += h->n;
    }
    __syncthreads();
    for (int k = 2; k <= np2; k <<= 1)
      for (int j = k >> 1; j > 0; j >>= 1) {
        for (int q = tid; q < (np2 >> 1); q += blockDim.x) {
          const int i = ((q & ~(j - 1)) << 1) | (q & (j - 1));
          const unsigned long long x = keys[i], y = keys[i + j];
          if ((x > y) == ((i & k) == 0)) {
            keys[i] = y;
            keys[i + j] = x;
          }
        }
        __syncthreads();
      }
    // the first item i with a non-zero mass whose running total (from the
    // mass before the bucket) reaches the target: each thread sums a
    // contiguous chunk, a block scan of the chunk sums, and the thread whose
    // chunk holds it walks its chunk
    {
      const int per = (n + static_cast<int>(blockDim.x) - 1) / static_cast<int>(blockDim.x);
      const int i0 = min(tid * per, n), i1 = min(i0 + per, n);
      unsigned long long local = 0;
      for (int i = i0; i < i1; ++i) local += fmass(ekey_y(keys[i]), st.m);
      unsigned long long inc = local;  // inclusive scan within the warp
      const int lane = tid & 31, wid = tid >> 5;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const unsigned long long y = __shfl_up_sync(0xffffffffu, inc, o);
        if (lane >= o) inc += y;
      }
      if (lane == 31) s_wsum[wid] = inc;
      if (tid == 0) s_cut = 0x7fffffff;
      __syncthreads();
      unsigned long long run = st.mass_before + inc - local;
      for (int w = 0; w < wid; ++w) run += s_wsum[w];
      for (int i = i0; i < i1; ++i) {
        const unsigned long long w = fmass(ekey_y(keys[i]), st.m);
        if (w > 0 && run + w >= st.T) {
          atomicMin(&s_cut, i);
          break;
        }
        run += w;
      }
      __syncthreads();
    }
    if (tid == 0) {
      const int cut = (s_cut == 0x7fffffff) ? -1 : s_cut;
      if (cut < 0) {
        finish(SS_ROW_LIMIT, -1, 0);
        return;
      }
      const float v = ekey_y(keys[cut]);
      const float min_p = a.p.min_p ? a.p.min_p[r] : 0.0f;
      const float lmp = (min_p > 0.0f) ? logf(min_p) : 0.0f;
      if (min_p > 0.0f && !(__fsub_rn(v, st.m) >= lmp)) {
        st.mode = kModeMinP;  // the min-p prefix is the shorter
      } else {
        st.cut_v = v;
        st.cut_t = ekey_t(keys[cut]);
      }
    }
    return;
  }
  // round 3
  if (tid != 0) return;
  float best = ninf();
  int32_t bt = 0x7fffffff, kept = 0;
  for (int s = 0; s < a.num_shards; ++s) {
    const Rec* h = rec(s);
    kept += h->count;
    if (h->best_t != 0x7fffffff && beats(h->best, h->best_t, best, bt)) {
      best = h->best;
      bt = h->best_t;
    }
  }
  finish(bt != 0x7fffffff ? SS_ROW_OK : SS_ROW_EMPTY_SET, bt, kept);
}

}  // namespace shard
}  // namespace ss

// -------------------------------------------------------------- C ABI --

extern "C" {

size_t ss_shard_round_record_bytes(void) { return ss::shard::kRecBytes; }

size_t ss_shard_round_state_bytes(int32_t num_rows) {
  return num_rows < 0 ? 0 : static_cast<size_t>(num_rows) * sizeof(ss::shard::RowState);
}

ss_status ss_shard_round(const ss_sample_args* args, int32_t vocab_offset, int32_t shard_len, int32_t round,
                         const void* state, void* records, ss_stream_t stream) {
  SS_NVTX_RANGE("ss_shard_round");
  using namespace ss::shard;
  if (!args) return SS_ERR_INVALID_ARG;
  const ss_sample_args& A = *args;
  if (A.num_rows < 0 || A.vocab < 1 || round < 0 || round >= kRounds) return SS_ERR_INVALID_ARG;
  if (A.dtype != SS_DTYPE_F32 && A.dtype != SS_DTYPE_BF16) return SS_ERR_INVALID_ARG;
  if (vocab_offset < 0 || shard_len < 1 || static_cast<int64_t>(vocab_offset) + shard_len > A.vocab)
    return SS_ERR_INVALID_ARG;
  if (A.num_rows == 0) return SS_OK;
  const int es = (A.dtype == SS_DTYPE_BF16) ? 2 : 4;
  if (!A.logits || (reinterpret_cast<uintptr_t>(A.logits) % es) != 0 || !records ||
      (reinterpret_cast<uintptr_t>(records) & 15u) != 0 || (round > 0 && !state))
    return SS_ERR_INVALID_ARG;
  if (A.row_stride < shard_len) return SS_ERR_INVALID_ARG;
  if (!A.params.temperature || !A.params.seed || !A.params.position) return SS_ERR_INVALID_ARG;
  if ((A.params.hist_offsets == nullptr) != (A.params.hist_ids == nullptr)) return SS_ERR_INVALID_ARG;
  if (A.params.bias_offsets && (!A.params.bias_ids || !A.params.bias_vals)) return SS_ERR_INVALID_ARG;
  if (A.params.bitmask && A.params.bitmask_stride < (static_cast<int64_t>(A.vocab) + 31) / 32) return SS_ERR_INVALID_ARG;
  SArgs a{};
  a.num_rows = A.num_rows;
  a.vocab = A.vocab;
  a.dtype = A.dtype;
  a.round = round;
  a.off = vocab_offset;
  a.len = shard_len;
  a.row_stride = A.row_stride;
  a.logits = A.logits;
  a.p = A.params;
  a.state = static_cast<const RowState*>(state);
  a.rec = static_cast<uint8_t*>(records);
  const size_t smem = (static_cast<size_t>((shard_len + 31) / 32) * 4 + 15) / 16 * 16 + kBuckets * 12;
  if (smem > 200 * 1024) return SS_ERR_UNSUPPORTED;
  cudaError_t e = cudaFuncSetAttribute(ss_shard_round_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e == cudaSuccess) {
    ss_shard_round_kernel<<<A.num_rows, kThreads, smem, reinterpret_cast<cudaStream_t>(stream)>>>(a);
    e = cudaGetLastError();
  }
  return e == cudaSuccess ? SS_OK : SS_ERR_CUDA;
}

ss_status ss_merge_round(const ss_sample_args* args, int32_t num_shards, void* const* records, int32_t round,
                         void* state, ss_stream_t stream) {
  SS_NVTX_RANGE("ss_merge_round");
  using namespace ss::shard;
  if (!args || !records || !state) return SS_ERR_INVALID_ARG;
  const ss_sample_args& A = *args;
  if (A.num_rows < 0 || num_shards < 1 || num_shards > kMaxShards || round < 0 || round >= kRounds)
    return SS_ERR_INVALID_ARG;
  if (A.num_rows == 0) return SS_OK;
  if (!A.out_token || !A.out_status || !A.params.temperature) return SS_ERR_INVALID_ARG;
  MArgs m{};
  m.num_rows = A.num_rows;
  m.num_shards = num_shards;
  m.round = round;
  m.vocab = A.vocab;
  for (int s = 0; s < num_shards; ++s) {
    if (!records[s] || (reinterpret_cast<uintptr_t>(records[s]) & 15u) != 0) return SS_ERR_INVALID_ARG;
    m.rec[s] = static_cast<const uint8_t*>(records[s]);
  }
  m.p = A.params;
  m.state = static_cast<RowState*>(state);
  m.out_token = A.out_token;
  m.out_status = A.out_status;
  m.out_kept = A.out_kept;
  const size_t smem = (round == 2) ? static_cast<size_t>(kMaxShards) * kList * 8 : 16;
  cudaError_t e = cudaFuncSetAttribute(ss_merge_round_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e == cudaSuccess) {
    ss_merge_round_kernel<<<A.num_rows, 256, smem, reinterpret_cast<cudaStream_t>(stream)>>>(m);
    e = cudaGetLastError();
  }
  return e == cudaSuccess ? SS_OK : SS_ERR_CUDA;
}

}  // extern "C"
