/*
 * ss_oracle.c -- CPU oracle (TEST INFRASTRUCTURE ONLY; see ss_oracle.h).
 *
 * Build: cc -std=c99 -O2 -ffp-contract=off -fPIC -shared (oracle/build.py).
 * -ffp-contract=off matters: the processed logits are defined as a sequence
 * of individually rounded fp32 operations, and a fused multiply-add would
 * round differently.
 *
 * Per row (SonicSampler abstract: the logit-processing feature list; order of
 * application is a reading, see the design notes):
 *   1. z_t = fp32(logits[t])                       (bf16 -> fp32 is exact)
 *   2. penalties, for every token t seen c_t > 0 times in the history:
 *        z = z > 0 ? z / rep : z * rep;  z = z - freq * c_t;  z = z - pres
 *   3. bias: z_t = z_t + b                      (ids must be distinct per row)
 *   4. grammar mask: bit (t & 31) of word t >> 5 equal to 0 -> z_t = -inf
 *   5. temperature: T = 0 is greedy (lowest index of the largest z);
 *      otherwise y_t = z_t * fp32(1 / T)
 *   6. order the allowed tokens by (y descending, index ascending)
 *   7. top-k keeps the first k, top-p the shortest prefix whose mass in the
 *      top-k-renormalised distribution reaches p, min-p the tokens with
 *      exp(y - y_max) >= min_p; K is the shortest of the three prefixes
 *   8. draw: argmax over K of y_t + g_t, g_t = -log(-log u_t)
 *      (FlashSampling page: Gumbel noise plus argmax is an exact sample)
 */
#include "ss_oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>

#define REL_MARGIN 1e-5
#define ABS_FLOOR 1e-30

/* ------------------------------------------------------------------ RNG -- */

static void philox_round(uint32_t c[4], uint32_t k0, uint32_t k1) {
  /* One Philox-4x32 round: two 32x32->64 products, the high halves xored
   * with the other two counter words and the key (SC'11, section 3). */
  uint64_t prod_a = (uint64_t)0xD2511F53u * (uint64_t)c[0];
  uint64_t prod_b = (uint64_t)0xCD9E8D57u * (uint64_t)c[2];
  uint32_t n0 = (uint32_t)(prod_b >> 32) ^ c[1] ^ k0;
  uint32_t n1 = (uint32_t)prod_b;
  uint32_t n2 = (uint32_t)(prod_a >> 32) ^ c[3] ^ k1;
  uint32_t n3 = (uint32_t)prod_a;
  c[0] = n0;
  c[1] = n1;
  c[2] = n2;
  c[3] = n3;
}

void or_philox4x32_10(const uint32_t ctr[4], const uint32_t key[2], uint32_t out[4]) {
  uint32_t c[4];
  uint32_t k0 = key[0], k1 = key[1];
  int r;
  memcpy(c, ctr, sizeof c);
  for (r = 0; r < 10; ++r) {
    philox_round(c, k0, k1);
    k0 += 0x9E3779B9u; /* Weyl key schedule */
    k1 += 0xBB67AE85u;
  }
  memcpy(out, c, sizeof c);
}

/* Counter (t >> 2, position, row, stream), key (seed lo, seed hi); lane t & 3.
 * u = (2 * (x >> 9) + 1) * 2^-24: 24 significant bits, so exact in fp32, and
 * strictly inside (0, 1). */
float or_uniform(uint64_t seed, int32_t row, uint32_t position, int32_t token, uint32_t stream) {
  uint32_t ctr[4], key[2], out[4];
  uint32_t x, odd;
  ctr[0] = (uint32_t)token >> 2;
  ctr[1] = position;
  ctr[2] = (uint32_t)row;
  ctr[3] = stream;
  key[0] = (uint32_t)(seed & 0xFFFFFFFFu);
  key[1] = (uint32_t)(seed >> 32);
  or_philox4x32_10(ctr, key, out);
  x = out[(uint32_t)token & 3u];
  odd = ((x >> 9) << 1) | 1u;
  return (float)ldexp((double)odd, -24);
}

double or_gumbel(uint64_t seed, int32_t row, uint32_t position, int32_t token, uint32_t stream) {
  double u = (double)or_uniform(seed, row, position, token, stream);
  return -log(-log(u));
}

/* The Gumbel noise of tokens 0 .. vocab-1 of one row, position and stream. */
void or_gumbel_row(uint64_t seed, int32_t row, uint32_t position, uint32_t stream, int32_t vocab, double* out) {
  int32_t t;
  for (t = 0; t < vocab; ++t) out[t] = or_gumbel(seed, row, position, t, stream);
}

/* ---------------------------------------------------------------- helpers -- */

static float ld_logit(const void* base, int32_t dtype, int64_t idx) {
  if (dtype == OR_DTYPE_BF16) {
    uint16_t h = ((const uint16_t*)base)[idx];
    uint32_t bits = (uint32_t)h << 16;
    float f;
    memcpy(&f, &bits, sizeof f);
    return f;
  }
  return ((const float*)base)[idx];
}

static int is_pos_inf_or_nan(float v) { return isnan(v) || (isinf(v) && v > 0); }

/* Order of step 6: larger y first, then smaller index. */
typedef struct {
  float y;
  int32_t t;
} yt_pair;

static int cmp_order(const void* a, const void* b) {
  const yt_pair* pa = (const yt_pair*)a;
  const yt_pair* pb = (const yt_pair*)b;
  if (pa->y > pb->y) return -1;
  if (pa->y < pb->y) return 1;
  return (pa->t < pb->t) ? -1 : (pa->t > pb->t);
}

/* ------------------------------------------------------------ row state -- */

typedef struct {
  int32_t vocab, dtype;
  const void* z;
  float temperature, top_p, min_p, rep, freq, pres;
  int32_t top_k;
  const int32_t* hist;
  int32_t hist_len;
  const int32_t* hist2; /* drafts before this target position */
  int32_t hist2_len;
  const int32_t* bias_ids;
  const float* bias_vals;
  int32_t bias_len;
  const int32_t* mask; /* NULL = no grammar mask */
  int bad_param;       /* request-level parameter error already found */
} row_in;

typedef struct {
  int32_t status;
  int greedy;
  float* y;          /* [V]; z for greedy rows; -inf = not allowed */
  int32_t* order;    /* allowed tokens in step-6 order */
  int32_t n_allowed;
  int32_t L;         /* |K| */
  int32_t L_lo, L_hi; /* |K| values a 1e-5 relative perturbation can give */
  float ymax;
  double* w;         /* [n_allowed] exp(y - ymax) by sorted position */
  double SK;         /* sum of w over K */
  int flag_k;        /* L_lo != L_hi: a top-p or min-p cut is within margin */
} row_state;

static void row_free(row_state* s) {
  free(s->y);
  free(s->order);
  free(s->w);
  memset(s, 0, sizeof *s);
}

static int param_invalid(const row_in* in) {
  if (in->bad_param) return 1;
  if (!(in->temperature >= 0.0f) || isinf(in->temperature)) return 1;
  if (in->top_k < 0) return 1;
  if (!(in->top_p > 0.0f)) return 1;
  if (!(in->min_p >= 0.0f && in->min_p <= 1.0f)) return 1;
  if (!(in->rep > 0.0f) || isinf(in->rep)) return 1;
  if (!isfinite(in->freq) || !isfinite(in->pres)) return 1;
  if (in->hist_len < 0 || in->bias_len < 0) return 1;
  for (int32_t e = 0; e < in->bias_len; ++e)
    if (!isfinite(in->bias_vals[e])) return 1;
  return 0;
}

static int index_invalid(const row_in* in) {
  int32_t V = in->vocab;
  for (int32_t e = 0; e < in->hist_len; ++e)
    if (in->hist[e] < 0 || in->hist[e] >= V) return 1;
  for (int32_t e = 0; e < in->hist2_len; ++e)
    if (in->hist2[e] < 0 || in->hist2[e] >= V) return 1;
  for (int32_t e = 0; e < in->bias_len; ++e) {
    if (in->bias_ids[e] < 0 || in->bias_ids[e] >= V) return 1;
    for (int32_t f = 0; f < e; ++f)
      if (in->bias_ids[f] == in->bias_ids[e]) return 1; /* ids must be distinct */
  }
  return 0;
}

/* Steps 1-7.  On return s->status is final; if it is OK, K = order[0..L). */
static void row_prepare(const row_in* in, row_state* s) {
  int32_t V = in->vocab, t, i, n = 0;
  int32_t* count;
  memset(s, 0, sizeof *s);
  s->greedy = (in->temperature == 0.0f);
  s->y = (float*)malloc(sizeof(float) * (size_t)(V > 0 ? V : 1));
  s->order = (int32_t*)malloc(sizeof(int32_t) * (size_t)(V > 0 ? V : 1));
  s->w = (double*)malloc(sizeof(double) * (size_t)(V > 0 ? V : 1));
  for (t = 0; t < V; ++t) s->y[t] = -INFINITY;
  if (param_invalid(in)) {
    s->status = OR_ROW_BAD_PARAM;
    return;
  }
  if (index_invalid(in)) {
    s->status = OR_ROW_BAD_INDEX;
    return;
  }

  /* 1. load */
  for (t = 0; t < V; ++t) s->y[t] = ld_logit(in->z, in->dtype, t);

  /* 2. penalties: occurrence counts over history + preceding drafts */
  count = (int32_t*)calloc((size_t)(V > 0 ? V : 1), sizeof(int32_t));
  for (i = 0; i < in->hist_len; ++i) count[in->hist[i]] += 1;
  for (i = 0; i < in->hist2_len; ++i) count[in->hist2[i]] += 1;
  for (t = 0; t < V; ++t) {
    if (count[t] > 0) {
      float z = s->y[t];
      z = (z > 0.0f) ? (z / in->rep) : (z * in->rep);
      z = z - in->freq * (float)count[t];
      z = z - in->pres;
      s->y[t] = z;
    }
  }
  free(count);

  /* 3. bias */
  for (i = 0; i < in->bias_len; ++i) s->y[in->bias_ids[i]] = s->y[in->bias_ids[i]] + in->bias_vals[i];

  /* 4. grammar mask, least significant bit first, 1 = allowed */
  if (in->mask) {
    for (t = 0; t < V; ++t) {
      uint32_t word = (uint32_t)in->mask[t >> 5];
      if (((word >> (t & 31)) & 1u) == 0u) s->y[t] = -INFINITY;
    }
  }

  /* 5. temperature */
  if (!s->greedy) {
    float inv_t = 1.0f / in->temperature;
    for (t = 0; t < V; ++t) s->y[t] = s->y[t] * inv_t;
  }

  /* allowed = not -inf; NaN or +inf among them is a data fault */
  for (t = 0; t < V; ++t) {
    if (s->y[t] == -INFINITY) continue;
    if (is_pos_inf_or_nan(s->y[t])) {
      s->status = OR_ROW_NONFINITE;
      return;
    }
    s->order[n++] = t;
  }
  s->n_allowed = n;
  if (n == 0) {
    s->status = OR_ROW_EMPTY_SET;
    return;
  }

  /* 6. order */
  {
    yt_pair* pairs = (yt_pair*)malloc(sizeof(yt_pair) * (size_t)n);
    for (i = 0; i < n; ++i) {
      pairs[i].y = s->y[s->order[i]];
      pairs[i].t = s->order[i];
    }
    qsort(pairs, (size_t)n, sizeof(yt_pair), cmp_order);
    for (i = 0; i < n; ++i) s->order[i] = pairs[i].t;
    free(pairs);
  }
  s->ymax = s->y[s->order[0]];

  if (s->greedy) { /* argmax with the lowest index survives every filter */
    s->L = s->L_lo = s->L_hi = 1;
    s->w[0] = 1.0;
    s->SK = 1.0;
    return;
  }

  /* 7. filters.  Besides L, record the range [L_lo, L_hi] of prefix lengths
   * the comparisons can give within the decision margin (1e-5 relative):
   * for top-p, each renormalised probability of the top-k prefix may move by
   * that much (so every prefix mass C may lie anywhere in [C(1-d), C(1+d)]);
   * for min-p, each ratio w = exp(y - ymax) may (the maximum's own w = 1 is
   * exact: its y - ymax is 0 in any arithmetic). */
  {
    int32_t Lk = (in->top_k > 0 && in->top_k < n) ? in->top_k : n;
    int32_t Lp = Lk, Lp_lo = Lk, Lp_hi = Lk, Lm = n, Lm_lo = n, Lm_hi = n;
    double Sk = 0.0;
    for (i = 0; i < n; ++i) s->w[i] = exp((double)s->y[s->order[i]] - (double)s->ymax);
    for (i = 0; i < Lk; ++i) Sk += s->w[i];

    if (in->top_p < 1.0f) {
      double p = (double)in->top_p, cum = 0.0, c;
      int got = 0, got_lo = 0, got_hi = 0;
      for (i = 0; i < Lk; ++i) {
        cum += s->w[i];
        c = cum / Sk; /* C_{i+1}: mass of the first i+1 tokens */
        /* shortest: every mass at its largest, C(1+d) >= p; longest: C(1-d) >= p */
        if (!got_lo && c * (1.0 + REL_MARGIN) >= p) { Lp_lo = i + 1; got_lo = 1; }
        if (!got && c >= p) { Lp = i + 1; got = 1; }
        if (!got_hi && c * (1.0 - REL_MARGIN) >= p) { Lp_hi = i + 1; got_hi = 1; break; }
      }
    }
    if (in->min_p > 0.0f) {
      double mp = (double)in->min_p;
      Lm = Lm_lo = Lm_hi = 0;
      while (Lm < n && s->w[Lm] >= mp) ++Lm;
      /* shortest: every w (but the exact 1s) at w(1-d); longest: at w(1+d) */
      while (Lm_lo < n && (s->w[Lm_lo] == 1.0 ? 1.0 >= mp : s->w[Lm_lo] * (1.0 - REL_MARGIN) >= mp)) ++Lm_lo;
      while (Lm_hi < n && (s->w[Lm_hi] == 1.0 ? 1.0 >= mp : s->w[Lm_hi] * (1.0 + REL_MARGIN) >= mp)) ++Lm_hi;
    }
    s->L = Lk < Lp ? Lk : Lp;
    if (Lm < s->L) s->L = Lm;
    s->L_lo = Lk < Lp_lo ? Lk : Lp_lo;
    if (Lm_lo < s->L_lo) s->L_lo = Lm_lo;
    s->L_hi = Lk < Lp_hi ? Lk : Lp_hi;
    if (Lm_hi < s->L_hi) s->L_hi = Lm_hi;
    s->flag_k = (s->L_lo != s->L_hi);
    s->SK = 0.0;
    for (i = 0; i < s->L; ++i) s->SK += s->w[i];
  }
}

/* Replace K by the first L tokens of the order, for an L inside [L_lo, L_hi]
 * (the tests pass the kept count the GPU chose when the oracle's own cut is
 * within margin).  Returns 1 when L was accepted. */
static int row_force_L(row_state* s, int32_t L) {
  int32_t i;
  if (s->status != OR_ROW_OK || s->greedy || L < s->L_lo || L > s->L_hi || L < 1) return 0;
  s->L = L;
  s->SK = 0.0;
  for (i = 0; i < L; ++i) s->SK += s->w[i];
  s->flag_k = 0;
  return 1;
}

/* P(t) of a prepared row; 0 outside K. */
static double row_prob(const row_state* s, int32_t t) {
  int32_t i;
  for (i = 0; i < s->L; ++i)
    if (s->order[i] == t) return s->w[i] / s->SK;
  return 0.0;
}

/* Step 8.  Gumbel-max over K.  Sets *flag when the decision is within the
 * margin: each y_t and each g_t may move by 1e-5 * max(1, |value|), and some
 * other token's highest score reaches the winner's lowest. */
static double margin_of(double v) { return REL_MARGIN * fmax(1.0, fabs(v)); }

static int32_t row_draw(const row_state* s, uint64_t seed, int32_t row, uint32_t pos, int* flag) {
  int32_t i, best = -1;
  double sb = -INFINITY, lo_best = 0.0;
  if (s->greedy) return s->order[0];
  for (i = 0; i < s->L; ++i) {
    int32_t t = s->order[i];
    double g = or_gumbel(seed, row, pos, t, OR_STREAM_DRAW);
    double sc = (double)s->y[t] + g;
    if (best < 0 || sc > sb || (sc == sb && t < best)) {
      best = t;
      sb = sc;
      lo_best = sc - margin_of((double)s->y[t]) - margin_of(g);
    }
  }
  for (i = 0; i < s->L; ++i) {
    int32_t t = s->order[i];
    double g, hi;
    if (t == best) continue;
    g = or_gumbel(seed, row, pos, t, OR_STREAM_DRAW);
    hi = (double)s->y[t] + g + margin_of((double)s->y[t]) + margin_of(g);
    if (hi >= lo_best) {
      *flag = 1;
      break;
    }
  }
  return best;
}

static void fill_row_in(row_in* r, const or_params* p, int32_t idx, int32_t V, int32_t dtype,
                        const void* zrow) {
  int64_t h0, h1, b0, b1;
  memset(r, 0, sizeof *r);
  r->vocab = V;
  r->dtype = dtype;
  r->z = zrow;
  r->temperature = p->temperature[idx];
  r->top_k = p->top_k ? p->top_k[idx] : 0;
  r->top_p = p->top_p ? p->top_p[idx] : 1.0f;
  r->min_p = p->min_p ? p->min_p[idx] : 0.0f;
  r->rep = p->repetition ? p->repetition[idx] : 1.0f;
  r->freq = p->frequency ? p->frequency[idx] : 0.0f;
  r->pres = p->presence ? p->presence[idx] : 0.0f;
  if (p->hist_offsets) {
    h0 = p->hist_offsets[idx];
    h1 = p->hist_offsets[idx + 1];
    r->hist = p->hist_ids + h0;
    r->hist_len = (int32_t)(h1 - h0);
  }
  if (p->bias_offsets) {
    b0 = p->bias_offsets[idx];
    b1 = p->bias_offsets[idx + 1];
    r->bias_ids = p->bias_ids + b0;
    r->bias_vals = p->bias_vals + b0;
    r->bias_len = (int32_t)(b1 - b0);
  }
  if (p->bitmask && (!p->use_bitmask || p->use_bitmask[idx])) r->mask = p->bitmask + (int64_t)idx * p->bitmask_stride;
  if (p->position[idx] < 0 || p->position[idx] > (int64_t)0xFFFFFFFFLL) r->bad_param = 1;
}

/* ------------------------------------------------------------ sampling -- */

int or_process_sample(const or_sample_in* in, or_sample_out* out) {
  int32_t r, V = in->vocab;
  size_t es = (in->dtype == OR_DTYPE_BF16) ? 2 : 4;
  for (r = 0; r < in->num_rows; ++r) {
    row_in ri;
    row_state s;
    int flag = 0;
    int32_t tok = -1;
    const char* zrow = (const char*)in->logits + (size_t)r * (size_t)in->row_stride * es;
    fill_row_in(&ri, &in->p, r, V, in->dtype, zrow);
    row_prepare(&ri, &s);
    if (out->kept_lo) out->kept_lo[r] = (s.status == OR_ROW_OK) ? s.L_lo : 0;
    if (out->kept_hi) out->kept_hi[r] = (s.status == OR_ROW_OK) ? s.L_hi : 0;
    if (out->kept_own) out->kept_own[r] = (s.status == OR_ROW_OK) ? s.L : 0;
    if (in->force_kept && in->force_kept[r] > 0) row_force_L(&s, in->force_kept[r]);
    if (s.status == OR_ROW_OK) {
      /* Philox counter word 2: the caller's row id, else the row's index */
      const int32_t rid = in->p.row_id ? (int32_t)in->p.row_id[r] : r;
      tok = row_draw(&s, in->p.seed[r], rid, (uint32_t)in->p.position[r], &flag);
      flag |= s.flag_k;
    }
    out->token[r] = tok;
    out->status[r] = s.status;
    if (out->kept) out->kept[r] = (s.status == OR_ROW_OK) ? s.L : 0;
    if (out->processed) memcpy(out->processed + (size_t)r * (size_t)V, s.y, sizeof(float) * (size_t)V);
    if (out->sub_margin) out->sub_margin[r] = (uint8_t)(flag != 0);
    row_free(&s);
  }
  return 0;
}

int32_t or_row_probs(const or_sample_in* in, int32_t row, const int32_t* extra_hist, int32_t extra_len,
                     double* probs_out) {
  row_in ri;
  row_state s;
  int32_t t, status;
  size_t es = (in->dtype == OR_DTYPE_BF16) ? 2 : 4;
  const char* zrow = (const char*)in->logits + (size_t)row * (size_t)in->row_stride * es;
  fill_row_in(&ri, &in->p, row, in->vocab, in->dtype, zrow);
  ri.hist2 = extra_hist;
  ri.hist2_len = extra_len;
  row_prepare(&ri, &s);
  for (t = 0; t < in->vocab; ++t) probs_out[t] = 0.0;
  if (s.status == OR_ROW_OK)
    for (t = 0; t < s.L; ++t) probs_out[s.order[t]] = s.w[t] / s.SK;
  status = s.status;
  row_free(&s);
  return status;
}

int32_t or_residual_probs(int32_t vocab, const double* P, const float* q, double* out) {
  double tot = 0.0;
  int32_t t;
  for (t = 0; t < vocab; ++t) {
    double r = P[t] - (double)q[t];
    out[t] = (r > 0.0) ? r : 0.0;
    tot += out[t];
  }
  if (!(tot > 0.0)) return 1;
  for (t = 0; t < vocab; ++t) out[t] /= tot;
  return 0;
}

/* ----------------------------------------------------- verification -- */

/* Residual draw on a rejected position: argmax over t with r_t > 0 of
 * log r_t + g_t (stream 2).  Returns -1 when no r_t > 0.  The sub-margin test
 * lets each P_t move by 1e-5 relative and each g_t by 1e-5 * max(1, |g_t|)
 * (q_t is an input, exact) and asks whether any other candidate's best case
 * reaches the winner's worst case, or the winner's residual can vanish. */
static int32_t residual_draw(const row_state* s, const float* qrow, uint64_t seed, int32_t row,
                             uint32_t pos, int* flag) {
  int32_t i, best = -1;
  double sb = -INFINITY, lo_best = -INFINITY;
  double* hi = (double*)malloc(sizeof(double) * (size_t)(s->L > 0 ? s->L : 1));
  double* lo = (double*)malloc(sizeof(double) * (size_t)(s->L > 0 ? s->L : 1));
  int32_t* tok = (int32_t*)malloc(sizeof(int32_t) * (size_t)(s->L > 0 ? s->L : 1));
  int any_contender = 0;
  for (i = 0; i < s->L; ++i) {
    int32_t t = s->order[i];
    double P = s->greedy ? 1.0 : s->w[i] / s->SK;
    double q = (double)qrow[t];
    double r = P - q;
    double d = REL_MARGIN * P; /* P may move by the margin; q is an input */
    double g = or_gumbel(seed, row, pos, t, OR_STREAM_RESIDUAL);
    double geps = margin_of(g);
    tok[i] = t;
    hi[i] = (r + d > 0.0) ? log(r + d) + g + geps : -INFINITY;
    lo[i] = (r - d > 0.0) ? log(r - d) + g - geps : -INFINITY;
    if (r + d > 0.0) any_contender = 1;
    if (r > 0.0) {
      double sc = log(r) + g;
      if (best < 0 || sc > sb || (sc == sb && t < best)) {
        best = t;
        sb = sc;
        lo_best = lo[i];
      }
    }
  }
  if (best < 0) {
    if (any_contender) *flag = 1;
  } else {
    for (i = 0; i < s->L; ++i)
      if (tok[i] != best && hi[i] >= lo_best) *flag = 1;
    if (lo_best == -INFINITY) *flag = 1;
  }
  free(hi);
  free(lo);
  free(tok);
  return best;
}

int or_spec_verify(const or_verify_in* in, or_verify_out* out) {
  int32_t i, V = in->vocab;
  size_t es = (in->dtype == OR_DTYPE_BF16) ? 2 : 4;
  int32_t width = in->max_draft + 1;
  for (i = 0; i < in->num_requests; ++i) {
    int32_t d0 = in->draft_offsets[i], d1 = in->draft_offsets[i + 1];
    int32_t k = d1 - d0, j, status = OR_ROW_OK, n_acc = 0;
    int flag = 0, bad_req = 0;
    int64_t pos64 = in->p.position[i];
    row_state* rows;
    int32_t* o = out->out_tokens + (size_t)i * (size_t)width;
    for (j = 0; j < width; ++j) o[j] = -1;
    if (k < 0 || k > in->max_draft || pos64 < 0 || pos64 + k > (int64_t)0xFFFFFFFFLL) bad_req = 1;
    if (bad_req) {
      out->num_accepted[i] = 0;
      out->status[i] = OR_ROW_BAD_PARAM;
      if (out->sub_margin) out->sub_margin[i] = 0;
      if (k >= 0 && k <= in->max_draft) {
        for (j = 0; j <= k; ++j) {
          int64_t trow = (int64_t)d0 + i + j;
          if (out->kept) out->kept[trow] = 0;
          if (out->processed)
            for (int32_t t = 0; t < V; ++t) out->processed[(size_t)trow * (size_t)V + (size_t)t] = -INFINITY;
        }
      }
      continue;
    }
    rows = (row_state*)calloc((size_t)k + 1, sizeof(row_state));
    for (j = 0; j <= k; ++j) {
      row_in ri;
      int64_t trow = (int64_t)d0 + i + j;
      const char* zrow = (const char*)in->target_logits + (size_t)trow * (size_t)in->row_stride * es;
      fill_row_in(&ri, &in->p, i, V, in->dtype, zrow);
      ri.hist2 = in->draft_tokens + d0;
      ri.hist2_len = j;
      if (j == 0) { /* every draft must be a token id */
        int32_t e;
        for (e = 0; e < k; ++e)
          if (in->draft_tokens[d0 + e] < 0 || in->draft_tokens[d0 + e] >= V) ri.hist2_len = k; /* flags it */
      }
      row_prepare(&ri, &rows[j]);
      if (out->kept_lo) out->kept_lo[trow] = (rows[j].status == OR_ROW_OK) ? rows[j].L_lo : 0;
      if (out->kept_hi) out->kept_hi[trow] = (rows[j].status == OR_ROW_OK) ? rows[j].L_hi : 0;
      if (out->kept_own) out->kept_own[trow] = (rows[j].status == OR_ROW_OK) ? rows[j].L : 0;
      if (in->force_kept && in->force_kept[trow] > 0) row_force_L(&rows[j], in->force_kept[trow]);
      if (rows[j].status > status) status = rows[j].status;
      if (out->kept) out->kept[trow] = (rows[j].status == OR_ROW_OK) ? rows[j].L : 0;
      if (out->processed) memcpy(out->processed + (size_t)trow * (size_t)V, rows[j].y, sizeof(float) * (size_t)V);
    }
    if (status == OR_ROW_OK) {
      uint64_t seed = in->p.seed[i];
      uint32_t pos = (uint32_t)pos64;
      /* Philox counter word 2: the caller's request id, else its index */
      const int32_t rid = in->p.row_id ? (int32_t)in->p.row_id[i] : i;
      int32_t final_tok = -1;
      for (j = 0; j < k; ++j) {
        int32_t x = in->draft_tokens[d0 + j];
        const float* qrow = in->draft_probs + (size_t)(d0 + j) * (size_t)in->draft_stride;
        double P = row_prob(&rows[j], x);
        double q = (double)qrow[x];
        double u = (double)or_uniform(seed, rid, pos + (uint32_t)j, 0, OR_STREAM_ACCEPT);
        double uq = u * q;
        flag |= rows[j].flag_k;
        /* accept iff u q < P; P may move by the margin, u and q are exact */
        if (uq >= P * (1.0 - REL_MARGIN) && uq < P * (1.0 + REL_MARGIN)) flag = 1;
        if (uq < P) {
          o[j] = x;
          ++n_acc;
          continue;
        }
        final_tok = residual_draw(&rows[j], qrow, seed, rid, pos + (uint32_t)j, &flag);
        if (final_tok < 0) final_tok = row_draw(&rows[j], seed, rid, pos + (uint32_t)j, &flag);
        break;
      }
      if (j == k) { /* every draft accepted: the bonus token from row k */
        flag |= rows[k].flag_k;
        final_tok = row_draw(&rows[k], seed, rid, pos + (uint32_t)k, &flag);
      }
      o[n_acc] = final_tok;
    } else {
      n_acc = 0;
      flag = 0;
    }
    out->num_accepted[i] = n_acc;
    out->status[i] = status;
    if (out->sub_margin) out->sub_margin[i] = (uint8_t)(flag != 0);
    for (j = 0; j <= k; ++j) row_free(&rows[j]);
    free(rows);
  }
  return 0;
}

/* Step after verification: append the emitted tokens of each accepted
 * request to its token buffer and advance its length and position. */
void or_commit_accepted(int32_t num_requests, int32_t max_draft, const int32_t* out_tokens,
                        const int32_t* num_accepted, const int32_t* status, int32_t* tokens, int32_t capacity,
                        int32_t* seq_len, int64_t* position, int32_t* next_token, int32_t* commit_status) {
  int32_t i, j;
  for (i = 0; i < num_requests; ++i) {
    const int32_t* emitted = out_tokens + (size_t)i * (size_t)(max_draft + 1);
    int32_t count;
    if (status[i] != 0) {
      commit_status[i] = status[i];
      continue;
    }
    count = num_accepted[i] + 1;
    if (count < 1 || count > max_draft + 1 || seq_len[i] < 0 || (int64_t)seq_len[i] + count > capacity) {
      commit_status[i] = 6;
      continue;
    }
    for (j = 0; j < count; ++j) tokens[(size_t)i * (size_t)capacity + (size_t)(seq_len[i] + j)] = emitted[j];
    seq_len[i] += count;
    position[i] += count;
    next_token[i] = emitted[count - 1];
    commit_status[i] = 0;
  }
}

/* ------------------------------------------------- tree verification -- */

/* Gumbel-max over t in K of log r_t + g_t (stream 2), r_t = p_t - q_t > 0,
 * for a dense residual base p (fp64).  `scale` bounds how much the rounding
 * of p may have grown through the normalisations before it (the product of
 * 1/Z); the sub-margin test perturbs r_t by REL_MARGIN * scale * (p_t + q_t)
 * and the noise by REL_MARGIN.  Returns -1 when no r_t > 0. */
static int32_t residual_draw_dense(const row_state* s, const double* p, const float* qrow, double scale,
                                   uint64_t seed, int32_t row, uint32_t pos, int* flag) {
  int32_t i, best = -1;
  double sb = -INFINITY, lo_best = -INFINITY;
  double* hi = (double*)malloc(sizeof(double) * (size_t)(s->L > 0 ? s->L : 1));
  int32_t* tok = (int32_t*)malloc(sizeof(int32_t) * (size_t)(s->L > 0 ? s->L : 1));
  int any_contender = 0;
  for (i = 0; i < s->L; ++i) {
    int32_t t = s->order[i];
    double q = (double)qrow[t];
    double r = p[t] - q;
    double d = REL_MARGIN * scale * (p[t] + fabs(q));
    double g = or_gumbel(seed, row, pos, t, OR_STREAM_RESIDUAL);
    double geps = REL_MARGIN * fmax(1.0, fabs(g));
    tok[i] = t;
    hi[i] = (r + d > 0.0) ? log(r + d) + g + geps : -INFINITY;
    if (r + d > 0.0) any_contender = 1;
    if (r > 0.0) {
      double sc = log(r) + g;
      if (best < 0 || sc > sb || (sc == sb && t < best)) {
        best = t;
        sb = sc;
        lo_best = (r - d > 0.0) ? log(r - d) + g - geps : -INFINITY;
      }
    }
  }
  if (best < 0) {
    if (any_contender) *flag = 1;
  } else {
    for (i = 0; i < s->L; ++i)
      if (tok[i] != best && hi[i] >= lo_best) *flag = 1;
    if (lo_best == -INFINITY) *flag = 1;
  }
  free(hi);
  free(tok);
  return best;
}

/* Depth of local node u (edges to the root); -1 when a parent on the way is
 * not a smaller index.  path (optional) receives the tokens of the nodes on
 * the way, u first, the root's child last. */
static int32_t tree_depth(const int32_t* par, const int32_t* tok, int32_t u, int32_t* path) {
  int32_t d = 0;
  while (u > 0) {
    int32_t pu = par[u];
    if (pu < 0 || pu >= u) return -1;
    if (path) path[d] = tok[u];
    ++d;
    u = pu;
  }
  return d;
}

int or_tree_verify(const or_tree_in* in, or_tree_out* out) {
  int32_t i, V = in->vocab, width = in->max_nodes;
  size_t es = (in->dtype == OR_DTYPE_BF16) ? 2 : 4;
  for (i = 0; i < in->num_requests; ++i) {
    int32_t g0 = in->node_offsets[i], nn = in->node_offsets[i + 1] - g0;
    const int32_t* par = in->parents + g0;
    const int32_t* tok = in->node_tokens + g0;
    int32_t* o = out->out_tokens + (size_t)i * (size_t)width;
    int32_t* op = out->out_path ? out->out_path + (size_t)i * (size_t)width : NULL;
    int32_t j, u, status = OR_ROW_OK, n_acc = 0, bad_tree = 0, bad_tok = 0;
    int64_t pos64 = in->p.position[i];
    int flag = 0;
    row_state* rows;
    int32_t* depth;
    for (j = 0; j < width; ++j) {
      o[j] = -1;
      if (op) op[j] = -1;
    }
    out->num_accepted[i] = 0;
    if (out->sub_margin) out->sub_margin[i] = 0;
    if (nn < 1 || nn > width || nn > 64) {
      out->status[i] = OR_ROW_BAD_PARAM;
      continue;
    }
    for (u = 1; u < nn; ++u) {
      if (par[u] < 0 || par[u] >= u) bad_tree = 1;
      if (tok[u] < 0 || tok[u] >= V) bad_tok = 1;
    }
    if (bad_tree) {
      out->status[i] = OR_ROW_BAD_PARAM;
      continue;
    }
    rows = (row_state*)calloc((size_t)nn, sizeof(row_state));
    depth = (int32_t*)calloc((size_t)nn, sizeof(int32_t));
    for (u = 0; u < nn; ++u) {
      row_in ri;
      int32_t path[64];
      const char* zrow = (const char*)in->target_logits + (size_t)(g0 + u) * (size_t)in->row_stride * es;
      depth[u] = tree_depth(par, tok, u, path);
      fill_row_in(&ri, &in->p, i, V, in->dtype, zrow);
      if (pos64 + (nn - 1) > (int64_t)0xFFFFFFFFLL) ri.bad_param = 1;
      ri.hist2 = path;
      ri.hist2_len = depth[u];
      row_prepare(&ri, &rows[u]);
      if (rows[u].status < OR_ROW_BAD_INDEX && bad_tok) rows[u].status = OR_ROW_BAD_INDEX;
      if (rows[u].status > status) status = rows[u].status;
    }
    if (status == OR_ROW_OK) {
      uint64_t seed = in->p.seed[i];
      const int32_t rid = in->p.row_id ? (int32_t)in->p.row_id[i] : i;
      double* p = (double*)malloc(sizeof(double) * (size_t)V);
      u = 0;
      for (;;) {
        const row_state* s = &rows[u];
        const float* qrow = in->draft_probs + (size_t)(g0 + u) * (size_t)in->draft_stride;
        uint32_t pos = (uint32_t)pos64 + (uint32_t)depth[u];
        int32_t kids[64], m = 0, c, next = -1, final_tok = -1, t;
        double scale = 1.0;
        for (c = u + 1; c < nn; ++c)
          if (par[c] == u) kids[m++] = c;
        flag |= s->flag_k;
        if (m == 0) { /* a leaf: the bonus token */
          final_tok = row_draw(s, seed, rid, pos, &flag);
        } else if (s->greedy) {
          for (c = 0; c < m; ++c)
            if (tok[kids[c]] == s->order[0]) {
              next = kids[c];
              break;
            }
          if (next < 0) final_tok = s->order[0];
        } else {
          for (t = 0; t < V; ++t) p[t] = 0.0;
          for (t = 0; t < s->L; ++t) p[s->order[t]] = s->w[t] / s->SK;
          for (c = 0; c < m; ++c) {
            int32_t x = tok[kids[c]];
            double q = (double)qrow[x];
            double uq = (double)or_uniform(seed, rid, pos, c, OR_STREAM_ACCEPT) * q;
            double Z = 0.0;
            if (fabs(uq - p[x]) <= REL_MARGIN * (1 + c) * scale * (p[x] + q) + ABS_FLOOR) flag = 1;
            if (uq < p[x]) {
              next = kids[c];
              break;
            }
            if (c == m - 1) {
              final_tok = residual_draw_dense(s, p, qrow, (1 + c) * scale, seed, rid, pos, &flag);
              if (final_tok < 0) final_tok = row_draw(s, seed, rid, pos, &flag);
              break;
            }
            for (t = 0; t < V; ++t) {
              double r = p[t] - (double)qrow[t];
              p[t] = (r > 0.0) ? r : 0.0;
              Z += p[t];
            }
            if (Z < 1e-6) flag = 1; /* rounding decides whether anything is left */
            if (!(Z > 0.0)) {
              final_tok = row_draw(s, seed, rid, pos, &flag);
              break;
            }
            for (t = 0; t < V; ++t) p[t] /= Z;
            scale /= Z;
          }
        }
        if (next >= 0) {
          o[n_acc] = tok[next];
          if (op) op[n_acc] = next;
          ++n_acc;
          u = next;
          continue;
        }
        o[n_acc] = final_tok;
        break;
      }
      free(p);
    } else {
      flag = 0;
    }
    out->num_accepted[i] = n_acc;
    out->status[i] = status;
    if (out->sub_margin) out->sub_margin[i] = (uint8_t)(flag != 0);
    for (u = 0; u < nn; ++u) row_free(&rows[u]);
    free(rows);
    free(depth);
  }
  return 0;
}
