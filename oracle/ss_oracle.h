/*
 * ss_oracle.h -- CPU oracle for batched LLM sampling and speculative
 * verification.  TEST INFRASTRUCTURE ONLY: the tests, the smoke check and the
 * CPU-baseline leg of the benchmark call it; the product path never does.
 *
 * Plain, slow, single-threaded C99.  It computes the *definition* of each
 * result (full sort, noise on every kept token, sequential rejection rule),
 * in the order the pages list the steps:
 *   - SonicSampler abstract (arxivdaily.com/papers/2607.20475): the feature
 *     list -- grammar-constrained decoding, repetition / frequency / presence
 *     penalties, logit bias, temperature, top-k / top-p / min-p, speculative
 *     verification, all per request in one batch.
 *   - "FlashSampling: schnelles, speichereffizientes Exact Sampling fuer LLMs"
 *     (meineki.news), paragraphs 2-3: exact sampling by adding Gumbel noise and
 *     taking the argmax; the argmax decomposes over vocabulary partitions.
 *   - "Accelerating Sonar through speculation" (Perplexity blog), section
 *     "Speculative decoding" (n drafts give up to n+1 tokens; the target's
 *     logits after the last accepted draft give one more token) and section
 *     "Draft-target" (acceptance compares the full draft and target
 *     distributions).  The accept/residual rule is that of the first work in
 *     the post's reference list, "Fast inference from transformers via
 *     speculative decoding".
 * Every numerical convention the pages leave open is a stated reading; the
 * readings are listed in the repository's design notes.
 *
 * This header is the oracle's own: nothing under the CUDA package includes it.
 */
#ifndef SS_ORACLE_H
#define SS_ORACLE_H
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Row status codes; the larger code wins when several apply. */
enum {
  OR_ROW_OK = 0,
  OR_ROW_EMPTY_SET = 1,  /* no token survives the mask */
  OR_ROW_NONFINITE = 2,  /* an allowed processed logit is NaN or +inf */
  OR_ROW_BAD_INDEX = 3,  /* history/draft/bias id outside [0,V), duplicate bias id */
  OR_ROW_BAD_PARAM = 4   /* invalid scalar parameter */
};

enum { OR_DTYPE_F32 = 0, OR_DTYPE_BF16 = 1 };

/* Philox stream ids (counter word 3). */
enum { OR_STREAM_DRAW = 0, OR_STREAM_ACCEPT = 1, OR_STREAM_RESIDUAL = 2 };

/* Per-row (or per-request) sampling parameters, host pointers.  A NULL
 * optional array means "feature off" for every row. */
typedef struct {
  const float* temperature;      /* [n] required; 0 = greedy                   */
  const int32_t* top_k;          /* [n] or NULL; <=0 or >= #allowed = off      */
  const float* top_p;            /* [n] or NULL; >= 1 = off                    */
  const float* min_p;            /* [n] or NULL; 0 = off                       */
  const float* repetition;       /* [n] or NULL (1 = off)                      */
  const float* frequency;        /* [n] or NULL (0 = off)                      */
  const float* presence;         /* [n] or NULL (0 = off)                      */
  const int32_t* hist_offsets;   /* [n+1] or NULL                              */
  const int32_t* hist_ids;
  const int32_t* bias_offsets;   /* [n+1] or NULL                              */
  const int32_t* bias_ids;
  const float* bias_vals;
  const int32_t* bitmask;        /* [n, bitmask_stride] words or NULL          */
  int64_t bitmask_stride;
  const uint8_t* use_bitmask;    /* [n] or NULL (= every row uses the mask)    */
  const uint64_t* seed;          /* [n] required                               */
  const int64_t* position;       /* [n] required                               */
  const uint32_t* row_id;        /* [n] or NULL (= the row's index): Philox counter word 2 */
} or_params;

typedef struct {
  int32_t num_rows, vocab;
  int64_t row_stride;            /* elements; 0 lets every row alias row 0     */
  int32_t dtype;
  const void* logits;
  or_params p;
  const int32_t* force_kept;     /* [n] or NULL: see or_process_sample         */
} or_sample_in;

typedef struct {
  int32_t* token;                /* [n]                                        */
  int32_t* status;               /* [n]                                        */
  int32_t* kept;                 /* [n] or NULL: |K| (1 for greedy)            */
  float* processed;              /* [n, vocab] or NULL                         */
  uint8_t* sub_margin;           /* [n] or NULL: a decision was within 1e-5    */
  int32_t* kept_lo;              /* [n] or NULL: smallest |K| within margin    */
  int32_t* kept_hi;              /* [n] or NULL: largest |K| within margin     */
  int32_t* kept_own;             /* [n] or NULL: |K| before force_kept         */
} or_sample_out;

typedef struct {
  int32_t num_requests, vocab, max_draft;
  int64_t row_stride;
  int32_t dtype;
  const void* target_logits;     /* row of (i,j) = draft_offsets[i] + i + j    */
  const int32_t* draft_offsets;  /* [R+1]                                      */
  const int32_t* draft_tokens;   /* [sum k]                                    */
  const float* draft_probs;      /* [sum k, draft_stride]                      */
  int64_t draft_stride;
  or_params p;                   /* per request                                */
  const int32_t* force_kept;     /* [rows] or NULL                             */
} or_verify_in;

typedef struct {
  int32_t* out_tokens;           /* [R, max_draft+1], -1 padded                */
  int32_t* num_accepted;         /* [R]                                        */
  int32_t* status;               /* [R]                                        */
  int32_t* kept;                 /* [rows] or NULL                             */
  float* processed;              /* [rows, vocab] or NULL                      */
  uint8_t* sub_margin;           /* [R] or NULL                                */
  int32_t* kept_lo;              /* [rows] or NULL                             */
  int32_t* kept_hi;              /* [rows] or NULL                             */
  int32_t* kept_own;             /* [rows] or NULL: |K| before force_kept      */
} or_verify_out;

/* Philox4x32-10 block function (Salmon, Moraes, Dror, Shaw, "Parallel random
 * numbers: as easy as 1, 2, 3", SC'11). */
void or_philox4x32_10(const uint32_t ctr[4], const uint32_t key[2], uint32_t out[4]);

/* The uniform of token t: u in [2^-24, 1-2^-24], exact in fp32. */
float or_uniform(uint64_t seed, int32_t row, uint32_t position, int32_t token, uint32_t stream);

/* Gumbel noise of that uniform, in fp64: -log(-log u). */
double or_gumbel(uint64_t seed, int32_t row, uint32_t position, int32_t token, uint32_t stream);

/* or_gumbel of tokens 0 .. vocab-1 (one row, position and stream) into out. */
void or_gumbel_row(uint64_t seed, int32_t row, uint32_t position, uint32_t stream, int32_t vocab, double* out);

/* Batched sampling over [num_rows, vocab] logits.  Returns 0.
 * When force_kept[r] > 0 lies in [kept_lo[r], kept_hi[r]] -- a kept-set size
 * that the top-p / min-p comparisons reach under a 1e-5 relative change of the
 * probabilities -- the row draws from the first force_kept[r] tokens of its
 * order instead of its own cut, and only the draw's own margin is flagged. */
int or_process_sample(const or_sample_in* in, or_sample_out* out);

/* Batched speculative verification.  Returns 0. */
int or_spec_verify(const or_verify_in* in, or_verify_out* out);

/* The step after verification, on the host-visible definition: for request
 * i whose status is 0, its num_accepted[i] + 1 emitted tokens
 * out_tokens[i * (max_draft + 1) + 0 .. num_accepted[i]] are appended to
 * tokens[i * capacity + seq_len[i] ...], seq_len[i] and position[i] advance
 * by their count and next_token[i] becomes the last of them; commit_status[i]
 * is 0.  A request whose tokens would not fit (or whose num_accepted lies
 * outside [0, max_draft], or whose seq_len is negative) is left unchanged
 * with commit_status 6 (limit); one whose status is not 0 is left unchanged
 * with that status copied.  (Accelerating Sonar through speculation, "MTP
 * schedule for a single token": the next target tokens are placed into their
 * slots on the GPU, with no GPU-to-CPU synchronisation.) */
void or_commit_accepted(int32_t num_requests, int32_t max_draft, const int32_t* out_tokens,
                        const int32_t* num_accepted, const int32_t* status, int32_t* tokens, int32_t capacity,
                        int32_t* seq_len, int64_t* position, int32_t* next_token, int32_t* commit_status);

/* The filtered, renormalised distribution of one sampling row (fp64, zero
 * outside the kept set K; one-hot for greedy rows).  `extra_hist` are tokens
 * appended to the row's history (the drafts preceding a target position).
 * Returns the row status. */
int32_t or_row_probs(const or_sample_in* in, int32_t row, const int32_t* extra_hist,
                     int32_t extra_len, double* probs_out /* [vocab] */);

/* Residual distribution max(P - q, 0) / sum, fp64.  Returns 0 if some entry is
 * positive, 1 if P <= q everywhere (the residual is empty). */
int32_t or_residual_probs(int32_t vocab, const double* P, const float* q, double* out);

/* ------------------------------------------------- tree verification --
 * Drafts arranged as a tree ("Accelerating Sonar through speculation",
 * section "EAGLE": several draft sequences explored as a tree, the longest
 * acceptable one kept, plus one token from the target).  The post gives no
 * acceptance rule for trees; the reading used here is recursive rejection
 * over each node's children: the children of node u are independent draws
 * from the draft distribution q_u at u; they are tried in index order, child
 * c_i is accepted with probability min(1, p_i(x)/q_u(x)) where p_0 = P_u and
 * p_{i+1} = max(p_i - q_u, 0) / Z_{i+1}, Z_{i+1} its sum; on acceptance the
 * walk continues at the child; when every child is rejected the emitted token
 * is drawn from max(p_{m-1} - q_u, 0); at a leaf it is drawn from P_u (the
 * bonus token).  A chain is exactly the linear rule of or_spec_verify.
 *
 * Request i owns nodes node_offsets[i] .. node_offsets[i+1]-1; local node 0
 * is the root (the state after the request's accepted prefix).  Node u's
 * target row is target_logits row node_offsets[i] + u; its history is the
 * request's history plus the tokens on the path from the root's child to u;
 * its Philox position is position[i] + depth(u).  Child c_i's uniform is
 * word i of stream OR_STREAM_ACCEPT at u's position; the residual at u uses
 * OR_STREAM_RESIDUAL and the bonus OR_STREAM_DRAW.  A greedy request (T = 0)
 * accepts the first child whose token is the argmax and otherwise emits the
 * argmax.  When a residual sums to zero before the last child, the walk ends
 * with the draw from P_u. */
typedef struct {
  int32_t num_requests, vocab, max_nodes;
  int64_t row_stride;
  int32_t dtype;
  const void* target_logits;     /* [sum n, row_stride]                          */
  const int32_t* node_offsets;   /* [R+1]                                        */
  const int32_t* parents;        /* [sum n] local index of the parent; the root's
                                    entry is not read; parent < child required  */
  const int32_t* node_tokens;    /* [sum n] draft token of each node (root: unused) */
  const float* draft_probs;      /* [sum n, draft_stride] q at each node         */
  int64_t draft_stride;
  or_params p;                   /* per request                                  */
} or_tree_in;

typedef struct {
  int32_t* out_tokens;           /* [R, max_nodes], -1 padded                    */
  int32_t* out_path;             /* [R, max_nodes] accepted local nodes, or NULL */
  int32_t* num_accepted;         /* [R]                                          */
  int32_t* status;               /* [R]                                          */
  uint8_t* sub_margin;           /* [R] or NULL                                  */
} or_tree_out;

/* Tree verification.  Status per request: node count outside [1, max_nodes]
 * or a parent not in [0, child) -> bad parameter; a node token outside
 * [0, V) -> bad index; otherwise the largest row status of its nodes.
 * Returns 0. */
int or_tree_verify(const or_tree_in* in, or_tree_out* out);

#ifdef __cplusplus
}
#endif
#endif
