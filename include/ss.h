/*
 * ss.h -- C ABI of the GB300 (sm_103a) batched sampling and speculative
 * verification library (libss.so).
 *
 * What is computed (all citations are to the pages this library implements):
 *   - SonicSampler: Unified Tile-Aware Kernels for LLM Sampling and Speculative
 *     Verification (abstract): one batched kernel applies, per request,
 *     grammar-constrained decoding, repetition / frequency / presence
 *     penalties, logit bias, temperature, top-k / top-p / min-p filtering and
 *     speculative verification, with a hierarchical two-stage top-k, and stays
 *     CUDA-Graph compatible.
 *   - FlashSampling (meineki.news), paragraphs 2-3: exact sampling as the argmax
 *     of logits plus Gumbel noise, reduced per vocabulary tile and then across
 *     tiles; the argmax decomposes over vocabulary partitions.
 *   - Accelerating Sonar through speculation (Perplexity blog), sections
 *     "Speculative decoding" and "Draft-target": drafts are accepted by
 *     comparing the full draft and target distributions, the longest accepted
 *     prefix is kept, and the target's logits after it give one more token
 *     (n drafts -> up to n+1 tokens).  The accept rule min(1, p/q) and the
 *     residual max(p - q, 0) are those of the post's first reference, "Fast
 *     inference from transformers via speculative decoding".
 *
 * Per row, in this order (the pages name the steps; the order and rounding are
 * this library's stated convention):
 *   z = logits row (fp32 or bf16, upcast exactly)
 *   penalties for each token seen c > 0 times in the row's history (and, for a
 *     verification target position j, in the drafts before j):
 *       z = z > 0 ? z / repetition : z * repetition
 *       z = z - frequency * c
 *       z = z - presence
 *   z = z + bias                        (bias ids of a row must be distinct)
 *   z = -inf where the grammar mask bit is 0
 *       (bit t & 31 of 32-bit word t >> 5, least significant bit first)
 *   temperature 0: greedy, token = lowest index of max z
 *   otherwise y = z * fp32(1 / temperature); order tokens by (y desc, index
 *   asc); K = shortest of the top-k prefix, the top-p prefix (mass in the
 *   top-k-renormalised distribution reaches top_p) and the min-p prefix
 *   (exp(y - y_max) >= min_p); token = argmax over K of y + g, with Gumbel
 *   noise g = -log(-log u) from Philox4x32-10:
 *     key (seed lo32, seed hi32), counter (t >> 2, position, row, stream),
 *     lane t & 3, u = (2 * (x >> 9) + 1) * 2^-24.
 *   stream 0 = draw / bonus token, 1 = accept uniform (t = 0), 2 = residual.
 * Verification of request i with k_i drafts x_0..x_{k_i-1}: for j = 0.. k_i-1
 *   accept x_j iff u_j * q_j(x_j) < P_j(x_j) (P_j = the distribution above at
 *   target position j); at the first rejection draw from max(P_j - q_j, 0)
 *   by argmax of log(P_j - q_j) + g (stream 2) over tokens with P_j > q_j; if
 *   all drafts are accepted, draw the bonus token from position k_i.
 *
 * Conventions of every entry point:
 *   - Pointers inside the argument structs are DEVICE pointers owned by the
 *     caller; the library keeps none of them after the call returns.
 *   - Calls are asynchronous on `stream`; results are valid once the stream
 *     reaches them.  They never synchronise, allocate or copy device to host,
 *     and launch a fixed number of kernels, so a call can be captured into a
 *     CUDA graph (the launch shape depends only on the host-side counts).
 *   - Host-detectable errors (NULL required pointer, bad sizes, misalignment,
 *     unsupported dtype, workspace too small) return an SS_ERR_* code and
 *     launch nothing.
 *   - Data-dependent errors are reported per row in out_status (SS_ROW_*),
 *     with token -1; a kernel never traps.
 *   - The logits pointer must be aligned to its element size.  Vocabulary
 *     slices that start on a 16-byte boundary (16-byte aligned pointer and
 *     row_stride * element size a multiple of 16) are staged with bulk TMA
 *     copies; others with plain loads, which is slower.
 *   - Every call that enqueues work opens one NVTX range named after the call
 *     (e.g. "ss_process_sample"), so that a timeline or a profiler's NVTX
 *     filter attributes the launches; without a tool attached it costs a few
 *     nanoseconds on the host.
 */
#ifndef SS_H
#define SS_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t; NULL is the legacy default stream. */
typedef struct CUstream_st* ss_stream_t;

typedef enum {
  SS_OK = 0,
  SS_ERR_INVALID_ARG = 1,  /* NULL pointer, bad size or stride, misaligned ptr */
  SS_ERR_UNSUPPORTED = 2,  /* vocabulary too large for one thread-block cluster */
  SS_ERR_CUDA = 3,         /* a CUDA runtime call failed; ss_last_cuda_error() */
  SS_ERR_WORKSPACE = 4,    /* workspace NULL or smaller than ss_workspace_size */
  SS_ERR_SCRATCH_LIMIT = 5 /* ss_spec_verify_noalloc: batch needs more than
                              SS_NOALLOC_SCRATCH_BYTES of scratch            */
} ss_status;

typedef enum { SS_DTYPE_F32 = 0, SS_DTYPE_BF16 = 1 } ss_dtype;

/* Per-row status written to out_status; when several apply the larger wins. */
enum {
  SS_ROW_OK = 0,
  SS_ROW_EMPTY_SET = 1,  /* every token is masked out                               */
  SS_ROW_NONFINITE = 2,  /* an allowed processed logit is NaN or +inf               */
  SS_ROW_BAD_INDEX = 3,  /* history / draft / bias id outside [0, V) or duplicate bias id */
  SS_ROW_BAD_PARAM = 4,  /* temperature < 0 or non-finite, top_k < 0, top_p <= 0 or NaN,
                            min_p outside [0, 1], repetition <= 0 or non-finite,
                            frequency / presence / bias value non-finite, negative list
                            length, position outside [0, 2^32 - 1 - k], k > max_draft */
  SS_ROW_TIMEOUT = 5,    /* a bounded wait for an asynchronous copy gave up         */
  SS_ROW_LIMIT = 6,      /* an implementation capacity: more distinct penalised /
                            biased tokens in one vocabulary slice than its table
                            holds (SS_MAX_PATCHED), or (bf16 logits) a cut the
                            kernel cannot place within its slot window or gather
                            buffers; never seen on the benchmark workloads       */
  SS_ROW_UNSUPPORTED = 7 /* vocabulary-sharded path only: top-p or min-p without
                            top-k, or top_k above the records' list capacity      */
};

/* Distinct penalised or biased tokens one vocabulary slice can hold. */
#define SS_MAX_PATCHED 1024

/* Per-row (process_sample) or per-request (spec_verify) parameters.  Arrays
 * have one entry per row/request; an optional array left NULL switches the
 * feature off for every row. */
typedef struct {
  const float* temperature;     /* required; 0 = greedy                          */
  const int32_t* top_k;         /* NULL or <= 0 or >= allowed count: off         */
  const float* top_p;           /* NULL or >= 1: off                             */
  const float* min_p;           /* NULL or 0: off                                */
  const float* repetition;      /* NULL: 1 (off)                                 */
  const float* frequency;       /* NULL: 0 (off)                                 */
  const float* presence;        /* NULL: 0 (off)                                 */
  const int32_t* hist_offsets;  /* [n+1] CSR offsets into hist_ids, or NULL      */
  const int32_t* hist_ids;      /* token history used by the three penalties     */
  const int32_t* bias_offsets;  /* [n+1] CSR offsets into bias_ids/vals, or NULL */
  const int32_t* bias_ids;
  const float* bias_vals;
  const int32_t* bitmask;       /* [n, bitmask_stride] allow bits, or NULL       */
  int64_t bitmask_stride;       /* words per row, >= ceil(V / 32)                */
  const uint8_t* use_bitmask;   /* NULL: every row uses its mask row             */
  const uint64_t* seed;         /* required: Philox key                          */
  const int64_t* position;      /* required: Philox counter word 1               */
  const uint32_t* row_id;       /* Philox counter word 2; NULL: the row's (request's)
                                   index in the call.  A stable id per request
                                   keeps its draws independent of its slot in the
                                   batch and of how a batch is split over GPUs. */
} ss_params;

/* ss_sample_args.flags / ss_verify_args.flags (0 = none). */
#define SS_SAMPLE_OVERLAP_PREVIOUS 1 /* the call may overlap the call before it (below) */
#define SS_VERIFY_OVERLAP_PREVIOUS 1 /* the same for ss_spec_verify / ss_spec_verify_noalloc */
#define SS_TREE_OVERLAP_PREVIOUS 1   /* the same for ss_tree_verify (ss_tree_args.flags) */

/* ss_process_sample: one token per row.  Row r is logits + r * row_stride. */
typedef struct {
  int32_t num_rows;
  int32_t vocab;                /* V >= 1                                         */
  int64_t row_stride;           /* elements; 0 (all rows alias row 0) or >= V     */
  int32_t dtype;                /* ss_dtype                                       */
  const void* logits;
  ss_params params;             /* indexed by row                                 */
  int32_t* out_token;           /* [num_rows], -1 when out_status != SS_ROW_OK    */
  int32_t* out_status;          /* [num_rows]                                     */
  int32_t* out_kept;            /* [num_rows] |K| (1 greedy, 0 error), or NULL    */
  float* debug_processed;       /* [num_rows, V] processed logits y (z for greedy
                                   rows, -inf where masked), or NULL              */
  int32_t flags;                /* 0, or SS_SAMPLE_OVERLAP_PREVIOUS: the call may
                                   begin while the kernel before it on the stream
                                   -- a bf16 sampling or verification call of this
                                   library -- is still
                                   running (programmatic dependent launch): it
                                   reads its inputs at once and orders only its
                                   writes after that call.  Set it only when no
                                   input of this call is written by that call
                                   (its out_token / out_status / out_kept /
                                   debug_processed); back-to-back calls over
                                   independent batches then overlap each other's
                                   first and last rows.  Honoured by bf16
                                   ss_process_sample; other bits are invalid;
                                   the other entry points taking this struct
                                   ignore it. */
} ss_sample_args;

/* ss_spec_verify: request i owns target rows draft_offsets[i] + i + j,
 * j = 0..k_i, k_i = draft_offsets[i+1] - draft_offsets[i] (0 allowed: then the
 * call returns exactly the ss_process_sample draw of that row). */
typedef struct {
  int32_t num_requests;
  int32_t vocab;
  int32_t max_draft;            /* upper bound of every k_i                       */
  int64_t row_stride;           /* elements between target rows (>= V)            */
  int32_t dtype;
  const void* target_logits;    /* [sum(k_i + 1), row_stride]                      */
  const int32_t* draft_offsets; /* [R+1], non-decreasing, draft_offsets[0] = 0    */
  const int32_t* draft_tokens;  /* [sum k_i]                                      */
  const float* draft_probs;     /* [sum k_i, draft_stride] q_j over the vocabulary */
  int64_t draft_stride;         /* elements, >= V                                 */
  ss_params params;             /* indexed by request                             */
  int32_t* out_tokens;          /* [R, max_draft + 1]: accepted drafts, then the
                                   residual or bonus token, then -1              */
  int32_t* out_num_accepted;    /* [R] in [0, k_i]; tokens emitted = this + 1     */
  int32_t* out_status;          /* [R] worst row status of the request            */
  int32_t* out_kept;            /* [sum(k_i + 1)] |K| per target row, or NULL     */
  float* debug_processed;       /* [sum(k_i + 1), V], or NULL                     */
  int32_t flags;                /* 0, or SS_VERIFY_OVERLAP_PREVIOUS: on bf16
                                   logits the call may begin while the kernel
                                   before it on the stream -- a bf16 sampling or
                                   verification call of this library -- is still
                                   running, as SS_SAMPLE_OVERLAP_PREVIOUS; its
                                   workspace is used only once that call has
                                   finished.  Set it only when no input of this
                                   call is an output of that call.  Other bits
                                   are invalid; ss_spec_verify_noalloc ignores
                                   it (it clears its scratch before the launch). */
  int32_t num_target_rows;      /* 0, or the number of target rows, sum(k_i + 1)
                                   with a k_i outside [0, max_draft] counted as
                                   0.  On bf16 logits the launch may then have
                                   one cluster per target row instead of one per
                                   (request, position up to max_draft): the
                                   library takes it when the full launch's idle
                                   clusters (positions past a request's drafts)
                                   would outnumber the rows past position 0,
                                   whose clusters find their request and
                                   position from draft_offsets.  Must be 0 or in
                                   [num_requests, num_requests * (max_draft +
                                   1)], else SS_ERR_INVALID_ARG; on bf16 logits a
                                   value in that range that is not the sum makes
                                   every request report SS_ROW_BAD_PARAM (tokens
                                   -1, none accepted; out_kept and
                                   debug_processed are not written), whichever
                                   launch is taken.  The fp32 path ignores it. */
} ss_verify_args;

/* Bytes of caller-owned device workspace ss_spec_verify needs for up to
 * `max_requests` requests with up to `max_draft` drafts each: per-position
 * results (16 B each) at its start, and two words per request at its end (an
 * arrival counter and a rejection word).  Returns 0 for a negative argument or
 * max_draft above 2^20.  A buffer sized for (R, k) serves any call with at
 * most R requests and k drafts, in any order of shapes: the per-request words
 * are placed from the buffer's end, so no shape puts them where another shape
 * left its results. */
size_t ss_workspace_size(int32_t max_requests, int32_t max_draft);

/* Zero a workspace before its first use (cudaMemsetAsync on `stream`).  Every
 * ss_spec_verify call leaves its per-request words at zero again, so this is
 * needed once per buffer.  Calls sharing one workspace must not overlap in
 * time. */
ss_status ss_workspace_init(void* workspace, size_t workspace_bytes, ss_stream_t stream);

/* Batched sampling.  bf16 logits: one launch of the histogram kernel (one
 * thread-block cluster per row).  fp32 logits: with 16 to 4096 rows and a
 * vocabulary whose cluster can double (ss_cluster_size <= 4), the rows with a
 * top-p cut and no top-k run on a second launch with twice the CTAs per row,
 * on a library-owned stream (one per host thread and device, created by the
 * first such call) forked from and joined back into `stream` with events;
 * otherwise one launch.  Either way the call is asynchronous on `stream`,
 * capturable in a CUDA graph, and its results do not depend on the split.  A
 * capture that starts before the thread's first such call records the single
 * launch. */
ss_status ss_process_sample(const ss_sample_args* args, ss_stream_t stream);

/* Self-test of the kernels' bounded waits (no counterpart in the pages; it
 * exists so that the timeout path can be exercised without a fault).  Runs
 * ss_process_sample on bf16 logits with one extra wait in every CTA, on a
 * barrier that nothing completes, given up after `polls` polls (each poll
 * sleeps a hardware-chosen interval, so keep it small: 100 to 1000).  Every
 * valid row then reports SS_ROW_TIMEOUT and token -1; the context stays
 * usable.  SS_ERR_UNSUPPORTED for fp32 logits or polls == 0; the other
 * errors are ss_process_sample's. */
ss_status ss_selftest_wait_timeout(const ss_sample_args* args, uint32_t polls, ss_stream_t stream);

/* Batched speculative verification; one kernel launch.  The workspace must
 * have been zeroed once (ss_workspace_init). */
ss_status ss_spec_verify(const ss_verify_args* args, void* workspace, size_t workspace_bytes,
                         ss_stream_t stream);

/* Size of the static device scratch behind ss_spec_verify_noalloc (1 MiB):
 * enough for ss_workspace_size(R, max_draft), e.g. 7000 requests with 7
 * drafts each. */
#define SS_NOALLOC_SCRATCH_BYTES (1u << 20)

/* ss_spec_verify_noalloc: ss_spec_verify without a caller workspace and
 * without allocating.  (The pages describe no such call; it exists for
 * callers that cannot allocate device memory -- e.g. a serving engine that
 * hands all GPU memory to its own pool at start-up, or a plugin whose host
 * interface provides no allocator -- and so cannot pass a workspace.)
 *
 * The scratch is one file-scope device array of SS_NOALLOC_SCRATCH_BYTES in
 * this library; every GPU that uses the library holds it until the process
 * exits.  A batch whose ss_workspace_size(num_requests, max_draft) exceeds it
 * is rejected with SS_ERR_SCRATCH_LIMIT and nothing is launched.  The call
 * itself allocates nothing: no cudaMalloc, cudaFree or allocating library
 * routine.
 *   - The first call on a device looks up the array's device address (once
 *     per device, with that device current); make that first call before any
 *     stream capture.
 *   - Every call clears the per-request words with cudaMemsetAsync on
 *     `stream`, then launches the verification kernel; the results are
 *     identical to ss_spec_verify's.
 *   - All calls on one device share the array: calls that overlap on the GPU
 *     (different streams, or host threads not ordered by a stream) race and
 *     produce undefined results.  Serialise them.
 * Arguments, outputs and the other errors are those of ss_spec_verify. */
ss_status ss_spec_verify_noalloc(const ss_verify_args* args, ss_stream_t stream);

/* ---------------------------------------------------- tree verification --
 * Drafts arranged as a tree ("Accelerating Sonar through speculation",
 * section "EAGLE": a draft model explores several sequences as a tree, the
 * longest acceptable one is kept and the target adds one more token).  The
 * post gives no acceptance rule for trees; this call implements recursive
 * rejection over each node's children, which reduces to the linear rule of
 * ss_spec_verify on a chain:
 *   - request i owns nodes node_offsets[i] .. node_offsets[i+1] - 1, n_i of
 *     them (1 <= n_i <= max_nodes); local node 0 is the root, the state after
 *     the request's accepted prefix; every other node u carries the draft
 *     token node_tokens[node_offsets[i] + u] and hangs under local node
 *     parents[node_offsets[i] + u], which must be smaller than u (the root's
 *     parent entry is not read);
 *   - node u's target row (target_logits row node_offsets[i] + u) is the
 *     target's next-token distribution after the tokens on the path from the
 *     root to u; its history is the request's history plus those tokens, its
 *     Philox position is position[i] + depth(u);
 *   - the children of u are taken to be independent draws from the draft
 *     distribution q_u (draft_probs row node_offsets[i] + u; leaves' rows are
 *     not read).  They are tried in index order: child c (the c-th child of
 *     u) is accepted with probability min(1, p_c(x)/q_u(x)), p_0 = P_u,
 *     p_{c+1} = max(p_c - q_u, 0) / Z (Z its sum), by u * q_u(x) < p_c(x) with
 *     u the Philox uniform of word c, stream 1, at u's position.  On
 *     acceptance the walk continues at the child.  When every child is
 *     rejected, the emitted token is the Gumbel-max draw (stream 2) from
 *     max(p_{m-1} - q_u, 0); when a residual sums to zero before the last
 *     child, it is the stream-0 draw from P_u.  At a leaf it is the stream-0
 *     draw from P_u (the bonus token).  A greedy request (temperature 0)
 *     accepts the first child carrying the argmax and otherwise emits it.
 * Outputs: out_tokens[i, 0 .. num_accepted[i]] the accepted drafts then the
 * final token, -1 after; out_path (or NULL) the accepted nodes' local
 * indices, -1 after; out_status the worst row status of the request (a node
 * count outside [1, max_nodes] or a parent not smaller than its child gives
 * SS_ROW_BAD_PARAM, a node token outside [0, V) SS_ROW_BAD_INDEX).
 * The workspace is that of ss_spec_verify for (num_requests, max_nodes - 1),
 * zeroed once; one kernel launch, asynchronous on `stream`. */
#define SS_TREE_MAX_NODES 64
typedef struct {
  int32_t num_requests;
  int32_t vocab;
  int32_t max_nodes;            /* in [1, SS_TREE_MAX_NODES], >= every n_i        */
  int64_t row_stride;           /* elements between target rows (>= V)            */
  int32_t dtype;
  const void* target_logits;    /* [sum n_i, row_stride]                           */
  const int32_t* node_offsets;  /* [R+1], non-decreasing, node_offsets[0] = 0     */
  const int32_t* parents;       /* [sum n_i] local parent index                   */
  const int32_t* node_tokens;   /* [sum n_i] draft token of each node             */
  const float* draft_probs;     /* [sum n_i, draft_stride] q at each node         */
  int64_t draft_stride;         /* elements, >= V                                 */
  ss_params params;             /* indexed by request                             */
  int32_t* out_tokens;          /* [R, max_nodes]                                 */
  int32_t* out_path;            /* [R, max_nodes], or NULL                        */
  int32_t* out_num_accepted;    /* [R]                                            */
  int32_t* out_status;          /* [R]                                            */
  int32_t* out_kept;            /* [sum n_i] |K| per node row, or NULL            */
  float* debug_processed;       /* [sum n_i, V], or NULL                          */
  int32_t flags;                /* 0, or SS_TREE_OVERLAP_PREVIOUS: the call may
                                   begin while the kernel before it on the stream
                                   -- a tree verification call of this library --
                                   is still running (programmatic dependent
                                   launch); its outputs, debug rows and workspace
                                   are written only once that call has finished.
                                   Set it only when no input of this call is an
                                   output of that call.  Other bits are invalid. */
  int32_t num_nodes_total;      /* 0, or the number of target rows, sum n_i
                                   (node_offsets[R]) with an n_i outside [1,
                                   max_nodes] counted as 1.  When the launch
                                   orders its node slots, costliest first (16 to
                                   4096 slots, R * max_nodes), it then stops at
                                   that many clusters instead of one per slot:
                                   the slots without a node come last in that
                                   order.  Must be 0 or in [num_requests,
                                   num_requests * max_nodes], else
                                   SS_ERR_INVALID_ARG; a value in that range
                                   that is not the sum makes every request
                                   report SS_ROW_BAD_PARAM (tokens and path -1,
                                   none accepted; out_kept and debug_processed
                                   are not written), whatever the launch. */
} ss_tree_args;

ss_status ss_tree_verify(const ss_tree_args* args, void* workspace, size_t workspace_bytes, ss_stream_t stream);

/* After a verification call, the next step's inputs without a device-to-host
 * copy (Accelerating Sonar through speculation, "MTP schedule for a single
 * token": once the target's inputs are shifted in, a kernel places the next
 * target tokens into their slots, avoiding the GPU-to-CPU synchronisation on
 * the accepted lengths).  For each request i whose status[i] is SS_ROW_OK,
 * its num_accepted[i] + 1 emitted tokens out_tokens[i * (max_draft + 1) +
 * 0 .. num_accepted[i]] (the accepted drafts and the residual or bonus token)
 * are appended to tokens[i * capacity + seq_len[i] ...]; seq_len[i] and
 * position[i] advance by that count and next_token[i] becomes the last of
 * them; commit_status[i] = SS_ROW_OK.  A request whose tokens would not fit
 * in `capacity` (or whose num_accepted lies outside [0, max_draft], or whose
 * seq_len is negative) is left unchanged with commit_status SS_ROW_LIMIT; one whose
 * status is not SS_ROW_OK is left unchanged with that status copied.  All
 * pointers are device pointers; tokens is [num_requests, capacity] int32,
 * seq_len int32, position int64, next_token and commit_status int32.
 * Asynchronous on `stream`; graph-capturable. */
ss_status ss_commit_accepted(int32_t num_requests, int32_t max_draft, const int32_t* out_tokens,
                             const int32_t* num_accepted, const int32_t* status, int32_t* tokens, int32_t capacity,
                             int32_t* seq_len, int64_t* position, int32_t* next_token, int32_t* commit_status,
                             ss_stream_t stream);

/* ---------------------------------------------------- vocabulary shards --
 * Sampling when each GPU holds only a slice of the vocabulary of every row
 * (a tensor-parallel LM head).  The draw is a Gumbel-max with noise keyed by
 * the global token id, and the maximum of per-partition maxima is the maximum
 * (FlashSampling news page: per-tile maxima, then a cross-tile reduction), so
 * a plain row needs one (score, token) pair per shard; a top-k row needs each
 * shard's top-k (two-stage top-k, SonicSampler abstract), after which the
 * merge applies top-p and min-p to the merged top-k exactly as the unsharded
 * call does.  The result is identical to ss_process_sample on the whole rows.
 * Rows with top-p or min-p but without top-k would need the whole
 * distribution and report SS_ROW_UNSUPPORTED.
 *
 * ss_sample_shard: args->vocab is the whole vocabulary V; args->logits holds
 * tokens [vocab_offset, vocab_offset + shard_len) of every row (row r at
 * logits + r * row_stride elements, row_stride >= shard_len or 0);
 * vocab_offset is a multiple of 32; history, bias and mask ids are global
 * (each shard applies the ones it holds).  out_token / out_status / out_kept
 * and debug_processed are not used (debug_processed must be NULL).  Writes
 * one record of ss_shard_record_bytes(list_cap) bytes per row to `records`
 * (device, 8-byte aligned, caller-owned); list_cap in [1, SS_SHARD_MAX_LIST]
 * bounds the top_k the rows may use.
 *
 * ss_merge_shards: the records of num_shards (1..8) shards that together
 * cover [0, V) exactly once, in any order (`records` is a host array of
 * device pointers); args supplies num_rows, the same params and the outputs
 * (out_token, out_status, out_kept as for ss_process_sample); logits is not
 * read.  Both calls are asynchronous on `stream`. */
#define SS_SHARD_MAX_LIST 1024
size_t ss_shard_record_bytes(int32_t list_cap);
ss_status ss_sample_shard(const ss_sample_args* args, int32_t vocab_offset, int32_t shard_len, int32_t list_cap,
                          void* records, ss_stream_t stream);
ss_status ss_merge_shards(const ss_sample_args* args, int32_t num_shards, void* const* records, int32_t list_cap,
                          ss_stream_t stream);

/* ---------------------------------- shards: top-p / min-p without top-k --
 * Rows whose kept set needs the whole distribution (top-p and / or min-p
 * without a top-k; also greedy and unfiltered rows) over vocabulary shards,
 * in four rounds.  Round i (0..3) is one ss_shard_round call per shard, then
 * one ss_merge_round call over every shard's records; on P GPUs the records
 * of a round are all-gathered before its merge.  What the rounds carry (the
 * FlashSampling news page's grouped variants need this much because a top-p
 * cut depends on the whole row's mass):
 *   0. the shard's largest processed logit, greedy argument, allowed count
 *      and status                    -> merge: the row maximum m; greedy and
 *                                       failed rows are finished here
 *   1. (top-p rows) the shard's fixed-point mass sum trunc(exp(y-m) 2^40)
 *      and a count / mass histogram over 1024 buckets of y below m
 *                                    -> merge: S, ceil(p S), the cut's bucket
 *   2. (top-p rows) the shard's tokens in that bucket (at most 1024)
 *                                    -> merge: the exact cut item, or the
 *                                       min-p threshold when that is shorter
 *   3. the shard's count of kept tokens and its best y + Gumbel noise
 *                                    -> merge: token, status and |K| to
 *                                       out_token / out_status / out_kept
 * The outputs equal ss_process_sample's on the whole rows.  args as for
 * ss_sample_shard (logits hold tokens [vocab_offset, vocab_offset +
 * shard_len) of every row, row_stride >= shard_len; ids are global).  Rows
 * with a top-k cut are left to ss_sample_shard / ss_merge_shards: the rounds
 * do not write their outputs, so a batch mixing both kinds runs the list
 * path's merge first, then the four rounds.  A row whose cut bucket holds
 * more than 1024 tokens in one shard reports SS_ROW_LIMIT.  records: ss_shard_round_record_bytes() per row, 16-byte
 * aligned, one buffer per shard (reused by every round); state:
 * ss_shard_round_state_bytes(num_rows), written by the merges and read by
 * the next round's shard calls.  All calls are asynchronous on `stream`. */
size_t ss_shard_round_record_bytes(void);
size_t ss_shard_round_state_bytes(int32_t num_rows);
ss_status ss_shard_round(const ss_sample_args* args, int32_t vocab_offset, int32_t shard_len, int32_t round,
                         const void* state, void* records, ss_stream_t stream);
ss_status ss_merge_round(const ss_sample_args* args, int32_t num_shards, void* const* records, int32_t round,
                         void* state, ss_stream_t stream);

/* ------------------------------------------------ fused LM head + draw --
 * The LM-head matrix multiply fused with the draw (FlashSampling news page:
 * the sample is taken inside the matrix multiply that produces the logits,
 * per-tile maxima of logit + Gumbel noise reduced across tiles, so the [B, V]
 * logits are never written).  logits[r, t] = sum_k hidden[r, k] * weight[t, k]
 * with bf16 inputs and fp32 accumulation on the tensor cores; then exactly
 * the sampling kernel's draw without filters: y = logit * fp32(1/T),
 * token = argmax over t of y + g(seed, row id, position, t) (stream 0),
 * temperature 0 = the lowest id of the largest logit.  Penalties, bias,
 * masks and the top-k / top-p / min-p filters need the materialised row:
 * use ss_process_sample for them.
 *   batch in [1, 128]; hidden a multiple of 64; hidden_states [batch, hidden]
 *   and weight [vocab, hidden] bf16, row-major, 16-byte aligned.
 *   scratch: device memory of ss_fused_scratch_bytes(batch) bytes, 8-byte
 *   aligned, cleared by the call (calls sharing it must not overlap).
 *   out_status: SS_ROW_OK, SS_ROW_BAD_PARAM (temperature < 0 or non-finite,
 *   position outside [0, 2^32 - 1]), SS_ROW_NONFINITE (a NaN / inf logit),
 *   SS_ROW_TIMEOUT (a bounded wait inside the kernel gave up).
 *   debug_logits: [batch, vocab] fp32 logits for tests, or NULL (slow). */
typedef struct {
  int32_t batch, hidden, vocab;
  const void* hidden_states;
  const void* weight;
  const float* temperature;     /* [batch] */
  const uint64_t* seed;         /* [batch] */
  const int64_t* position;      /* [batch] */
  const uint32_t* row_id;       /* [batch] or NULL: the row's index */
  void* scratch;
  size_t scratch_bytes;
  int32_t* out_token;           /* [batch] */
  int32_t* out_status;          /* [batch] */
  float* debug_logits;
} ss_fused_args;
size_t ss_fused_scratch_bytes(int32_t batch);
ss_status ss_fused_lmhead_sample(const ss_fused_args* args, ss_stream_t stream);

/* Cluster size (CTAs per vocabulary row) the kernels use for this vocabulary
 * and dtype, or 0 if unsupported.  A row is split over at most 8 CTAs of at
 * most 61,440 tokens and 160 KiB each, whose slice and working tables must
 * fit one CTA's 227 KiB of shared memory, so the largest vocabulary is
 * 491,520 for bf16 and 321,536 for f32; larger ones return
 * SS_ERR_UNSUPPORTED. */
int32_t ss_cluster_size(int32_t vocab, int32_t dtype);

/* The cudaError_t of the last SS_ERR_CUDA on this thread. */
int32_t ss_last_cuda_error(void);

const char* ss_status_string(ss_status status);
const char* ss_version(void);

#ifdef __cplusplus
}
#endif
#endif /* SS_H */
