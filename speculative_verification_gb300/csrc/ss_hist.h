// ss_hist.h -- host entry points of the bf16 histogram kernel (ss_hist.cu),
// called by the C ABI in ss_kernel.cu for bf16 logits.
#pragma once
#include <cuda_runtime.h>
#include <stdint.h>

#include "ss.h"

namespace ss {

// Largest draft length a verification call may declare.
constexpr int32_t kMaxDraft = 1 << 20;

// CTAs per row the histogram kernel uses for this vocabulary (bf16 only),
// or 0 when it does not take it (the general kernel does).
int hist_cluster_size(int32_t vocab, int32_t dtype);

// cudaError_t of the last failed launch on this thread.
int32_t hist_last_error();

// Batched sampling; arguments already validated by the caller.  With
// stall_polls > 0 every CTA also waits, for at most that many polls, on a
// barrier nothing completes (the bounded-wait self-test).
ss_status hist_sample(const ss_sample_args& args, cudaStream_t stream, uint32_t stall_polls = 0);

// Linear verification; `results` holds R * (max_draft + 1) int4 and
// `counters` 2R words that are zero on entry (the kernel leaves them at
// zero): R arrival counters, then R rejection words.
ss_status hist_verify(const ss_verify_args& args, int4* results, int32_t* counters, cudaStream_t stream);

}  // namespace ss
