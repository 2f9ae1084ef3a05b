// ss_fused.cu -- the LM-head matrix multiply fused with the exact draw.
//
// FlashSampling (news page, paragraphs 2-3): sampling is folded into the
// matrix multiply that produces the logits; each tile of logits is turned
// into its own maximum of "logit + Gumbel noise" (and the token holding it)
// in the epilogue, and the maxima of the tiles are reduced across tiles, so
// the [B, V] logits are never written to or read back from memory.  The
// result is the same Gumbel-max draw as the sampling kernel's: noise keyed by
// (seed, row id, position, token) through Philox4x32-10, y = logit * (1/T),
// temperature 0 = greedy (lowest id of the largest logit).
//
// sm_103a design: one persistent CTA per SM walks vocabulary tiles of 128
// tokens.  Warp 0 streams 64-wide K slices of the hidden states ([B, d]:
// 64 rows when B <= 64, the rest of the 128-row tile kept zero) and of the
// tile's weight rows
// with 2-D tensor copies (128-byte swizzle) into a 7-stage shared-memory
// ring; warp 1 issues tcgen05.mma (M = 128 rows, N = 128 tokens, K = 16,
// bf16 in, fp32 accumulate) into one of two tensor-memory accumulators;
// warps 4-11 (two per 32-lane quarter of tensor memory, each on half of the
// columns) read the finished accumulator with tcgen05.ld, add the noise and
// keep each row's best, while
// the next tile accumulates into the other buffer.  Rows end with one 64-bit
// atomic maximum per CTA on (order key of the score, inverted token id).
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>
#include <stdint.h>
#include <string.h>

#include "ss.h"
#include "ss_nvtx.h"
#include "ss_philox.cuh"
#include "ss_ptx.cuh"

namespace ss {
void set_last_cuda_error(int32_t e);  // ss_kernel.cu: the value ss_last_cuda_error() reports
}

namespace ssf {
using namespace ss;

constexpr int kBM = 128;                     // batch rows per MMA (rows past the batch are zero)
constexpr int kBN = 128;                     // vocabulary tokens per tile
constexpr int kBK = 64;                      // K per stage: one 128-byte swizzle span of bf16
constexpr int kUK = 16;                      // K of one tcgen05.mma for 16-bit inputs
constexpr int kStages = 7;
constexpr int kTileA = kBM * kBK * 2;        // 16 KiB
constexpr int kTileB = kBN * kBK * 2;        // 16 KiB
constexpr int kStageBytes = kTileA + kTileB;
constexpr int kEpiWarps = 8;                 // two per tensor-memory lane quarter, each half of the columns
constexpr int kThreadsF = 128 + 32 * kEpiWarps;
constexpr int kTmemCols = 2 * kBN;           // two fp32 accumulators of 128 columns
constexpr uint32_t kPolls = 1u << 24;        // bounded waits
constexpr size_t kSmemBytes = static_cast<size_t>(kStages) * kStageBytes + 1024;  // + alignment slack

struct FArgs {
  int32_t batch, hidden, vocab;
  const float* temperature;
  const uint64_t* seed;
  const int64_t* position;
  const uint32_t* row_id;
  unsigned long long* best;  // [batch] packed (score key, ~token)
  int32_t* flags;            // [batch] bit 0: non-finite logit seen, bit 1: bad parameters
  int32_t* error;            // [1] a bounded wait gave up
  float* debug_logits;       // [batch, vocab] or NULL
  int32_t a_rows;            // rows of hidden states each copy brings (64 when batch <= 64, else 128)
};

__device__ __forceinline__ float f_neg_inf() { return __int_as_float(0xff800000); }

__device__ __forceinline__ uint32_t f_order_key(float y) {
  const uint32_t b = __float_as_uint(y + 0.0f);
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

__device__ __forceinline__ bool wait_bounded(uint64_t* bar, uint32_t parity, int32_t* error) {
  for (uint32_t i = 0; i < kPolls; ++i)
    if (mbar_try_wait(bar, parity)) return true;
  atomicExch(error, 1);
  return false;
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

// 2-D tiled tensor copy global -> shared (x = innermost coordinate, in
// elements; a multiple of 8 for 16-bit data), completion on `bar`.
__device__ __forceinline__ void tma_2d(void* dst, const CUtensorMap* map, int32_t x, int32_t y, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
          smem_addr(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_addr(bar))
      : "memory");
}

// Shared-memory matrix descriptor of a K-major tile whose rows are 128 bytes
// (64 bf16) with the 128-byte swizzle, as the tensor copy writes it: 8-row
// groups 1024 bytes apart (stride byte offset), descriptor version 1,
// layout type 2 (128-byte swizzle).  Moving 16 elements along K inside the
// swizzle span advances the start address by 32 bytes.
__device__ __forceinline__ uint64_t smem_desc(uint32_t addr) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((addr & 0x3ffffu) >> 4);          // start address
  d |= static_cast<uint64_t>(1) << 16;                          // leading byte offset (unused when swizzled)
  d |= static_cast<uint64_t>(1024 >> 4) << 32;                  // stride byte offset
  d |= static_cast<uint64_t>(1) << 46;                          // version
  d |= static_cast<uint64_t>(2) << 61;                          // 128-byte swizzle
  return d;
}

// Instruction descriptor of kind::f16: fp32 accumulator, bf16 A and B, both
// K-major, N = kBN, M = kBM.
constexpr uint32_t kIdesc = (1u << 4) | (1u << 7) | (1u << 10) | (static_cast<uint32_t>(kBN >> 3) << 17) |
                            (static_cast<uint32_t>(kBM >> 4) << 24);

__device__ __forceinline__ void umma(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a), "l"(b), "r"(kIdesc), "r"(accumulate)
      : "memory");
}

// Arrive on `bar` once every tcgen05.mma this thread issued so far is done.
__device__ __forceinline__ void umma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_addr(bar))
               : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// 32 consecutive fp32 columns of this warp's 32 tensor-memory lanes.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&v)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
      "%15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
      : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]), "=r"(v[8]),
        "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15]), "=r"(v[16]),
        "=r"(v[17]), "=r"(v[18]), "=r"(v[19]), "=r"(v[20]), "=r"(v[21]), "=r"(v[22]), "=r"(v[23]), "=r"(v[24]),
        "=r"(v[25]), "=r"(v[26]), "=r"(v[27]), "=r"(v[28]), "=r"(v[29]), "=r"(v[30]), "=r"(v[31])
      : "r"(taddr)
      : "memory");
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

__global__ void __launch_bounds__(kThreadsF, 1)
    ss_fused_kernel(const __grid_constant__ CUtensorMap tm_h, const __grid_constant__ CUtensorMap tm_w, const FArgs a) {
  extern __shared__ uint8_t fsmem_raw[];
  __shared__ __align__(8) uint64_t full[kStages], empty[kStages], tfull[2], tempty[2];
  __shared__ uint32_t tmem_slot;
  uint8_t* ring = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(fsmem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int num_tiles = (a.vocab + kBN - 1) / kBN;
  const int k_steps = a.hidden / kBK;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(full + s, 1);
      mbar_init(empty + s, 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(tfull + i, 1);
      mbar_init(tempty + i, 32 * kEpiWarps);
    }
    fence_barrier_init();
  }
  if (a.a_rows < kBM) {
    // the copies fill rows [0, a_rows) of each stage's A tile; the rest stays
    // zero for the whole launch (the MMA reads 128 rows)
    for (int s = 0; s < kStages; ++s) {
      uint4* z = reinterpret_cast<uint4*>(ring + s * kStageBytes + a.a_rows * kBK * 2);
      for (int i = threadIdx.x; i < (kBM - a.a_rows) * kBK * 2 / 16; i += kThreadsF) z[i] = make_uint4(0u, 0u, 0u, 0u);
    }
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // visible to the tensor cores
  }
  if (warp == 1) {  // the whole warp allocates the accumulators
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_addr(&tmem_slot)),
                 "r"(kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    tc_fence_before();
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_slot;

  if (warp == 0) {
    if (lane == 0) {  // producer: tensor copies into the ring
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      for (int tile = blockIdx.x; tile < num_tiles && ok; tile += gridDim.x)
        for (int k = 0; k < k_steps && ok; ++k) {
          ok = wait_bounded(empty + stage, phase ^ 1u, a.error);
          if (!ok) break;
          uint8_t* sa = ring + stage * kStageBytes;
          mbar_arrive_expect_tx(full + stage, static_cast<uint32_t>(a.a_rows * kBK * 2 + kTileB));
          tma_2d(sa, &tm_h, k * kBK, 0, full + stage);
          tma_2d(sa + kTileA, &tm_w, k * kBK, tile * kBN, full + stage);
          if (++stage == kStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
    }
  } else if (warp == 1) {
    if (lane == 0) {  // MMA issuer
      int stage = 0, acc = 0;
      uint32_t phase = 0, acc_phase = 0;
      bool ok = true;
      for (int tile = blockIdx.x; tile < num_tiles && ok; tile += gridDim.x) {
        ok = wait_bounded(tempty + acc, acc_phase ^ 1u, a.error);
        if (!ok) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem + static_cast<uint32_t>(acc * kBN);
        for (int k = 0; k < k_steps; ++k) {
          ok = wait_bounded(full + stage, phase, a.error);
          if (!ok) break;
          tc_fence_after();
          const uint32_t sa = smem_addr(ring + stage * kStageBytes);
#pragma unroll
          for (int kk = 0; kk < kBK / kUK; ++kk)
            umma(d_tmem, smem_desc(sa + kk * 32), smem_desc(sa + kTileA + kk * 32), (k > 0 || kk > 0) ? 1u : 0u);
          umma_commit(empty + stage);  // the stage is free once these MMAs are done
          if (++stage == kStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
        umma_commit(tfull + acc);  // the accumulator is complete
        if (++acc == 2) {
          acc = 0;
          acc_phase ^= 1u;
        }
      }
    }
  } else if (warp >= 4) {  // epilogue: one batch row per thread, half of each tile's columns
    const int q = warp & 3;                       // tensor-memory lane quarter (warp % 4)
    const int half = (warp - 4) >> 2;             // which 64 columns of the tile
    constexpr int kHalfCols = kBN / 2;
    const int r = q * 32 + lane;
    const bool live = r < a.batch;
    float inv_t = 1.0f;
    bool greedy = true;
    uint64_t seed = 0;
    uint32_t rowid = 0, pos = 0;
    if (live) {
      const float T = a.temperature[r];
      greedy = (T == 0.0f);
      inv_t = greedy ? 1.0f : __fdiv_rn(1.0f, T);
      seed = a.seed[r];
      rowid = a.row_id ? a.row_id[r] : static_cast<uint32_t>(r);
      pos = static_cast<uint32_t>(a.position[r]);
    }
    const uint32_t key0 = static_cast<uint32_t>(seed), key1 = static_cast<uint32_t>(seed >> 32);
    float bv = f_neg_inf();
    int32_t bi = 0x7fffffff;
    bool nonfinite = false;
    int acc = 0;
    uint32_t acc_phase = 0;
    bool ok = true;
    for (int tile = blockIdx.x; tile < num_tiles && ok; tile += gridDim.x) {
      ok = wait_bounded(tfull + acc, acc_phase, a.error);
      if (!ok) break;
      tc_fence_after();
      for (int c = half * (kHalfCols / 32); c < (half + 1) * (kHalfCols / 32); ++c) {
        uint32_t v[32];
        __syncwarp();  // tcgen05.ld is warp-collective: reconverge after the per-row work
        tmem_ld32(tmem + static_cast<uint32_t>(acc * kBN + c * 32) + (static_cast<uint32_t>(q * 32) << 16), v);
        if (!live) continue;
        const int t_base = tile * kBN + c * 32;
#pragma unroll
        for (int g4 = 0; g4 < 8; ++g4) {
          const int t0 = t_base + g4 * 4;
          float y[4];
          uint32_t cand = 0;
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float z = __uint_as_float(v[g4 * 4 + e]);
            y[e] = greedy ? z : __fmul_rn(z, inv_t);
            const bool in = (t0 + e) < a.vocab;
            if (in && !(fabsf(z) <= 3.0e38f)) nonfinite = true;
            if (a.debug_logits && in) a.debug_logits[static_cast<int64_t>(r) * a.vocab + t0 + e] = z;
            const bool could = greedy ? !(y[e] < bv) : !(y[e] + kGumbelMax + 1e-3f + fabsf(y[e]) * 1e-6f < bv);
            cand |= static_cast<uint32_t>(in && could) << e;
          }
          if (!cand) continue;
          if (greedy) {
#pragma unroll
            for (int e = 0; e < 4; ++e)
              if (((cand >> e) & 1u) && (y[e] > bv || (y[e] == bv && t0 + e < bi))) {
                bv = y[e];
                bi = t0 + e;
              }
            continue;
          }
          const Philox4 pr = philox4x32_10(static_cast<uint32_t>(t0) >> 2, pos, rowid, 0u, key0, key1);
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            if (!((cand >> e) & 1u)) continue;
            const uint32_t num = uniform_numerator(pr.w[e]);
            if (y[e] + gumbel_upper_bound(num) + 1e-3f + fabsf(y[e]) * 1e-6f < bv) continue;
            const float s = __fadd_rn(y[e], gumbel_from_numerator(num));
            if (s > bv || (s == bv && t0 + e < bi)) {
              bv = s;
              bi = t0 + e;
            }
          }
        }
      }
      tc_fence_before();
      mbar_arrive(tempty + acc);
      if (++acc == 2) {
        acc = 0;
        acc_phase ^= 1u;
      }
    }
    if (live) {
      if (bi != 0x7fffffff)
        atomicMax(a.best + r, (static_cast<unsigned long long>(f_order_key(bv)) << 32) |
                                  static_cast<unsigned long long>(0xffffffffu - static_cast<uint32_t>(bi)));
      if (nonfinite) atomicOr(a.flags + r, 1);
    }
  }
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols) : "memory");
  }
}

__global__ void ss_fused_finish(int32_t batch, const unsigned long long* best, const int32_t* flags,
                                const int32_t* error, int32_t* out_token, int32_t* out_status) {
  const int r = blockIdx.x * blockDim.x + threadIdx.x;
  if (r >= batch) return;
  const unsigned long long k = best[r];
  int32_t st = SS_ROW_OK;
  if (flags[r] & 2) st = SS_ROW_BAD_PARAM;
  else if (*error) st = SS_ROW_TIMEOUT;
  else if (flags[r] & 1) st = SS_ROW_NONFINITE;
  else if (k == 0ull) st = SS_ROW_EMPTY_SET;
  out_status[r] = st;
  out_token[r] = (st == SS_ROW_OK) ? static_cast<int32_t>(0xffffffffu - static_cast<uint32_t>(k)) : -1;
}

// Rows whose temperature or position is invalid (reported as BAD_PARAM).
__global__ void ss_fused_check(int32_t batch, const float* temperature, const int64_t* position, int32_t* flags) {
  const int r = blockIdx.x * blockDim.x + threadIdx.x;
  if (r >= batch) return;
  const float T = temperature[r];
  const int64_t p = position[r];
  if (!(T >= 0.0f) || isinf(T) || p < 0 || p > 0xffffffffll) atomicOr(flags + r, 2);
}

static PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }
  return fn;
}

// [rows, cols] bf16 row-major tensor, boxes of box_rows x 64 with the
// 128-byte swizzle; rows past the tensor read as zero.
static bool make_map(CUtensorMap* m, const void* base, int64_t rows, int64_t cols, uint32_t box_rows) {
  auto fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(cols) * 2};
  const cuuint32_t box[2] = {static_cast<cuuint32_t>(kBK), box_rows};
  const cuuint32_t estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace ssf

extern "C" {

size_t ss_fused_scratch_bytes(int32_t batch) {
  if (batch < 1 || batch > ssf::kBM) return 0;
  return static_cast<size_t>(batch) * (8 + 4) + 16;
}

ss_status ss_fused_lmhead_sample(const ss_fused_args* args, ss_stream_t stream) {
  SS_NVTX_RANGE("ss_fused_lmhead_sample");
  using namespace ssf;
  if (!args) return SS_ERR_INVALID_ARG;
  const ss_fused_args& A = *args;
  if (A.batch < 1 || A.batch > kBM || A.hidden < kBK || (A.hidden % kBK) != 0 || A.vocab < 1) return SS_ERR_INVALID_ARG;
  if (!A.hidden_states || !A.weight || !A.temperature || !A.seed || !A.position || !A.out_token || !A.out_status ||
      !A.scratch)
    return SS_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(A.hidden_states) & 15u) || (reinterpret_cast<uintptr_t>(A.weight) & 15u) ||
      (reinterpret_cast<uintptr_t>(A.scratch) & 7u))
    return SS_ERR_INVALID_ARG;
  if (A.scratch_bytes < ss_fused_scratch_bytes(A.batch)) return SS_ERR_WORKSPACE;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  CUtensorMap mh, mw;
  const int a_rows = (A.batch <= 64) ? 64 : kBM;
  if (!make_map(&mh, A.hidden_states, A.batch, A.hidden, static_cast<uint32_t>(a_rows)) ||
      !make_map(&mw, A.weight, A.vocab, A.hidden, kBN))
    return SS_ERR_UNSUPPORTED;
  uint8_t* sc = static_cast<uint8_t*>(A.scratch);
  unsigned long long* best = reinterpret_cast<unsigned long long*>(sc);
  int32_t* flags = reinterpret_cast<int32_t*>(sc + static_cast<size_t>(A.batch) * 8);
  int32_t* error = flags + A.batch;
  cudaError_t e = cudaMemsetAsync(A.scratch, 0, ss_fused_scratch_bytes(A.batch), s);
  int dev = 0, sms = 0;
  if (e == cudaSuccess) e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(reinterpret_cast<const void*>(&ss_fused_kernel), cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(kSmemBytes));
  if (e == cudaSuccess) {
    const int tiles = (A.vocab + kBN - 1) / kBN;
    FArgs f{};
    f.batch = A.batch;
    f.hidden = A.hidden;
    f.vocab = A.vocab;
    f.temperature = A.temperature;
    f.seed = A.seed;
    f.position = A.position;
    f.row_id = A.row_id;
    f.best = best;
    f.flags = flags;
    f.error = error;
    f.debug_logits = A.debug_logits;
    f.a_rows = a_rows;
    ss_fused_check<<<(A.batch + 127) / 128, 128, 0, s>>>(A.batch, A.temperature, A.position, flags);
    ss_fused_kernel<<<tiles < sms ? tiles : sms, kThreadsF, kSmemBytes, s>>>(mh, mw, f);
    ss_fused_finish<<<(A.batch + 127) / 128, 128, 0, s>>>(A.batch, best, flags, error, A.out_token, A.out_status);
    e = cudaGetLastError();
  }
  if (e != cudaSuccess) {
    ss::set_last_cuda_error(static_cast<int32_t>(e));
    return SS_ERR_CUDA;
  }
  return SS_OK;
}

}  // extern "C"
