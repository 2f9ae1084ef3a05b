// ss_philox.cuh -- counter-based Philox4x32-10 (Salmon, Moraes, Dror, Shaw,
// "Parallel random numbers: as easy as 1, 2, 3", SC'11) and the Gumbel noise
// built on it.  Key (seed lo32, seed hi32); counter (t >> 2, position, row,
// stream); token t uses output word t & 3.
#pragma once
#include <stdint.h>

namespace ss {

struct Philox4 {
  uint32_t w[4];
};

__device__ __forceinline__ Philox4 philox4x32_10(uint32_t c0, uint32_t c1, uint32_t c2, uint32_t c3, uint32_t k0,
                                                 uint32_t k1) {
#pragma unroll
  for (int round = 0; round < 10; ++round) {
    // S-box of one round: two 32x32 -> 64-bit products; the high halves are
    // mixed with the other counter words and the round key.
    // one 32 x 32 -> 64-bit multiply each (a single wide multiply-add)
    const uint64_t a = static_cast<uint64_t>(0xD2511F53u) * c0;
    const uint64_t b = static_cast<uint64_t>(0xCD9E8D57u) * c2;
    const uint32_t a_hi = static_cast<uint32_t>(a >> 32), a_lo = static_cast<uint32_t>(a);
    const uint32_t b_hi = static_cast<uint32_t>(b >> 32), b_lo = static_cast<uint32_t>(b);
    const uint32_t n0 = b_hi ^ c1 ^ k0;
    const uint32_t n2 = a_hi ^ c3 ^ k1;
    c0 = n0;
    c1 = b_lo;
    c2 = n2;
    c3 = a_lo;
    k0 += 0x9E3779B9u;  // Weyl sequence key schedule
    k1 += 0xBB67AE85u;
  }
  Philox4 r;
  r.w[0] = c0;
  r.w[1] = c1;
  r.w[2] = c2;
  r.w[3] = c3;
  return r;
}

// Odd 24-bit numerator n of u = n * 2^-24 in [2^-24, 1 - 2^-24].
__device__ __forceinline__ uint32_t uniform_numerator(uint32_t x) { return ((x >> 9) << 1) | 1u; }

// u = n * 2^-24, built from the bits: 1 + (n >> 1) * 2^-23 minus 1 is
// (n - 1) * 2^-24 exactly, and adding 2^-24 is exact too (n < 2^24).  This
// avoids the integer -> float conversion instruction, which sm_103 issues at
// a small fraction of the add rate.
__device__ __forceinline__ float uniform_from_numerator(uint32_t n) {
  return __fadd_rn(__fsub_rn(__uint_as_float(0x3f800000u | (n >> 1)), 1.0f), 5.9604644775390625e-08f);
}

// Gumbel noise -log(-log u) with the accurate single-precision logf.
__device__ __forceinline__ float gumbel_from_numerator(uint32_t n) {
  const float u = uniform_from_numerator(n);
  return -logf(-logf(u));
}

// Cheap upper bound of the Gumbel noise: -log(u) >= 1 - u, so
// g <= -log(1 - u) = ln2 * (24 - log2(2^24 - n)) <= ln2 * (clz(2^24 - n) - 7).
__device__ __forceinline__ float gumbel_upper_bound(uint32_t n) {
  const uint32_t m = (1u << 24) - n;  // in [1, 2^24 - 1]
  // clz(m) - 7 is in [1, 24]: converted with the 2^23 bit-pattern trick
  return 0.69314718f * __fsub_rn(__uint_as_float(0x4b000000u + static_cast<uint32_t>(__clz(m) - 7)), 8388608.0f);
}

// Largest Gumbel value any token can get: -log(-log(1 - 2^-24)) = 16.6355...
constexpr float kGumbelMax = 16.63554f;

__device__ __forceinline__ uint32_t philox_word(uint64_t seed, uint32_t row, uint32_t pos, uint32_t token,
                                                uint32_t stream) {
  Philox4 r = philox4x32_10(token >> 2, pos, row, stream, static_cast<uint32_t>(seed),
                            static_cast<uint32_t>(seed >> 32));
  return r.w[token & 3u];
}

}  // namespace ss
