// philox.cuh -- Philox4x32-10 counter-based generator on the device, written
// from its published definition (Salmon, Moraes, Dror, Shaw, "Parallel Random
// Numbers: As Easy as 1, 2, 3", SC'11): ten rounds, each multiplying words 0
// and 2 by fixed odd constants, taking the high/low halves of the products and
// mixing the high halves with words 1 and 3 and the round key; the key is
// advanced by the Weyl increments between rounds.
//
// Token-sampling noise of the Markov head (the pages ask for a counter-based
// generator keyed on request, position and token): counter = (v >> 2, k, b, 0),
// key = (seed low, seed high); word v & 3 becomes
// u = ((word >> 9) + 0.5) * 2^-23, an odd multiple of 2^-24 in (0, 1).
#pragma once

#include <cstdint>

namespace dspark {

struct Philox4 {
  uint32_t w[4];
};

__device__ __forceinline__ Philox4 philox4x32_10(uint32_t c0, uint32_t c1, uint32_t c2,
                                                 uint32_t c3, uint32_t k0, uint32_t k1) {
#pragma unroll
  for (int round = 0; round < 10; ++round) {
    const uint32_t lo_a = 0xD2511F53u * c0;
    const uint32_t hi_a = __umulhi(0xD2511F53u, c0);
    const uint32_t lo_b = 0xCD9E8D57u * c2;
    const uint32_t hi_b = __umulhi(0xCD9E8D57u, c2);
    const uint32_t n0 = hi_b ^ c1 ^ k0;
    const uint32_t n2 = hi_a ^ c3 ^ k1;
    c0 = n0;
    c1 = lo_b;
    c2 = n2;
    c3 = lo_a;
    k0 += 0x9E3779B9u;
    k1 += 0xBB67AE85u;
  }
  Philox4 r;
  r.w[0] = c0;
  r.w[1] = c1;
  r.w[2] = c2;
  r.w[3] = c3;
  return r;
}

// u = ((word >> 9) + 0.5) * 2^-23 computed without an int->float conversion:
// 1 + n * 2^-23 is built from the mantissa bits, and subtracting 1 - 2^-24 is
// exact (the result is an odd multiple of 2^-24 below 1).
__device__ __forceinline__ float philox_uniform(uint32_t word) {
  const float one_plus = __uint_as_float(0x3F800000u | (word >> 9));
  return one_plus - 0.99999994039535522461f;  // 1 - 2^-24
}

// Accurate E = -ln(u) for u in (0, 1): -log(u) below 1/2; above it, with
// t = 1 - u exact, -log1p(-t), so the small values (large Gumbel noise) keep
// their relative accuracy.
__device__ __forceinline__ float neg_log_uniform_accurate(float u) {
  return (u < 0.5f) ? -logf(u) : -log1pf(-(1.0f - u));
}

}  // namespace dspark
