// philox.cuh -- Philox4x32-10 counter-based generator on the device, written
// from its published definition (Salmon, Moraes, Dror, Shaw, "Parallel Random
// Numbers: As Easy as 1, 2, 3", SC'11): ten rounds, each multiplying words 0
// and 2 by fixed odd constants, taking the high/low halves of the products and
// mixing the high halves with words 1 and 3 and the round key; the key is
// advanced by the Weyl increments between rounds.
//
// Noise of the Markov head's draw (a counter-based generator keyed on request
// b, position k and 16-token block beta = v >> 4): key = (seed low, seed high),
// counter = (beta >> 3, k, b, 1 + (beta & 3)); with h = (beta >> 2) & 1, word 2h
// is the block's stage-1 uniform (the race between blocks) and word 2h + 1 its
// stage-2 uniform (the inverse CDF inside the block).  A word becomes
// u = ((word & 0x7FFFFF) + 0.5) * 2^-23, an odd multiple of 2^-24 in (0, 1).
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

// One block with counter (c0, c1, c2, c3) and a precomputed key schedule.
__device__ __forceinline__ void philox4x32_10_rk(uint32_t c0, uint32_t c1, uint32_t c2,
                                                 uint32_t c3, const uint32_t (&rk0)[10],
                                                 const uint32_t (&rk1)[10], uint32_t (&out)[4]) {
#pragma unroll
  for (int round = 0; round < 10; ++round) {
    const uint64_t pa = static_cast<uint64_t>(0xD2511F53u) * c0;
    const uint64_t pb = static_cast<uint64_t>(0xCD9E8D57u) * c2;
    const uint32_t n0 = static_cast<uint32_t>(pb >> 32) ^ c1 ^ rk0[round];
    const uint32_t n2 = static_cast<uint32_t>(pa >> 32) ^ c3 ^ rk1[round];
    c0 = n0;
    c1 = static_cast<uint32_t>(pb);
    c2 = n2;
    c3 = static_cast<uint32_t>(pa);
  }
  out[0] = c0;
  out[1] = c1;
  out[2] = c2;
  out[3] = c3;
}

// Philox key schedule: round i uses (k0 + i * 0x9E3779B9, k1 + i * 0xBB67AE85).
__host__ __device__ inline void philox_round_keys(uint32_t k0, uint32_t k1, uint32_t (&rk0)[10],
                                                  uint32_t (&rk1)[10]) {
  for (int i = 0; i < 10; ++i) {
    rk0[i] = k0 + static_cast<uint32_t>(i) * 0x9E3779B9u;
    rk1[i] = k1 + static_cast<uint32_t>(i) * 0xBB67AE85u;
  }
}

// Two blocks with counters (c0, c1, c2, c3a) and (c0, c1, c2, c3b) and a precomputed key
// schedule, interleaved round by round for instruction-level parallelism.  Round 0 of
// both shares the products of words 0 and 2 (equal in both counters).
__device__ __forceinline__ void philox4x32_10_rk2(uint32_t c0, uint32_t c1, uint32_t c2,
                                                  uint32_t c3a, uint32_t c3b,
                                                  const uint32_t (&rk0)[10],
                                                  const uint32_t (&rk1)[10], uint32_t (&oa)[4],
                                                  uint32_t (&ob)[4]) {
  const uint64_t pa0 = static_cast<uint64_t>(0xD2511F53u) * c0;
  const uint64_t pb0 = static_cast<uint64_t>(0xCD9E8D57u) * c2;
  uint32_t a0 = static_cast<uint32_t>(pb0 >> 32) ^ c1 ^ rk0[0];
  uint32_t a1 = static_cast<uint32_t>(pb0);
  uint32_t a2 = static_cast<uint32_t>(pa0 >> 32) ^ c3a ^ rk1[0];
  uint32_t a3 = static_cast<uint32_t>(pa0);
  uint32_t b0 = a0, b1 = a1, b3 = a3;
  uint32_t b2 = static_cast<uint32_t>(pa0 >> 32) ^ c3b ^ rk1[0];
#pragma unroll
  for (int round = 1; round < 10; ++round) {
    const uint64_t qa = static_cast<uint64_t>(0xD2511F53u) * a0;
    const uint64_t qb = static_cast<uint64_t>(0xCD9E8D57u) * a2;
    const uint64_t ra = static_cast<uint64_t>(0xD2511F53u) * b0;
    const uint64_t rb = static_cast<uint64_t>(0xCD9E8D57u) * b2;
    const uint32_t na0 = static_cast<uint32_t>(qb >> 32) ^ a1 ^ rk0[round];
    const uint32_t na2 = static_cast<uint32_t>(qa >> 32) ^ a3 ^ rk1[round];
    const uint32_t nb0 = static_cast<uint32_t>(rb >> 32) ^ b1 ^ rk0[round];
    const uint32_t nb2 = static_cast<uint32_t>(ra >> 32) ^ b3 ^ rk1[round];
    a1 = static_cast<uint32_t>(qb);
    a3 = static_cast<uint32_t>(qa);
    b1 = static_cast<uint32_t>(rb);
    b3 = static_cast<uint32_t>(ra);
    a0 = na0;
    a2 = na2;
    b0 = nb0;
    b2 = nb2;
  }
  oa[0] = a0;
  oa[1] = a1;
  oa[2] = a2;
  oa[3] = a3;
  ob[0] = b0;
  ob[1] = b1;
  ob[2] = b2;
  ob[3] = b3;
}

// t = 1 - u for the uniform u of `word`: with n = word & 0x7FFFFF,
// u = (n + 0.5) 2^-23 and 1 - u = (n' + 0.5) 2^-23 with n' = 2^23 - 1 - n, the
// low 23 bits of ~word; built exactly like u.
__device__ __forceinline__ float philox_one_minus_uniform(uint32_t word) {
  const float one_plus = __uint_as_float(0x3F800000u | (~word & 0x7FFFFFu));
  return one_plus - 0.99999994039535522461f;  // 1 - 2^-24, exact result
}

// 1 + n' 2^-23 (the operand of the subtraction above), one logic op.
__device__ __forceinline__ float philox_one_plus_complement(uint32_t word) {
  return __uint_as_float(0x3F800000u | (~word & 0x7FFFFFu));
}

// u = ((word & 0x7FFFFF) + 0.5) * 2^-23 computed without an int->float
// conversion: 1 + n * 2^-23 is built from the mantissa bits, and subtracting
// 1 - 2^-24 is exact (the result is an odd multiple of 2^-24 below 1).
__device__ __forceinline__ float philox_uniform(uint32_t word) {
  const float one_plus = __uint_as_float(0x3F800000u | (word & 0x7FFFFFu));
  return one_plus - 0.99999994039535522461f;  // 1 - 2^-24
}

// E = -ln(u) for the uniform u of `word`, to about 1e-6 relative, without a
// branch: with t = 1 - u (exact), the Taylor series of -ln(1 - t) to t^8 / 8
// for t < 1/8 (remainder below t^8 / 8 relative), else -log2(u) ln 2 from the
// hardware base-2 logarithm (|ln u| >= 0.13 there, so its absolute error of
// about 2^-22 stays near 1e-6 relative).
__device__ __forceinline__ float neg_log_uniform_fast(uint32_t word) {
  const float t = philox_one_minus_uniform(word);
  float sr = fmaf(t, 0.125f, 0.142857142857f);
  sr = fmaf(t, sr, 0.166666666667f);
  sr = fmaf(t, sr, 0.2f);
  sr = fmaf(t, sr, 0.25f);
  sr = fmaf(t, sr, 0.333333333333f);
  sr = fmaf(t, sr, 0.5f);
  sr = fmaf(t, sr, 1.0f);
  sr *= t;
  float l2;
  asm("lg2.approx.f32 %0, %1;" : "=f"(l2) : "f"(1.0f - t));
  return (t < 0.125f) ? sr : -l2 * 0.69314718055994531f;
}

// Accurate E = -ln(u) for u in (0, 1): -log(u) below 1/2; above it, with
// t = 1 - u exact, -log1p(-t), so the small values (the race's fast arrivals) keep
// their relative accuracy.
__device__ __forceinline__ float neg_log_uniform_accurate(float u) {
  return (u < 0.5f) ? -logf(u) : -log1pf(-(1.0f - u));
}

}  // namespace dspark
