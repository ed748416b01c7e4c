// headlogit.cuh -- the draft head's calibrated logit of one token, warp-cooperative:
// l(v) = U[v] + sum_i e_i W2[i, v], e = W1[prev] (bf16), or W1[prev] * gate rounded to
// bf16 (the operand the draft kernel's MMA multiplies).  Source: DSpark explainer, "The
// Markov head"; equivalence page, "What the two methods do".
#pragma once

#include <cstdint>
#include <cuda_bf16.h>

namespace dspark {

__device__ __forceinline__ float head_logit(const float* urow, const uint16_t* W1,
                                            const uint16_t* W2, const float* hrow, int V, int r,
                                            int prev, int v, int lane) {
  float acc = 0.f;
  for (int i = lane; i < r; i += 32) {
    float e = __uint_as_float(static_cast<uint32_t>(__ldg(W1 + static_cast<size_t>(prev) * r + i)) << 16);
    if (hrow) e = __bfloat162float(__float2bfloat16_rn(e * __ldg(hrow + i)));
    acc = fmaf(e, __uint_as_float(static_cast<uint32_t>(__ldg(W2 + static_cast<size_t>(i) * V + v)) << 16),
               acc);
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xFFFFFFFFu, acc, off);
  return acc + __ldg(urow + v);
}

}  // namespace dspark
