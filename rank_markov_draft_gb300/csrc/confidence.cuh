// confidence.cuh -- the confidence head's logit, one warp per (request,
// position).  Source: DSpark explainer, "Confidence-scheduled verification":
// c_k = sigmoid(w^T [h_k ; W1[x_{k-1}]]); vLLM speculators "DSpark" guide,
// "Confidence Head" (the Markov embedding is concatenated only with
// --confidence-head-with-markov).
#pragma once

#include <cstdint>

namespace dspark {

__device__ __forceinline__ float bf16x2_dot(uint32_t a, uint32_t b) {
  return __uint_as_float(a << 16) * __uint_as_float(b << 16) +
         __uint_as_float(a & 0xFFFF0000u) * __uint_as_float(b & 0xFFFF0000u);
}

// Warp-cooperative dot of n bf16 values (n a multiple of 8, 16-byte aligned rows).
__device__ __forceinline__ float warp_dot_bf16(const uint16_t* x, const uint16_t* y, int n,
                                               int lane) {
  float z = 0.f;
  for (int j = lane * 8; j < n; j += 256) {
    const uint4 xv = __ldg(reinterpret_cast<const uint4*>(x + j));
    const uint4 yv = __ldg(reinterpret_cast<const uint4*>(y + j));
    z += bf16x2_dot(xv.x, yv.x) + bf16x2_dot(xv.y, yv.y) + bf16x2_dot(xv.z, yv.z) +
         bf16x2_dot(xv.w, yv.w);
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) z += __shfl_xor_sync(0xFFFFFFFFu, z, off);
  return z;
}

// z = w[:d] . h + (emb ? w[d:d+r] . emb : 0) + bias; every lane gets the value.
__device__ __forceinline__ float confidence_logit(const uint16_t* h, int d, const uint16_t* w,
                                                  const uint16_t* emb, int r, float bias,
                                                  int lane) {
  float z = warp_dot_bf16(h, w, d, lane);
  if (emb != nullptr) z += warp_dot_bf16(emb, w + d, r, lane);
  return z + bias;
}

__device__ __forceinline__ float sigmoidf_accurate(float z) { return 1.0f / (1.0f + expf(-z)); }

}  // namespace dspark
