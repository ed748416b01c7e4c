// confidence.cu -- standalone confidence head and prefix survival.
//
// Source: DSpark explainer, "Confidence-scheduled verification":
// c_k = sigmoid(w^T [h_k ; W1[x_{k-1}]]), prefix survival a_j = prod_{i<=j} c_i;
// with sequential temperature scaling, c_k = sigmoid(z_k / tau_k);
// vLLM speculators "DSpark" guide, "Confidence Head".  verify_len is the
// longest prefix whose survival stays at or above the threshold.
// One warp per request walks the K positions in order (the survival product is
// sequential; each position's logit is a warp-cooperative dot product).

#include <cstdint>

#include "confidence.cuh"
#include "internal.h"
#include "sm103.cuh"

namespace dspark {
namespace {

__global__ void __launch_bounds__(128) confidence_kernel(
    const uint16_t* __restrict__ h, const uint16_t* __restrict__ W1,
    const int32_t* __restrict__ anchors, const int32_t* __restrict__ tokens,
    const uint16_t* __restrict__ w, float bias, int with_markov, int B, int K, int d, int r,
    int V, float threshold, const float* __restrict__ tau, float* __restrict__ conf,
    float* __restrict__ cumprod,
    int32_t* __restrict__ verify_len, int* status) {
  const int lane = threadIdx.x & 31;
  const int b = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (b >= B) return;
  float surv = 1.f;
  int len = 0;
  bool open = true;
  for (int k = 0; k < K; ++k) {
    const size_t o = static_cast<size_t>(b) * K + k;
    const uint16_t* emb = nullptr;
    if (with_markov) {
      int prev = (k == 0) ? anchors[b] : tokens[o - 1];
      if (prev < 0 || prev >= V) {
        if (lane == 0) record_error(status, kStatusDeviceOob);
        prev = 0;
      }
      emb = W1 + static_cast<size_t>(prev) * r;
    }
    const float z = confidence_logit(h + o * d, d, w, emb, r, bias, lane);
    const float c = sigmoidf_accurate(tau ? z / __ldg(tau + k) : z);
    surv *= c;
    if (open && surv >= threshold) {
      len = k + 1;
    } else {
      open = false;
    }
    if (lane == 0) {
      conf[o] = c;
      cumprod[o] = surv;
    }
  }
  if (lane == 0) verify_len[b] = len;
}

}  // namespace

cudaError_t launch_confidence(const uint16_t* h, const uint16_t* W1, const int32_t* anchors,
                              const int32_t* tokens, const uint16_t* w, float bias,
                              int with_markov, int B, int K, int d, int r, int V,
                              float threshold, const float* tau, float* conf, float* cumprod,
                              int32_t* verify_len, int* status, cudaStream_t stream) {
  const int warps = 4;
  confidence_kernel<<<(B + warps - 1) / warps, warps * 32, 0, stream>>>(
      h, W1, anchors, tokens, w, bias, with_markov, B, K, d, r, V, threshold, tau, conf,
      cumprod, verify_len, status);
  return cudaGetLastError();
}

}  // namespace dspark
