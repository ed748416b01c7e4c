// calibrate.cu -- sequential temperature scaling (STS) of the confidence head.
//
// Source: DSpark explainer, "Confidence-scheduled verification": the raw head
// is calibrated with one temperature per position, fitted left to right
// against cumulative prefix-survival probabilities (the ranking is kept).
// tau_k minimises, over N calibration rows, the binary cross-entropy between
// the model's prefix survival a_k = prod_{i<=k} sigmoid(z_i / tau_i) (earlier
// temperatures fixed) and the target survival y_k = prod_{i<=k} label_i, with
// z_i the logit of the raw confidence.  The 1-D search over ln tau: 32 evenly
// spaced points, the best (ties to the smaller) kept and the interval between
// its neighbours searched again, 8 rounds.
//
// One CTA: 256 threads share the rows; each thread keeps the 32 grid losses
// of its rows as compensated fp32 sums, the block adds them in fp64, and
// thread 0 narrows the interval.  Positions run in order (each needs the
// earlier temperatures), the fitted 1 / tau_i kept in shared memory.

#include <cstdint>

#include "internal.h"

namespace dspark {
namespace {

constexpr int kStsThreads = 256;
constexpr int kStsG = 32;
constexpr int kStsR = 8;

__device__ __forceinline__ float logit_clamped(float c) {
  const float lo = 5.9604645e-08f;  // 2^-24
  c = fminf(fmaxf(c, lo), 1.0f - lo);
  return logf(c) - log1pf(-c);
}

__device__ __forceinline__ float sigmoid_f(float z) { return 1.0f / (1.0f + expf(-z)); }

__global__ void __launch_bounds__(kStsThreads, 1) sts_fit_kernel(const float* __restrict__ conf,
                                                              const float* __restrict__ label,
                                                              int N, int K, float tau_lo,
                                                              float tau_hi, float* __restrict__ tau,
                                                              float* __restrict__ loss) {
  __shared__ float s_inv_tau[kMaxK];
  __shared__ float s_inv[kStsG];
  __shared__ double s_part[kStsThreads / 32][kStsG];
  __shared__ double s_L[kStsG];
  __shared__ double s_x0, s_x1, s_xb, s_Lb;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  for (int k = 0; k < K; ++k) {
    if (tid == 0) {
      s_x0 = log(static_cast<double>(tau_lo));
      s_x1 = log(static_cast<double>(tau_hi));
    }
    __syncthreads();
    for (int round = 0; round < kStsR; ++round) {
      const double x0 = s_x0, step = (s_x1 - s_x0) / (kStsG - 1);
      if (tid < kStsG) s_inv[tid] = static_cast<float>(exp(-(x0 + step * tid)));
      __syncthreads();
      float acc[kStsG], comp[kStsG];
#pragma unroll
      for (int g = 0; g < kStsG; ++g) acc[g] = comp[g] = 0.f;
      for (int n = tid; n < N; n += kStsThreads) {
        const float* crow = conf + static_cast<size_t>(n) * K;
        const float* lrow = label + static_cast<size_t>(n) * K;
        float a = 1.f, y = 1.f;
        for (int i = 0; i < k; ++i) {
          a *= sigmoid_f(logit_clamped(__ldg(crow + i)) * s_inv_tau[i]);
          y *= __ldg(lrow + i);
        }
        y *= __ldg(lrow + k);
        const float z = logit_clamped(__ldg(crow + k));
#pragma unroll
        for (int g = 0; g < kStsG; ++g) {
          const float q = fminf(fmaxf(a * sigmoid_f(z * s_inv[g]), 1e-7f), 1.0f - 1e-7f);
          const float l = -(y * logf(q) + (1.f - y) * log1pf(-q));
          // compensated sum
          const float t = l - comp[g];
          const float s = acc[g] + t;
          comp[g] = (s - acc[g]) - t;
          acc[g] = s;
        }
      }
#pragma unroll
      for (int g = 0; g < kStsG; ++g) {
        double v = static_cast<double>(acc[g]) - static_cast<double>(comp[g]);
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, off);
        if (lane == 0) s_part[warp][g] = v;
      }
      __syncthreads();
      if (tid < kStsG) {
        double v = 0.0;
        for (int w = 0; w < kStsThreads / 32; ++w) v += s_part[w][tid];
        s_L[tid] = v;
      }
      __syncthreads();
      if (tid == 0) {
        int best = 0;
        for (int g = 1; g < kStsG; ++g)
          if (s_L[g] < s_L[best]) best = g;
        s_xb = x0 + step * best;
        s_Lb = s_L[best];
        const double nx0 = x0 + step * (best > 0 ? best - 1 : 0);
        const double nx1 = x0 + step * (best < kStsG - 1 ? best + 1 : kStsG - 1);
        s_x0 = nx0;
        s_x1 = nx1;
      }
      __syncthreads();
    }
    if (tid == 0) {
      const double t = exp(s_xb);
      tau[k] = static_cast<float>(t);
      if (loss != nullptr) loss[k] = static_cast<float>(s_Lb / N);
      s_inv_tau[k] = static_cast<float>(1.0 / t);
    }
    __syncthreads();
  }
}

}  // namespace

cudaError_t launch_sts_fit(const float* conf, const float* label, int N, int K, float tau_lo,
                           float tau_hi, float* tau, float* loss, cudaStream_t stream) {
  sts_fit_kernel<<<1, kStsThreads, 0, stream>>>(conf, label, N, K, tau_lo, tau_hi, tau, loss);
  return cudaGetLastError();
}

}  // namespace dspark
