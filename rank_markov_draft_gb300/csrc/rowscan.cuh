// rowscan.cuh -- one CTA's pass over a row of target logits: the log-sum-exp of P / Tt in
// natural-log units, or the row's argmax (first index of the maximum) when the target is
// greedy (Tt = 0).  Sources: "DSpark: Repair the Joint, Meter the Verify", "Watch the Mass
// Land Wrong" (the target's distribution p = softmax(P / Tt) that verification tests
// against); DSpark explainer, "Confidence-scheduled verification" (the same p in the
// acceptance label).  The row is read once, streaming (__ldcs), four float4 loads in flight
// per thread; the result is final in thread 0.
#pragma once

#include <cstdint>

#include "sm103.cuh"

namespace dspark {

constexpr int kScanThreads = 256;
constexpr float kScanLog2e = 1.4426950408889634f;
constexpr float kScanLn2 = 0.69314718055994531f;

// Merge (ma, sa) with (mb, sb): log-sum-exp partials in base 2.
__device__ __forceinline__ void lse2_merge(float& ma, float& sa, float mb, float sb) {
  if (mb == -INFINITY) return;
  if (ma == -INFINITY) {
    ma = mb;
    sa = sb;
    return;
  }
  if (mb > ma) {
    sa = sa * ex2_approx(ma - mb) + sb;
    ma = mb;
  } else {
    sa += sb * ex2_approx(mb - ma);
  }
}

struct RowScanSmem {
  float m[kScanThreads / 32], s[kScanThreads / 32];
  int i[kScanThreads / 32];
};

// Called by every thread of a kScanThreads-thread CTA (it synchronises the CTA); thread 0
// returns with `argmax` (greedy) or `lse` set.  V a multiple of 4, `row` 16-byte aligned.
__device__ __forceinline__ void scan_target_row(const float* __restrict__ row, int V, float inv_tt,
                                                bool greedy, RowScanSmem& sm, float& lse,
                                                int& argmax) {
  const float4* p4 = reinterpret_cast<const float4*>(row);
  const int n4 = V / 4;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (greedy) {
    float bv = -INFINITY;
    int bi = 0x7FFFFFFF;
    for (int i = threadIdx.x; i < n4; i += kScanThreads) {
      const float4 x = __ldcs(p4 + i);
      const float xs[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
      for (int c = 0; c < 4; ++c)
        if (xs[c] > bv || (xs[c] == bv && 4 * i + c < bi)) {
          bv = xs[c];
          bi = 4 * i + c;
        }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      const float ov = __shfl_xor_sync(0xFFFFFFFFu, bv, off);
      const int oi = __shfl_xor_sync(0xFFFFFFFFu, bi, off);
      if (ov > bv || (ov == bv && oi < bi)) {
        bv = ov;
        bi = oi;
      }
    }
    if (lane == 0) {
      sm.m[warp] = bv;
      sm.i[warp] = bi;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
      for (int w = 1; w < kScanThreads / 32; ++w)
        if (sm.m[w] > bv || (sm.m[w] == bv && sm.i[w] < bi)) {
          bv = sm.m[w];
          bi = sm.i[w];
        }
      argmax = bi;
    }
    return;
  }
  // online log-sum-exp of y = P * log2(e) / Tt
  const float sc = inv_tt * kScanLog2e;
  float m = -INFINITY, s = 0.f;
  for (int i0 = threadIdx.x; i0 < n4; i0 += 4 * kScanThreads) {
    float4 x[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int i = i0 + u * kScanThreads;
      x[u] = (i < n4) ? __ldcs(p4 + i) : make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
    }
    float cm = -INFINITY;
#pragma unroll
    for (int u = 0; u < 4; ++u)
      cm = fmaxf(cm, fmaxf(fmaxf(x[u].x, x[u].y), fmaxf(x[u].z, x[u].w)) * sc);
    if (cm == -INFINITY) continue;
    if (cm > m) {
      s = (m == -INFINITY) ? 0.f : s * ex2_approx(m - cm);
      m = cm;
    }
#pragma unroll
    for (int u = 0; u < 4; ++u)
      s += ex2_approx(x[u].x * sc - m) + ex2_approx(x[u].y * sc - m) +
           ex2_approx(x[u].z * sc - m) + ex2_approx(x[u].w * sc - m);
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1)
    lse2_merge(m, s, __shfl_xor_sync(0xFFFFFFFFu, m, off), __shfl_xor_sync(0xFFFFFFFFu, s, off));
  if (lane == 0) {
    sm.m[warp] = m;
    sm.s[warp] = s;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    for (int w = 1; w < kScanThreads / 32; ++w) lse2_merge(m, s, sm.m[w], sm.s[w]);
    lse = (m + log2f(s)) * kScanLn2;
  }
}

}  // namespace dspark
