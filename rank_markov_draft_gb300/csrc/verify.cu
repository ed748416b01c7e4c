// verify.cu -- speculative verification of a drafted block on sm_103a.
//
// Source: "DSpark: Repair the Joint, Meter the Verify", "Watch the Mass Land
// Wrong" (the target accepts a drafted token with probability min(1, p/q) and
// resamples when it rejects); DSpark explainer, "Confidence-scheduled
// verification" (that probability is 1 - TV(p^d_k, p^t_k)), "Hardware-aware
// prefix scheduling" (every retained token goes through the target's
// accept-or-correct rule; truncation changes the work, not the output) and
// "Two bottlenecks after you already have a parallel drafter" (a bonus token
// when the whole draft survives).  The first rejection is corrected by a draw
// from the normalised residual max(0, p - q); a fully accepted window draws
// the bonus from the target's next row.
//
// Kernels (all stream-ordered, no host synchronisation):
//   verify_stats_kernel  one CTA per (request, position <= window) row of the
//                        target logits: log-sum-exp of P / Tt (argmax when
//                        Tt = 0), a pure HBM scan of the row;
//   verify_accept_kernel one warp per request, lanes = positions: every
//                        acceptance test at once (the draft's own
//                        log-probabilities give q(x)), the first failure ends
//                        the prefix; records where the draw happens and what
//                        feeds it;
//   verify_prep_kernel   one warp per request: the offsets that turn the draft
//                        head's logits and the target logits at the draw
//                        position into log2 q and log2 p (the draft's
//                        normaliser from its own log-probability of the
//                        rejected token, rebuilt l(x) by a dot product), and
//                        the draw position's predecessor and gate row;
// then the draft kernel's residual mode streams each request's base-logit row
// and target row at its draw position, read in place, and draws from
// max(0, p - q) (p alone for a bonus) by the block race.
// Noise: acceptance uniform of position k: Philox4x32-10 counter (k, 0, b, 13),
// word 0; the draw's block race at position j: counter (beta >> 3, j, b,
// 9 + (beta & 3)), words 2h (stage 1) and 2h + 1 (stage 2), h = (beta >> 2) & 1.

#include <cstdint>
#include <cuda_bf16.h>

#include "headlogit.cuh"
#include "internal.h"
#include "philox.cuh"
#include "sm103.cuh"

namespace dspark {
namespace {

constexpr float kLog2eV = 1.4426950408889634f;
constexpr float kLn2V = 0.69314718055994531f;
constexpr int kStatsThreads = 256;

__device__ __forceinline__ float uniform_of(uint32_t word) { return philox_uniform(word); }

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

__global__ void __launch_bounds__(kStatsThreads) verify_stats_kernel(
    const float* __restrict__ P, const int32_t* __restrict__ ell, int K, int kmax, int V,
    float inv_tt, int greedy, float* __restrict__ lse_t, int32_t* __restrict__ argmax_t) {
  const int row = blockIdx.x;             // b * (K + 1) + k
  const int b = row / (K + 1), k = row - b * (K + 1);
  const int L = min(ell ? min(max(__ldg(ell + b), 0), K) : K, kmax);
  if (k > L) return;
  const float4* p4 = reinterpret_cast<const float4*>(P + static_cast<size_t>(row) * V);
  const int n4 = V / 4;
  __shared__ float s_m[kStatsThreads / 32], s_s[kStatsThreads / 32];
  __shared__ int s_i[kStatsThreads / 32];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (greedy) {
    float bv = -INFINITY;
    int bi = 0x7FFFFFFF;
    for (int i = threadIdx.x; i < n4; i += kStatsThreads) {
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
      s_m[warp] = bv;
      s_i[warp] = bi;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
      for (int w = 1; w < kStatsThreads / 32; ++w)
        if (s_m[w] > bv || (s_m[w] == bv && s_i[w] < bi)) {
          bv = s_m[w];
          bi = s_i[w];
        }
      argmax_t[row] = bi;
    }
    return;
  }
  // online log-sum-exp of y = P * log2(e) / Tt, four float4 loads in flight
  const float sc = inv_tt * kLog2eV;
  float m = -INFINITY, s = 0.f;
  for (int i0 = threadIdx.x; i0 < n4; i0 += 4 * kStatsThreads) {
    float4 x[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int i = i0 + u * kStatsThreads;
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
    s_m[warp] = m;
    s_s[warp] = s;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    for (int w = 1; w < kStatsThreads / 32; ++w) lse2_merge(m, s, s_m[w], s_s[w]);
    lse_t[row] = (m + log2f(s)) * kLn2V;  // natural-log units of P / Tt
  }
}

// One warp per request: lanes evaluate the acceptance tests of positions
// lane, lane + 32 (K <= 64) at once; the first failed test ends the prefix.
__global__ void verify_accept_kernel(const float* __restrict__ P, const int32_t* __restrict__ tokens,
                                     const float* __restrict__ logq, const int32_t* __restrict__ anchors,
                                     const int32_t* __restrict__ ell, const float* __restrict__ lse_t,
                                     const int32_t* __restrict__ argmax_t, int B, int K, int V,
                                     float inv_tt, int target_greedy, int draft_greedy,
                                     uint32_t seed_lo, uint32_t seed_hi, int32_t* __restrict__ n_acc,
                                     int32_t* __restrict__ next_token, float* __restrict__ accept_prob,
                                     VerifySel* __restrict__ sel, int* status) {
  const int lane = threadIdx.x & 31;
  const int b = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (b >= B) return;
  const int L = ell ? min(max(__ldg(ell + b), 0), K) : K;
  uint32_t ok_lo = 0u, ok_hi = 0u;  // bit k: position k's token survives its test
#pragma unroll
  for (int half = 0; half < 2; ++half) {
    const int k = half * 32 + lane;
    bool pass = true;
    if (k < L) {
      int x = __ldg(tokens + static_cast<size_t>(b) * K + k);
      if (x < 0 || x >= V) {
        record_error(status, kStatusDeviceOob);
        x = 0;
      }
      const size_t row = static_cast<size_t>(b) * (K + 1) + k;
      const float pr = target_greedy ? ((x == argmax_t[row]) ? 1.f : 0.f)
                                     : expf(__ldg(P + row * V + x) * inv_tt - lse_t[row]);
      const float q = draft_greedy ? 1.f : expf(__ldg(logq + static_cast<size_t>(b) * K + k));
      const float a = (q > 0.f) ? fminf(1.f, pr / q) : 1.f;
      if (accept_prob) accept_prob[static_cast<size_t>(b) * K + k] = a;
      const Philox4 rnd = philox4x32_10(static_cast<uint32_t>(k), 0u, static_cast<uint32_t>(b),
                                        13u, seed_lo, seed_hi);
      pass = uniform_of(rnd.w[0]) < a;
    } else if (k < K && accept_prob) {
      accept_prob[static_cast<size_t>(b) * K + k] = -1.f;
    }
    const uint32_t bal = __ballot_sync(0xFFFFFFFFu, pass);
    if (half == 0) ok_lo = bal; else ok_hi = bal;
  }
  // first failed test below L
  int n = L;
  if (~ok_lo != 0u && __ffs(~ok_lo) - 1 < L) {
    n = __ffs(~ok_lo) - 1;
  } else if (~ok_hi != 0u && 32 + __ffs(~ok_hi) - 1 < L) {
    n = 32 + __ffs(~ok_hi) - 1;
  }
  if (lane == 0) {
    const int rejected = n < L ? 1 : 0;
    const int pos = n;
    n_acc[b] = n;
    VerifySel s;
    s.pos = pos;
    s.residual = rejected;
    s.x = rejected ? __ldg(tokens + static_cast<size_t>(b) * K + pos) : -1;
    int prev = (pos == 0) ? __ldg(anchors + b) : __ldg(tokens + static_cast<size_t>(b) * K + pos - 1);
    if (prev < 0 || prev >= V) {
      record_error(status, kStatusDeviceOob);
      prev = 0;
    }
    if (s.x >= V || (rejected && s.x < 0)) s.x = 0;
    s.prev = prev;
    sel[b] = s;
    if (target_greedy) next_token[b] = argmax_t[static_cast<size_t>(b) * (K + 1) + pos];
  }
}

// Base-logit (and gate) row and target row of each request's draw position, for
// the draft kernel's residual mode.
// One warp per request: the residual mode's per-row constants, and the predecessor and
// gate row of the draw position (the one position the residual mode drafts over).
__global__ void verify_prep_kernel(const float* __restrict__ U, const uint16_t* __restrict__ W1,
                                   const uint16_t* __restrict__ W2, const float* __restrict__ H,
                                   const float* __restrict__ logq, const float* __restrict__ lse_t,
                                   const VerifySel* __restrict__ sel, int B, int K, int V, int r,
                                   float inv_td, int draft_greedy, ResRow* __restrict__ rows,
                                   uint16_t* __restrict__ H_sel, int32_t* __restrict__ prev_sel) {
  const int lane = threadIdx.x & 31;
  const int b = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (b >= B) return;
  const VerifySel s = sel[b];
  if (H != nullptr) {  // a bonus row needs no q: any valid gate row will do
    const float* hs = H + (static_cast<size_t>(b) * K + min(s.pos, K - 1)) * r;
    for (int i = lane; i < r; i += 32)
      H_sel[static_cast<size_t>(b) * r + i] = __bfloat16_as_ushort(__float2bfloat16_rn(hs[i]));
  }
  if (lane == 0) prev_sel[b] = s.prev;
  ResRow rr;
  rr.pos = s.pos;
  rr.offp2 = -lse_t[static_cast<size_t>(b) * (K + 1) + s.pos] * kLog2eV;
  rr.offq2 = -INFINITY;  // bonus, or a greedy draft: no draft mass to subtract
  rr.excl = (s.residual && draft_greedy) ? s.x : -1;
  if (s.residual && !draft_greedy) {
    const size_t row = static_cast<size_t>(b) * K + s.pos;
    const float lx = head_logit(U + row * V, W1, W2, H ? H + row * r : nullptr, V, r, s.prev,
                                s.x, lane);
    rr.offq2 = (__ldg(logq + row) - lx * inv_td) * kLog2eV;
  }
  if (lane == 0) rows[b] = rr;
}

}  // namespace

cudaError_t launch_target_stats(const float* P, const int32_t* ell, int B, int K, int kmax, int V,
                                float target_temperature, float* lse_t, int32_t* argmax_t,
                                cudaStream_t stream) {
  const int greedy_t = target_temperature > 0.f ? 0 : 1;
  const float inv_tt = greedy_t ? 1.f : 1.0f / target_temperature;
  verify_stats_kernel<<<B * (K + 1), kStatsThreads, 0, stream>>>(P, ell, K, kmax, V, inv_tt,
                                                                 greedy_t, lse_t, argmax_t);
  return cudaGetLastError();
}

cudaError_t launch_verify(const VerifyArgs& v, cudaStream_t stream, int* launches) {
  *launches = 0;
  const int greedy_t = v.target_temperature > 0.f ? 0 : 1;
  const int greedy_d = v.draft_temperature > 0.f ? 0 : 1;
  const float inv_tt = greedy_t ? 1.f : 1.0f / v.target_temperature;
  cudaError_t e = launch_target_stats(v.P, v.ell, v.B, v.K, v.K, v.V, v.target_temperature,
                                      v.lse_t, v.argmax_t, stream);
  if (e != cudaSuccess) return e;
  ++*launches;
  verify_accept_kernel<<<(v.B + 3) / 4, 128, 0, stream>>>(
      v.P, v.tokens, v.logq, v.anchors, v.ell, v.lse_t, v.argmax_t, v.B, v.K, v.V, inv_tt,
      greedy_t, greedy_d, v.seed_lo, v.seed_hi, v.n_acc, v.next_token, v.accept_prob, v.sel,
      v.status);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  ++*launches;
  return cudaSuccess;
}

cudaError_t launch_verify_prep(const VerifyArgs& v, cudaStream_t stream) {
  const int greedy_d = v.draft_temperature > 0.f ? 0 : 1;
  const float inv_td = greedy_d ? 1.f : 1.0f / v.draft_temperature;
  verify_prep_kernel<<<(v.B + 7) / 8, 256, 0, stream>>>(v.U, v.W1, v.W2, v.H, v.logq, v.lse_t,
                                                        v.sel, v.B, v.K, v.V, v.r, inv_td,
                                                        greedy_d, v.rows, v.H_sel, v.prev_sel);
  return cudaGetLastError();
}

}  // namespace dspark
