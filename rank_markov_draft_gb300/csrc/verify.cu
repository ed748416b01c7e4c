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
//                        Tt = 0), a pure HBM scan of the row, then that
//                        position's acceptance test (the draft's own
//                        log-probabilities give q(x)); the request's last CTA
//                        to finish ends the prefix at the first failed test
//                        and, for a sampled target, computes the offsets that
//                        turn the draft head's logits and the target logits at
//                        the draw position into log2 q and log2 p (the draft's
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
#include "rowscan.cuh"
#include "sm103.cuh"

namespace dspark {
namespace {

constexpr float kLog2eV = kScanLog2e;

__device__ __forceinline__ float uniform_of(uint32_t word) { return philox_uniform(word); }

// One CTA per row (b, k) of P [B, K+1, V]: the row's log-sum-exp of P / Tt (its argmax when
// Tt = 0) for the rows k <= L_b = ell_b (the window; K without ell); later rows only take
// part in the count.  The CTA of a drafted position k < L_b then runs that position's
// acceptance test, and the last CTA of request b to finish resolves the request (the
// accepted prefix ends at the first failed test) and, for a sampled target (v.rows set),
// prepares the draw at that position for the draft kernel's residual mode: the offsets that
// turn the draft head's logits and the target logits there into log2 q and log2 p (the
// draft's normaliser from its own log-probability of the rejected token, l(x) rebuilt by a
// dot product), and the draw position's predecessor and gate row.
__global__ void __launch_bounds__(kScanThreads) verify_stats_kernel(const VerifyArgs v,
                                                                    float inv_tt, float inv_td,
                                                                    int greedy, int draft_greedy) {
  // the residual draw that follows may start its prologue while the last rows are scanned
  griddep_launch_dependents();
  const int K = v.K, V = v.V;
  const int row = blockIdx.x;  // b * (K + 1) + k
  const int b = row / (K + 1), k = row - b * (K + 1);
  const int L = v.ell ? min(max(__ldg(v.ell + b), 0), K) : K;
  const float* __restrict__ P = v.P;
  __shared__ RowScanSmem sm;
  __shared__ int s_last;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // the row's statistic, final in thread 0
  int bi = 0;
  float lse = 0.f;
  if (k <= L) {
    scan_target_row(P + static_cast<size_t>(row) * V, V, inv_tt, greedy != 0, sm, lse, bi);
    if (threadIdx.x == 0) {
      if (greedy)
        v.argmax_t[row] = bi;
      else
        v.lse_t[row] = lse;
    }
  }
  if (threadIdx.x == 0) {
    if (k < L) {  // the acceptance test of drafted position k: accept with min(1, p / q)
      int x = __ldg(v.tokens + static_cast<size_t>(b) * K + k);
      if (x < 0 || x >= V) {
        record_error(v.status, kStatusDeviceOob);
        x = 0;
      }
      const float pr = greedy ? (x == bi ? 1.f : 0.f)
                              : expf(__ldg(P + static_cast<size_t>(row) * V + x) * inv_tt - lse);
      const float q = draft_greedy ? 1.f : expf(__ldg(v.logq + static_cast<size_t>(b) * K + k));
      const float a = (q > 0.f) ? fminf(1.f, pr / q) : 1.f;
      if (v.accept_prob) v.accept_prob[static_cast<size_t>(b) * K + k] = a;
      const Philox4 rnd = philox4x32_10(static_cast<uint32_t>(k), 0u, static_cast<uint32_t>(b),
                                        13u, v.seed_lo, v.seed_hi);
      if (!(uniform_of(rnd.w[0]) < a)) atomicOr(v.fail_mask + b, 1ull << k);
    } else if (k < K && v.accept_prob) {
      v.accept_prob[static_cast<size_t>(b) * K + k] = -1.f;
    }
    // publish this CTA's results, then count it; the (K + 1)-th CTA of request b resolves it
    __threadfence();
    const int before = atomicAdd(v.count + b, 1);
    s_last = before == K;
    if (before == K) v.count[b] = 0;  // every CTA of b has counted: ready for the next call
  }
  __syncthreads();
  if (!s_last || warp != 0) return;
  __threadfence();
  const unsigned long long fails = __ldcg(v.fail_mask + b);
  const int n = fails != 0ull ? __ffsll(static_cast<long long>(fails)) - 1 : L;  // < L if any
  // the draw: position n, from the residual at a rejection, else the bonus from p
  const bool rejected = n < L;
  const int pos = n;
  int x = rejected ? __ldg(v.tokens + static_cast<size_t>(b) * K + pos) : -1;
  int prev = (pos == 0) ? __ldg(v.anchors + b) : __ldg(v.tokens + static_cast<size_t>(b) * K + pos - 1);
  if (prev < 0 || prev >= V) {
    if (lane == 0) record_error(v.status, kStatusDeviceOob);
    prev = 0;
  }
  if (x >= V || (rejected && x < 0)) x = 0;
  if (lane == 0) {
    v.n_acc[b] = n;
    v.fail_mask[b] = 0ull;  // ready for the next call
    if (greedy) v.next_token[b] = __ldcg(v.argmax_t + static_cast<size_t>(b) * (K + 1) + pos);
  }
  if (v.rows == nullptr) return;
  if (v.H != nullptr) {  // a bonus row needs no q: any valid gate row will do
    const float* hs = v.H + (static_cast<size_t>(b) * K + min(pos, K - 1)) * v.r;
    for (int i = lane; i < v.r; i += 32)
      v.H_sel[static_cast<size_t>(b) * v.r + i] = __bfloat16_as_ushort(__float2bfloat16_rn(hs[i]));
  }
  if (lane == 0) v.prev_sel[b] = prev;
  ResRow rr;
  rr.pos = pos;
  rr.offp2 = -__ldcg(v.lse_t + static_cast<size_t>(b) * (K + 1) + pos) * kLog2eV;
  rr.offq2 = -INFINITY;  // bonus, or a greedy draft: no draft mass to subtract
  rr.excl = (rejected && draft_greedy) ? x : -1;
  if (rejected && !draft_greedy) {
    const size_t drow = static_cast<size_t>(b) * K + pos;
    const float lx = head_logit(v.U + drow * V, v.W1, v.W2, v.H ? v.H + drow * v.r : nullptr, V,
                                v.r, prev, x, lane);
    rr.offq2 = (__ldg(v.logq + drow) - lx * inv_td) * kLog2eV;
  }
  if (lane == 0) v.rows[b] = rr;
}

}  // namespace

cudaError_t launch_verify(const VerifyArgs& v, cudaStream_t stream, int* launches) {
  *launches = 0;
  const int greedy_t = v.target_temperature > 0.f ? 0 : 1;
  const int greedy_d = v.draft_temperature > 0.f ? 0 : 1;
  const float inv_tt = greedy_t ? 1.f : 1.0f / v.target_temperature;
  const float inv_td = greedy_d ? 1.f : 1.0f / v.draft_temperature;
  verify_stats_kernel<<<v.B * (v.K + 1), kScanThreads, 0, stream>>>(v, inv_tt, inv_td, greedy_t,
                                                                   greedy_d);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  ++*launches;
  return cudaSuccess;
}

}  // namespace dspark
