// label.cu -- acceptance label of each drafted position, per-row preparation.
//
// Source: DSpark explainer, "Confidence-scheduled verification": the label the
// confidence head is trained on is c*_k = 1 - TV(p^d_k, p^t_k), the acceptance
// probability of position k under speculative decoding, with p^d_k the draft
// head's softmax given the drafted predecessor and p^t_k the target's.  It is
// summed as sum_v min(p^d_k(v), p^t_k(v)).
//
// The sum over the vocabulary runs in the draft kernel's label mode, which
// needs both distributions' normalisers before its single pass: the target's
// comes from a scan of each target row (the kernel here, one CTA a row, which
// then prepares that row), the draft's from the draft's
// own log-probability of the drafted token, log q(x) = l(x) / Td - log Z_q, so
// that log2 q(v) = l(v) log2(e) / Td + offq2 with
//     offq2 = (log q(x) - l(x) / Td) log2(e),
// l(x) rebuilt here as U[x] + sum_i e_i W2[i, x] from the same bf16 operand
// (e = W1[prev] rounded, or W1[prev] * gate rounded to bf16) the kernel's MMA
// multiplies.  Where one side is greedy its distribution is one-hot and the
// label is a single probability, computed here outright:
//     draft greedy:  p^t(x)   (1 if x is the target's argmax, when both are)
//     target greedy: q(a), a the target's argmax.

#include <cstdint>

#include "headlogit.cuh"
#include "internal.h"
#include "rowscan.cuh"
#include "sm103.cuh"

namespace dspark {
namespace {

constexpr float kLog2eL = kScanLog2e;

// One CTA per drafted row (b, k), k < K: the scan of target row (b, k) (its log-sum-exp of
// P / Tt, or its argmax when the target is greedy), then, on warp 0, that row's
// preparation: the predecessor, the draft's log2 q offset and, where one side is greedy,
// the label itself.
__global__ void __launch_bounds__(kScanThreads) label_prep_kernel(const LabelPrepArgs a) {
  // the label pass that follows may start its prologue while the last rows are scanned
  griddep_launch_dependents();
  const int row = blockIdx.x;  // b * K + k
  const int b = row / a.K, k = row - b * a.K;
  const size_t trow = static_cast<size_t>(b) * (a.K + 1) + k;  // target row of position k
  __shared__ RowScanSmem sm;
  __shared__ float s_lse;
  __shared__ int s_argmax;
  float lse = 0.f;
  int am = 0;
  scan_target_row(a.P + trow * a.V, a.V, a.inv_tt, a.inv_tt == 0.f, sm, lse, am);
  if (threadIdx.x == 0) {
    if (a.inv_tt == 0.f)
      a.argmax_t[trow] = am;
    else
      a.lse_t[trow] = lse;
    s_lse = lse;
    s_argmax = am;
  }
  __syncthreads();
  if (threadIdx.x >= 32) return;
  const int lane = threadIdx.x;
  lse = s_lse;
  am = s_argmax;
  int x = __ldg(a.tokens + row);
  int prev = (k == 0) ? __ldg(a.anchors + b) : __ldg(a.tokens + row - 1);
  if (x < 0 || x >= a.V || prev < 0 || prev >= a.V) {
    if (lane == 0) record_error(a.status, kStatusDeviceOob);
    x = 0;
    prev = 0;
  }
  if (lane == 0) a.prev[row] = prev;
  if (a.inv_td == 0.f) {
    if (lane == 0) {
      a.label[row] = (a.inv_tt == 0.f) ? ((x == am) ? 1.f : 0.f)
                                       : expf(__ldg(a.P + trow * a.V + x) * a.inv_tt - lse);
    }
    return;
  }
  const float* urow = a.U + (static_cast<size_t>(b) * a.K + k) * a.V;
  const float* hrow = a.H ? a.H + (static_cast<size_t>(b) * a.K + k) * a.r : nullptr;
  const float lx = head_logit(urow, a.W1, a.W2, hrow, a.V, a.r, prev, x, lane);
  const float offq2 = (__ldg(a.logq + row) - lx * a.inv_td) * kLog2eL;
  if (lane == 0) a.offq2[row] = offq2;
  if (a.inv_tt == 0.f) {
    if (am < 0 || am >= a.V) {  // a target row without a finite logit
      if (lane == 0) record_error(a.status, kStatusDeviceOob);
      am = 0;
    }
    const float la = head_logit(urow, a.W1, a.W2, hrow, a.V, a.r, prev, am, lane);
    if (lane == 0) a.label[row] = fminf(1.f, exp2f(la * a.inv_td * kLog2eL + offq2));
  }
}

}  // namespace

cudaError_t launch_label_prep(const LabelPrepArgs& a, cudaStream_t stream) {
  label_prep_kernel<<<a.B * a.K, kScanThreads, 0, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace dspark
