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
// comes from the row scan of the target logits, the draft's from the draft's
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
#include "sm103.cuh"

namespace dspark {
namespace {

constexpr float kLog2eL = 1.4426950408889634f;

__global__ void label_prep_kernel(const LabelPrepArgs a) {
  const int lane = threadIdx.x & 31;
  const int row = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);  // b * K + k
  if (row >= a.B * a.K) return;
  const int b = row / a.K, k = row - b * a.K;
  int x = __ldg(a.tokens + row);
  int prev = (k == 0) ? __ldg(a.anchors + b) : __ldg(a.tokens + row - 1);
  if (x < 0 || x >= a.V || prev < 0 || prev >= a.V) {
    if (lane == 0) record_error(a.status, kStatusDeviceOob);
    x = 0;
    prev = 0;
  }
  const size_t trow = static_cast<size_t>(b) * (a.K + 1) + k;  // target row of position k
  if (lane == 0) a.prev[row] = prev;
  if (a.inv_td == 0.f) {
    if (lane == 0) {
      a.label[row] = (a.inv_tt == 0.f)
                         ? ((x == __ldg(a.argmax_t + trow)) ? 1.f : 0.f)
                         : expf(__ldg(a.P + trow * a.V + x) * a.inv_tt - __ldg(a.lse_t + trow));
    }
    return;
  }
  const float* urow = a.U + (static_cast<size_t>(b) * a.K + k) * a.V;
  const float* hrow = a.H ? a.H + (static_cast<size_t>(b) * a.K + k) * a.r : nullptr;
  const float lx = head_logit(urow, a.W1, a.W2, hrow, a.V, a.r, prev, x, lane);
  const float offq2 = (__ldg(a.logq + row) - lx * a.inv_td) * kLog2eL;
  if (lane == 0) a.offq2[row] = offq2;
  if (a.inv_tt == 0.f) {
    int am = __ldg(a.argmax_t + trow);
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
  const int rows = a.B * a.K;
  label_prep_kernel<<<(rows + 7) / 8, 256, 0, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace dspark
