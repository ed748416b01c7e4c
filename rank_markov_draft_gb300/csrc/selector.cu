// selector.cu -- Selector-style top-k execution of the Markov head.
//
// Source: "DFlash-2's Selector and DSpark's Markov Head: An Equivalence
// Observation", sections "Where the parallelism comes from" (fix the top-16
// candidate sets of the base logits; precompute the 16 x 16 calibrations of
// adjacent positions in parallel; then a light sequential walk) and "Two
// implications" (the same top-k execution for a trained Markov head, with
// A = W1 and B = W2^T); the score S_t(a, b) = U_t(b) + <A(a) (.) H(h_t), B(b)>
// is from "What the two methods do".
//
// Three kernels:
//   topk_kernel        one CTA per (request, position) row of U, a pure
//                      streaming scan: each warp keeps a sorted top-k list in
//                      its lanes and only touches it for the rare element that
//                      beats the current k-th entry; the CTA merges its 8 lists.
//   pair_scores_kernel one CTA per (request, position): gathers the k
//                      predecessor rows of A (times the gate) and the k
//                      candidate rows of B into shared memory, then computes
//                      the k x k dot products on CUDA cores (0.5 GFLOP for a
//                      256 x 16 block: not worth the tensor cores).
//   walk_kernel        one warp per request, lanes = candidates: Gumbel-max
//                      with noise keyed by the candidate's token id, softmax
//                      over the k candidates, optional fused confidence head.

#include <cstdint>

#include "confidence.cuh"
#include "internal.h"
#include "philox.cuh"
#include "sm103.cuh"

namespace dspark {
namespace {

__device__ __forceinline__ bool better(float av, int ai, float bv, int bi) {
  return av > bv || (av == bv && ai < bi);
}

// Warp-resident sorted list: lane j < topk holds entry j (best first).
struct WarpTopk {
  float lv;
  int li;
  float tv;  // current k-th value (threshold)
  int ti;

  __device__ __forceinline__ void init() {
    lv = -INFINITY;
    li = 0x7FFFFFFF;
    tv = -INFINITY;
    ti = 0x7FFFFFFF;
  }

  // Insert (x, xi), known to beat the threshold; all 32 lanes call this with
  // the same (x, xi).
  __device__ __forceinline__ void insert(float x, int xi, int lane, int topk) {
    const bool above = (lane < topk) && better(lv, li, x, xi);
    const int pos = __popc(__ballot_sync(0xFFFFFFFFu, above));
    const float uv = __shfl_up_sync(0xFFFFFFFFu, lv, 1);
    const int ui = __shfl_up_sync(0xFFFFFFFFu, li, 1);
    if (lane > pos && lane < topk) {
      lv = uv;
      li = ui;
    }
    if (lane == pos) {
      lv = x;
      li = xi;
    }
    tv = __shfl_sync(0xFFFFFFFFu, lv, topk - 1);
    ti = __shfl_sync(0xFFFFFFFFu, li, topk - 1);
  }

  // Offer one candidate per lane (valid = false: none); inserts every one
  // that beats the running threshold.
  __device__ __forceinline__ void offer(float x, int xi, bool valid, int lane, int topk) {
    unsigned mask = __ballot_sync(0xFFFFFFFFu, valid && better(x, xi, tv, ti));
    while (mask) {
      const int src = __ffs(mask) - 1;
      mask &= mask - 1;
      const float cx = __shfl_sync(0xFFFFFFFFu, x, src);
      const int ci = __shfl_sync(0xFFFFFFFFu, xi, src);
      if (better(cx, ci, tv, ti)) insert(cx, ci, lane, topk);
    }
  }
};

constexpr int kTopkWarps = 8;

__global__ void __launch_bounds__(kTopkWarps * 32) topk_kernel(const float* __restrict__ U, int V,
                                                               int topk, int32_t* __restrict__ cand,
                                                               float* __restrict__ cval) {
  __shared__ float s_v[kTopkWarps][32];
  __shared__ int s_i[kTopkWarps][32];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const size_t row = blockIdx.x;
  const float* u = U + row * V;
  // contiguous segment per warp, a multiple of 4 tokens
  const int seg = ((V + kTopkWarps - 1) / kTopkWarps + 3) & ~3;
  const int s0 = warp * seg;
  const int s1 = min(V, s0 + seg);
  WarpTopk list;
  list.init();
  constexpr int kUnroll = 4;
  for (int base = s0; base < s1; base += 128 * kUnroll) {
    float4 x[kUnroll];
#pragma unroll
    for (int r = 0; r < kUnroll; ++r) {
      const int idx = base + r * 128 + lane * 4;
      x[r] = (idx < s1) ? __ldcs(reinterpret_cast<const float4*>(u + idx))
                        : make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
    }
#pragma unroll
    for (int r = 0; r < kUnroll; ++r) {
      const int idx = base + r * 128 + lane * 4;
      const bool in = idx < s1;
      list.offer(x[r].x, idx + 0, in, lane, topk);
      list.offer(x[r].y, idx + 1, in, lane, topk);
      list.offer(x[r].z, idx + 2, in, lane, topk);
      list.offer(x[r].w, idx + 3, in, lane, topk);
    }
  }
  s_v[warp][lane] = list.lv;
  s_i[warp][lane] = list.li;
  __syncthreads();
  if (warp == 0) {
    for (int w = 1; w < kTopkWarps; ++w) {
      const float x = s_v[w][lane];
      const int xi = s_i[w][lane];
      list.offer(x, xi, lane < topk && xi != 0x7FFFFFFF, lane, topk);
    }
    if (lane < topk) {
      cand[row * topk + lane] = list.li;
      cval[row * topk + lane] = list.lv;
    }
  }
}

__global__ void __launch_bounds__(256) pair_scores_kernel(
    const int32_t* __restrict__ cand, const float* __restrict__ cval,
    const uint16_t* __restrict__ A, const uint16_t* __restrict__ Bt,
    const int32_t* __restrict__ anchors, const float* __restrict__ H, int K, int V, int r,
    int topk, float* __restrict__ S, int* status) {
  extern __shared__ float sm[];
  const int ld = r + 1;  // padded rows: conflict-free column walks
  float* sAp = sm;                 // [topk][r + 1]
  float* sBc = sm + topk * ld;     // [topk][r + 1]
  __shared__ int s_prev[kMaxTopk], s_cand[kMaxTopk];
  const size_t bt = blockIdx.x;
  const int b = static_cast<int>(bt / K), t = static_cast<int>(bt % K);
  if (threadIdx.x < topk) {
    int pv = (t == 0) ? anchors[b] : cand[(bt - 1) * topk + threadIdx.x];
    int cv = cand[bt * topk + threadIdx.x];
    if (pv < 0 || pv >= V || cv < 0 || cv >= V) {
      record_error(status, kStatusDeviceOob);
      pv = min(max(pv, 0), V - 1);
      cv = min(max(cv, 0), V - 1);
    }
    s_prev[threadIdx.x] = pv;
    s_cand[threadIdx.x] = cv;
  }
  __syncthreads();
  const float* g = (H != nullptr) ? H + bt * r : nullptr;
  const int units = r / 8;  // 8 bf16 per 16-byte load
  for (int idx = threadIdx.x; idx < topk * units; idx += blockDim.x) {
    const int i = idx / units, q0 = (idx % units) * 8;
    const uint4 av = __ldg(reinterpret_cast<const uint4*>(A + static_cast<size_t>(s_prev[i]) * r + q0));
    const uint4 bv = __ldg(reinterpret_cast<const uint4*>(Bt + static_cast<size_t>(s_cand[i]) * r + q0));
    const uint32_t aw[4] = {av.x, av.y, av.z, av.w};
    const uint32_t bw[4] = {bv.x, bv.y, bv.z, bv.w};
#pragma unroll
    for (int h = 0; h < 4; ++h) {
      float a0 = __uint_as_float(aw[h] << 16), a1 = __uint_as_float(aw[h] & 0xFFFF0000u);
      if (g != nullptr) {
        a0 *= __ldg(g + q0 + 2 * h);
        a1 *= __ldg(g + q0 + 2 * h + 1);
      }
      sAp[i * ld + q0 + 2 * h] = a0;
      sAp[i * ld + q0 + 2 * h + 1] = a1;
      sBc[i * ld + q0 + 2 * h] = __uint_as_float(bw[h] << 16);
      sBc[i * ld + q0 + 2 * h + 1] = __uint_as_float(bw[h] & 0xFFFF0000u);
    }
  }
  __syncthreads();
  for (int pidx = threadIdx.x; pidx < topk * topk; pidx += blockDim.x) {
    const int i = pidx / topk, j = pidx % topk;
    const float* ar = sAp + i * ld;
    const float* br = sBc + j * ld;
    float acc = 0.f;
    for (int q = 0; q < r; ++q) acc = fmaf(ar[q], br[q], acc);
    S[(bt * topk + i) * topk + j] = __ldg(cval + bt * topk + j) + acc;
  }
}

__global__ void __launch_bounds__(128) walk_kernel(
    const int32_t* __restrict__ cand, const float* __restrict__ S,
    const int32_t* __restrict__ anchors, const uint16_t* __restrict__ A, int B, int K, int V,
    int r, int topk, float inv_t, int sample, uint32_t seed_lo, uint32_t seed_hi,
    int32_t* __restrict__ tokens, float* __restrict__ logprobs, dspark_conf_args conf,
    int conf_on, int* status) {
  const int lane = threadIdx.x & 31;
  const int b = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (b >= B) return;
  int slot = 0;
  int prev_tok = anchors[b];
  float surv = 1.f;
  int len = 0;
  bool open = true;
  for (int t = 0; t < K; ++t) {
    const size_t bt = static_cast<size_t>(b) * K + t;
    const bool live = lane < topk;
    const float sv = live ? S[(bt * topk + slot) * topk + lane] : -INFINITY;
    const int c = live ? cand[bt * topk + lane] : 0x7FFFFFFF;
    const float z = sv * inv_t;
    float s = z;
    if (sample && live) {
      const Philox4 rnd = philox4x32_10(static_cast<uint32_t>(c) >> 2, static_cast<uint32_t>(t),
                                        static_cast<uint32_t>(b), 0u, seed_lo, seed_hi);
      const float u = philox_uniform(rnd.w[c & 3]);
      s = z - logf(neg_log_uniform_accurate(u));
    }
    // argmax by (score desc, token id asc)
    float best_s = live ? s : -INFINITY;
    int best_c = c, best_j = lane;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      const float os = __shfl_xor_sync(0xFFFFFFFFu, best_s, off);
      const int oc = __shfl_xor_sync(0xFFFFFFFFu, best_c, off);
      const int oj = __shfl_xor_sync(0xFFFFFFFFu, best_j, off);
      if (better(os, oc, best_s, best_c)) {
        best_s = os;
        best_c = oc;
        best_j = oj;
      }
    }
    float m = live ? z : -INFINITY;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, off));
    float e = live ? expf(z - m) : 0.f;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) e += __shfl_xor_sync(0xFFFFFFFFu, e, off);
    const float zw = __shfl_sync(0xFFFFFFFFu, z, best_j);
    if (best_c < 0 || best_c >= V) {
      if (lane == 0) record_error(status, kStatusDeviceOob);
      best_c = 0;
    }
    if (lane == 0) {
      tokens[bt] = best_c;
      logprobs[bt] = zw - (m + logf(e));
    }
    if (conf_on) {
      const uint16_t* emb = conf.with_markov ? A + static_cast<size_t>(prev_tok) * r : nullptr;
      const float zc = confidence_logit(conf.h + bt * conf.d, conf.d, conf.w, emb, r, conf.bias,
                                        lane);
      const float cc = sigmoidf_accurate(zc);
      surv *= cc;
      if (open && surv >= conf.threshold) {
        len = t + 1;
      } else {
        open = false;
      }
      if (lane == 0) {
        conf.conf[bt] = cc;
        conf.cumprod[bt] = surv;
      }
    }
    slot = best_j;
    prev_tok = best_c;
  }
  if (conf_on && lane == 0) conf.verify_len[b] = len;
}

}  // namespace

cudaError_t launch_topk(const float* U, int rows, int V, int topk, int32_t* cand, float* cval,
                        cudaStream_t stream) {
  topk_kernel<<<rows, kTopkWarps * 32, 0, stream>>>(U, V, topk, cand, cval);
  return cudaGetLastError();
}

cudaError_t launch_pair_scores(const int32_t* cand, const float* cval, const uint16_t* A,
                               const uint16_t* Bt, const int32_t* anchors, const float* H,
                               int B, int K, int V, int r, int topk, float* S, int* status,
                               cudaStream_t stream) {
  const size_t smem = 2ull * topk * (r + 1) * sizeof(float);
  cudaError_t err = cudaFuncSetAttribute(reinterpret_cast<const void*>(&pair_scores_kernel),
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
  if (err != cudaSuccess) return err;
  pair_scores_kernel<<<B * K, 256, smem, stream>>>(cand, cval, A, Bt, anchors, H, K, V, r, topk,
                                                  S, status);
  return cudaGetLastError();
}

cudaError_t launch_walk(const int32_t* cand, const float* S, const int32_t* anchors,
                        const uint16_t* A, int B, int K, int V, int r, int topk, float inv_t,
                        int sample, uint32_t seed_lo, uint32_t seed_hi, int32_t* tokens,
                        float* logprobs, const dspark_conf_args* conf, int* status,
                        cudaStream_t stream) {
  dspark_conf_args c{};
  if (conf != nullptr) c = *conf;
  const int warps = 4;
  walk_kernel<<<(B + warps - 1) / warps, warps * 32, 0, stream>>>(
      cand, S, anchors, A, B, K, V, r, topk, inv_t, sample, seed_lo, seed_hi, tokens, logprobs, c,
      conf != nullptr ? 1 : 0, status);
  return cudaGetLastError();
}

}  // namespace dspark
