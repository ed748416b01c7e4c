// schedule.cu -- load-aware greedy prefix scheduler on the GPU.
//
// Source: DSpark explainer, "Hardware-aware prefix scheduling": R requests,
// request r verifies a prefix of length ell_r, the target batch is
// B = sum_r (1 + ell_r) tokens and, with survival a_{r,j} of extension (r, j),
// Theta(S) = (R + sum_S a_{r,j}) SPS(B); starting at B = R, candidate
// extensions are ranked globally by survival probability and admitted while
// Theta increases (strictly); request r cannot admit j + 1 without j.  The
// ranking is (survival desc, position asc, request asc): survival never grows
// along a request (a product of probabilities), so this keeps prefixes whole.
//
// One CTA: the R x K candidates are packed into 64-bit keys (ordered survival
// bits | inverted position | inverted request), sorted descending by a bitonic
// network in shared memory, their survivals summed by a block scan in that
// order, and the first admission that would not raise Theta cuts the list; each
// request's length is one past its last admitted position (no atomics).

#include <cstdint>

#include "internal.h"

namespace dspark {
namespace {

constexpr int kSchedThreads = 1024;

__device__ __forceinline__ uint32_t ordered_bits32(float f) {
  const uint32_t b = __float_as_uint(f);
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

__device__ __forceinline__ float from_ordered32(uint32_t o) {
  return __uint_as_float((o & 0x80000000u) ? (o & 0x7FFFFFFFu) : ~o);
}

__global__ void __launch_bounds__(kSchedThreads) schedule_kernel(const float* __restrict__ a, int R,
                                                                 int K, const float* __restrict__ sps,
                                                                 int n_pow2, int32_t* __restrict__ ell,
                                                                 float* __restrict__ theta) {
  extern __shared__ __align__(16) unsigned long long s_key[];  // [n_pow2]
  float* s_sum = reinterpret_cast<float*>(s_key + n_pow2);     // [n_pow2] inclusive prefix sums
  __shared__ int s_cut;
  __shared__ float s_part[kSchedThreads / 32];
  const int n = R * K;
  const int tid = threadIdx.x;
  for (int i = tid; i < R; i += kSchedThreads) ell[i] = 0;
  for (int i = tid; i < n_pow2; i += kSchedThreads) {
    unsigned long long key = 0ull;  // padding sorts after every candidate
    if (i < n) {
      const int r = i / K, k = i - r * K;
      key = (static_cast<unsigned long long>(ordered_bits32(a[i])) << 32) |
            (static_cast<unsigned long long>(0xFFFFu - static_cast<uint32_t>(k)) << 16) |
            static_cast<unsigned long long>(0xFFFFu - static_cast<uint32_t>(r));
    }
    s_key[i] = key;
  }
  if (tid == 0) s_cut = n;
  __syncthreads();
  // bitonic sort, descending: every stage is n_pow2 / 2 compare-exchanges, one pair per
  // thread at a time; a stage with stride < 32 keeps each warp inside its own 64-key
  // block (pairs 32w .. 32w + 31 cover keys 64w .. 64w + 63), so it needs only a warp
  // barrier, and a block barrier is taken only after a stage with a larger stride
  const int pairs = n_pow2 >> 1;
  for (int size = 2; size <= n_pow2; size <<= 1) {
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      for (int t = tid; t < pairs; t += kSchedThreads) {
        // pair t: (t / stride) * 2 * stride + t % stride (stride is a power of two)
        const int i = 2 * t - (t & (stride - 1)), j = i + stride;
        const unsigned long long x = s_key[i], y = s_key[j];
        const bool desc = (i & size) == 0;
        if (desc ? (x < y) : (x > y)) {
          s_key[i] = y;
          s_key[j] = x;
        }
      }
      if (stride >= 32 || pairs > kSchedThreads || (stride == 1 && size >= 64)) {
        __syncthreads();
      } else {
        __syncwarp();
      }
    }
  }
  __syncthreads();
  // inclusive prefix sums of the survivals in rank order: each thread sums a
  // contiguous slice, the slice totals are scanned by warp 0
  const int per = (n_pow2 + kSchedThreads - 1) / kSchedThreads;
  const int i0 = tid * per, i1 = min(n, i0 + per);
  float run = 0.f;
  for (int i = i0; i < i1; ++i) {
    run += from_ordered32(static_cast<uint32_t>(s_key[i] >> 32));
    s_sum[i] = run;
  }
  // exclusive scan of the per-thread totals
  const int lane = tid & 31, warp = tid >> 5;
  float tot = run, incl = run;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const float o = __shfl_up_sync(0xFFFFFFFFu, incl, off);
    if (lane >= off) incl += o;
  }
  if (lane == 31) s_part[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    float w = s_part[lane];
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const float o = __shfl_up_sync(0xFFFFFFFFu, w, off);
      if (lane >= off) w += o;
    }
    s_part[lane] = w;  // inclusive over warps
  }
  __syncthreads();
  const float base = incl - tot + (warp > 0 ? s_part[warp - 1] : 0.f);
  for (int i = i0; i < i1; ++i) s_sum[i] += base;
  __syncthreads();
  // the first candidate whose admission would not raise Theta: each thread's first such
  // candidate (its indices ascend), the warp's minimum, one shared atomic per warp
  int mine = n;
  for (int i = tid; i < n; i += kSchedThreads) {
    const float prev = static_cast<float>(R) + (i > 0 ? s_sum[i - 1] : 0.f);
    const float cur = static_cast<float>(R) + s_sum[i];
    const float th_prev = prev * sps[R + i];
    const float th_next = cur * sps[R + i + 1];
    if (!(th_next > th_prev)) {
      mine = i;
      break;
    }
  }
  mine = __reduce_min_sync(0xFFFFFFFFu, mine);
  if (lane == 0 && mine < n) atomicMin(&s_cut, mine);
  __syncthreads();
  const int cut = s_cut;
  if (tid == 0 && theta != nullptr)
    *theta = (static_cast<float>(R) + (cut > 0 ? s_sum[cut - 1] : 0.f)) * sps[R + cut];
  __syncthreads();
  // every candidate's rank (reusing the prefix sums' storage); the admitted positions of a
  // request form a prefix, so its last admitted position k gives ell = k + 1 (no atomics)
  int* s_rank = reinterpret_cast<int*>(s_sum);
  for (int i = tid; i < n; i += kSchedThreads) {
    const unsigned long long key = s_key[i];
    const int r = static_cast<int>(0xFFFFu - static_cast<uint32_t>(key & 0xFFFFull));
    const int k = static_cast<int>(0xFFFFu - static_cast<uint32_t>((key >> 16) & 0xFFFFull));
    s_rank[r * K + k] = i;
  }
  __syncthreads();
  for (int idx = tid; idx < n; idx += kSchedThreads) {
    const int r = idx / K, k = idx - r * K;
    if (s_rank[idx] < cut && (k + 1 == K || s_rank[idx + 1] >= cut)) ell[r] = k + 1;
  }
}

}  // namespace

size_t schedule_smem_bytes(int n_pow2) { return static_cast<size_t>(n_pow2) * (8 + 4); }

cudaError_t launch_schedule(const float* a, int R, int K, const float* sps, int32_t* ell,
                            float* theta, cudaStream_t stream) {
  int n_pow2 = 1;
  while (n_pow2 < R * K) n_pow2 <<= 1;
  const size_t smem = schedule_smem_bytes(n_pow2);
  cudaError_t e = cudaFuncSetAttribute(reinterpret_cast<const void*>(&schedule_kernel),
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  schedule_kernel<<<1, kSchedThreads, smem, stream>>>(a, R, K, sps, n_pow2, ell, theta);
  return cudaGetLastError();
}

}  // namespace dspark
