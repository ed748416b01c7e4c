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
// bits | inverted position | inverted request) and sorted descending by a
// bitonic network held in registers (E keys a thread: strides inside a thread
// in registers, inside a warp by shuffles, wider ones through shared memory);
// their survivals are summed by a block scan in that order, the first admission
// that would not raise Theta cuts the list, and each request's length is the
// number of its admitted candidates.

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

__device__ __forceinline__ unsigned long long shfl_xor_u64(unsigned long long v, int m) {
  const uint32_t lo = __shfl_xor_sync(0xFFFFFFFFu, static_cast<uint32_t>(v), m);
  const uint32_t hi = __shfl_xor_sync(0xFFFFFFFFu, static_cast<uint32_t>(v >> 32), m);
  return (static_cast<unsigned long long>(hi) << 32) | lo;
}

// one compare-exchange in a bitonic stage (size, stride), sorting descending: the lower index
// of a pair in a descending block keeps the larger key, and so does the upper index of a pair
// in an ascending block.  For stride >= E the answer is the same for all of a thread's keys
// (their indices differ only below bit log2 E), so it is taken once per stage.
__device__ __forceinline__ bool bitonic_keeps_max(int i, int size, int stride) {
  return ((i & stride) == 0) == ((i & size) == 0);
}

__device__ __forceinline__ unsigned long long bitonic_keep(unsigned long long x,
                                                           unsigned long long y, bool keep_max) {
  return ((x > y) == keep_max) ? x : y;  // equal keys: either
}

// E keys per thread, thread t holding sorted positions t * E .. t * E + E - 1; the block has
// n_pow2 / E threads (at least one warp)
template <int E>
__global__ void __launch_bounds__(kSchedThreads) schedule_kernel(const float* __restrict__ a, int R,
                                                                 int K, const float* __restrict__ sps,
                                                                 int32_t* __restrict__ ell,
                                                                 float* __restrict__ theta) {
  extern __shared__ __align__(16) unsigned long long s_key[];  // [n_pow2]: exchange, then counts
  __shared__ float s_part[kSchedThreads / 32];
  __shared__ int s_min[kSchedThreads / 32];
  const int T = blockDim.x, n_pow2 = T * E, n = R * K;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nw = T >> 5;
  if (n == 0) {  // nothing to admit: B = R
    for (int i = tid; i < R; i += T) ell[i] = 0;
    if (tid == 0 && theta != nullptr) *theta = static_cast<float>(R) * sps[R];
    return;
  }
  const int i0 = tid * E;
  // the SPS values this thread's cut test reads, loaded before the sort (E + 1 entries)
  constexpr bool kPreload = E <= 4;
  float sp[kPreload ? E + 1 : 1];
  if (kPreload) {
#pragma unroll
    for (int e = 0; e <= E; ++e) sp[e] = i0 + e <= n ? __ldg(sps + R + i0 + e) : 0.f;
  }
  // keys: ordered survival bits | inverted position | inverted request (0 pads, sorting last)
  unsigned long long x[E];
  {
    int r = i0 / K, k = i0 - r * K;
#pragma unroll
    for (int e = 0; e < E; ++e) {
      x[e] = 0ull;
      if (i0 + e < n)
        x[e] = (static_cast<unsigned long long>(ordered_bits32(__ldg(a + i0 + e))) << 32) |
               (static_cast<unsigned long long>(0xFFFFu - static_cast<uint32_t>(k)) << 16) |
               static_cast<unsigned long long>(0xFFFFu - static_cast<uint32_t>(r));
      if (++k == K) {
        k = 0;
        ++r;
      }
    }
  }
  // bitonic sort, descending: strides of 32 E and more exchange through shared memory, the
  // others between the lanes of a warp (stride / E) or inside a thread (stride < E)
  for (int size = 2; size <= n_pow2; size <<= 1) {
    int stride = size >> 1;
    for (; stride >= 32 * E; stride >>= 1) {
      __syncthreads();  // the last stage's readers are done
#pragma unroll
      for (int e = 0; e < E; ++e) s_key[i0 + e] = x[e];
      __syncthreads();
      const bool keep_max = bitonic_keeps_max(i0, size, stride);
#pragma unroll
      for (int e = 0; e < E; ++e) x[e] = bitonic_keep(x[e], s_key[(i0 + e) ^ stride], keep_max);
    }
    for (; stride >= E; stride >>= 1) {
      const int m = stride / E;
      const bool keep_max = bitonic_keeps_max(i0, size, stride);
#pragma unroll
      for (int e = 0; e < E; ++e) x[e] = bitonic_keep(x[e], shfl_xor_u64(x[e], m), keep_max);
    }
#pragma unroll
    for (int s = E / 2; s > 0; s >>= 1) {
      if (s < size) {
#pragma unroll
        for (int e = 0; e < E; ++e) {
          if ((e & s) == 0) {
            const bool desc = ((i0 + e) & size) == 0;
            const unsigned long long p = x[e], q = x[e + s];
            const unsigned long long hi = p > q ? p : q, lo = p > q ? q : p;
            x[e] = desc ? hi : lo;
            x[e + s] = desc ? lo : hi;
          }
        }
      }
    }
  }
  // inclusive prefix sums of the survivals in rank order: the thread's own run, then an
  // exclusive scan of the thread totals
  float run[E];
  float tot = 0.f;
#pragma unroll
  for (int e = 0; e < E; ++e) {
    tot += i0 + e < n ? from_ordered32(static_cast<uint32_t>(x[e] >> 32)) : 0.f;
    run[e] = tot;
  }
  float incl = tot;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const float o = __shfl_up_sync(0xFFFFFFFFu, incl, off);
    if (lane >= off) incl += o;
  }
  if (lane == 31) s_part[warp] = incl;
  __syncthreads();  // also: every thread is past its last read of the exchange buffer
  if (warp == 0) {
    float w = lane < nw ? s_part[lane] : 0.f;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const float o = __shfl_up_sync(0xFFFFFFFFu, w, off);
      if (lane >= off) w += o;
    }
    if (lane < nw) s_part[lane] = w;  // inclusive over warps
  }
  int* s_cnt = reinterpret_cast<int*>(s_key);  // admitted candidates per request (R <= n)
  for (int i = tid; i < R; i += T) s_cnt[i] = 0;
  __syncthreads();
  const float base = incl - tot + (warp > 0 ? s_part[warp - 1] : 0.f);
  // the first candidate whose admission would not raise Theta = (R + sum) * SPS(R + i)
  const float Rf = static_cast<float>(R);
  int mine = n;
  float th_cut = 0.f;  // Theta with this thread's admitted prefix, at its first failure
#pragma unroll
  for (int e = 0; e < E; ++e) {
    const int i = i0 + e;
    if (i < n && mine == n) {
      const float s0 = kPreload ? sp[e] : __ldg(sps + R + i);
      const float s1 = kPreload ? sp[e + 1] : __ldg(sps + R + i + 1);
      const float th_prev = (Rf + (base + (e > 0 ? run[e - 1] : 0.f))) * s0;
      const float th_next = (Rf + (base + run[e])) * s1;
      if (!(th_next > th_prev)) {
        mine = i;
        th_cut = th_prev;
      }
    }
  }
  const int wmin = __reduce_min_sync(0xFFFFFFFFu, mine);
  if (lane == 0) s_min[warp] = wmin;
  __syncthreads();
  int cut = n;
  for (int w = 0; w < nw; ++w) cut = min(cut, s_min[w]);
  if (theta != nullptr) {
    if (cut < n && mine == cut) *theta = th_cut;  // the thread that holds the cut
    if (cut == n) {  // everything admitted: the holder of the last candidate
#pragma unroll
      for (int e = 0; e < E; ++e)
        if (i0 + e == n - 1) *theta = (Rf + (base + run[e])) * __ldg(sps + R + n);
    }
  }
  // each request's length is the number of its admitted candidates
#pragma unroll
  for (int e = 0; e < E; ++e)
    if (i0 + e < cut)
      atomicAdd(&s_cnt[static_cast<int>(0xFFFFu - static_cast<uint32_t>(x[e] & 0xFFFFull))], 1);
  __syncthreads();
  for (int i = tid; i < R; i += T) ell[i] = s_cnt[i];
}

}  // namespace

size_t schedule_smem_bytes(int n_pow2) { return static_cast<size_t>(n_pow2) * 8; }

template <int E>
static cudaError_t launch_schedule_e(const float* a, int R, int K, const float* sps, int32_t* ell,
                                     float* theta, int n_pow2, cudaStream_t stream) {
  const size_t smem = schedule_smem_bytes(n_pow2);
  cudaError_t e = cudaFuncSetAttribute(reinterpret_cast<const void*>(&schedule_kernel<E>),
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  schedule_kernel<E><<<1, n_pow2 / E, smem, stream>>>(a, R, K, sps, ell, theta);
  return cudaGetLastError();
}

cudaError_t launch_schedule(const float* a, int R, int K, const float* sps, int32_t* ell,
                            float* theta, cudaStream_t stream) {
  int n_pow2 = 32;  // at least one warp of one key each
  while (n_pow2 < R * K) n_pow2 <<= 1;
  switch (n_pow2 <= kSchedThreads ? 1 : n_pow2 / kSchedThreads) {
    case 1: return launch_schedule_e<1>(a, R, K, sps, ell, theta, n_pow2, stream);
    case 2: return launch_schedule_e<2>(a, R, K, sps, ell, theta, n_pow2, stream);
    case 4: return launch_schedule_e<4>(a, R, K, sps, ell, theta, n_pow2, stream);
    case 8: return launch_schedule_e<8>(a, R, K, sps, ell, theta, n_pow2, stream);
    case 16: return launch_schedule_e<16>(a, R, K, sps, ell, theta, n_pow2, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace dspark
