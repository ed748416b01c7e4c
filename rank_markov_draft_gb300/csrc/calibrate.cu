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
// One thread-block cluster (16 CTAs where the device allows it, else 8) splits
// the rows; the positions and rounds run in order (each round needs the last
// one's interval, each position the earlier temperatures).  Lane g of every
// warp evaluates grid point g, so a warp takes one row at a time for all 32
// points (the row's logit z_k, survival before k and label product through k
// are broadcast from shared memory, where each CTA keeps them for its rows and
// advances them once per position).  Each lane keeps a compensated fp32 sum;
// the CTA adds its warps as float pairs (hi + lo), and after one cluster
// barrier per round every CTA adds the CTAs' partials in rank order from
// distributed shared memory, so all of them take the same decision with no
// broadcast.  Only the interval of ln tau is kept in fp64, by one warp.

#include <cstdint>

#include "internal.h"

namespace dspark {
namespace {

constexpr int kStsThreads = 1024;
constexpr int kStsWarps = kStsThreads / 32;
constexpr int kStsG = 32;            // grid points per round: one per lane
constexpr int kStsR = 8;             // rounds per position
constexpr int kStsTileRows = 8192;   // rows a CTA holds in shared memory at once
constexpr int kStsRowsPerCta = 256;  // fewer rows than this per CTA: a smaller cluster
constexpr int kStsMaxCluster = 16;
static_assert(kStsWarps == kStsG, "warp w reduces grid point w over the CTA's warps");

__device__ __forceinline__ float logit_clamped(float c) {
  const float lo = 5.9604645e-08f;  // 2^-24
  c = fminf(fmaxf(c, lo), 1.0f - lo);
  return logf(c) - log1pf(-c);
}

__device__ __forceinline__ float sigmoid_f(float z) { return 1.0f / (1.0f + expf(-z)); }

__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

__device__ __forceinline__ uint32_t cluster_size() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(r));
  return r;
}

// every thread of every CTA in the cluster; writes before it are visible after it
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
  asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// a loss as an unevaluated sum hi + lo of two floats, |lo| <= ulp(hi) / 2: fp32 arithmetic
// throughout (fp64 runs at a small fraction of the fp32 rate on this part)
struct Pair {
  float hi, lo;
};

// the sum of two pairs: Knuth's two-sum of the high parts (its error term is exact, so the
// result does not depend on the order of the operands), then renormalised
__device__ __forceinline__ Pair pair_add(Pair a, Pair b) {
  const float s = a.hi + b.hi;
  const float bb = s - a.hi;
  const float e = (a.hi - (s - bb)) + (b.hi - bb);
  const float lo = e + (a.lo + b.lo);
  const float hi = s + lo;
  return {hi, lo - (hi - s)};
}

__device__ __forceinline__ bool pair_less(Pair a, Pair b) {
  return a.hi < b.hi || (a.hi == b.hi && a.lo < b.lo);
}

__device__ __forceinline__ Pair pair_shfl_xor(Pair a, int off) {
  return {__shfl_xor_sync(0xFFFFFFFFu, a.hi, off), __shfl_xor_sync(0xFFFFFFFFu, a.lo, off)};
}

// (volatile: kept after the cluster barrier, and the loads of one round issued together)
__device__ __forceinline__ Pair ld_cluster_pair(const Pair* p, uint32_t rank) {
  const uint32_t local = static_cast<uint32_t>(__cvta_generic_to_shared(p));
  uint32_t remote;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(local), "r"(rank));
  Pair v;
  asm volatile("ld.shared::cluster.v2.f32 {%0, %1}, [%2];" : "=f"(v.hi), "=f"(v.lo) : "r"(remote));
  return v;
}

// the interval [x0, x0 + 31 step] of a round as the 32 grid points' 1 / tau = exp(-x), one per
// lane of a warp (x in fp64: the last rounds' steps are below fp32's resolution of ln tau)
__device__ __forceinline__ void grid_inverses(double x0, double step, int lane, float* s_inv) {
  s_inv[lane] = expf(-static_cast<float>(x0 + step * lane));
}

// row state at position k from scratch: z_k, the survival before k under the fitted
// temperatures, the label product through k (the same products, in the same order, as the
// per-position update below)
__device__ __forceinline__ void row_from_scratch(const float* __restrict__ crow,
                                                 const float* __restrict__ lrow, int k,
                                                 const float* s_inv_tau, float& z, float& a,
                                                 float& y) {
  a = 1.f;
  y = 1.f;
  for (int i = 0; i < k; ++i) {
    a *= sigmoid_f(logit_clamped(__ldg(crow + i)) * s_inv_tau[i]);
    y *= __ldg(lrow + i);
  }
  y *= __ldg(lrow + k);
  z = logit_clamped(__ldg(crow + k));
}

__global__ void __launch_bounds__(kStsThreads, 1) sts_fit_kernel(
    const float* __restrict__ conf, const float* __restrict__ label, int N, int K, float tau_lo,
    float tau_hi, int rows_per_cta, int tile_cap, float* __restrict__ tau,
    float* __restrict__ loss) {
  extern __shared__ __align__(16) float s_rows[];  // [3][tile_cap]: z, survival before k, y
  __shared__ float s_inv_tau[kMaxK];
  __shared__ Pair s_part[kStsWarps][kStsG];
  __shared__ Pair s_cta[2][kStsG];  // this CTA's partial losses, by round parity
  __shared__ float s_inv[kStsG];    // this round's grid points as 1 / tau
  __shared__ double s_x0, s_step, s_xb;  // the round's interval; the position's best point
  __shared__ Pair s_Lb;
  float* s_z = s_rows;
  float* s_a = s_rows + tile_cap;
  float* s_y = s_rows + 2 * tile_cap;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const uint32_t rank = cluster_rank(), ncta = cluster_size();
  const int r0 = min(N, static_cast<int>(rank) * rows_per_cta);
  const int nr = min(N, r0 + rows_per_cta) - r0;
  const bool cached = nr <= tile_cap;  // the rows stay in shared memory for the whole fit
  if (cached) {
    for (int i = tid; i < nr; i += kStsThreads) {
      const size_t o = static_cast<size_t>(r0 + i) * K;
      s_z[i] = logit_clamped(__ldg(conf + o));
      s_a[i] = 1.f;
      s_y[i] = __ldg(label + o);
    }
  }
  double lx0 = 0.0, lstep = 0.0;  // the first round's interval (warp 0 only)
  if (warp == 0) {
    lx0 = log(static_cast<double>(tau_lo));
    lstep = (log(static_cast<double>(tau_hi)) - lx0) * (1.0 / (kStsG - 1));
  }
  int gr = 0;  // rounds so far (parity of the partial buffer)
  for (int k = 0; k < K; ++k) {
    if (warp == 0) {
      grid_inverses(lx0, lstep, lane, s_inv);
      if (lane == 0) {
        s_x0 = lx0;
        s_step = lstep;
      }
    }
    __syncthreads();
    for (int round = 0; round < kStsR; ++round, ++gr) {
      const float inv = s_inv[lane];
      float acc = 0.f, comp = 0.f;
      for (int t0 = 0; t0 < nr; t0 += tile_cap) {
        const int cnt = min(tile_cap, nr - t0);
        if (!cached) {
          __syncthreads();  // the previous tile's readers are done
          for (int i = tid; i < cnt; i += kStsThreads) {
            const size_t o = static_cast<size_t>(r0 + t0 + i) * K;
            row_from_scratch(conf + o, label + o, k, s_inv_tau, s_z[i], s_a[i], s_y[i]);
          }
          __syncthreads();
        }
        for (int i = warp; i < cnt; i += kStsWarps) {
          const float z = s_z[i], a = s_a[i], y = s_y[i];
          const float q = fminf(fmaxf(a * sigmoid_f(z * inv), 1e-7f), 1.0f - 1e-7f);
          // a 0/1 target leaves one of the two terms (the other is an exact zero: both logs
          // are finite on the clamped q); the branch is uniform across the warp's lanes
          float l;
          if (y == 1.f)
            l = -logf(q);
          else if (y == 0.f)
            l = -log1pf(-q);
          else
            l = -(y * logf(q) + (1.f - y) * log1pf(-q));
          const float t = l - comp;  // compensated sum
          const float s = acc + t;
          comp = (s - acc) - t;
          acc = s;
        }
      }
      {
        const float hi = acc - comp;  // the lane's sum acc - comp as a normalised pair
        s_part[warp][lane] = {hi, (acc - hi) - comp};
      }
      __syncthreads();
      Pair* mine = s_cta[gr & 1];
      {  // warp w adds grid point w over the CTA's warps (a fixed shuffle tree)
        Pair v = s_part[lane][warp];
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) v = pair_add(v, pair_shfl_xor(v, off));
        if (lane == 0) mine[warp] = v;
      }
      cluster_sync_all();
      if (warp == 0) {
        Pair part[kStsMaxCluster];
#pragma unroll
        for (int c = 0; c < kStsMaxCluster; ++c)
          part[c] = c < static_cast<int>(ncta) ? ld_cluster_pair(mine + lane, c) : Pair{0.f, 0.f};
        Pair L = part[0];  // every CTA adds the partials in rank order: the same sums everywhere
#pragma unroll
        for (int c = 1; c < kStsMaxCluster; ++c) L = pair_add(L, part[c]);
        Pair bv = L;
        int bi = lane;
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {  // the smallest loss, ties to the smaller point
          const Pair ov = pair_shfl_xor(bv, off);
          const int oi = __shfl_xor_sync(0xFFFFFFFFu, bi, off);
          if (pair_less(ov, bv) || (ov.hi == bv.hi && ov.lo == bv.lo && oi < bi)) {
            bv = ov;
            bi = oi;
          }
        }
        const double x0 = s_x0, step = s_step;
        const double nx0 = x0 + step * (bi > 0 ? bi - 1 : 0);
        const double nx1 = x0 + step * (bi < kStsG - 1 ? bi + 1 : kStsG - 1);
        const double nstep = (nx1 - nx0) * (1.0 / (kStsG - 1));
        __syncwarp();  // every lane has read s_x0 and s_step
        if (round + 1 < kStsR) grid_inverses(nx0, nstep, lane, s_inv);
        if (lane == 0) {
          s_xb = x0 + step * bi;
          s_Lb = bv;
          s_x0 = nx0;
          s_step = nstep;
        }
      }
      __syncthreads();
    }
    if (tid == 0) {
      const double t = exp(s_xb);
      s_inv_tau[k] = static_cast<float>(1.0 / t);
      if (rank == 0) {
        tau[k] = static_cast<float>(t);
        if (loss != nullptr)
          loss[k] = static_cast<float>((static_cast<double>(s_Lb.hi) + s_Lb.lo) / N);
      }
    }
    __syncthreads();
    if (cached && k + 1 < K) {  // advance the rows to position k + 1
      const float inv_tau = s_inv_tau[k];
      for (int i = tid; i < nr; i += kStsThreads) {
        const size_t o = static_cast<size_t>(r0 + i) * K + k + 1;
        s_a[i] *= sigmoid_f(s_z[i] * inv_tau);
        s_y[i] *= __ldg(label + o);
        s_z[i] = logit_clamped(__ldg(conf + o));
      }
    }
    __syncthreads();
  }
  cluster_sync_all();  // no CTA leaves while another may still read its partials
}

}  // namespace

cudaError_t launch_sts_fit(const float* conf, const float* label, int N, int K, float tau_lo,
                           float tau_hi, float* tau, float* loss, cudaStream_t stream) {
  const void* fn = reinterpret_cast<const void*>(&sts_fit_kernel);
  cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           3 * kStsTileRows * static_cast<int>(sizeof(float)));
  if (e != cudaSuccess) return e;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.blockDim = dim3(kStsThreads, 1, 1);
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  // the largest cluster the device can hold: 16 (non-portable) where allowed, else 8
  int ncta = 8;
  {
    attr[0].val.clusterDim.x = 16;
    cfg.gridDim = dim3(16, 1, 1);
    cfg.dynamicSmemBytes = 3 * kStsTileRows * sizeof(float);
    int clusters = 0;
    if (cudaOccupancyMaxActiveClusters(&clusters, fn, &cfg) == cudaSuccess && clusters >= 1)
      ncta = 16;
    else
      (void)cudaGetLastError();  // a refused query leaves no error behind
  }
  ncta = max(1, min(ncta, (N + kStsRowsPerCta - 1) / kStsRowsPerCta));
  const int rows_per_cta = (N + ncta - 1) / ncta;
  const int tile_cap = min(rows_per_cta, kStsTileRows);
  attr[0].val.clusterDim.x = ncta;
  cfg.gridDim = dim3(ncta, 1, 1);
  cfg.dynamicSmemBytes = 3 * static_cast<size_t>(tile_cap) * sizeof(float);
  return cudaLaunchKernelEx(&cfg, sts_fit_kernel, conf, label, N, K, tau_lo, tau_hi, rows_per_cta,
                            tile_cap, tau, loss);
}

}  // namespace dspark
