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
// Kernels:
//   topk_stream_kernel persistent CTAs over (row, piece) units: a bulk-copy
//                      ring streams U through shared memory at HBM speed; each
//                      warp keeps a sorted top-k list in its lanes and touches
//                      it only for elements above a CTA-wide floor; the lists
//                      are merged by rank (topk_merge_kernel merges pieces of
//                      rows split across CTAs when rows are few).
//   pair_scores16_kernel (k <= 16) one warp per (request, position): bulk-copies
//                      the k predecessor rows of A (and the gate row) and the k
//                      candidate rows of B into shared memory and accumulates
//                      4 x 4 register tiles of the k x k dot products on CUDA
//                      cores (0.5 GFLOP for a 256 x 16 block: not worth the
//                      tensor cores); pair_scores_kernel covers k up to 32.
//   walk_kernel        one CTA per request: the candidates' noise and score
//                      tables are staged in shared memory by all warps, then
//                      one warp walks the positions (lanes = candidates) with
//                      the Markov head's own two-stage block race restricted
//                      to the candidates, softmax over the k candidates; the
//                      optional confidence head runs for all positions at once.

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

constexpr int kTopkWarps = 8;                          // scanning warps
constexpr int kTopkThreads = (kTopkWarps + 1) * 32;   // + one copy warp
constexpr int kTopkChunk = 4096;                      // floats per ring stage (16 KB)
constexpr int kTopkStages = 3;                     // 48 KB: four CTAs per SM
constexpr uint32_t kTopkRingBytes = kTopkStages * kTopkChunk * 4;
constexpr int kNoIndex = 0x7FFFFFFF;
constexpr uint32_t kTopkBar = 1;                      // named barrier of the scanning warps

__device__ __forceinline__ uint32_t ordered_u32(float f) {
  const uint32_t b = __float_as_uint(f);
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

__device__ __forceinline__ float from_ordered_u32(uint32_t o) {
  return __uint_as_float((o & 0x80000000u) ? (o & 0x7FFFFFFFu) : ~o);
}

struct TopkArgs {
  const float* U;      // [rows][V]
  int rows, V, topk;
  int pieces;          // pieces per row (1: each CTA scans whole rows)
  int piece_len;       // tokens per piece, a multiple of 4
  int32_t* cand;       // pieces == 1: [rows][topk]
  float* cval;
  int32_t* part_i;     // pieces > 1: [rows * pieces][topk]
  float* part_v;
  int* status;
  uint64_t timeout_ns;
};

// Streaming top-k of each row of U.  Work unit = (row, piece); CTA c takes
// units c, c + grid, ...  One lane of the copy warp streams the unit's floats
// through a 3-stage shared-memory ring with bulk copies; each scanning warp
// takes a 512-float slice of every stage and keeps a sorted top-k list in its
// lanes.  A warp touches its list only for elements at or above a floor, a
// lower bound on the unit's k-th value built from values the CTA has seen:
//   * the k-th value of any full list (k real elements lie at or above it);
//   * the smallest of the warps' m-th values, m = ceil(k / 8) (the m best of
//     every list are >= k distinct elements), which tracks the k-th value of
//     everything the CTA has seen so far;
//   * on a unit's first chunk, the k-th largest of the warp's 32 lane maxima.
// At the end of a unit the 8 lists are merged by rank: each candidate counts
// the candidates ahead of it and lands in that output slot.
__global__ void __launch_bounds__(kTopkThreads) topk_stream_kernel(const __grid_constant__ TopkArgs a) {
  extern __shared__ __align__(128) uint8_t topk_smem[];
  float* ring = reinterpret_cast<float*>(topk_smem);
  __shared__ __align__(8) uint64_t full[kTopkStages];
  __shared__ __align__(8) uint64_t empty[kTopkStages];
  __shared__ float s_v[kTopkWarps][32];
  __shared__ int s_i[kTopkWarps][32];
  __shared__ uint32_t s_floor;  // ordered bits of the best k-th value held by a full list
  __shared__ uint32_t s_mth[kTopkWarps];  // ordered bits of each warp's m-th best value
  __shared__ int s_abort;
  __shared__ uint32_t s_sink;  // scratch word of the stage releases
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int units = a.rows * a.pieces;
  volatile int* abort_flag = &s_abort;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kTopkStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kTopkWarps);
    }
    s_floor = ordered_u32(-INFINITY);
    for (int w = 0; w < kTopkWarps; ++w) s_mth[w] = ordered_u32(-INFINITY);
    s_abort = 0;
    fence_mbar_init();
  }
  __syncthreads();
  // m = ceil(k / warps): the m best entries of every warp's list are >= k distinct
  // elements, so the smallest of the warps' m-th values bounds the k-th value too
  const int mth = (a.topk + kTopkWarps - 1) / kTopkWarps;

  if (warp == kTopkWarps) {
    // ------------------------------------------------------------ copy warp
    if (lane != 0) return;
    const uint64_t pol = l2_policy_evict_first();
    uint32_t issued = 0;
    bool ok = true;
    for (int unit = blockIdx.x; unit < units && ok; unit += gridDim.x) {
      const int row = unit / a.pieces, piece = unit - row * a.pieces;
      const int e0 = piece * a.piece_len, e1 = min(a.V, e0 + a.piece_len);
      const float* src = a.U + static_cast<size_t>(row) * a.V;
      for (int c0 = e0; c0 < e1; c0 += kTopkChunk) {
        const int s = static_cast<int>(issued % kTopkStages);
        if (!mbar_wait(&empty[s], ((issued / kTopkStages) & 1u) ^ 1u, a.timeout_ns, abort_flag,
                       200u)) {
          ok = false;
          break;
        }
        const uint32_t bytes = static_cast<uint32_t>(min(kTopkChunk, e1 - c0)) * 4u;
        mbar_arrive_expect_tx(&full[s], bytes);
        bulk_load(ring + s * kTopkChunk, src + c0, bytes, &full[s], pol);
        ++issued;
      }
    }
    if (!ok) {
      s_abort = 1;
      record_error(a.status, kStatusTimeout);
      // every copy in flight must land before the CTA exits
      for (uint32_t j = issued > kTopkStages ? issued - kTopkStages : 0u; j < issued; ++j)
        mbar_wait(&full[j % kTopkStages], (j / kTopkStages) & 1u, a.timeout_ns, nullptr);
    }
    return;
  }

  // -------------------------------------------------------------- scanning warps
  uint32_t consumed = 0;
  bool ok = true;
  for (int unit = blockIdx.x; unit < units; unit += gridDim.x) {
    const int row = unit / a.pieces, piece = unit - row * a.pieces;
    const int e0 = piece * a.piece_len, e1 = min(a.V, e0 + a.piece_len);
    WarpTopk list;
    list.init();
    for (int c0 = e0; c0 < e1; c0 += kTopkChunk, ++consumed) {
      const int s = static_cast<int>(consumed % kTopkStages);
      if (ok) ok = mbar_wait(&full[s], (consumed / kTopkStages) & 1u, a.timeout_ns, abort_flag);
      ok = __all_sync(0xFFFFFFFFu, ok);
      if (!ok) continue;  // keep walking the units so the named barriers below still meet
      const int n = min(kTopkChunk, e1 - c0);
      const float* chunk = ring + s * kTopkChunk;
      float4 x[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int off = warp * 512 + j * 128 + lane * 4;
        x[j] = (off < n) ? *reinterpret_cast<const float4*>(chunk + off)
                         : make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
      }
      // free the stage once every lane's slice is in registers
      arrive_after_reads(&empty[s],
                         __float_as_uint(x[0].x) ^ __float_as_uint(x[1].x) ^
                             __float_as_uint(x[2].x) ^ __float_as_uint(x[3].x),
                         &s_sink, lane);
      float mx = fmaxf(fmaxf(fmaxf(x[0].x, x[0].y), fmaxf(x[0].z, x[0].w)),
                       fmaxf(fmaxf(x[1].x, x[1].y), fmaxf(x[1].z, x[1].w)));
      mx = fmaxf(mx, fmaxf(fmaxf(fmaxf(x[2].x, x[2].y), fmaxf(x[2].z, x[2].w)),
                           fmaxf(fmaxf(x[3].x, x[3].y), fmaxf(x[3].z, x[3].w))));
      uint32_t mmin = s_mth[0];
#pragma unroll
      for (int w = 1; w < kTopkWarps; ++w) mmin = min(mmin, s_mth[w]);
      float floor_v = fmaxf(list.tv, from_ordered_u32(max(s_floor, mmin)));
      if (c0 == e0) {
        // First chunk of the unit, list still empty: the k-th largest of the 32
        // lane maxima (k distinct elements of the unit) bounds the unit's k-th
        // value from below, so the warp starts filtering at once instead of
        // inserting most of its first slice.
        int ge = 0;
#pragma unroll
        for (int i = 0; i < 32; ++i) ge += (__shfl_sync(0xFFFFFFFFu, mx, i) >= mx) ? 1 : 0;
        float seed = (ge >= a.topk) ? mx : -INFINITY;
#pragma unroll
        for (int off = 16; off > 0; off >>= 1)
          seed = fmaxf(seed, __shfl_xor_sync(0xFFFFFFFFu, seed, off));
        if (lane == 0 && seed > -INFINITY) atomicMax(&s_floor, ordered_u32(seed));
        floor_v = fmaxf(floor_v, seed);
      }
      if (!__any_sync(0xFFFFFFFFu, mx >= floor_v)) continue;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int off = warp * 512 + j * 128 + lane * 4;
        const bool in = off < n;
        const int idx = c0 + off;
        list.offer(x[j].x, idx + 0, in && x[j].x >= floor_v, lane, a.topk);
        list.offer(x[j].y, idx + 1, in && x[j].y >= floor_v, lane, a.topk);
        list.offer(x[j].z, idx + 2, in && x[j].z >= floor_v, lane, a.topk);
        list.offer(x[j].w, idx + 3, in && x[j].w >= floor_v, lane, a.topk);
      }
      if (lane == 0 && list.ti != kNoIndex) atomicMax(&s_floor, ordered_u32(list.tv));
      const float vm = __shfl_sync(0xFFFFFFFFu, list.lv, mth - 1);
      const int im = __shfl_sync(0xFFFFFFFFu, list.li, mth - 1);
      if (lane == 0 && im != kNoIndex) s_mth[warp] = ordered_u32(vm);
    }
    // ---- merge the warps' lists: candidate c = (warp c / k, slot c % k) goes to
    // output slot rank(c), the number of candidates ahead of it (distinct ids)
    s_v[warp][lane] = list.lv;
    s_i[warp][lane] = list.li;
    named_bar_sync(kTopkBar, kTopkWarps * 32);
    const int ncand = kTopkWarps * a.topk;
    if (threadIdx.x < ncand && !*abort_flag) {
      const int cw = threadIdx.x / a.topk, cs = threadIdx.x - cw * a.topk;
      const float cv = s_v[cw][cs];
      const int ci = s_i[cw][cs];
      if (ci != kNoIndex) {
        int rank = 0;
        for (int w = 0; w < kTopkWarps; ++w) {
          for (int j = 0; j < a.topk; ++j) {
            const float v = s_v[w][j];
            const int vi = s_i[w][j];
            rank += (vi != kNoIndex && better(v, vi, cv, ci)) ? 1 : 0;
          }
        }
        if (rank < a.topk) {
          if (a.pieces == 1) {
            a.cand[static_cast<size_t>(row) * a.topk + rank] = ci;
            a.cval[static_cast<size_t>(row) * a.topk + rank] = cv;
          } else {
            a.part_i[static_cast<size_t>(unit) * a.topk + rank] = ci;
            a.part_v[static_cast<size_t>(unit) * a.topk + rank] = cv;
          }
        }
      }
    }
    if (threadIdx.x < kTopkWarps) s_mth[threadIdx.x] = ordered_u32(-INFINITY);
    if (threadIdx.x == 0) s_floor = ordered_u32(-INFINITY);
    named_bar_sync(kTopkBar, kTopkWarps * 32);
  }
}

// Row-wise merge of the pieces' lists (one warp per row).
__global__ void __launch_bounds__(128) topk_merge_kernel(const int32_t* __restrict__ part_i,
                                                         const float* __restrict__ part_v,
                                                         int rows, int pieces, int topk,
                                                         int32_t* __restrict__ cand,
                                                         float* __restrict__ cval) {
  const int lane = threadIdx.x & 31;
  const int row = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (row >= rows) return;
  const int n = pieces * topk;
  const size_t base = static_cast<size_t>(row) * n;
  WarpTopk list;
  list.init();
  for (int e0 = 0; e0 < n; e0 += 32) {
    const int e = e0 + lane;
    const int vi = (e < n) ? __ldg(part_i + base + e) : kNoIndex;
    const float v = (e < n) ? __ldg(part_v + base + e) : -INFINITY;
    list.offer(v, vi, vi != kNoIndex, lane, topk);
  }
  if (lane < topk) {
    cand[static_cast<size_t>(row) * topk + lane] = list.li;
    cval[static_cast<size_t>(row) * topk + lane] = list.lv;
  }
}

constexpr int kPairWarps = 4;  // (request, position) pairs per CTA, one per warp

// Shared bytes of one warp of pair_scores16_kernel: 32 gathered bf16 rows of
// r + 8 elements (the 16-byte pad spreads the 4 x 4 register tiles' loads over
// all banks) and, when gated, the fp32 gate row.
__host__ __device__ __forceinline__ int pair16_warp_bytes(int r, bool gated) {
  return 32 * (2 * r + 16) + (gated ? 4 * r : 0);
}

// k <= 16 candidates: one warp per (request, position).  Lanes 0..15 bulk-copy
// the k predecessor rows of A, lanes 16..31 the k candidate rows of B (and
// lane 0 the gate row) into shared memory on one mbarrier; then lane
// (half, blk) accumulates a 4 x 4 tile of S (rows blk % 4 + 4m, columns
// blk / 4 + 4n) over half of the rank, and the halves are summed by a shuffle.
__global__ void __launch_bounds__(kPairWarps * 32) pair_scores16_kernel(
    const int32_t* __restrict__ cand, const float* __restrict__ cval,
    const uint16_t* __restrict__ A, const uint16_t* __restrict__ Bt,
    const int32_t* __restrict__ anchors, const float* __restrict__ H, int BK, int K, int V,
    int r, int topk, float* __restrict__ S, int* status, uint64_t timeout_ns) {
  extern __shared__ __align__(128) uint8_t pair_smem[];
  __shared__ __align__(8) uint64_t bar[kPairWarps];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const bool gated = H != nullptr;
  const int row_bytes = 2 * r + 16;
  uint8_t* wbase = pair_smem + warp * pair16_warp_bytes(r, gated);
  if (lane == 0) {
    mbar_init(&bar[warp], 1);
    fence_mbar_init();
  }
  __syncwarp();
  const size_t bt = static_cast<size_t>(blockIdx.x) * kPairWarps + warp;
  if (bt >= static_cast<size_t>(BK)) return;
  const int b = static_cast<int>(bt / K), t = static_cast<int>(bt % K);
  // lanes i and 16 + i fetch row i; rows past k repeat row 0 (their outputs are dropped)
  const int i = (lane & 15) < topk ? (lane & 15) : 0;
  int tok;
  if (lane < 16) {
    tok = (t == 0) ? __ldg(anchors + b) : __ldg(cand + (bt - 1) * topk + i);
  } else {
    tok = __ldg(cand + bt * topk + i);
  }
  if (tok < 0 || tok >= V) {
    record_error(status, kStatusDeviceOob);
    tok = min(max(tok, 0), V - 1);
  }
  const uint64_t pol = l2_policy_evict_last();
  if (lane == 0) mbar_arrive_expect_tx(&bar[warp], 32u * 2u * r + (gated ? 4u * r : 0u));
  __syncwarp();
  bulk_load(wbase + lane * row_bytes, (lane < 16 ? A : Bt) + static_cast<size_t>(tok) * r,
            2u * r, &bar[warp], pol);
  if (gated && lane == 0) bulk_load(wbase + 32 * row_bytes, H + bt * r, 4u * r, &bar[warp], pol);
  if (!mbar_wait(&bar[warp], 0, timeout_ns, nullptr)) {
    record_error(status, kStatusTimeout);
    return;
  }
  const int half = lane >> 4, blk = lane & 15;
  const int ib = blk & 3, jb = blk >> 2;
  const float* hrow = reinterpret_cast<const float*>(wbase + 32 * row_bytes);
  float acc[4][4];
#pragma unroll
  for (int m = 0; m < 4; ++m)
#pragma unroll
    for (int n = 0; n < 4; ++n) acc[m][n] = 0.f;
  // half h takes rank elements [64 c + 32 h, 64 c + 32 h + 32) of every 64
  for (int q0 = half * 32; q0 < r; q0 += 64) {
#pragma unroll
    for (int sub = 0; sub < 4; ++sub) {
      const int q = q0 + sub * 8;
      if (q >= r) break;
      uint4 av[4], bv[4];
#pragma unroll
      for (int m = 0; m < 4; ++m) {
        av[m] = *reinterpret_cast<const uint4*>(wbase + (ib + 4 * m) * row_bytes + 2 * q);
        bv[m] = *reinterpret_cast<const uint4*>(wbase + (16 + jb + 4 * m) * row_bytes + 2 * q);
      }
      float g[8];
      if (gated) {
        const float4 g0 = *reinterpret_cast<const float4*>(hrow + q);
        const float4 g1 = *reinterpret_cast<const float4*>(hrow + q + 4);
        g[0] = g0.x; g[1] = g0.y; g[2] = g0.z; g[3] = g0.w;
        g[4] = g1.x; g[5] = g1.y; g[6] = g1.z; g[7] = g1.w;
      }
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        float a[4], bb[4];
#pragma unroll
        for (int m = 0; m < 4; ++m) {
          const uint32_t aw = (e >> 1) == 0 ? av[m].x : (e >> 1) == 1 ? av[m].y
                            : (e >> 1) == 2 ? av[m].z : av[m].w;
          const uint32_t bw = (e >> 1) == 0 ? bv[m].x : (e >> 1) == 1 ? bv[m].y
                            : (e >> 1) == 2 ? bv[m].z : bv[m].w;
          a[m] = (e & 1) ? __uint_as_float(aw & 0xFFFF0000u) : __uint_as_float(aw << 16);
          bb[m] = (e & 1) ? __uint_as_float(bw & 0xFFFF0000u) : __uint_as_float(bw << 16);
          if (gated) a[m] *= g[e];
        }
#pragma unroll
        for (int m = 0; m < 4; ++m)
#pragma unroll
          for (int n = 0; n < 4; ++n) acc[m][n] = fmaf(a[m], bb[n], acc[m][n]);
      }
    }
  }
#pragma unroll
  for (int m = 0; m < 4; ++m)
#pragma unroll
    for (int n = 0; n < 4; ++n) acc[m][n] += __shfl_xor_sync(0xFFFFFFFFu, acc[m][n], 16);
  if (half == 0) {
#pragma unroll
    for (int m = 0; m < 4; ++m) {
      const int ii = ib + 4 * m;
#pragma unroll
      for (int n = 0; n < 4; ++n) {
        const int jj = jb + 4 * n;
        if (ii < topk && jj < topk)
          S[(bt * topk + ii) * topk + jj] = __ldg(cval + bt * topk + jj) + acc[m][n];
      }
    }
  }
}

// k in 17..32: one CTA per (request, position), operands widened to fp32 in
// shared memory, one thread per score.
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

constexpr int kWalkWarps = 8;
constexpr int kWalkWindowBytes = 32768;  // score tables staged per window

// One CTA per request.  The draw at position t depends on the path only through
// the predecessor slot i (the row S_t(i, .)); the candidates' noise depends on
// their blocks of token ids, not on the path.  So, per window of positions:
//   1. the k x k score tables and, per candidate, its token, its block's
//      -ln E, its block's stage-2 uniform and the mask of candidates sharing its
//      16-token block are staged in shared memory (one warp per position);
//   2. every thread draws for one (position, predecessor slot) pair at a time --
//      the head's block race restricted to the candidates: candidates of one
//      block race with their summed mass, then the inverse CDF in token order --
//      and records the chosen slot and its log-softmax over the k candidates;
//   3. thread 0 follows the chain slot_{t+1} = next(t, slot_t).
// After the walk, the confidence head runs for all positions at once (one warp
// per position) and thread 0 forms the survival products.
__global__ void __launch_bounds__(kWalkWarps * 32) walk_kernel(
    const int32_t* __restrict__ cand, const float* __restrict__ S,
    const int32_t* __restrict__ anchors, const uint16_t* __restrict__ A, int B, int K, int V,
    int r, int topk, int window, float inv_t, int sample, uint32_t seed_lo, uint32_t seed_hi,
    int32_t* __restrict__ tokens, float* __restrict__ logprobs, dspark_conf_args conf,
    int conf_on, int* status) {
  extern __shared__ __align__(16) float walk_smem[];
  const int tile = topk * topk;
  float* s_S = walk_smem;                                   // [window][topk][topk]
  float* s_L = s_S + window * tile;                         // [window][32] -ln E of the block
  float* s_U2 = s_L + window * 32;                          // [window][32] stage-2 uniform
  int* s_C = reinterpret_cast<int*>(s_U2 + window * 32);    // [window][32] candidate token
  uint32_t* s_M = reinterpret_cast<uint32_t*>(s_C + window * 32);  // [window][32] block mates
  int* s_next = reinterpret_cast<int*>(s_M + window * 32);  // [window][32] slot drawn from row i
  float* s_lp = reinterpret_cast<float*>(s_next + window * 32);  // [window][32] its logprob
  __shared__ int s_tok[kMaxK];
  __shared__ float s_conf[kMaxK];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int b = blockIdx.x;
  int slot = 0;
  for (int t0 = 0; t0 < K; t0 += window) {
    const int nt = min(window, K - t0);
    const size_t base = (static_cast<size_t>(b) * K + t0) * tile;
    // the window's score tables: 16-byte asynchronous copies, all in flight at once
    // (nt * topk^2 floats; topk^2 is a multiple of 4 except for odd topk)
    if ((tile & 3) == 0 && (reinterpret_cast<uintptr_t>(S) & 15u) == 0) {
      for (int e = threadIdx.x * 4; e < nt * tile; e += blockDim.x * 4)
        cp_async_16(s_S + e, S + base + e);
      cp_async_commit();
    } else {
      for (int e = threadIdx.x; e < nt * tile; e += blockDim.x) s_S[e] = __ldg(S + base + e);
    }
    for (int w = warp; w < nt; w += kWalkWarps) {
      const int t = t0 + w;
      const size_t bt = static_cast<size_t>(b) * K + t;
      const bool live = lane < topk;
      const int c = live ? __ldg(cand + bt * topk + lane) : 0x7FFFFFFF;
      const int blk = live ? (c >> 4) : -1 - lane;  // distinct for dead lanes
      float lnE = 0.f, u2 = 0.f;
      if (sample && live) {
        const uint32_t ub = static_cast<uint32_t>(blk);
        const Philox4 rnd = philox4x32_10(ub >> 3, static_cast<uint32_t>(t),
                                          static_cast<uint32_t>(b), 1u + (ub & 3u), seed_lo,
                                          seed_hi);
        const int h = (ub >> 2) & 1u;
        lnE = -logf(neg_log_uniform_accurate(philox_uniform(h ? rnd.w[2] : rnd.w[0])));
        u2 = philox_uniform(h ? rnd.w[3] : rnd.w[1]);
      }
      s_L[w * 32 + lane] = lnE;
      s_U2[w * 32 + lane] = u2;
      s_C[w * 32 + lane] = c;
      s_M[w * 32 + lane] = __match_any_sync(0xFFFFFFFFu, blk) & (live ? 0xFFFFFFFFu : 0u);
    }
    cp_async_wait_all();
    __syncthreads();
    // every (position, predecessor slot) draw of the window
    for (int d = threadIdx.x; d < nt * topk; d += blockDim.x) {
      const int w = d / topk, i = d - w * topk;
      const float* row = s_S + (w * topk + i) * topk;
      const float* L = s_L + w * 32;
      const int* C = s_C + w * 32;
      const uint32_t* M = s_M + w * 32;
      float m = -INFINITY;
      for (int j = 0; j < topk; ++j) m = fmaxf(m, row[j] * inv_t);
      float tot = 0.f;
      for (int j = 0; j < topk; ++j) tot += expf(row[j] * inv_t - m);
      int pick = 0;
      if (!sample) {
        // greedy: argmax by (score desc, token id asc)
        float bz = row[0] * inv_t;
        for (int j = 1; j < topk; ++j) {
          const float z = row[j] * inv_t;
          if (z > bz || (z == bz && C[j] < C[pick])) {
            bz = z;
            pick = j;
          }
        }
      } else {
        // stage 1: each block (represented by its lowest slot) races with its mass
        float best = -INFINITY, bestZ = 0.f;
        int bestj = 0;
        for (int j = 0; j < topk; ++j) {
          const uint32_t mates = M[j];
          if ((__ffs(mates) - 1) != j) continue;  // not the block's first slot
          float Z = 0.f;
          for (uint32_t mm = mates; mm != 0u; mm &= mm - 1u) {
            const int jj = __ffs(mm) - 1;
            Z += expf(row[jj] * inv_t - m);
          }
          const float sc = (Z > 0.f) ? logf(Z) + L[j] : -INFINITY;
          if (sc > best || (sc == best && (C[j] >> 4) < (C[bestj] >> 4))) {
            best = sc;
            bestZ = Z;
            bestj = j;
          }
        }
        // stage 2: inverse CDF over the block's candidates in token order
        const float target = s_U2[w * 32 + bestj] * bestZ;
        uint32_t left = M[bestj];
        float Cum = 0.f;
        int last = bestj;
        pick = -1;
        while (left != 0u) {
          int jmin = __ffs(left) - 1;
          for (uint32_t mm = left & (left - 1u); mm != 0u; mm &= mm - 1u) {
            const int jj = __ffs(mm) - 1;
            if (C[jj] < C[jmin]) jmin = jj;
          }
          left &= ~(1u << jmin);
          const float e = expf(row[jmin] * inv_t - m);
          if (e > 0.f) {
            Cum += e;
            last = jmin;
            if (target < Cum) {
              pick = jmin;
              break;
            }
          }
        }
        if (pick < 0) pick = last;  // target at the very top (rounding): the last live one
      }
      s_next[w * 32 + i] = pick;
      s_lp[w * 32 + i] = row[pick] * inv_t - (m + logf(tot));
    }
    __syncthreads();
    if (threadIdx.x == 0) {
      for (int w = 0; w < nt; ++w) {
        const int t = t0 + w;
        const size_t bt = static_cast<size_t>(b) * K + t;
        const int j = s_next[w * 32 + slot];
        int c = s_C[w * 32 + j];
        if (c < 0 || c >= V) {
          record_error(status, kStatusDeviceOob);
          c = 0;
        }
        tokens[bt] = c;
        logprobs[bt] = s_lp[w * 32 + slot];
        s_tok[t] = c;
        slot = j;
      }
    }
    __syncthreads();
  }
  if (!conf_on) return;
  for (int t = warp; t < K; t += kWalkWarps) {
    const size_t bt = static_cast<size_t>(b) * K + t;
    const int prev_tok = (t == 0) ? __ldg(anchors + b) : s_tok[t - 1];
    const uint16_t* emb = conf.with_markov ? A + static_cast<size_t>(prev_tok) * r : nullptr;
    const float zc = confidence_logit(conf.h + bt * conf.d, conf.d, conf.w, emb, r, conf.bias,
                                      lane);
    if (lane == 0) s_conf[t] = sigmoidf_accurate(conf.tau ? zc / __ldg(conf.tau + t) : zc);
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    float surv = 1.f;
    int len = 0;
    bool open = true;
    for (int t = 0; t < K; ++t) {
      const size_t bt = static_cast<size_t>(b) * K + t;
      const float cc = s_conf[t];
      surv *= cc;
      if (open && surv >= conf.threshold) {
        len = t + 1;
      } else {
        open = false;
      }
      conf.conf[bt] = cc;
      conf.cumprod[bt] = surv;
    }
    conf.verify_len[b] = len;
  }
}

}  // namespace

cudaError_t launch_topk(const float* U, int rows, int V, int topk, int32_t* cand, float* cval,
                        int32_t* part_i, float* part_v, int part_units, int* status,
                        uint64_t timeout_ns, int* launches, cudaStream_t stream) {
  *launches = 0;
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  int sms = 0, occ = 0;
  if ((err = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
    return err;
  const void* fn = reinterpret_cast<const void*>(&topk_stream_kernel);
  if ((err = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  static_cast<int>(kTopkRingBytes))) != cudaSuccess)
    return err;
  // four 48 KB rings per SM need the largest shared-memory carveout
  if ((err = cudaFuncSetAttribute(fn, cudaFuncAttributePreferredSharedMemoryCarveout,
                                  cudaSharedmemCarveoutMaxShared)) != cudaSuccess)
    return err;
  if ((err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, fn, kTopkThreads,
                                                           kTopkRingBytes)) != cudaSuccess)
    return err;
  const int capacity = sms * (occ > 0 ? occ : 1);
  // Few rows: split each into pieces (of at least one ring stage) so that the
  // grid fills the GPU; the pieces' lists are merged by a second kernel.
  int pieces = 1;
  if (rows < 2 * capacity && part_i != nullptr && part_units >= 2 * rows) {
    const int want = (2 * capacity + rows - 1) / rows;
    const int most = (V + kTopkChunk - 1) / kTopkChunk;
    pieces = min(min(want, most), part_units / rows);
  }
  int piece_len = V;
  if (pieces > 1) {
    piece_len = (((V + pieces - 1) / pieces) + 3) & ~3;
    pieces = (V + piece_len - 1) / piece_len;
  }
  TopkArgs a{U, rows, V, topk, pieces, piece_len, cand, cval, part_i, part_v, status, timeout_ns};
  const int units = rows * pieces;
  const int grid = min(units, capacity);
  topk_stream_kernel<<<grid, kTopkThreads, kTopkRingBytes, stream>>>(a);
  if ((err = cudaGetLastError()) != cudaSuccess) return err;
  *launches = 1;
  if (pieces == 1) return cudaSuccess;
  topk_merge_kernel<<<(rows + 3) / 4, 128, 0, stream>>>(part_i, part_v, rows, pieces, topk, cand,
                                                        cval);
  if ((err = cudaGetLastError()) != cudaSuccess) return err;
  *launches = 2;
  return cudaSuccess;
}

cudaError_t launch_pair_scores(const int32_t* cand, const float* cval, const uint16_t* A,
                               const uint16_t* Bt, const int32_t* anchors, const float* H,
                               int B, int K, int V, int r, int topk, float* S, int* status,
                               uint64_t timeout_ns, cudaStream_t stream) {
  cudaError_t err;
  const int BK = B * K;
  if (topk <= 16) {
    const size_t smem = static_cast<size_t>(kPairWarps) * pair16_warp_bytes(r, H != nullptr);
    err = cudaFuncSetAttribute(reinterpret_cast<const void*>(&pair_scores16_kernel),
                               cudaFuncAttributeMaxDynamicSharedMemorySize,
                               static_cast<int>(smem));
    if (err != cudaSuccess) return err;
    err = cudaFuncSetAttribute(reinterpret_cast<const void*>(&pair_scores16_kernel),
                               cudaFuncAttributePreferredSharedMemoryCarveout,
                               cudaSharedmemCarveoutMaxShared);
    if (err != cudaSuccess) return err;
    pair_scores16_kernel<<<(BK + kPairWarps - 1) / kPairWarps, kPairWarps * 32, smem, stream>>>(
        cand, cval, A, Bt, anchors, H, BK, K, V, r, topk, S, status, timeout_ns);
    return cudaGetLastError();
  }
  const size_t smem = 2ull * topk * (r + 1) * sizeof(float);
  err = cudaFuncSetAttribute(reinterpret_cast<const void*>(&pair_scores_kernel),
                             cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (err != cudaSuccess) return err;
  pair_scores_kernel<<<BK, 256, smem, stream>>>(cand, cval, A, Bt, anchors, H, K, V, r, topk, S,
                                                status);
  return cudaGetLastError();
}

cudaError_t launch_walk(const int32_t* cand, const float* S, const int32_t* anchors,
                        const uint16_t* A, int B, int K, int V, int r, int topk, float inv_t,
                        int sample, uint32_t seed_lo, uint32_t seed_hi, int32_t* tokens,
                        float* logprobs, const dspark_conf_args* conf, int* status,
                        cudaStream_t stream) {
  dspark_conf_args c{};
  if (conf != nullptr) c = *conf;
  const int tile_bytes = topk * topk * 4;
  const int window = max(1, min(K, kWalkWindowBytes / tile_bytes));
  const size_t smem = static_cast<size_t>(window) * (tile_bytes + 6 * 32 * 4);
  cudaError_t err = cudaFuncSetAttribute(reinterpret_cast<const void*>(&walk_kernel),
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
  if (err != cudaSuccess) return err;
  walk_kernel<<<B, kWalkWarps * 32, smem, stream>>>(cand, S, anchors, A, B, K, V, r, topk, window,
                                                    inv_t, sample, seed_lo, seed_hi, tokens,
                                                    logprobs, c, conf != nullptr ? 1 : 0, status);
  return cudaGetLastError();
}

}  // namespace dspark
