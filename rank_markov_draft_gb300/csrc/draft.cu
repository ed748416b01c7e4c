// draft.cu -- persistent Markov-head draft kernel for sm_103a.
//
// What it computes (DSpark explainer, "Semi-autoregressive generation" and
// "The Markov head"; equivalence page, "What the two methods do"): for a
// chunk of up to 128 requests and block positions k = 0 .. K-1,
//     l[b, v] = U[b, k, v] + sum_i e_b[i] * W2[i, v],   e_b = W1[x_{k-1}[b]] (. H[b, k])
//     x_k[b]  ~ softmax(l[b, :] / T), drawn by the two-stage block race below
//               (T = 0: argmax l)
//     logprob = l[b, x_k] / T' - log sum_v exp(l[b, v] / T')
// with x_{-1} = the anchor ("Sample From Anchor" in the vLLM guide).  The
// local softmax is exact, as rejection sampling needs ("Why the normalization
// has to be local", "Repair the Joint, Meter the Verify").
//
// Layout of the work (one CTA per SM, cooperative launch, all K steps in one
// launch):
//   * the vocabulary is split into 64-token tiles; CTA c owns a fixed,
//     contiguous range of tiles for every step;
//   * warp 0 (one lane) streams W2 tiles [r x 64] and U tiles [rows x 64]
//     with TMA into shared memory rings; these never depend on sampled
//     tokens, so the producer runs ahead across step boundaries;
//   * warp 1 (one lane) issues tcgen05.mma: D[128 requests x 64 tokens] =
//     E[128 x r] * W2tile[r x 64] into one of four TMEM accumulators;
//     E is the gathered Markov embedding of every request, gathered into
//     shared memory (K-major, 128B swizzle) and copied once per position into
//     TMEM (row m in lane m, two bf16 per column), from where the MMAs read it
//     (each MMA would otherwise re-read its A slice from shared memory); W2 is
//     the MN-major tile exactly as TMA wrote it;
//   * warps 2..17 (the epilogue) read the accumulator (one request per TMEM
//     lane, 16 tokens per thread) and U from shared memory, and keep, per
//     request, a running log-sum-exp and a running block-race winner, so the
//     full-vocabulary logits never reach HBM;
//   * at the end of a step each CTA publishes, per request, a 64-bit key
//     (epoch | ordered score | inverted token id) by atomicMax and its
//     log-sum-exp partial; after a bounded grid barrier every CTA decodes the
//     winning tokens from the keys and gathers the next step's embeddings;
//   * after the last step, CTA c reduces request c's partials into tokens and
//     log-probabilities and runs the fused confidence head.
//
// Teacher-forced modes take every position's predecessor from the caller, so
// positions do not depend on one another: the next position's embeddings are
// gathered as soon as the MMAs are done with the current ones and the grid
// barrier is waited on only before the final reduction.  The label mode
// (DSpark explainer, "Confidence-scheduled verification": c*_k = 1 - TV of the
// draft head's and the target's distributions) streams the target's rows
// beside U and sums 2^min(log2 q(v), log2 p(v)) over the vocabulary, both
// normalisers known beforehand (the target's from a row scan, the draft's
// from its own log-probability of the drafted token).  Its ring slots hold U
// and target for half a tile (32 tokens each), two slots per tile, so the
// same 96 KB of shared memory keeps twice the bytes per tile in flight; every
// epilogue warp reads both halves (8 tokens of each per thread), so each slot
// has one group of readers that takes its fills in order.
//
// Sampling epilogue (an exact draw from softmax(l / T) in two stages over
// 16-token blocks; each thread's 16 columns of a tile are one block beta):
//   y = l * log2(e) / T, w = 2^(y - m) (shared with the log-sum-exp), and the
//   block's mass relative to m is s = sum w;
//   stage 1, a race between blocks: the block maximising
//     G = m + log2(s) - log2(E),  E = -ln u1 (a unit exponential)
//   wins with probability Z_beta / Z (argmax Z_beta / E_beta);
//   stage 2, only for a block that can still beat the best G any thread has
//   reached for the request: the first token whose cumulative w exceeds
//   u2 * s.  Both uniforms come from one Philox call per two of the thread's
//   tiles.  The (G, token) winner is merged across threads and CTAs as a key.
//
// Every wait is bounded (mbarrier waits and the grid barrier give up after
// timeout_ns, set the device status word and make the CTA exit cleanly after
// draining its own TMA copies and MMAs and freeing its TMEM).

#include <cstdint>
#include <cuda_bf16.h>

#ifndef BOUND_REFRESH
#define BOUND_REFRESH 2
#endif
#include "confidence.cuh"
#include "internal.h"
#include "philox.cuh"
#include "sm103.cuh"

namespace dspark {
namespace {

constexpr int kTileV = kDraftTileV;              // 64 tokens per tile (MMA N)
constexpr int kRows = kBatchChunk;               // 128 requests (MMA M)
constexpr int kNumW2Stages = 2;
constexpr int kNumUStages = 3;                   // U ring slots of 32 KB (B > 64)
constexpr int kNumUStagesSmall = 4;              // slots of 16 KB when B <= 64 (box <= 64 rows)
constexpr int kNumAcc = 4;                       // TMEM accumulators, 64 columns each
constexpr int kEpiWarps = 16;
constexpr int kEpiThreads = kEpiWarps * 32;      // 512
constexpr int kThreads = 64 + kEpiThreads;       // 576
constexpr uint32_t kABytes = kRows * kMaxRank * 2;           // 64 KB
constexpr uint32_t kW2StageBytes = kMaxRank * kTileV * 2;    // 32 KB
constexpr uint32_t kUBoxBytes = kRows * 32 * 4;              // 16 KB (32 tokens x 128 rows)
constexpr uint32_t kUStageBytes = 2 * kUBoxBytes;            // 32 KB
constexpr uint32_t kOffA = 0;
constexpr uint32_t kOffW2 = kOffA + kABytes;
constexpr uint32_t kOffU = kOffW2 + kNumW2Stages * kW2StageBytes;
constexpr uint32_t kOffBar = kOffU + kNumUStages * kUStageBytes;
constexpr uint32_t kBarRegion = 2048;
constexpr uint32_t kSmemBytes = kOffBar + kBarRegion + 1024;  // + alignment slack
// TMEM: kNumAcc accumulators of 64 columns, then the MMA's A operand ([128 x r] bf16,
// two elements per column: r / 2 <= 128 columns)
constexpr uint32_t kTmemA = kNumAcc * kTileV;                // 256
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kEpiBarrier = 1;                          // named barrier id
constexpr int kBoundRefresh = BOUND_REFRESH;  // tiles between reads of the global bound
constexpr uint32_t kBackoffControlNs = 200;  // sleep between polls of the TMA / MMA lanes
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.69314718055994531f;
constexpr uint32_t kTokenBits = 18;                          // V <= 2^18
constexpr uint32_t kTokenMask = (1u << kTokenBits) - 1u;

static_assert(kSmemBytes <= 232448, "draft kernel shared memory above the sm_103 limit");
static_assert(kTmemA + kMaxRank / 2 <= kTmemCols, "TMEM columns");
static_assert((kNumAcc & (kNumAcc - 1)) == 0, "accumulator count must be a power of two");
static_assert((2 * kNumW2Stages + 2 * kNumUStagesSmall + 2 * kNumAcc + 5) * 8 + 2 * kMaxK * 4 +
                      kRows * 8 + 16 <=
                  kBarRegion,
              "barrier region too small");

__device__ __forceinline__ uint32_t ordered_bits(float f) {
  const uint32_t b = __float_as_uint(f);
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

// Key order: larger epoch, then larger score, then smaller token id.
__device__ __forceinline__ unsigned long long make_key(uint32_t epoch, float score, int v) {
  return (static_cast<unsigned long long>(epoch) << 50) |
         (static_cast<unsigned long long>(ordered_bits(score)) << kTokenBits) |
         static_cast<unsigned long long>(kTokenMask - static_cast<uint32_t>(v));
}

__device__ __forceinline__ int key_token(unsigned long long key) {
  return static_cast<int>(kTokenMask - static_cast<uint32_t>(key & kTokenMask));
}

__device__ __forceinline__ uint32_t key_epoch(unsigned long long key) {
  return static_cast<uint32_t>(key >> 50);
}

// Optional phase trace: global-timer stamps of CTA `cta` at step k (thread etid 0).
__device__ __forceinline__ void trace_stamp(const DraftParams& p, int cta, int k, int slot) {
  if (p.trace != nullptr)
    p.trace[(static_cast<size_t>(cta) * p.K + k) * kTraceSlots + slot] = globaltimer_ns();
}

__device__ __forceinline__ float bf16_lo(uint32_t x) { return __uint_as_float(x << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t x) { return __uint_as_float(x & 0xFFFF0000u); }

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  const __nv_bfloat16 a = __float2bfloat16_rn(lo);
  const __nv_bfloat16 b = __float2bfloat16_rn(hi);
  return static_cast<uint32_t>(__bfloat16_as_ushort(a)) |
         (static_cast<uint32_t>(__bfloat16_as_ushort(b)) << 16);
}

// Small batches: with B <= 32 (64) requests, the 128 MMA rows hold 4 (2) copies
// of the batch, row m serving request m mod rows_per_copy, so that the TMEM lane
// quadrants of every epilogue warp hold real rows; the copies split the tiles.
__device__ __forceinline__ int rows_per_copy(int B) { return B <= 32 ? 32 : (B <= 64 ? 64 : 128); }

// Gather the step's Markov embeddings into the K-major, 128B-swizzled MMA
// operand: row b (request b mod rows_per_copy), 64-element K chunk c at
// c * 16 KB, 8-row groups of 1024 B, 16-byte unit u of row b stored at unit
// (u ^ (b & 7)).  Thread etid handles row etid / 4 and K chunk etid % 4.
__device__ __forceinline__ void gather_embeddings(uint8_t* sA, const DraftParams& p, int k,
                                                  int etid, int32_t tok) {
  const int b = etid >> 2, c = etid & 3;
  const int req = b & (rows_per_copy(p.B) - 1);
  const bool live = req < p.B;
  uint4 vals[8];
#pragma unroll
  for (int u = 0; u < 8; ++u) {
    const int kel = c * 64 + u * 8;
    if (live && kel < p.r) {
      vals[u] = __ldg(reinterpret_cast<const uint4*>(p.W1 + static_cast<size_t>(tok) * p.r + kel));
    } else {
      vals[u] = make_uint4(0u, 0u, 0u, 0u);
    }
  }
  if (p.H != nullptr && live) {
    const float* hrow = p.H + (static_cast<size_t>(req) * p.K + k) * p.r;
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int kel = c * 64 + u * 8;
      if (kel < p.r) {
        const float4 g0 = __ldg(reinterpret_cast<const float4*>(hrow + kel));
        const float4 g1 = __ldg(reinterpret_cast<const float4*>(hrow + kel + 4));
        uint4 x = vals[u];
        x.x = pack_bf16(bf16_lo(x.x) * g0.x, bf16_hi(x.x) * g0.y);
        x.y = pack_bf16(bf16_lo(x.y) * g0.z, bf16_hi(x.y) * g0.w);
        x.z = pack_bf16(bf16_lo(x.z) * g1.x, bf16_hi(x.z) * g1.y);
        x.w = pack_bf16(bf16_lo(x.w) * g1.z, bf16_hi(x.w) * g1.w);
        vals[u] = x;
      }
    }
  }
  uint8_t* base = sA + c * 16384 + (b >> 3) * 1024 + (b & 7) * 128;
#pragma unroll
  for (int u = 0; u < 8; ++u) {
    *reinterpret_cast<uint4*>(base + ((u ^ (b & 7)) << 4)) = vals[u];
  }
}

// Asynchronous form of gather_embeddings without a gate: the thread's 128-byte
// piece of W1[tok] goes to the operand by 16-byte cp.async copies (rows of no
// request and K chunks past r are zeroed with plain stores).
__device__ __forceinline__ void copy_embedding_async(uint8_t* sA, const DraftParams& p, int etid,
                                                     int32_t tok) {
  const int b = etid >> 2, c = etid & 3;
  const int req = b & (rows_per_copy(p.B) - 1);
  const bool live = req < p.B;
  uint8_t* base = sA + c * 16384 + (b >> 3) * 1024 + (b & 7) * 128;
#pragma unroll
  for (int u = 0; u < 8; ++u) {
    const int kel = c * 64 + u * 8;
    uint8_t* dst = base + ((u ^ (b & 7)) << 4);
    if (live && kel < p.r) {
      cp_async_16(dst, p.W1 + static_cast<size_t>(tok) * p.r + kel);
    } else {
      *reinterpret_cast<uint4*>(dst) = make_uint4(0u, 0u, 0u, 0u);
    }
  }
  cp_async_commit();
}

// Score of a key (the ordered float in its middle bits); -inf for "no key".
__device__ __forceinline__ float key_score(unsigned long long key) {
  if (key == 0ull) return -INFINITY;
  const uint32_t ob = static_cast<uint32_t>(key >> kTokenBits);
  const uint32_t bits = (ob & 0x80000000u) ? (ob & 0x7FFFFFFFu) : ~ob;
  return __uint_as_float(bits);
}

__device__ __forceinline__ void load_partial(const DraftPartial* src, unsigned long long& key,
                                             float& m2, float& sum, float& lbest) {
  key = __ldcg(reinterpret_cast<const unsigned long long*>(src));
  const float2 ms = __ldcg(reinterpret_cast<const float2*>(&src->m2));
  m2 = ms.x;
  sum = ms.y;
  lbest = __ldcg(&src->lbest);
}

// Merge (m_b, s_b) into (m_a, s_a): log-sum-exp in base 2.
__device__ __forceinline__ void lse_merge(float& ma, float& sa, float mb, float sb) {
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
    sa = sa + sb * ex2_approx(mb - ma);
  }
}

// One 16-token block's part in the two-stage race (w: the block's weights relative to
// 2^m2, s = their sum, y: their scaled logits): stage 1 scores the block by
// G = m2 + log2(s) - log2(E), E = -ln u1; a block that can still beat the best key
// known for the request (this thread's, the CTA's, or the global one as last read)
// runs stage 2, the first token whose cumulative weight exceeds u2 * s.
__device__ __forceinline__ void race_block(const float (&w)[16], const float (&y)[16], float m2,
                                           float bsum, uint32_t word1, uint32_t word2, int vbase,
                                           uint32_t epoch, float inv_scale2,
                                           unsigned long long* bound, unsigned long long gkey,
                                           unsigned long long& bkey, float& yb, int& vb,
                                           float& lb) {
  const float G = m2 + lg2_approx(bsum) - lg2_approx(neg_log_uniform_fast(word1));
  const unsigned long long sb = *bound;
  const float S = key_score(sb > gkey ? sb : gkey);
  if (bsum > 0.f && G >= S) {
    float C[16];
    C[0] = w[0];
#pragma unroll
    for (int j = 1; j < 16; ++j) C[j] = C[j - 1] + w[j];
    const float target = philox_uniform(word2) * C[15];
    int js = -1, jl = 0;
#pragma unroll
    for (int j = 15; j >= 0; --j) {
      if (target < C[j]) js = j;
      if (jl == 0 && w[j] > 0.f) jl = j;
    }
    if (js < 0) js = jl;  // target at the very top (rounding): the last live token
    float yj = 0.f;
#pragma unroll
    for (int j = 0; j < 16; ++j)
      if (j == js) yj = y[j];
    const unsigned long long key = make_key(epoch, G, vbase + js);
    if (key > bkey) {
      bkey = key;
      yb = G;
      vb = vbase + js;
      lb = yj * inv_scale2;
      atomicMax(bound, key);
    }
  }
}

template <int MODE, bool COPIES>
__global__ void __launch_bounds__(kThreads, 1) draft_kernel(const __grid_constant__ DraftArgs args) {
  const DraftParams& p = args.p;
  // teacher-forced modes take the predecessors from the caller
  constexpr bool kTF = MODE == kModeTeacherForced || MODE == kModeLabel || MODE == kModeResidual;
  // ring slots of half tiles holding U and the target rows
  constexpr bool kHalf = MODE == kModeLabel || MODE == kModeResidual;
  // modes that draw a token by the block race
  constexpr bool kRace = MODE == kModeSample || MODE == kModeResidual;
  // modes whose per-request winners are published as 64-bit keys
  constexpr bool kKeys = !kTF || MODE == kModeResidual;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* sA = smem + kOffA;
  uint8_t* sW = smem + kOffW2;
  uint8_t* sU = smem + kOffU;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kOffBar);
  uint64_t* w_full = bars;                          // [kNumW2Stages]
  uint64_t* w_empty = w_full + kNumW2Stages;        // [kNumW2Stages]
  uint64_t* u_full = w_empty + kNumW2Stages;        // [kNumUStagesSmall]
  uint64_t* u_empty = u_full + kNumUStagesSmall;    // [kNumUStagesSmall]
  uint64_t* acc_full = u_empty + kNumUStagesSmall;  // [kNumAcc]
  uint64_t* acc_empty = acc_full + kNumAcc;         // [kNumAcc]
  uint64_t* a_full = acc_empty + kNumAcc;
  uint64_t* a_empty = a_full + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(a_empty + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(a_empty + 2);
  int32_t* s_tok = reinterpret_cast<int32_t*>(a_empty + 3);  // [kMaxK]
  float* s_conf = reinterpret_cast<float*>(s_tok + kMaxK);  // [kMaxK]
  // best key (epoch | score | token) any thread of this CTA reached for each
  // request in the current step: a lower bound on the step's winner
  unsigned long long* s_bound = reinterpret_cast<unsigned long long*>(s_conf + kMaxK);  // [128]
  uint32_t* s_sink = reinterpret_cast<uint32_t*>(s_bound + kRows);  // scratch word (U releases)

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int cta = blockIdx.x, ncta = gridDim.x;
  const int t_begin = static_cast<int>(static_cast<int64_t>(cta) * p.n_tiles / ncta);
  const int t_end = static_cast<int>(static_cast<int64_t>(cta + 1) * p.n_tiles / ncta);
  const int nt = t_end - t_begin;
  const int nkk = p.r / 16;
  // Small batches use 4 U slots of 16 KB (a multiple of the batch copies, so every
  // use of a slot -- and of an accumulator -- is read by the same copy and its
  // warps see each mbarrier phase in order); larger ones 3 slots of 32 KB.
  // (COPIES: B <= 64; the B > 64 instantiation keeps these compile-time constants)
  const int nus = COPIES ? kNumUStagesSmall : kNumUStages;
  const uint32_t ubox = COPIES ? kUBoxBytes / 2 : kUBoxBytes;  // one 32-token box

  if (threadIdx.x == 0) {
    for (int s = 0; s < kNumW2Stages; ++s) {
      mbar_init(&w_full[s], 1);
      mbar_init(&w_empty[s], 1);
    }
    // a tile is read (and released) by the epilogue warps of one copy of the batch
    const uint32_t readers =
        COPIES ? static_cast<uint32_t>(kEpiWarps * rows_per_copy(p.B) / kRows) : kEpiWarps;
    for (int s = 0; s < nus; ++s) {
      mbar_init(&u_full[s], 1);
      mbar_init(&u_empty[s], readers);
    }
    for (int s = 0; s < kNumAcc; ++s) {
      mbar_init(&acc_full[s], 1);
      mbar_init(&acc_empty[s], readers);
    }
    mbar_init(a_full, 1);
    mbar_init(a_empty, 1);
    *abort_flag = 0;
    fence_mbar_init();
    if (nkk > 0) tma_prefetch_desc(&args.tm_w2);
    tma_prefetch_desc(&args.tm_u);
    if (kHalf) tma_prefetch_desc(&args.tm_p);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  if (warp == 0 && MODE == kModeResidual) {
    // ------------------------------------------------ TMA producer, residual mode
    // The draw rows are read in place: each request's base-logit row and target row at
    // its own draw position (tile::gather4 over 2-D row maps of U [B K, V] and
    // P [B (K + 1), V]), lane l fetching requests 4 l .. 4 l + 3 of every half tile into
    // the same slot layout as the 3-D boxes; lane 0 waits for the slots and loads W2.
    const uint64_t pol_w = l2_policy_evict_last();
    const uint64_t pol_u = l2_policy_evict_first();
    const uint32_t w_bytes = static_cast<uint32_t>(p.r) * kTileV * 2u;
    const uint32_t u_bytes = 2u * static_cast<uint32_t>(p.box_rows) * 128u;
    const bool mine = 4 * lane < p.box_rows;
    // the lane's four requests (past the batch: request 0 again, never read) and their draw
    // positions, a byte each (a position is at most K <= 64)
    uint32_t pos4 = 0;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int b = 4 * lane + q < p.B ? 4 * lane + q : 0;
      pos4 |= static_cast<uint32_t>(p.rows[b].pos) << (8 * q);
    }
    // row of request q of the lane in U (a bonus row reads no q: any valid row) or P
    auto draw_row = [&](int q, bool target) {
      const int gb = p.b_global0 + (4 * lane + q < p.B ? 4 * lane + q : 0);
      const int pos = static_cast<int>((pos4 >> (8 * q)) & 0xFFu);
      return target ? gb * (p.res_K + 1) + pos : gb * p.res_K + min(pos, p.res_K - 1);
    };
    bool ok = true;
    int w_issued = 0, u_issued = 0;
    for (int k = 0; k < p.K && ok; ++k) {
      for (int t = 0; t < nt; ++t) {
        const int i = k * nt + t;
        const int v0 = (t_begin + t) * kTileV;
        if (lane == 0 && nkk > 0) {
          const int s = i % kNumW2Stages;
          ok = mbar_wait(&w_empty[s], ((i / kNumW2Stages) & 1) ^ 1, p.timeout_ns, abort_flag,
                         kBackoffControlNs);
          if (ok) {
            mbar_arrive_expect_tx(&w_full[s], w_bytes);
            tma_load_2d(sW + s * kW2StageBytes, &args.tm_w2, v0, 0, &w_full[s], pol_w);
            w_issued = i + 1;
          }
        }
        ok = __shfl_sync(0xFFFFFFFFu, ok, 0);
        for (int h = 0; h < 2 && ok; ++h) {
          const int j = 2 * i + h, su = j % nus;
          if (lane == 0) {
            ok = mbar_wait(&u_empty[su], ((j / nus) & 1) ^ 1, p.timeout_ns, abort_flag,
                           kBackoffControlNs);
            if (ok) mbar_arrive_expect_tx(&u_full[su], u_bytes);
          }
          ok = __shfl_sync(0xFFFFFFFFu, ok, 0);
          if (!ok) break;
          if (mine) {
            uint8_t* dst = sU + su * 2 * ubox + lane * 512;
            tma_gather4_2d(dst, &args.tm_u, v0 + 32 * h, draw_row(0, false), draw_row(1, false),
                           draw_row(2, false), draw_row(3, false), &u_full[su], pol_u);
            tma_gather4_2d(dst + ubox, &args.tm_p, v0 + 32 * h, draw_row(0, true),
                           draw_row(1, true), draw_row(2, true), draw_row(3, true), &u_full[su],
                           pol_u);
          }
          u_issued = j + 1;
        }
        if (!ok) break;
      }
    }
    if (!ok && lane == 0) {
      *abort_flag = 1;
      record_error(p.status, kStatusTimeout);
      // Drain: every copy the warp started completes on the full barriers of its fills.
      for (int i = w_issued - 1; i >= 0 && i >= w_issued - kNumW2Stages; --i)
        mbar_wait(&w_full[i % kNumW2Stages], (i / kNumW2Stages) & 1, p.timeout_ns, nullptr);
      for (int i = u_issued - 1; i >= 0 && i >= u_issued - nus; --i)
        mbar_wait(&u_full[i % nus], (i / nus) & 1, p.timeout_ns, nullptr);
    }
  } else if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      const uint64_t pol_w = l2_policy_evict_last();
      const uint64_t pol_u = l2_policy_evict_first();
      const uint32_t w_bytes = static_cast<uint32_t>(p.r) * kTileV * 2u;
      const uint32_t u_bytes = 2u * static_cast<uint32_t>(p.box_rows) * 128u;
      bool ok = true;
      int w_issued = 0, u_issued = 0;  // u_issued: ring slot fills
      for (int k = 0; k < p.K && ok; ++k) {
        for (int t = 0; t < nt; ++t) {
          const int i = k * nt + t;
          const int v0 = (t_begin + t) * kTileV;
          if (nkk > 0) {
            const int s = i % kNumW2Stages;
            if (!mbar_wait(&w_empty[s], ((i / kNumW2Stages) & 1) ^ 1, p.timeout_ns, abort_flag,
                           kBackoffControlNs)) {
              ok = false;
              break;
            }
            mbar_arrive_expect_tx(&w_full[s], w_bytes);
            tma_load_2d(sW + s * kW2StageBytes, &args.tm_w2, v0, 0, &w_full[s], pol_w);
            w_issued = i + 1;
          }
          if (kHalf) {
            // two fills per tile: U and target tokens [v0 + 32 h, v0 + 32 h + 32)
            for (int h = 0; h < 2 && ok; ++h) {
              const int j = 2 * i + h, su = j % nus;
              if (!mbar_wait(&u_empty[su], ((j / nus) & 1) ^ 1, p.timeout_ns, abort_flag,
                             kBackoffControlNs)) {
                ok = false;
                break;
              }
              mbar_arrive_expect_tx(&u_full[su], u_bytes);
              tma_load_3d(sU + su * 2 * ubox, &args.tm_u, v0 + 32 * h, k, 0, &u_full[su], pol_u);
              tma_load_3d(sU + su * 2 * ubox + ubox, &args.tm_p, v0 + 32 * h, k, 0, &u_full[su],
                          pol_u);
              u_issued = j + 1;
            }
            if (!ok) break;
            continue;
          }
          const int su = i % nus;
          if (!mbar_wait(&u_empty[su], ((i / nus) & 1) ^ 1, p.timeout_ns, abort_flag,
                         kBackoffControlNs)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&u_full[su], u_bytes);
          tma_load_3d(sU + su * 2 * ubox, &args.tm_u, v0, k, 0, &u_full[su], pol_u);
          tma_load_3d(sU + su * 2 * ubox + ubox, &args.tm_u, v0 + 32, k, 0, &u_full[su],
                      pol_u);
          u_issued = i + 1;
        }
      }
      if (!ok) {
        *abort_flag = 1;
        record_error(p.status, kStatusTimeout);
        // Drain: every copy this thread started must land before the CTA exits.
        // The last issue of each ring slot is the one in [issued - stages, issued).
        for (int i = w_issued - 1; i >= 0 && i >= w_issued - kNumW2Stages; --i)
          mbar_wait(&w_full[i % kNumW2Stages], (i / kNumW2Stages) & 1, p.timeout_ns, nullptr);
        for (int i = u_issued - 1; i >= 0 && i >= u_issued - nus; --i)
          mbar_wait(&u_full[i % nus], (i / nus) & 1, p.timeout_ns, nullptr);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t idesc = idesc_bf16_f32(kRows, kTileV, /*a_mn=*/false, /*b_mn=*/true);
      const uint32_t a0 = smem_addr(sA);
      bool ok = true;
      int last_i = -1;
      for (int k = 0; k < p.K && ok; ++k) {
        if (!mbar_wait(a_full, k & 1, p.timeout_ns, abort_flag, 32u)) {
          ok = false;
          break;
        }
        tc_fence_after();
        for (int t = 0; t < nt; ++t) {
          const int i = k * nt + t;
          const int s = i % kNumW2Stages, buf = i % kNumAcc;
          if (nkk > 0 &&
              !mbar_wait(&w_full[s], (i / kNumW2Stages) & 1, p.timeout_ns, abort_flag,
                        kBackoffControlNs)) {
            ok = false;
            break;
          }
          if (!mbar_wait(&acc_empty[buf], ((i / kNumAcc) & 1) ^ 1, p.timeout_ns, abort_flag,
                         kBackoffControlNs)) {
            ok = false;
            break;
          }
          tc_fence_after();
          if (nkk > 0) {
            const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(buf * kTileV);
            const uint32_t b0 = smem_addr(sW + s * kW2StageBytes);
            for (int kk = 0; kk < nkk; ++kk) {
              const uint64_t bd = smem_desc(b0 + kk * 2048, 1024, 1024);
              umma_bf16_ts(d_tmem, tmem_base + kTmemA + static_cast<uint32_t>(kk * 8), bd, idesc,
                           kk > 0 ? 1u : 0u);
            }
            umma_commit(&w_empty[s]);
            umma_commit(&acc_full[buf]);
            last_i = i;
          } else {
            mbar_arrive(&acc_full[buf]);  // rank 0: the bias is zero, nothing to multiply
          }
        }
        if (!ok) break;
        if (nkk > 0) {
          umma_commit(a_empty);
        } else {
          mbar_arrive(a_empty);
        }
      }
      if (!ok) {
        *abort_flag = 1;
        record_error(p.status, kStatusTimeout);
      }
      // Drain: the last MMA batch must finish before TMEM is released.
      if (last_i >= 0)
        mbar_wait(&acc_full[last_i % kNumAcc], (last_i / kNumAcc) & 1, p.timeout_ns, nullptr);
    }
  } else {
    // ------------------------------------------------------------ epilogue warps
    const int e = warp - 2;          // 0 .. 15
    const int q = warp & 3;          // TMEM lane quadrant this warp may access
    const int g = e >> 2;            // 16-token column group of the 64-token tile
    const int rpc = COPIES ? rows_per_copy(p.B) : kRows;
    const int ncopy = COPIES ? kRows / rpc : 1;  // copies of the batch in the MMA rows
    const int b = (q * 32 + lane) & (rpc - 1);  // request of this thread's TMEM lane
    const int copy = (q * 32) / rpc;  // its copy: it reads tiles i (global index) with
                                      // i % ncopy == copy
    const int etid = threadIdx.x - 64;
    const bool row_ok = b < p.B;
    const uint32_t b_global = static_cast<uint32_t>(p.b_global0 + b);
    const float scale2 = p.inv_t * kLog2e;
    const float inv_scale2 = 1.0f / scale2;  // logit of the winner from its scaled value
    float* merge = reinterpret_cast<float*>(sA);  // reused after a step's MMAs completed
    // this thread's four 16-byte pieces of its U row within a stage (128B swizzle)
    uint32_t u_off[4];
#pragma unroll
    for (int c = 0; c < 4; ++c)
      u_off[c] = (g >> 1) * ubox + b * 128 + ((((g & 1) * 4 + c) ^ (b & 7)) << 4);
    bool fail = false;
    bool aborted = false;
    int u_stage = 0;        // U ring slot of the next tile
    uint32_t u_phase = 0;   // its mbarrier phase parity

    unsigned long long spec_key = 0ull;  // winner key this thread's row was gathered for
    for (int k = 0; k < p.K; ++k) {
      // ---- the step's embeddings: position 0 is gathered here; later positions were
      // gathered speculatively before the previous grid barrier and are re-checked now
      if (etid == 0) trace_stamp(p, cta, k, 0);
      {
        const int grow = (etid >> 2) & (rpc - 1);  // request of this thread's gather row
        if (k == 0) {
          int32_t tok = 0;
          if (grow < p.B) {
            tok = kTF ? __ldg(p.prev + static_cast<size_t>(grow) * p.K) : __ldg(p.anchors + grow);
            if (tok < 0 || tok >= p.V) {
              record_error(p.status, kStatusDeviceOob);
              tok = 0;
            }
          }
          if (!fail) gather_embeddings(sA, p, 0, etid, tok);
        } else if (!kTF && grow < p.B) {
          cp_async_wait_all();  // the speculative copy must land before any rewrite
          const unsigned long long key = __ldcg(p.keys + (k - 1) * kRows + grow);
          if (key != spec_key) {  // the winner changed after the speculative gather
            int32_t tok = key_token(key);
            if (key_epoch(key) != p.epoch || tok < 0 || tok >= p.V) {
              record_error(p.status, kStatusDeviceOob);
              tok = 0;
            }
            if (!fail) gather_embeddings(sA, p, k, etid, tok);
          }
        }
        if (etid < kRows) s_bound[etid] = 0ull;
        cp_async_wait_all();
      }
      fence_proxy_async_smem();
      named_bar_sync(kEpiBarrier, kEpiThreads);
      {
        // copy the operand into TMEM: each warp its lane quadrant's rows m = q*32 + lane,
        // K chunk e / 4 (64 bf16 = 32 columns); the previous position's MMAs finished
        // with the TMEM copy before the speculative gather (a_empty)
        const int m = q * 32 + lane, cc = e >> 2;
        const uint8_t* src = sA + cc * 16384 + (m >> 3) * 1024 + (m & 7) * 128;
        uint32_t wv[32];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const uint4 x = *reinterpret_cast<const uint4*>(src + ((u ^ (m & 7)) << 4));
          wv[4 * u + 0] = x.x;
          wv[4 * u + 1] = x.y;
          wv[4 * u + 2] = x.z;
          wv[4 * u + 3] = x.w;
        }
        tmem_st_x32(tmem_base + (static_cast<uint32_t>(q * 32) << 16) + kTmemA +
                        static_cast<uint32_t>(cc * 32),
                    wv);
        tmem_wait_st();
        tc_fence_before();
        named_bar_sync(kEpiBarrier, kEpiThreads);
      }
      if (etid == 0) {
        mbar_arrive(a_full);
        trace_stamp(p, cta, k, 1);
      }

      // ---- stream the step's tiles
      float m2 = (MODE == kModeLabel) ? 0.f : -INFINITY, sum = 0.f;  // label: a plain sum
      float offq2 = 0.f, offp2 = 0.f;  // label: log2 q = l * scale2 + offq2, log2 p likewise
      int res_pos = 0, res_excl = -1;  // residual: draw position, excluded token
      if (MODE == kModeLabel && row_ok) {
        const size_t o = static_cast<size_t>(b) * p.K + k;
        offq2 = __ldg(p.offq2 + o);
        offp2 = -__ldg(p.lse_t + o + b) * kLog2e;  // target row b * (K + 1) + k
      }
      if (MODE == kModeResidual && row_ok) {
        const ResRow rr = p.rows[b];
        offq2 = rr.offq2;
        offp2 = rr.offp2;
        res_pos = rr.pos;
        res_excl = rr.excl;
      }
      float yb = -INFINITY, lb = 0.f;  // best score (G, or y when greedy) and its logit
      int vb = 0x7FFFFFFF;
      unsigned long long bkey = 0ull;  // key of (yb, vb)
      unsigned long long gkey = 0ull;  // global key of this request and step, as last read
      uint32_t nz[4] = {0u, 0u, 0u, 0u};  // Philox words of this thread's current tile pair
      unsigned long long kpre = 0ull;  // global key, read one tile ahead of its use
      int tt = -1;                      // tiles of this step this thread has taken
      int nz_pair = -1;                 // tile pair whose Philox words nz holds
      for (int t = 0; t < nt && !fail; ++t) {
        const int i = k * nt + t;
        const int buf = i & (kNumAcc - 1);
        const int su = u_stage;
        const uint32_t uph = u_phase;
        if (++u_stage == nus) {
          u_stage = 0;
          u_phase ^= 1u;
        }
        if (COPIES && (i & (ncopy - 1)) != copy) continue;  // another copy's tile
        ++tt;
        if (kRace && row_ok) {
          // every other tile, refresh the bound with the key read a tile earlier, so
          // the load's latency is covered by a whole tile's work
          if (tt > 0 && (tt & (kBoundRefresh - 1)) == 0 && key_epoch(kpre) == p.epoch &&
              kpre > gkey)
            gkey = kpre;
          if (((tt + 1) & (kBoundRefresh - 1)) == 0) kpre = __ldcg(p.keys + k * kRows + b);
        }
        if (MODE == kModeResidual) {
          // the verification draw: this thread's 16 tokens [16 g, 16 g + 16) of tile i
          // (one block) come from fill 2 i + g / 2; every warp waits for and releases
          // both fills, so each slot keeps one group of readers taking its fills in order
          bool ok = mbar_wait(&acc_full[buf], (i / kNumAcc) & 1, p.timeout_ns, abort_flag);
          ok = __all_sync(0xFFFFFFFFu, ok);
          if (!ok) {
            fail = true;
            *abort_flag = 1;
            break;
          }
          tc_fence_after();
          uint32_t acc[16];
          if (nkk > 0) {
            tmem_ld_x16(tmem_base + (static_cast<uint32_t>(q * 32) << 16) +
                            static_cast<uint32_t>(buf * kTileV + g * 16),
                        acc);
            tmem_wait_ld();
          } else {
#pragma unroll
            for (int j = 0; j < 16; ++j) acc[j] = 0u;
          }
          float uval[16], pt[16];
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const int j = 2 * i + h, sh = j % nus;
            bool okh = mbar_wait(&u_full[sh], static_cast<uint32_t>(j / nus) & 1u, p.timeout_ns,
                                 abort_flag);
            okh = __all_sync(0xFFFFFFFFu, okh);
            if (!okh) {
              fail = true;
              *abort_flag = 1;
              break;
            }
            uint32_t dep = 0u;
            if (h == (g >> 1)) {
              const uint8_t* row = sU + sh * 2 * ubox + b * 128;
#pragma unroll
              for (int c = 0; c < 4; ++c) {
                const uint32_t off = static_cast<uint32_t>((((g & 1) * 4 + c) ^ (b & 7)) << 4);
                const float4 x = *reinterpret_cast<const float4*>(row + off);
                const float4 z = *reinterpret_cast<const float4*>(row + ubox + off);
                uval[4 * c + 0] = x.x;
                uval[4 * c + 1] = x.y;
                uval[4 * c + 2] = x.z;
                uval[4 * c + 3] = x.w;
                pt[4 * c + 0] = z.x;
                pt[4 * c + 1] = z.y;
                pt[4 * c + 2] = z.z;
                pt[4 * c + 3] = z.w;
                dep ^= __float_as_uint(x.x) ^ __float_as_uint(z.x);
              }
            }
            arrive_after_reads(&u_empty[sh], dep, s_sink, lane);
          }
          if (fail) break;
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&acc_empty[buf]);
          if (!row_ok) continue;
          const int tile = t_begin + t;
          const int vbase = tile * kTileV + g * 16;
          // weights max(0, p - q) (p alone for a bonus draw), relative to 2^0
          float w[16];
          float bsum = 0.f;
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const float lj = uval[j] + __uint_as_float(acc[j]);
            const float pj = ex2_approx(fmaf(pt[j], p.target_scale2, offp2));
            const float qj = ex2_approx(fmaf(lj, scale2, offq2));  // 0 when offq2 = -inf
            float wj = fmaxf(0.f, pj - qj);
            if (vbase + j >= p.V || vbase + j == res_excl) wj = 0.f;
            w[j] = wj;
            bsum += wj;
          }
          if ((tile >> 1) != nz_pair) {
            nz_pair = tile >> 1;
            philox4x32_10_rk(static_cast<uint32_t>(tile >> 1), static_cast<uint32_t>(res_pos),
                             b_global, 9u + static_cast<uint32_t>(g), p.round_key0, p.round_key1,
                             nz);
          }
          race_block(w, w, 0.f, bsum, (tile & 1) ? nz[2] : nz[0], (tile & 1) ? nz[3] : nz[1],
                     vbase, p.epoch, inv_scale2, &s_bound[b], gkey, bkey, yb, vb, lb);
          if ((tt & 1) == 1 && g == 0) {
            const unsigned long long mine = s_bound[b];
            if (mine > gkey) {
              atomicMax(p.keys + k * kRows + b, mine);
              gkey = mine;
            }
          }
          continue;
        }
        if (kHalf) {
          // label: tile i is ring fills 2 i (tokens 0-31) and 2 i + 1 (32-63), each
          // holding U and the target; this thread takes tokens 8 g .. 8 g + 7 of both
          bool ok = mbar_wait(&acc_full[buf], (i / kNumAcc) & 1, p.timeout_ns, abort_flag);
          ok = __all_sync(0xFFFFFFFFu, ok);
          if (!ok) {
            fail = true;
            *abort_flag = 1;
            break;
          }
          tc_fence_after();
          uint32_t acc[16];
          if (nkk > 0) {
            const uint32_t ta = tmem_base + (static_cast<uint32_t>(q * 32) << 16) +
                                static_cast<uint32_t>(buf * kTileV + g * 8);
            tmem_ld_x8(ta, acc);
            tmem_ld_x8(ta + 32, acc + 8);
            tmem_wait_ld();
          } else {
#pragma unroll
            for (int j = 0; j < 16; ++j) acc[j] = 0u;
          }
          float uval[16], pt[16];
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const int j = 2 * i + h, sh = j % nus;
            bool okh = mbar_wait(&u_full[sh], static_cast<uint32_t>(j / nus) & 1u, p.timeout_ns,
                                 abort_flag);
            okh = __all_sync(0xFFFFFFFFu, okh);
            if (!okh) {
              fail = true;
              *abort_flag = 1;
              break;
            }
            const uint8_t* row = sU + sh * 2 * ubox + b * 128;
            uint32_t dep = 0u;
#pragma unroll
            for (int c = 0; c < 2; ++c) {
              const uint32_t off = static_cast<uint32_t>(((2 * g + c) ^ (b & 7)) << 4);
              const float4 x = *reinterpret_cast<const float4*>(row + off);
              const float4 y = *reinterpret_cast<const float4*>(row + ubox + off);
              uval[8 * h + 4 * c + 0] = x.x;
              uval[8 * h + 4 * c + 1] = x.y;
              uval[8 * h + 4 * c + 2] = x.z;
              uval[8 * h + 4 * c + 3] = x.w;
              pt[8 * h + 4 * c + 0] = y.x;
              pt[8 * h + 4 * c + 1] = y.y;
              pt[8 * h + 4 * c + 2] = y.z;
              pt[8 * h + 4 * c + 3] = y.w;
              dep ^= __float_as_uint(x.x) ^ __float_as_uint(y.x);
            }
            arrive_after_reads(&u_empty[sh], dep, s_sink, lane);
          }
          if (fail) break;
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&acc_empty[buf]);
          if (!row_ok) continue;
          // past V the boxes read zeros; the target side is masked to p = 0
          const int vt = (t_begin + t) * kTileV;
          if (vt + kTileV > p.V) {
#pragma unroll
            for (int j = 0; j < 16; ++j)
              if (vt + (j >> 3) * 32 + g * 8 + (j & 7) >= p.V) pt[j] = -INFINITY;
          }
          // sum of min(q, p) over the thread's columns
          const float2 sq = make_float2(scale2, scale2), oq = make_float2(offq2, offq2);
          const float2 sp = make_float2(p.target_scale2, p.target_scale2);
          const float2 op = make_float2(offp2, offp2);
          float2 acc2 = make_float2(0.f, 0.f);
#pragma unroll
          for (int j = 0; j < 16; j += 2) {
            const float2 lj = __fadd2_rn(make_float2(uval[j], uval[j + 1]),
                                         make_float2(__uint_as_float(acc[j]),
                                                     __uint_as_float(acc[j + 1])));
            const float2 aq = __ffma2_rn(lj, sq, oq);
            const float2 ap = __ffma2_rn(make_float2(pt[j], pt[j + 1]), sp, op);
            acc2 = __fadd2_rn(acc2, make_float2(ex2_approx(fminf(aq.x, ap.x)),
                                                ex2_approx(fminf(aq.y, ap.y))));
          }
          sum += acc2.x + acc2.y;
          continue;
        }
        bool ok = mbar_wait(&acc_full[buf], (i / kNumAcc) & 1, p.timeout_ns, abort_flag);
        ok = ok && mbar_wait(&u_full[su], uph, p.timeout_ns, abort_flag);
        ok = __all_sync(0xFFFFFFFFu, ok);
        if (!ok) {
          fail = true;
          *abort_flag = 1;
          break;
        }
        tc_fence_after();
        if (tt == 0 && etid == 0) trace_stamp(p, cta, k, 2);
        uint32_t acc[16];
        if (nkk > 0) {
          tmem_ld_x16(tmem_base + (static_cast<uint32_t>(q * 32) << 16) +
                          static_cast<uint32_t>(buf * kTileV + g * 16),
                      acc);
          tmem_wait_ld();
        } else {
#pragma unroll
          for (int j = 0; j < 16; ++j) acc[j] = 0u;
        }
        float uval[16];
        {
          const uint8_t* ubase = sU + su * 2 * ubox;
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            const float4 x = *reinterpret_cast<const float4*>(ubase + u_off[c]);
            uval[4 * c + 0] = x.x;
            uval[4 * c + 1] = x.y;
            uval[4 * c + 2] = x.z;
            uval[4 * c + 3] = x.w;
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&acc_empty[buf]);  // tcgen05.wait::ld returned the values
        arrive_after_reads(&u_empty[su],
                           __float_as_uint(uval[0]) ^ __float_as_uint(uval[4]) ^
                               __float_as_uint(uval[8]) ^ __float_as_uint(uval[12]),
                           s_sink, lane);
        if (!row_ok) continue;

        const int vbase = (t_begin + t) * kTileV + g * 16;
        const bool full_chunk = vbase + 16 <= p.V;  // warp-uniform
        float y[16];
#pragma unroll
        for (int j = 0; j < 16; j += 2) {
          const float2 lj = __fadd2_rn(make_float2(uval[j], uval[j + 1]),
                                       make_float2(__uint_as_float(acc[j]),
                                                   __uint_as_float(acc[j + 1])));
          if (MODE == kModeTeacherForced) {
            uval[j] = lj.x;  // keep the logits for the store below
            uval[j + 1] = lj.y;
          }
          const float2 yj = __fmul2_rn(lj, make_float2(scale2, scale2));
          y[j] = yj.x;
          y[j + 1] = yj.y;
        }
        if (!full_chunk) {
#pragma unroll
          for (int j = 0; j < 16; ++j)
            if (vbase + j >= p.V) y[j] = -INFINITY;
        }
        if (MODE == kModeTeacherForced) {
          float* dst = p.logits + (static_cast<size_t>(b) * p.K + k) * p.V + vbase;
          if (full_chunk) {
#pragma unroll
            for (int c = 0; c < 4; ++c)
              reinterpret_cast<float4*>(dst)[c] =
                  make_float4(uval[4 * c], uval[4 * c + 1], uval[4 * c + 2], uval[4 * c + 3]);
          } else {
            for (int j = 0; j < 16 && vbase + j < p.V; ++j) dst[j] = uval[j];
          }
        }
        // chunk maximum (tree)
        float mx[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) mx[j] = fmaxf(y[j], y[j + 8]);
#pragma unroll
        for (int j = 0; j < 4; ++j) mx[j] = fmaxf(mx[j], mx[j + 4]);
        const float cmax = fmaxf(fmaxf(mx[0], mx[2]), fmaxf(mx[1], mx[3]));
        if (cmax == -INFINITY) continue;  // nothing in this chunk can be drawn
        if (cmax > m2) {
          sum *= ex2_approx(m2 - cmax);
          m2 = cmax;
        }
        float w[16];
        float bsum;  // the block's mass relative to 2^m2
#pragma unroll
        for (int j = 0; j < 16; j += 2) {
          const float2 dj = __fadd2_rn(make_float2(y[j], y[j + 1]), make_float2(-m2, -m2));
          w[j] = ex2_approx(dj.x);
          w[j + 1] = ex2_approx(dj.y);
        }
        {
          float2 s0 = __fadd2_rn(make_float2(w[0], w[1]), make_float2(w[2], w[3]));
          float2 s1 = __fadd2_rn(make_float2(w[4], w[5]), make_float2(w[6], w[7]));
          float2 s2 = __fadd2_rn(make_float2(w[8], w[9]), make_float2(w[10], w[11]));
          float2 s3 = __fadd2_rn(make_float2(w[12], w[13]), make_float2(w[14], w[15]));
          s0 = __fadd2_rn(__fadd2_rn(s0, s1), __fadd2_rn(s2, s3));
          bsum = s0.x + s0.y;
          sum += bsum;
        }
        if (MODE == kModeSample) {
          const int tile = t_begin + t;
          if ((tile >> 1) != nz_pair) {
            nz_pair = tile >> 1;
            philox4x32_10_rk(static_cast<uint32_t>(tile >> 1), static_cast<uint32_t>(k), b_global,
                             1u + static_cast<uint32_t>(g), p.round_key0, p.round_key1, nz);
          }
          race_block(w, y, m2, bsum, (tile & 1) ? nz[2] : nz[0], (tile & 1) ? nz[3] : nz[1], vbase,
                     p.epoch, inv_scale2, &s_bound[b], gkey, bkey, yb, vb, lb);
          if ((tt & 1) == 1 && g == 0) {
            // share this CTA's best with the other CTAs (rate-limited)
            const unsigned long long mine = s_bound[b];
            if (mine > gkey) {
              atomicMax(p.keys + k * kRows + b, mine);
              gkey = mine;
            }
          }
        } else if (MODE == kModeGreedy) {
          if (cmax > yb) {
            int jb = 15;
#pragma unroll
            for (int j = 15; j >= 0; --j)
              if (y[j] == cmax) jb = j;
            yb = cmax;
            vb = vbase + jb;
            lb = 0.f;
#pragma unroll
            for (int j = 0; j < 16; ++j)
              if (j == jb) lb = y[j];
            lb *= inv_scale2;
            atomicMax(&s_bound[b], make_key(p.epoch, yb, vb));
          }
          if ((tt & 1) == 1 && g == 0) {
            // publish this CTA's best so far (lets other CTAs gather the next
            // position's embeddings speculatively before the grid barrier)
            const unsigned long long mine = s_bound[b];
            if (mine > gkey) {
              atomicMax(p.keys + k * kRows + b, mine);
              gkey = mine;
            }
          }
        }
      }

      // ---- merge the column groups (and copies) of each request, publish the CTA's
      // partial; record slot sl = copy * 4 + g, rpc rows per record field
      if (etid == 0) trace_stamp(p, cta, k, 3);
      // sampling a full batch: the global key of this thread's gather row is read now, so
      // that the merge hides the load (greedy draws and batch copies keep the later,
      // fresher read: measured faster there)
      constexpr bool kEarlyKey = MODE == kModeSample && !COPIES;
      const int grow_pre = (etid >> 2) & (rpc - 1);
      const unsigned long long gk_pre =
          (kEarlyKey && k + 1 < p.K && grow_pre < p.B)
              ? __ldcg(p.keys + k * kRows + grow_pre)
              : 0ull;
      const float score = yb;
      const int slot = copy * 4 + g;
      // the merge records live in the operand's memory: with several copies a warp can
      // get here while the MMAs of other copies' last tiles still read it
      if (!fail && !mbar_wait(a_empty, k & 1, p.timeout_ns, abort_flag)) {
        fail = true;
        *abort_flag = 1;
      }
      if (!fail) {
        merge[(slot * 5 + 0) * rpc + b] = m2;
        merge[(slot * 5 + 1) * rpc + b] = sum;
        merge[(slot * 5 + 2) * rpc + b] = score;
        merge[(slot * 5 + 3) * rpc + b] = __int_as_float(vb);
        merge[(slot * 5 + 4) * rpc + b] = lb;
      }
      named_bar_sync(kEpiBarrier, kEpiThreads);
      if (!fail && slot == 0 && row_ok) {
        float M = merge[0 * rpc + b], S = merge[1 * rpc + b];
        float best_s = merge[2 * rpc + b], best_l = merge[4 * rpc + b];
        int best_v = __float_as_int(merge[3 * rpc + b]);
        for (int ss = 1; ss < 4 * ncopy; ++ss) {
          lse_merge(M, S, merge[(ss * 5 + 0) * rpc + b], merge[(ss * 5 + 1) * rpc + b]);
          const float s2 = merge[(ss * 5 + 2) * rpc + b];
          const int v2 = __float_as_int(merge[(ss * 5 + 3) * rpc + b]);
          if (v2 != 0x7FFFFFFF && (s2 > best_s || (s2 == best_s && v2 < best_v))) {
            best_s = s2;
            best_v = v2;
            best_l = merge[(ss * 5 + 4) * rpc + b];
          }
        }
        unsigned long long key = 0ull;
        if (kKeys && best_v != 0x7FFFFFFF) {
          key = make_key(p.epoch, best_s, best_v);
          atomicMax(p.keys + k * kRows + b, key);
          if (!kTF && key >= gkey && k + 1 < p.K) {
            // this CTA may hold the winner: pull its Markov embedding into L2 so that
            // every CTA's gather for the next position hits L2
            const char* row = reinterpret_cast<const char*>(p.W1 + static_cast<size_t>(best_v) * p.r);
            for (int off = 0; off < p.r * 2; off += 128)
              asm volatile("prefetch.global.L2 [%0];" ::"l"(row + off));
          }
        }
        DraftPartial* dst = p.partials + (static_cast<size_t>(k) * kRows + b) * ncta + cta;
        dst->key = key;
        dst->m2 = M;
        dst->sum = S;
        dst->lbest = best_l;
      }
      named_bar_sync(kEpiBarrier, kEpiThreads);

      // ---- arrive at the grid barrier (the wait comes after the speculative gather)
      if (etid == 0 && !fail) {
        const bool skip = (p.debug_skip_cta == cta) && (k == 0);
        // the release add orders every epilogue thread's partial and key writes
        // (synchronised by the named barrier above) before the arrival
        if (!skip) red_release_gpu_add(p.bar, 1u);
      }

      if (etid == 0) trace_stamp(p, cta, k, 7);
      // ---- speculative gather for the next position: the likely winner is the better
      // of the global key (read before the merge) and this CTA's best (complete now);
      // without a gate its row is copied asynchronously and lands while the grid
      // barrier completes
      if (k + 1 < p.K && !fail) {
        if (!mbar_wait(a_empty, k & 1, p.timeout_ns, abort_flag)) {  // MMAs done reading E
          fail = true;
          *abort_flag = 1;
        } else {
          const int grow = (etid >> 2) & (rpc - 1);
          int32_t tok = 0;
          if (grow < p.B) {
            if (kTF) {
              tok = __ldg(p.prev + static_cast<size_t>(grow) * p.K + k + 1);
              if (tok < 0 || tok >= p.V) {
                record_error(p.status, kStatusDeviceOob);
                tok = 0;
              }
            } else {
              const unsigned long long gk =
                  kEarlyKey ? gk_pre : __ldcg(p.keys + k * kRows + grow);
              const unsigned long long lk = s_bound[grow];
              spec_key = (key_epoch(gk) == p.epoch && gk > lk) ? gk : lk;
              tok = key_token(spec_key);
              if (key_epoch(spec_key) != p.epoch || tok < 0 || tok >= p.V) {
                spec_key = ~0ull;  // never matches: refetched after the barrier
                tok = 0;
              }
            }
          }
          if (p.H == nullptr) {
            copy_embedding_async(sA, p, etid, tok);
          } else {
            gather_embeddings(sA, p, k + 1, etid, tok);
          }
        }
      }

      // ---- grid barrier (bounded); teacher-forced positions are independent, so
      // those modes wait only before the final reduction
      bool bar_fail = false;
      if (etid == 0) trace_stamp(p, cta, k, 4);
      if (etid == 0 && !fail && (!kTF || k + 1 == p.K)) {
        const uint32_t target = p.bar_base + static_cast<uint32_t>((k + 1) * ncta);
        uint64_t deadline = 0;
        for (uint32_t it = 0;; ++it) {
          const uint32_t cur = ld_acquire_gpu(p.bar);
          if (static_cast<int32_t>(cur - target) >= 0) break;
          if ((it & 15u) == 15u) {
            const uint64_t now = globaltimer_ns();
            if (deadline == 0) {
              deadline = now + p.timeout_ns;
            } else if (now > deadline || *abort_flag) {
              bar_fail = true;
              break;
            }
          }
        }
        trace_stamp(p, cta, k, 5);  // the acquire load above orders the reads that follow
      }
      const bool any = named_bar_or(kEpiBarrier, kEpiThreads, fail || bar_fail || *abort_flag);
      if (any) {
        if (etid == 0) {
          *abort_flag = 1;
          record_error(p.status, kStatusTimeout);
        }
        aborted = true;
        break;
      }
    }

    // ---- final reduction: CTA c owns requests c, c + grid, ...
    if (!aborted) {
      for (int bb = cta; bb < p.B; bb += ncta) {
        for (int k = e; k < p.K; k += kEpiWarps) {
          const DraftPartial* src = p.partials + (static_cast<size_t>(k) * kRows + bb) * ncta;
          const unsigned long long gkey =
              kKeys ? __ldcg(p.keys + k * kRows + bb) : 0ull;
          float M = -INFINITY, S = 0.f, lwin = 0.f;
          int found = 0;
          for (int c = lane; c < ncta; c += 32) {
            unsigned long long key;
            float m2, s, lbest;
            load_partial(src + c, key, m2, s, lbest);
            lse_merge(M, S, m2, s);
            if (kKeys && key == gkey) {
              lwin = lbest;
              found = 1;
            }
          }
#pragma unroll
          for (int off = 16; off > 0; off >>= 1) {
            const float Mo = __shfl_xor_sync(0xFFFFFFFFu, M, off);
            const float So = __shfl_xor_sync(0xFFFFFFFFu, S, off);
            lse_merge(M, S, Mo, So);
          }
          const unsigned who = __ballot_sync(0xFFFFFFFFu, found);
          lwin = __shfl_sync(0xFFFFFFFFu, lwin, who ? __ffs(who) - 1 : 0);
          if (lane == 0) {
            const float lse_nat = (M + log2f(S)) * kLn2;
            const size_t o = static_cast<size_t>(bb) * p.K + k;
            if (MODE == kModeTeacherForced) {
              p.lse[o] = lse_nat;
            } else if (MODE == kModeLabel) {
              const float tot = (M == -INFINITY) ? 0.f : S * exp2f(M);
              p.label[o] = fminf(fmaxf(tot, 0.f), 1.f);
            } else {
              int v = key_token(gkey);
              if (who == 0 || key_epoch(gkey) != p.epoch || v < 0 || v >= p.V) {
                record_error(p.status, kStatusDeviceOob);
                v = 0;
              }
              p.tokens[o] = v;
              if (MODE != kModeResidual) p.logprobs[o] = lwin * p.inv_t - lse_nat;
              s_tok[k] = v;
            }
          }
        }
        if (!kTF && p.conf != nullptr) {
          named_bar_sync(kEpiBarrier, kEpiThreads);
          const int d = p.conf_d;
          for (int k = e; k < p.K; k += kEpiWarps) {
            const int32_t prev_tok = (k == 0) ? __ldg(p.anchors + bb) : s_tok[k - 1];
            const uint16_t* emb =
                p.conf_with_markov ? p.W1 + static_cast<size_t>(prev_tok) * p.r : nullptr;
            const float z = confidence_logit(p.conf_h + (static_cast<size_t>(bb) * p.K + k) * d,
                                             d, p.conf_w, emb, p.r, p.conf_bias, lane);
            if (lane == 0)
              s_conf[k] = sigmoidf_accurate(p.conf_tau ? z / __ldg(p.conf_tau + k) : z);
          }
          named_bar_sync(kEpiBarrier, kEpiThreads);
          if (etid == 0) {
            float surv = 1.f;
            int len = 0;
            bool open = true;
            for (int k = 0; k < p.K; ++k) {
              const float c = s_conf[k];
              surv *= c;
              const size_t o = static_cast<size_t>(bb) * p.K + k;
              p.conf[o] = c;
              p.cumprod[o] = surv;
              if (open && surv >= p.conf_threshold) {
                len = k + 1;
              } else {
                open = false;
              }
            }
            p.verify_len[bb] = len;
          }
        }
        named_bar_sync(kEpiBarrier, kEpiThreads);
      }
      if (etid == 0) trace_stamp(p, cta, p.K - 1, 6);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem_base, kTmemCols);
  }
}

}  // namespace

int draft_smem_bytes() { return static_cast<int>(kSmemBytes); }
int draft_threads() { return kThreads; }

cudaError_t launch_draft(const DraftArgs& args, int mode, int grid, cudaStream_t stream) {
  const void* fn = nullptr;
  const bool copies = args.p.B <= 64;  // small batches fill the MMA rows with copies
  switch (mode) {
    case kModeSample:
      fn = copies ? reinterpret_cast<const void*>(&draft_kernel<kModeSample, true>)
                  : reinterpret_cast<const void*>(&draft_kernel<kModeSample, false>);
      break;
    case kModeGreedy:
      fn = copies ? reinterpret_cast<const void*>(&draft_kernel<kModeGreedy, true>)
                  : reinterpret_cast<const void*>(&draft_kernel<kModeGreedy, false>);
      break;
    case kModeTeacherForced:
      fn = copies ? reinterpret_cast<const void*>(&draft_kernel<kModeTeacherForced, true>)
                  : reinterpret_cast<const void*>(&draft_kernel<kModeTeacherForced, false>);
      break;
    case kModeLabel:  // half-tile ring slots: always the 128-row instantiation
      fn = reinterpret_cast<const void*>(&draft_kernel<kModeLabel, false>);
      break;
    case kModeResidual:
      fn = reinterpret_cast<const void*>(&draft_kernel<kModeResidual, false>);
      break;
    default: return cudaErrorInvalidValue;
  }
  cudaError_t err = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(kSmemBytes));
  if (err != cudaSuccess) return err;
  void* kargs[] = {const_cast<DraftArgs*>(&args)};
  return cudaLaunchCooperativeKernel(fn, dim3(grid), dim3(kThreads), kargs, kSmemBytes, stream);
}

}  // namespace dspark
