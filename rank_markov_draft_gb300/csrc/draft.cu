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
//   * the vocabulary is split into 128-token tiles (the MMA's N); CTA c owns
//     a fixed, contiguous range of tiles for every step.  A tcgen05.mma of
//     M = 128 rows and K = 16 costs about the same time for N = 64, 128 or 256,
//     so the tile is as wide as the tensor memory allows: three 128-column
//     accumulators plus the 128 columns of the A operand fill the 512 columns;
//   * warp 0 (one lane) streams U in 64-token sub-tiles [rows x 64] fp32 with TMA
//     into its ring (two sub-tiles a tile); it never depends on sampled tokens,
//     so it runs ahead across step boundaries.  Above 64 requests a sub-tile is
//     two "row-pair" boxes of 64 rows x 64 tokens (256 contiguous bytes of each
//     row, which DRAM serves far better than 128-byte pieces of rows 9.7 MB
//     apart); otherwise two boxes of 32 tokens x every row;
//   * the tiles of a step are streamed in ascending order at even steps and in
//     descending order at odd ones, so a step starts on the W2 tiles the
//     previous one used last;
//   * warp 1 (one lane) streams W2 in slices of [128 rank rows x 128 tokens]
//     bf16 (a tile is one slice per 128 of the rank) into a 3-slot ring (a
//     fourth slot with batch copies, in the U ring's free tail), slices ahead
//     of its own MMAs, and issues tcgen05.mma: D[128 requests x
//     128 tokens] = E[128 x r] * W2tile[r x 128] into one of three TMEM
//     accumulators.  E, the step's operand for every request (the gathered
//     Markov embedding, gated or not, or the RNN head's state), lives in TMEM
//     (row m in lane m, two bf16 per column), written there by the epilogue
//     threads straight from global memory (no shared-memory staging); W2 is
//     the MN-major slice exactly as TMA wrote it;
//   * warps 2..9 (the epilogue, two warps per TMEM lane quadrant) read the
//     accumulator (one request per TMEM lane, 32 tokens -- two 16-token blocks
//     -- of each 64-token sub-tile per thread) and U from shared memory, and
//     keep, per request, a running log-sum-exp and each thread's best block of
//     the race (its values parked in shared memory), so the full-vocabulary
//     logits never reach HBM; stage 2 of the race runs once per step per
//     thread, in that best block;
//   * warps 10 and 11 exist in two builds only: in the sampling build above 64
//     requests they draw the race's stage-1 noise of every epilogue thread's
//     blocks a tile ahead into a two-tile shared-memory ring (noise warps); in
//     the residual build they share the gathered-row copies with warp 0;
//   * at the end of a step each CTA publishes, per request, a 64-bit key
//     (epoch | ordered score | inverted token id) by atomicMax (only where it
//     can still raise the key) and its log-sum-exp partial; it arrives at a
//     bounded grid barrier and, while the others finish, gathers the next
//     step's operand for the winners known so far (the gated head loads its
//     gate rows before the winners' keys; the RNN head parks the decayed state
//     a (.) s in free accumulator columns); after the barrier the operand goes
//     to TMEM, re-gathered only for rows whose winner changed;
//   * after the last step, CTA c reduces request c's partials into tokens and
//     log-probabilities and runs the fused confidence head.
//
// Small batches (B <= 64): the 128 MMA rows hold two copies of the batch (row
// m serves request m mod 64); copy c takes the 64-token sub-tile c of every
// tile, so every TMEM lane quadrant holds real rows.
//
// Template parameters: MODE, COPIES (batch copies, B <= 64) and GATED (the launch
// may carry gates; the plain build compiles the operand path without them).
//
// Teacher-forced modes take every position's predecessor from the caller, so
// positions do not depend on one another: the next position's operand is
// written during the current position's last tile, as soon as its MMAs are done
// with the operand, and the grid barrier is waited on only before the final
// reduction.  The label mode
// (DSpark explainer, "Confidence-scheduled verification": c*_k = 1 - TV of the
// draft head's and the target's distributions) streams the target's rows
// beside U and sums 2^min(log2 q(v), log2 p(v)) over the vocabulary, both
// normalisers known beforehand (the target's from a row scan, the draft's
// from its own log-probability of the drafted token).  Its ring slots hold U
// and target for half a sub-tile, two slots per sub-tile: 32 tokens of every
// row, or with row-pair boxes 64 tokens of rows [64 h, 64 h + 64); every
// epilogue warp waits for and releases both (reading the one that holds its
// tokens), so each slot has one group of readers that takes its fills in order.
//
// Sampling epilogue (an exact draw from softmax(l / T) in two stages over
// 16-token blocks; each thread's 16 columns of a sub-tile are one block beta):
//   y = l * log2(e) / T, w = 2^(y - m) (shared with the log-sum-exp), and the
//   block's mass relative to m is s = sum w;
//   stage 1, a race between blocks: the block maximising
//     G = m + log2(s) - log2(E),  E = -ln u1 (a unit exponential)
//   wins with probability Z_beta / Z (argmax Z_beta / E_beta);
//   stage 2, once per step in the thread's best block (its 16 weights kept in
//   shared memory while the sweep goes on): the first token whose cumulative
//   w exceeds u2 * s.  The four blocks' uniforms of a thread in a tile come
//   from two interleaved Philox calls.  The (G, token) winner is merged across
//   threads and CTAs as a key.
//
// Every wait is bounded (mbarrier waits and the grid barrier give up after
// timeout_ns, set the device status word and make the CTA exit cleanly after
// draining its own TMA copies and MMAs and freeing its TMEM).

#include <cstdint>
#include <cuda_bf16.h>

#include "checks.cuh"
#include "confidence.cuh"
#include "internal.h"
#include "philox.cuh"
#include "sm103.cuh"

namespace dspark {
namespace {

constexpr int kTileN = kDraftTileN;              // 128 tokens per MMA tile (MMA N)
constexpr int kSubV = 64;                        // tokens per epilogue sub-tile (U ring slot)
constexpr int kRows = kBatchChunk;               // 128 requests (MMA M)
constexpr int kNumW2Slots = 3;                   // W2 ring: slices of [128 rows x 128 tokens]
// With batch copies (B <= 64) the U ring's four 16 KB slots leave the last 32 KB of its region
// free: a fourth W2 slot goes there
constexpr int kNumW2SlotsMax = 4;
constexpr int kKSlice = kDraftSliceRows / 16;    // MMAs (K = 16 each) per W2 slice
constexpr int kNumUStages = 3;                   // U ring slots of 32 KB (B > 64)
constexpr int kNumUStagesSmall = 4;              // slots of 16 KB when B <= 64 (box <= 64 rows)
constexpr int kNumAcc = 3;                       // TMEM accumulators, 128 columns each
constexpr int kCtlWarps = 2;                     // U producer; MMA issuer and W2 producer
// Eight epilogue warps: two per TMEM lane quadrant, each thread taking 32 tokens (two
// 16-token blocks) of every 64-token sub-tile.  Ten warps in all (twelve in the builds with
// two more warps, below) leave up to 168 registers a thread (three warps on a scheduler),
// enough for two blocks at once.
constexpr int kEpiWarps = 8;
constexpr int kEpiThreads = kEpiWarps * 32;      // 256
constexpr int kThreads = kCtlWarps * 32 + kEpiThreads;  // 320
// The residual draw reads its rows with tile::gather4, whose copies one warp issues at about
// one per 45 ns whatever their size: two more warps (10 and 11, still three warps on a
// scheduler at most) share each fill's copies with warp 0.
constexpr int kResCopyWarps = 2;
constexpr int kResProducers = 1 + kResCopyWarps;
// The sampling mode above 64 requests runs two more warps too (noise warps): they draw the
// race's stage-1 exponentials of every epilogue thread's blocks, a tile ahead, into a
// two-tile ring in shared memory, taking the two Philox calls per thread and tile off the
// epilogue warps (with batch copies, a thread using one sub-tile of each tile, the handoff
// measured slower than the calls).
constexpr int kNoiseWarps = 2;
template <int MODE, bool COPIES>
__host__ __device__ constexpr bool noise_warps() {
  return MODE == kModeSample && !COPIES;
}
template <int MODE, bool COPIES>
__host__ __device__ constexpr int threads_of() {
  return kThreads + (MODE == kModeResidual              ? kResCopyWarps * 32
                     : noise_warps<MODE, COPIES>()      ? kNoiseWarps * 32
                                                        : 0);
}
constexpr uint32_t kW2SlotBytes = kDraftSliceRows * kTileN * 2;  // 32 KB
constexpr uint32_t kUBoxBytes = kRows * 32 * 4;              // 16 KB (32 tokens x 128 rows)
constexpr uint32_t kUStageBytes = 2 * kUBoxBytes;            // 32 KB
// merge records: (2 column groups x batch copies) slots x 5 fields x rows per copy
constexpr uint32_t kMergeBytes = 2 * 5 * kRows * 4;          // 5 KB
constexpr uint32_t kOffW2 = 0;
constexpr uint32_t kOffU = kOffW2 + kNumW2Slots * kW2SlotBytes;
// each epilogue thread's best block of the position so far: 16 floats, stored as four
// float4 planes [4][threads] so that a warp's stores are contiguous
constexpr uint32_t kBestBytes = kEpiThreads * 16 * 4;        // 16 KB
constexpr uint32_t kOffMerge = kOffU + kNumUStages * kUStageBytes;
constexpr uint32_t kOffBest = kOffMerge + kMergeBytes;
constexpr uint32_t kOffBar = kOffBest + kBestBytes;
constexpr uint32_t kBarRegion = 2048;
// the noise ring: two tiles of one float4 (log2 E of its four blocks) per epilogue thread
constexpr uint32_t kOffNoise = kOffBar + kBarRegion;
constexpr uint32_t kNoiseBytes = 2 * kEpiThreads * 16;       // 8 KB
constexpr uint32_t kSmemBytes = kOffNoise + kNoiseBytes + 1024;  // + alignment slack
// TMEM: kNumAcc accumulators of 128 columns, then the MMA's A operand ([128 x r] bf16,
// two elements per column: r / 2 <= 128 columns)
constexpr uint32_t kTmemA = kNumAcc * kTileN;                // 384
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kEpiBarrier = 1;                          // named barrier id
constexpr uint32_t kBackoffControlNs = 200;  // sleep between polls of the TMA / MMA lanes
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.69314718055994531f;
constexpr uint32_t kTokenBits = 18;                          // V <= 2^18
constexpr uint32_t kTokenMask = (1u << kTokenBits) - 1u;

static_assert(kSmemBytes <= 232448, "draft kernel shared memory above the sm_103 limit");
static_assert(kTmemA + kMaxRank / 2 <= kTmemCols, "TMEM columns");
static_assert(kNumUStagesSmall * kUStageBytes / 2 <= kNumUStages * kUStageBytes, "U ring");
static_assert(kTileN == 2 * kSubV, "a tile is two sub-tiles");
static_assert((2 * kNumW2SlotsMax + 2 * kNumUStagesSmall + 2 * kNumAcc + 6) * 8 + 2 * kMaxK * 4 +
                      kRows * 8 + 8 + 4 * 8 <=
                  kBarRegion,
              "barrier region too small");

// On-chip offset checks of the debug library (compiled away in the release library): a
// failed check records DSPARK_ERR_DEVICE_OOB and yields the region's first offset, so the
// access stays in bounds and the launch ends with its status set.
__device__ __forceinline__ uint32_t tmem_checked(uint32_t addr, uint32_t tmem_base, uint32_t width,
                                                 uint32_t col_lo, uint32_t col_hi, uint32_t lane0,
                                                 int* status) {
  if constexpr (kDeviceChecks) {
    const uint32_t rel = addr - tmem_base;
    if (!tmem_span_ok(rel, width, col_lo, col_hi, lane0)) {
      record_error(status, kStatusDeviceOob);
      return tmem_base + tmem_or_first(rel, width, col_lo, col_hi, lane0);
    }
  }
  return addr;
}

__device__ __forceinline__ uint32_t smem_checked(uint32_t off, uint32_t len, uint32_t limit,
                                                 int* status) {
  if constexpr (kDeviceChecks) {
    if (!span_ok(off, len, limit)) {
      record_error(status, kStatusDeviceOob);
      return span_or_first(off, len, limit);
    }
  }
  return off;
}

// (the same for an access that is skipped, not redirected, when its check fails)
__device__ __forceinline__ bool smem_range_ok(uint32_t off, uint32_t len, uint32_t limit,
                                              int* status) {
  if constexpr (kDeviceChecks) {
    if (!span_ok(off, len, limit)) {
      record_error(status, kStatusDeviceOob);
      return false;
    }
  }
  return true;
}

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

// Small batches: with B <= 64 requests the 128 MMA rows hold two copies of the batch,
// row m serving request m mod 64, so that every TMEM lane quadrant holds real rows.
__device__ __forceinline__ int rows_per_copy(int B) { return B <= 64 ? 64 : kRows; }

// bf16 pair arithmetic on packed 32-bit words (two bf16 each, element 2j in the low half).
__device__ __forceinline__ uint32_t bf16x2_mul(uint32_t a, uint32_t b) {
  const __nv_bfloat162 r = __hmul2(*reinterpret_cast<const __nv_bfloat162*>(&a),
                                   *reinterpret_cast<const __nv_bfloat162*>(&b));
  return *reinterpret_cast<const uint32_t*>(&r);
}

// a * s + g * w per element, in fp32, rounded to bf16 (the RNN head's state update).
__device__ __forceinline__ uint32_t bf16x2_state(uint32_t a, uint32_t s, uint32_t g, uint32_t w) {
  return pack_bf16(fmaf(bf16_lo(a), bf16_lo(s), bf16_lo(g) * bf16_lo(w)),
                   fmaf(bf16_hi(a), bf16_hi(s), bf16_hi(g) * bf16_hi(w)));
}

// The bf16 gate row piece of chunk cc (elements [64 cc, 64 cc + 64)) of request req at
// position k: eight 16-byte pieces (zeros past r or for a dead row).
__device__ __forceinline__ void load_gate_chunk(const DraftParams& p, int k, int req, bool live,
                                                int cc, uint4 (&gv)[8]) {
  const uint16_t* hrow = p.H + (static_cast<size_t>(req) * p.K + k) * p.r;
#pragma unroll
  for (int u = 0; u < 8; ++u) {
    const int kel = cc * 64 + u * 8;
    gv[u] = (live && kel < p.r) ? __ldg(reinterpret_cast<const uint4*>(hrow + kel))
                                : make_uint4(0u, 0u, 0u, 0u);
  }
}

// One K chunk (elements [64 cc, 64 cc + 64)) of the Markov embedding of token `tok` --
// gated (gv given): times the chunk's bf16 gate, rounded to bf16 -- packed the way the
// MMA reads its A operand from TMEM: elements 2j and 2j + 1 of the chunk in column j.  A
// dead row (no request) and elements past r are zero.
__device__ __forceinline__ void load_embedding(const DraftParams& p, bool live, int cc,
                                               int32_t tok, bool gated, const uint4 (&gv)[8],
                                               uint32_t (&wv)[32]) {
  uint4 vals[8];
#pragma unroll
  for (int u = 0; u < 8; ++u) {
    const int kel = cc * 64 + u * 8;
    if (live && kel < p.r) {
      vals[u] = __ldg(reinterpret_cast<const uint4*>(p.W1 + static_cast<size_t>(tok) * p.r + kel));
    } else {
      vals[u] = make_uint4(0u, 0u, 0u, 0u);
    }
  }
  if (gated) {
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      vals[u].x = bf16x2_mul(vals[u].x, gv[u].x);
      vals[u].y = bf16x2_mul(vals[u].y, gv[u].y);
      vals[u].z = bf16x2_mul(vals[u].z, gv[u].z);
      vals[u].w = bf16x2_mul(vals[u].w, gv[u].w);
    }
  }
#pragma unroll
  for (int u = 0; u < 8; ++u) {
    wv[4 * u + 0] = vals[u].x;
    wv[4 * u + 1] = vals[u].y;
    wv[4 * u + 2] = vals[u].z;
    wv[4 * u + 3] = vals[u].w;
  }
}

// The gated operand in two steps, so that the gate rows -- known before the winner is --
// load while the winner's key is read: the chunk's gate, packed like load_embedding's output,
// then (gate_times_embedding) its product with the chunk of W1[tok], rounded to bf16.
__device__ __forceinline__ void load_gate_packed(const DraftParams& p, int k, int req, bool live,
                                                 int cc, uint32_t (&wv)[32]) {
  uint4 gv[8];
  load_gate_chunk(p, k, req, live, cc, gv);
#pragma unroll
  for (int u = 0; u < 8; ++u) {
    wv[4 * u + 0] = gv[u].x;
    wv[4 * u + 1] = gv[u].y;
    wv[4 * u + 2] = gv[u].z;
    wv[4 * u + 3] = gv[u].w;
  }
}

__device__ __forceinline__ void gate_times_embedding(const DraftParams& p, bool live, int cc,
                                                     int32_t tok, uint32_t (&wv)[32]) {
#pragma unroll
  for (int u = 0; u < 8; ++u) {
    const int kel = cc * 64 + u * 8;
    if (live && kel < p.r) {
      const uint4 v =
          __ldg(reinterpret_cast<const uint4*>(p.W1 + static_cast<size_t>(tok) * p.r + kel));
      wv[4 * u + 0] = bf16x2_mul(v.x, wv[4 * u + 0]);
      wv[4 * u + 1] = bf16x2_mul(v.y, wv[4 * u + 1]);
      wv[4 * u + 2] = bf16x2_mul(v.z, wv[4 * u + 2]);
      wv[4 * u + 3] = bf16x2_mul(v.w, wv[4 * u + 3]);
    } else {
      wv[4 * u + 0] = wv[4 * u + 1] = wv[4 * u + 2] = wv[4 * u + 3] = 0u;
    }
  }
}

// One K chunk of the RNN head's next state, s_k = a_k (.) s_{k-1} + g_k (.) W1[tok]
// (a_k = A[req, k], g_k = H[req, k] or 1, both bf16), rounded to bf16 and packed like
// load_embedding's output.  sp holds the same chunk of s_{k-1} as the previous position's
// operand (bf16 pairs, read back from TMEM; zeros before position 0): the state is carried
// as the bf16 MMA operand.  A dead row and elements past r are zero.
__device__ __forceinline__ void load_rnn_state(const DraftParams& p, int k, int req, bool live,
                                               int cc, int32_t tok, const uint32_t (&sp)[32],
                                               uint32_t (&wv)[32]) {
  const size_t row = (static_cast<size_t>(req) * p.K + k) * p.r;
#pragma unroll
  for (int half = 0; half < 2; ++half) {  // four 16-byte pieces of each input at a time
    uint4 w[4], a[4], g[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int kel = cc * 64 + (4 * half + q) * 8;
      const bool in = live && kel < p.r;
      const uint4 z = make_uint4(0u, 0u, 0u, 0u);
      const uint4 one = make_uint4(0x3F803F80u, 0x3F803F80u, 0x3F803F80u, 0x3F803F80u);
      w[q] = in ? __ldg(reinterpret_cast<const uint4*>(p.W1 + static_cast<size_t>(tok) * p.r + kel))
                : z;
      a[q] = in ? __ldg(reinterpret_cast<const uint4*>(p.A + row + kel)) : z;
      g[q] = (in && p.H != nullptr) ? __ldg(reinterpret_cast<const uint4*>(p.H + row + kel)) : one;
    }
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int u = 4 * half + q;
      wv[4 * u + 0] = bf16x2_state(a[q].x, sp[4 * u + 0], g[q].x, w[q].x);
      wv[4 * u + 1] = bf16x2_state(a[q].y, sp[4 * u + 1], g[q].y, w[q].y);
      wv[4 * u + 2] = bf16x2_state(a[q].z, sp[4 * u + 2], g[q].z, w[q].z);
      wv[4 * u + 3] = bf16x2_state(a[q].w, sp[4 * u + 3], g[q].w, w[q].w);
    }
  }
}

// The RNN head's drafted update in two steps around the grid barrier.  Before it, for one K
// chunk: t = a_{k} (.) s_{k-1} (exact in fp32: both factors are bf16) into 64 TMEM columns at
// taddr (element e in column e), and the input gate g_k (1 without one) packed into gw.  After
// it (rnn_finish_chunk): s_k = bf16(t + g_k (.) W1[tok]), the value load_rnn_state makes.
__device__ __forceinline__ void rnn_decay_chunk(const DraftParams& p, int k, int req, bool live,
                                                int cc, const uint32_t (&sp)[32], uint32_t taddr,
                                                uint32_t (&gw)[32]) {
  const size_t row = (static_cast<size_t>(req) * p.K + k) * p.r;
#pragma unroll
  for (int piece = 0; piece < 2; ++piece) {
    uint32_t t[32];
#pragma unroll
    for (int qq = 0; qq < 4; ++qq) {
      const int kel = cc * 64 + (4 * piece + qq) * 8;
      const bool in = live && kel < p.r;
      const uint4 z = make_uint4(0u, 0u, 0u, 0u);
      const uint4 one = make_uint4(0x3F803F80u, 0x3F803F80u, 0x3F803F80u, 0x3F803F80u);
      const uint4 a = in ? __ldg(reinterpret_cast<const uint4*>(p.A + row + kel)) : z;
      const uint4 g = in ? (p.H != nullptr ? __ldg(reinterpret_cast<const uint4*>(p.H + row + kel))
                                           : one)
                         : z;
      const int j0 = 16 * piece + 4 * qq;
      const uint32_t av[4] = {a.x, a.y, a.z, a.w}, gv[4] = {g.x, g.y, g.z, g.w};
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        t[8 * qq + 2 * c] = __float_as_uint(bf16_lo(av[c]) * bf16_lo(sp[j0 + c]));
        t[8 * qq + 2 * c + 1] = __float_as_uint(bf16_hi(av[c]) * bf16_hi(sp[j0 + c]));
        gw[j0 + c] = gv[c];
      }
    }
    tmem_st_x32(taddr + static_cast<uint32_t>(32 * piece), t);
  }
}

// (All lanes take part: the TMEM loads are warp-wide; `update` false leaves gw as it is.)
__device__ __forceinline__ void rnn_finish_chunk(const DraftParams& p, bool update, int cc,
                                                 int32_t tok, uint32_t taddr, uint32_t (&wv)[32]) {
#pragma unroll
  for (int piece = 0; piece < 2; ++piece) {
    uint32_t t[32];
    tmem_ld_x32(taddr + static_cast<uint32_t>(32 * piece), t);
    tmem_wait_ld();
    if (!update) continue;
#pragma unroll
    for (int qq = 0; qq < 4; ++qq) {
      const int kel = cc * 64 + (4 * piece + qq) * 8;
      const uint4 w =
          kel < p.r
              ? __ldg(reinterpret_cast<const uint4*>(p.W1 + static_cast<size_t>(tok) * p.r + kel))
              : make_uint4(0u, 0u, 0u, 0u);
      const uint32_t wvv[4] = {w.x, w.y, w.z, w.w};
      const int j0 = 16 * piece + 4 * qq;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const uint32_t g = wv[j0 + c];
        wv[j0 + c] = pack_bf16(
            fmaf(bf16_lo(g), bf16_lo(wvv[c]), __uint_as_float(t[8 * qq + 2 * c])),
            fmaf(bf16_hi(g), bf16_hi(wvv[c]), __uint_as_float(t[8 * qq + 2 * c + 1])));
      }
    }
  }
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

// Store four float4 to shared memory if `pred` (predicated, no branch).
__device__ __forceinline__ void st_shared_v4_if(bool pred, float4* dst, float4 v) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.u32 p, %0, 0;\n\t"
      "@p st.shared.v4.f32 [%1], {%2, %3, %4, %5};\n\t}" ::"r"(pred ? 1u : 0u),
      "r"(smem_addr(dst)), "f"(v.x), "f"(v.y), "f"(v.z), "f"(v.w)
      : "memory");
}

// Keep the better of this thread's best block so far and a new one: the block's score
// (the race's G, or the greedy maximum), its first token, its stage-2 uniform word and
// its 16 values (logits, or the weights themselves in the residual draw), which go to
// this thread's slot of the shared best-block store.  Ties keep the earlier block, which
// holds the smaller token ids.
__device__ __forceinline__ void keep_best(float score, int vbase, uint32_t word2, const float* v,
                                          float4* slot, int stride, float& best, int& best_v,
                                          uint32_t& best_w) {
  const bool better = score > best;
  best = better ? score : best;
  best_v = better ? vbase : best_v;
  best_w = better ? word2 : best_w;
#pragma unroll
  for (int c = 0; c < 4; ++c)
    st_shared_v4_if(better, slot + c * stride,
                    make_float4(v[4 * c], v[4 * c + 1], v[4 * c + 2], v[4 * c + 3]));
}

// Stage 2 of the race in the thread's best block, once per position: the first token whose
// cumulative weight exceeds u2 times the block's mass; w are the block's weights (any
// common scale).  Returns the index in the block.
__device__ __forceinline__ int race_stage2(const float (&w)[16], uint32_t word2) {
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
  return js < 0 ? jl : js;  // target at the very top (rounding): the last live token
}

// Largest of 16 values (three-input maxima).
__device__ __forceinline__ float max16(const float* x) {
  const float a0 = fmax3(x[0], x[1], x[2]), a1 = fmax3(x[3], x[4], x[5]);
  const float a2 = fmax3(x[6], x[7], x[8]), a3 = fmax3(x[9], x[10], x[11]);
  const float a4 = fmax3(x[12], x[13], x[14]);
  return fmaxf(fmax3(a0, a1, a2), fmax3(a3, a4, x[15]));
}

// Sum of 16 values as a pairwise tree of packed additions.
__device__ __forceinline__ float sum16(const float* w) {
  float2 s0 = __fadd2_rn(make_float2(w[0], w[1]), make_float2(w[2], w[3]));
  float2 s1 = __fadd2_rn(make_float2(w[4], w[5]), make_float2(w[6], w[7]));
  float2 s2 = __fadd2_rn(make_float2(w[8], w[9]), make_float2(w[10], w[11]));
  float2 s3 = __fadd2_rn(make_float2(w[12], w[13]), make_float2(w[14], w[15]));
  s0 = __fadd2_rn(__fadd2_rn(s0, s1), __fadd2_rn(s2, s3));
  return s0.x + s0.y;
}

// GATED: the launch may carry a gate (gated head) or decay and input gates (RNN head); the
// plain instantiations compile the operand path without them
template <int MODE, bool COPIES, bool GATED>
__global__ void __launch_bounds__(threads_of<MODE, COPIES>(), 1)
    draft_kernel(const __grid_constant__ DraftArgs args) {
  const DraftParams& p = args.p;
  // teacher-forced modes take the predecessors from the caller
  constexpr bool kTF = MODE == kModeTeacherForced || MODE == kModeLabel || MODE == kModeResidual;
  // ring slots of half sub-tiles holding U and the target rows
  constexpr bool kHalf = MODE == kModeLabel || MODE == kModeResidual;
  // modes that draw a token by the block race
  constexpr bool kRace = MODE == kModeSample || MODE == kModeResidual;
  // modes whose per-request winners are published as 64-bit keys
  constexpr bool kKeys = !kTF || MODE == kModeResidual;
  // modes that can run the RNN head (verification and labels take no decay gate)
  constexpr bool kRnnOk = !kHalf;
  // the race's stage-1 noise comes from the noise warps
  constexpr bool kNoise = noise_warps<MODE, COPIES>();
  // W2 ring slots: a fourth one in the U region's free tail with batch copies
  constexpr int kW2Slots = COPIES ? kNumW2SlotsMax : kNumW2Slots;
  static_assert(kNumUStagesSmall * kUStageBytes / 2 + kW2SlotBytes <= kNumUStages * kUStageBytes,
                "the fourth W2 slot lies in the U region");
  // byte offset of W2 slot `slot` from the (aligned) shared memory base
  auto w2_slot_off = [](int slot) -> uint32_t {
    return slot < kNumW2Slots ? kOffW2 + static_cast<uint32_t>(slot) * kW2SlotBytes
                              : kOffU + kNumUStagesSmall * kUStageBytes / 2;
  };
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* sW = smem + kOffW2;
  uint8_t* sU = smem + kOffU;
  float* merge = reinterpret_cast<float*>(smem + kOffMerge);
  float4* s_best = reinterpret_cast<float4*>(smem + kOffBest);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kOffBar);
  uint64_t* w_full = bars;                          // [kNumW2SlotsMax]
  uint64_t* w_empty = w_full + kNumW2SlotsMax;      // [kNumW2SlotsMax]
  uint64_t* u_full = w_empty + kNumW2SlotsMax;      // [kNumUStagesSmall]
  uint64_t* u_empty = u_full + kNumUStagesSmall;    // [kNumUStagesSmall]
  uint64_t* acc_full = u_empty + kNumUStagesSmall;  // [kNumAcc]
  uint64_t* acc_empty = acc_full + kNumAcc;         // [kNumAcc]
  uint64_t* a_full = acc_empty + kNumAcc;
  uint64_t* a_empty = a_full + 1;
  uint64_t* mma_drain = a_empty + 1;  // an aborting MMA lane waits here for its MMAs
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(mma_drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(mma_drain + 2);
  int32_t* s_tok = reinterpret_cast<int32_t*>(mma_drain + 3);  // [kMaxK]
  float* s_conf = reinterpret_cast<float*>(s_tok + kMaxK);  // [kMaxK]
  // best key (epoch | score | token) any thread of this CTA reached for each
  // request in the current step: a lower bound on the step's winner
  unsigned long long* s_bound = reinterpret_cast<unsigned long long*>(s_conf + kMaxK);  // [128]
  uint32_t* s_sink = reinterpret_cast<uint32_t*>(s_bound + kRows);  // scratch word (U releases)
  uint64_t* noise_full = reinterpret_cast<uint64_t*>(s_bound + kRows) + 1;  // [2]
  uint64_t* noise_empty = noise_full + 2;                                  // [2]
  float4* s_noise = reinterpret_cast<float4*>(smem + kOffNoise);  // [2][kEpiThreads]

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int cta = blockIdx.x, ncta = gridDim.x;
  const int t_begin = static_cast<int>(static_cast<int64_t>(cta) * p.n_tiles / ncta);
  const int t_end = static_cast<int>(static_cast<int64_t>(cta + 1) * p.n_tiles / ncta);
  const int nt = t_end - t_begin;
  // The tiles of a position in the order they are streamed: ascending at even positions,
  // descending at odd ones, so a position starts on the W2 tiles the previous one used last
  // (still in L2 when the streams evict W2 from it)
  auto tile_of = [&](int k, int t) { return t_begin + ((k & 1) ? nt - 1 - t : t); };
  const int nkk = p.r / 16;
  // W2 slices per tile and rows per slice
  const int sr = p.r < kDraftSliceRows ? p.r : kDraftSliceRows;
  const int ns = nkk > 0 ? (p.r + kDraftSliceRows - 1) / kDraftSliceRows : 0;
  // Small batches use 4 U slots of 16 KB (sub-tile j in slot j % 4, read by copy j % 2
  // only, so each slot keeps one group of readers); larger ones 3 slots of 32 KB.
  const int nus = COPIES ? kNumUStagesSmall : kNumUStages;
  const uint32_t ubox = COPIES ? kUBoxBytes / 2 : kUBoxBytes;  // one 32-token box

  if (threadIdx.x == 0) {
    for (int s = 0; s < kW2Slots; ++s) {
      mbar_init(&w_full[s], 1);
      mbar_init(&w_empty[s], 1);
    }
    // a sub-tile's U slot is read (and released) by the epilogue warps of one copy
    const uint32_t u_readers = COPIES ? static_cast<uint32_t>(kEpiWarps / 2) : kEpiWarps;
    static_assert(kEpiWarps % 2 == 0, "the copies split the epilogue warps");
    for (int s = 0; s < nus; ++s) {
      mbar_init(&u_full[s], MODE == kModeResidual ? kResProducers : 1);
      mbar_init(&u_empty[s], u_readers);
    }
    for (int s = 0; s < kNumAcc; ++s) {
      mbar_init(&acc_full[s], 1);
      mbar_init(&acc_empty[s], kEpiWarps);  // every epilogue warp reads every accumulator
    }
    if (kNoise) {
      for (int s = 0; s < 2; ++s) {
        mbar_init(&noise_full[s], kNoiseWarps);
        mbar_init(&noise_empty[s], kEpiWarps);
      }
    }
    mbar_init(a_full, kEpiWarps);  // every epilogue warp's operand rows are in TMEM
    mbar_init(a_empty, 1);
    mbar_init(mma_drain, 1);
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
  // launched as a programmatic dependent of the scan that writes its per-row inputs (label and
  // residual modes): the prologue above overlapped the scan's last CTAs; nothing the scan
  // writes is read before this point
  griddep_wait();

  if (kNoise && warp >= kCtlWarps + kEpiWarps) {
    // ------------------------------------------------------------ noise warps
    // Noise warp n draws for epilogue warps 4 n .. 4 n + 3 (those of column group g = n):
    // lane l for the epilogue threads 128 n + 32 j + l, j = 0..3, each the same Philox calls
    // (counter (tile, k, request, 1 + 2 g) and (.., 2 + 2 g)) the thread would make, reduced
    // to the four blocks' log2 E; the stage-2 word of a thread's best block is drawn again
    // by the thread after the sweep.
    const int n = warp - (kCtlWarps + kEpiWarps);
    const int rpc = COPIES ? rows_per_copy(p.B) : kRows;
    const uint32_t tag = 1u + 2u * static_cast<uint32_t>(n);
    uint32_t bg[4];
    bool rok[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int q = (4 * n + j + kCtlWarps) & 3;  // the epilogue warp's TMEM lane quadrant
      const int b = (q * 32 + lane) & (rpc - 1);
      rok[j] = b < p.B;
      bg[j] = static_cast<uint32_t>(p.b_global0 + b);
    }
    bool ok = true;
    for (int k = 0; k < p.K && ok; ++k) {
      for (int t = 0; t < nt; ++t) {
        const int i = k * nt + t, slot = i & 1;
        if (lane == 0)
          ok = mbar_wait(&noise_empty[slot], ((i >> 1) & 1) ^ 1, p.timeout_ns, abort_flag,
                         kBackoffControlNs);
        ok = __shfl_sync(0xFFFFFFFFu, ok, 0);
        if (!ok) break;
        const uint32_t tile = static_cast<uint32_t>(tile_of(k, t));
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          float4 e4 = make_float4(0.f, 0.f, 0.f, 0.f);
          if (rok[j]) {
            uint32_t za[4], zb[4];
            philox4x32_10_rk2(tile, static_cast<uint32_t>(k), bg[j], tag, tag + 1u, p.round_key0,
                              p.round_key1, za, zb);
            e4 = make_float4(lg2_approx(neg_log_uniform_fast(za[0])),
                             lg2_approx(neg_log_uniform_fast(zb[0])),
                             lg2_approx(neg_log_uniform_fast(za[2])),
                             lg2_approx(neg_log_uniform_fast(zb[2])));
          }
          s_noise[smem_checked(static_cast<uint32_t>(slot * kEpiThreads + 128 * n + 32 * j + lane),
                               1, 2 * kEpiThreads, p.status)] = e4;
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&noise_full[slot]);
      }
    }
    if (!ok && lane == 0) {
      *abort_flag = 1;
      record_error(p.status, kStatusTimeout);
    }
  } else if (MODE == kModeResidual && (warp == 0 || warp >= kCtlWarps + kEpiWarps)) {
    // --------------------------------------------------- U producers, residual mode
    // The draw rows are read in place: each request's base-logit row and target row at its
    // own draw position (tile::gather4 over 2-D row maps of U [B K, V] and P [B (K + 1), V],
    // four rows an op, into the slot layout of the 3-D boxes). A fill's 64 copies (32 per
    // tensor, copy i of a tensor taking rows 4 i .. 4 i + 3) are shared by three warps:
    // lane l of producer w issues copy o = 3 l + w; each warp arrives on the slot's full
    // barrier with the bytes of its own copies, and every warp takes every fill in order.
    const int w = warp == 0 ? 0 : warp - (kCtlWarps + kEpiWarps) + 1;
    const int o = kResProducers * lane + w;  // this lane's copy of every fill
    const bool target = o >= 32;
    const int rg = o & 31;                   // rows 4 rg .. 4 rg + 3
    const bool mine = o < 64 && 4 * rg < p.box_rows;
    const uint32_t w_bytes =
        static_cast<uint32_t>(__popc(__ballot_sync(0xFFFFFFFFu, mine))) * 512u;
    const uint64_t pol_u = l2_policy_evict_first();
    // the copy's four rows (past the batch: request 0 again, never read); a bonus row reads
    // no base logit: any valid row
    int y[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int b = 4 * rg + i < p.B ? 4 * rg + i : 0;
      const int gb = p.b_global0 + b, pos = mine ? p.rows[b].pos : 0;
      y[i] = target ? gb * (p.res_K + 1) + pos : gb * p.res_K + min(pos, p.res_K - 1);
    }
    bool ok = true;
    int issued = 0;
    for (int k = 0; k < p.K && ok; ++k) {
      for (int t = 0; t < nt && ok; ++t) {
        for (int f = 0; f < 4; ++f) {  // sub-tile f / 2, half f % 2
          const int j = 4 * (k * nt + t) + f, su = j % nus;
          if (lane == 0) {
            ok = mbar_wait(&u_empty[su], ((j / nus) & 1) ^ 1, p.timeout_ns, abort_flag,
                           kBackoffControlNs);
            if (ok) mbar_arrive_expect_tx(&u_full[su], w_bytes);
          }
          ok = __shfl_sync(0xFFFFFFFFu, ok, 0);
          if (!ok) break;
          const int x = tile_of(k, t) * kTileN + 32 * f;
          if (mine) {
            uint8_t* dst = sU + smem_checked(su * 2 * ubox + (target ? ubox : 0u) + rg * 512, 512,
                                             kNumUStages * kUStageBytes, p.status);
            tma_gather4_2d(dst, target ? &args.tm_p : &args.tm_u, x, y[0], y[1], y[2], y[3],
                           &u_full[su], pol_u);
          }
          issued = j + 1;
        }
      }
    }
    if (!ok && lane == 0) {
      *abort_flag = 1;
      record_error(p.status, kStatusTimeout);
      for (int j = issued - 1; j >= 0 && j >= issued - nus; --j)
        mbar_wait(&u_full[j % nus], (j / nus) & 1, p.timeout_ns, nullptr);
    }
  } else if (warp == 0) {
    // ------------------------------------------------------------ U producer
    if (lane == 0) {
      const uint64_t pol_u = l2_policy_evict_first();
      // a fill: 64 tokens of box_rows rows (row-pair boxes: one box of up to 64 rows, or two
      // of 64 rows, the rows past the batch filled with zeros), or U and target for 32 tokens
      const bool pair2 = p.u_rowpair && (kHalf || p.box_rows > 64);
      const uint32_t u_bytes = pair2 ? 2u * 64u * 256u : 2u * static_cast<uint32_t>(p.box_rows) * 128u;
      // fills per tile: two sub-tiles (U boxes of 32 tokens, two per fill), or four half
      // sub-tiles of U and target (label mode)
      constexpr int kFills = kHalf ? 4 : 2;
      bool ok = true;
      int issued = 0;
      for (int k = 0; k < p.K && ok; ++k) {
        for (int t = 0; t < nt && ok; ++t) {
          for (int f = 0; f < kFills; ++f) {
            const int j = kFills * (k * nt + t) + f, su = j % nus;
            if (!mbar_wait(&u_empty[su], ((j / nus) & 1) ^ 1, p.timeout_ns, abort_flag,
                           kBackoffControlNs)) {
              ok = false;
              break;
            }
            mbar_arrive_expect_tx(&u_full[su], u_bytes);
            uint8_t* dst = sU + smem_checked(su * 2 * ubox, 2 * ubox, kNumUStages * kUStageBytes,
                                             p.status);
            if (kHalf && p.u_rowpair) {  // U and target tokens [x, x + 64), rows [64 h, +64)
              const int c0 = (tile_of(k, t) * kTileN + kSubV * (f >> 1)) / 32, h = f & 1;
              tma_load_4d(dst, &args.tm_u, 0, c0, k, 64 * h, &u_full[su], pol_u);
              tma_load_4d(dst + ubox, &args.tm_p, 0, c0, k, 64 * h, &u_full[su], pol_u);
            } else if (kHalf) {  // U and target tokens [x, x + 32)
              const int x = tile_of(k, t) * kTileN + 32 * f;
              tma_load_3d(dst, &args.tm_u, x, k, 0, &u_full[su], pol_u);
              tma_load_3d(dst + ubox, &args.tm_p, x, k, 0, &u_full[su], pol_u);
            } else if (p.u_rowpair) {  // U tokens [x, x + 64): chunks x / 32, x / 32 + 1
              const int c0 = (tile_of(k, t) * kTileN + kSubV * f) / 32;
              tma_load_4d(dst, &args.tm_u, 0, c0, k, 0, &u_full[su], pol_u);
              if (pair2) tma_load_4d(dst + 16384, &args.tm_u, 0, c0, k, 64, &u_full[su], pol_u);
            } else {  // U tokens [x, x + 64)
              const int x = tile_of(k, t) * kTileN + kSubV * f;
              tma_load_3d(dst, &args.tm_u, x, k, 0, &u_full[su], pol_u);
              tma_load_3d(dst + ubox, &args.tm_u, x + 32, k, 0, &u_full[su], pol_u);
            }
            issued = j + 1;
          }
        }
      }
      if (!ok) {
        *abort_flag = 1;
        record_error(p.status, kStatusTimeout);
        for (int j = issued - 1; j >= 0 && j >= issued - nus; --j)
          mbar_wait(&u_full[j % nus], (j / nus) & 1, p.timeout_ns, nullptr);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------- MMA issuer and W2 producer (one lane)
    // W2 slices are loaded kW2Slots - 1 ahead of the MMAs: slice j + kW2Slots - 1 goes into the
    // slot of slice j - 1 as soon as slice j's MMAs are issued (they queue behind slice
    // j - 1's in the tensor pipe, so waiting for that slot never starves the pipe).
    if (lane == 0) {
      const uint32_t idesc = idesc_bf16_f32(kRows, kTileN, /*a_mn=*/false, /*b_mn=*/true);
      // B operand: a W2 slice as TMA wrote it, MN-major with 128-byte swizzle -- two
      // 64-token column blocks sr * 128 bytes apart, 8-row groups 1024 bytes apart
      const uint32_t lbo = static_cast<uint32_t>(sr) * 128u;
      const uint64_t pol_w = l2_policy_evict_last();
      const uint32_t w_bytes = 2u * kDraftBoxV * static_cast<uint32_t>(sr) * 2u;
      const int total = p.K * nt * ns;  // W2 slices of the launch
      int loaded = 0;                   // slices whose loads were issued
      bool ok = true;
      bool issued_any = false;
      // load slice j (the (j / ns) % nt-th tile its position streams, rows [128 (j % ns), ...))
      // into its slot
      auto load_slice = [&](int j) -> bool {
        const int slot = j % kW2Slots;
        if (!mbar_wait(&w_empty[slot], ((j / kW2Slots) & 1) ^ 1, p.timeout_ns, abort_flag,
                       kBackoffControlNs))
          return false;
        const int s = j % ns, t = (j / ns) % nt, kj = j / (ns * nt);
        const int v0 = tile_of(kj, t) * kTileN;
        uint8_t* dst = smem + smem_checked(w2_slot_off(slot), w_bytes, kSmemBytes - 1024, p.status);
        mbar_arrive_expect_tx(&w_full[slot], w_bytes);
        tma_load_2d(dst, &args.tm_w2, v0, s * kDraftSliceRows, &w_full[slot], pol_w);
        tma_load_2d(dst + sr * 128, &args.tm_w2, v0 + kDraftBoxV, s * kDraftSliceRows,
                    &w_full[slot], pol_w);
        return true;
      };
      while (ok && loaded < total && loaded < kW2Slots) ok = load_slice(loaded++);
      for (int k = 0; k < p.K && ok; ++k) {
        if (!mbar_wait(a_full, k & 1, p.timeout_ns, abort_flag, 32u)) {
          ok = false;
          break;
        }
        tc_fence_after();
        for (int t = 0; t < nt; ++t) {
          const int i = k * nt + t;
          const int buf = i % kNumAcc;
          if (!mbar_wait(&acc_empty[buf], ((i / kNumAcc) & 1) ^ 1, p.timeout_ns, abort_flag,
                         kBackoffControlNs)) {
            ok = false;
            break;
          }
          tc_fence_after();
          if (nkk == 0) {
            mbar_arrive(&acc_full[buf]);  // rank 0: the bias is zero, nothing to multiply
            continue;
          }
          const uint32_t d_tmem = tmem_checked(tmem_base + static_cast<uint32_t>(buf * kTileN),
                                               tmem_base, kTileN, 0, kTmemA, 0, p.status);
          for (int s = 0; s < ns && ok; ++s) {
            const int j = i * ns + s, slot = j % kW2Slots;
            if (!mbar_wait(&w_full[slot], (j / kW2Slots) & 1, p.timeout_ns, abort_flag,
                           kBackoffControlNs)) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint32_t b0 = smem_addr(smem + w2_slot_off(slot));
            const int kk_end = nkk < (s + 1) * kKSlice ? nkk : (s + 1) * kKSlice;
            for (int kk = s * kKSlice; kk < kk_end; ++kk) {
              const uint64_t bd = smem_desc(b0 + (kk - s * kKSlice) * 2048, lbo, 1024);
              const uint32_t a_tmem =
                  tmem_checked(tmem_base + kTmemA + static_cast<uint32_t>(kk * 8), tmem_base, 8,
                               kTmemA, kTmemCols, 0, p.status);
              umma_bf16_ts(d_tmem, a_tmem, bd, idesc, kk > 0 ? 1u : 0u);
            }
            issued_any = true;
            umma_commit(&w_empty[slot]);
            if (loaded < total && loaded <= j + kW2Slots - 1) ok = load_slice(loaded++);
          }
          if (!ok) break;
          umma_commit(&acc_full[buf]);
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
        // Drain: every copy and every MMA this lane issued must finish before the CTA
        // exits and TMEM is released (on the normal path the epilogue waited for all)
        for (int j = loaded - 1; j >= 0 && j >= loaded - kW2Slots; --j)
          mbar_wait(&w_full[j % kW2Slots], (j / kW2Slots) & 1, p.timeout_ns, nullptr);
        if (issued_any) {
          umma_commit(mma_drain);
          mbar_wait(mma_drain, 0, p.timeout_ns, nullptr);
        }
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue warps
    const int e = warp - kCtlWarps;  // 0 .. 7
    const int q = warp & 3;          // TMEM lane quadrant this warp may access
    const int g = e >> 2;            // 32-token half of a 64-token sub-tile
    const int rpc = COPIES ? rows_per_copy(p.B) : kRows;
    const int ncopy = COPIES ? kRows / rpc : 1;  // copies of the batch in the MMA rows
    const int b = (q * 32 + lane) & (rpc - 1);   // request of this thread's TMEM lane
    const int copy = (q * 32) / rpc;  // its copy: it reads sub-tile `copy` of every tile
    const int sub_lo = COPIES ? copy : 0;
    constexpr int nsub = COPIES ? 1 : 2;
    const int etid = threadIdx.x - kCtlWarps * 32;
    const bool row_ok = b < p.B;
    const uint32_t b_global = static_cast<uint32_t>(p.b_global0 + b);
    const float scale2 = p.inv_t * kLog2e;
    const uint32_t lane_base = tmem_base + (static_cast<uint32_t>(q * 32) << 16);
    // the 128-byte line of a ring slot that holds this thread's 32 U values (the half-tile
    // modes: row b of a 32-token box; 32-token boxes: row b of box g; row-pair boxes: chunk
    // g of row b mod 64 in box b / 64, whose 64-row boxes are 16 KB apart); the 128B
    // swizzle puts 16-byte unit u of line L at unit u ^ (L & 7)
    // (the label pass with row-pair boxes: a fill holds 64 tokens of U and of the target for
    // rows [64 h, 64 h + 64), U's 64-row box then the target's, 16 KB apart; a thread reads
    // fill h = b / 64, line 2 (b mod 64) + g)
    const uint32_t u_line =
        kHalf ? (p.u_rowpair ? static_cast<uint32_t>(2 * (b & 63) + g) : static_cast<uint32_t>(b))
              : (p.u_rowpair ? static_cast<uint32_t>((b >> 6) * 128 + 2 * (b & 63) + g)
                             : static_cast<uint32_t>(g) * (ubox / 128u) + static_cast<uint32_t>(b));
    const int u_fill = (kHalf && p.u_rowpair) ? (b >> 6) : g;  // the half-tile fill it reads
    const uint32_t row_off = u_line * 128u;
    const uint32_t swz = u_line & 7u;
    bool fail = false;
    bool aborted = false;

    // this thread's piece of the MMA operand: K chunks 2g and 2g + 1 of its row
    uint32_t wv0[32], wv1[32];
    unsigned long long spec_key = 0ull;  // winner key this thread's row was gathered for
    auto store_operand = [&]() {
      const uint32_t op = tmem_checked(lane_base + kTmemA + static_cast<uint32_t>(g * 64),
                                       tmem_base, 64, kTmemA, kTmemCols, q * 32, p.status);
      tmem_st_x32(op, wv0);
      tmem_st_x32(op + 32u, wv1);
    };
    // gated head (not the RNN head): the gate row pieces of the operand's next position are
    // pulled into L1 ahead of the winner's key, so that their loads in gather_operand hit
    const bool gated_op = GATED && p.H != nullptr && (!kRnnOk || p.A == nullptr);
    const bool rnn_op = GATED && kRnnOk && p.A != nullptr;
    auto prefetch_gates = [&](int kpos, bool live) {
      if (!gated_op || !live) return;
      const uint16_t* hrow = p.H + (static_cast<size_t>(b) * p.K + kpos) * p.r + 128 * g;
      if (128 * g < p.r) asm volatile("prefetch.global.L1 [%0];" ::"l"(hrow));
      if (128 * g + 64 < p.r) asm volatile("prefetch.global.L1 [%0];" ::"l"(hrow + 64));
    };
    // the operand of position kpos: the Markov embedding of tok (gated: times the gate), or
    // the RNN head's next state; `update` false leaves this lane's registers as they are
    // (the RNN state's read-back from TMEM is a warp-wide load, so every lane takes part)
    auto gather_operand = [&](int kpos, bool live, int32_t tok, bool update = true) {
      if (!rnn_op) {
        if (!update) return;
        uint4 gv[8];
        load_gate_chunk(p, kpos, b, live && gated_op, 2 * g, gv);
        load_embedding(p, live, 2 * g, tok, gated_op, gv, wv0);
        load_gate_chunk(p, kpos, b, live && gated_op, 2 * g + 1, gv);
        load_embedding(p, live, 2 * g + 1, tok, gated_op, gv, wv1);
        return;
      }
      uint32_t sp[32];
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        if (kpos == 0) {
#pragma unroll
          for (int j = 0; j < 32; ++j) sp[j] = 0u;  // s_{-1} = 0
        } else {
          tmem_ld_x32(tmem_checked(lane_base + kTmemA + static_cast<uint32_t>(g * 64 + 32 * half),
                                   tmem_base, 32, kTmemA, kTmemCols, q * 32, p.status),
                      sp);
          tmem_wait_ld();
        }
        if (update) load_rnn_state(p, kpos, b, live, 2 * g + half, tok, sp, half ? wv1 : wv0);
      }
    };
    for (int k = 0; k < p.K; ++k) {
      // ---- the step's operand: position 0 is gathered here; later positions were written
      // speculatively before the previous grid barrier and are re-checked now
      if (etid == 0) trace_stamp(p, cta, k, 0);
      if (!fail) {
        if (k == 0) {
          int32_t tok = 0;
          if (row_ok) {
            tok = kTF ? __ldg(p.prev + static_cast<size_t>(b) * p.K) : __ldg(p.anchors + b);
            if (tok < 0 || tok >= p.V) {
              record_error(p.status, kStatusDeviceOob);
              tok = 0;
            }
          }
          gather_operand(0, row_ok, tok);
        } else if (!kTF) {
          bool changed = false;
          int32_t tok = 0;
          if (row_ok) {
            const unsigned long long key = __ldcg(p.keys + (k - 1) * kRows + b);
            if (key != spec_key) {  // the winner changed after the speculative gather
              changed = true;
              tok = key_token(key);
              if (key_epoch(key) != p.epoch || tok < 0 || tok >= p.V) {
                record_error(p.status, kStatusDeviceOob);
                tok = 0;
              }
            }
          }
          if (rnn_op && !kTF) {
            // the RNN head's state: the decayed part made before the barrier, plus the input
            // (every live row: its state is never speculated)
            tc_fence_after();
#pragma unroll
            for (int half = 0; half < 2; ++half)
              rnn_finish_chunk(p, changed, 2 * g + half, tok,
                               tmem_checked(lane_base + static_cast<uint32_t>(g * 128 + 64 * half),
                                            tmem_base, 64, 0, kTmemA, q * 32, p.status),
                               half ? wv1 : wv0);
          } else if (__any_sync(0xFFFFFFFFu, changed)) {
            tc_fence_after();
            gather_operand(k, true, tok, changed);
          }
        }
        // (teacher-forced modes wrote the operand of positions k > 0 during the previous
        // position's last tile)
        if (!kTF || k == 0) store_operand();
      }
      tmem_wait_st();
      tc_fence_before();
      if (etid < kRows) s_bound[etid] = 0ull;
      named_bar_sync(kEpiBarrier, kEpiThreads);
      if (lane == 0 && (!kTF || k == 0)) mbar_arrive(a_full);
      if (etid == 0) trace_stamp(p, cta, k, 1);

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
      // this thread's best block of the position so far (score, first token, stage-2 word);
      // its values are in the shared best-block store
      float best = -INFINITY;
      int best_v = 0;
      uint32_t best_w = 0u;
      // (four float4 planes of kEpiThreads entries: the entry in plane 0 decides)
      float4* my_best = s_best + smem_checked(static_cast<uint32_t>(etid) * 16u, 16,
                                              kEpiThreads * 16u, p.status) / 16u;
      // Philox words of this thread's two blocks (2g, 2g + 1 within a sub-tile) of a tile:
      // words 0, 1 serve sub-tile 0, words 2, 3 sub-tile 1; lE = log2(E) of the four blocks
      uint32_t nza[4] = {0u, 0u, 0u, 0u}, nzb[4] = {0u, 0u, 0u, 0u};
      float lE[4] = {0.f, 0.f, 0.f, 0.f};
      bool first = true;
      for (int t = 0; t < nt && !fail; ++t) {
        const int i = k * nt + t;
        const int buf = i % kNumAcc;
        const int tile = tile_of(k, t);
        if (kNoise) {
          // the stage-1 exponentials of this thread's blocks, drawn by the noise warps
          const int slot = i & 1;
          bool okn = mbar_wait(&noise_full[slot], static_cast<uint32_t>(i >> 1) & 1u,
                               p.timeout_ns, abort_flag);
          okn = __all_sync(0xFFFFFFFFu, okn);
          if (!okn) {
            fail = true;
            *abort_flag = 1;
            break;
          }
          const float4 e4 = s_noise[smem_checked(static_cast<uint32_t>(slot * kEpiThreads + etid),
                                                 1, 2 * kEpiThreads, p.status)];
          lE[0] = e4.x;
          lE[1] = e4.y;
          lE[2] = e4.z;
          lE[3] = e4.w;
          arrive_after_reads(&noise_empty[slot], __float_as_uint(e4.x) ^ __float_as_uint(e4.w),
                             s_sink, lane);
        } else if (kRace && row_ok) {
          const uint32_t c1 = static_cast<uint32_t>(MODE == kModeResidual ? res_pos : k);
          const uint32_t tag = (MODE == kModeResidual ? 9u : 1u) + 2u * static_cast<uint32_t>(g);
          philox4x32_10_rk2(static_cast<uint32_t>(tile), c1, b_global, tag, tag + 1u,
                            p.round_key0, p.round_key1, nza, nzb);
          // stage 1's exponentials E = -ln u1 of the thread's blocks, as log2 E (the noise
          // needs no accumulator: it is drawn while the tile's MMAs may still be running)
#pragma unroll
          for (int s = 0; s < 2; ++s) {
            lE[2 * s] = lg2_approx(neg_log_uniform_fast(nza[2 * s]));
            lE[2 * s + 1] = lg2_approx(neg_log_uniform_fast(nzb[2 * s]));
          }
        }
        if (kTF && t == nt - 1 && k + 1 < p.K) {
          // teacher-forced: the predecessors are known, so the next position's operand goes to
          // TMEM as soon as this position's MMAs are done with it (their last tile's), and the
          // MMAs of the next position start while this one's last tile, merge and partial run
          bool oka = mbar_wait(a_empty, k & 1, p.timeout_ns, abort_flag);
          oka = __all_sync(0xFFFFFFFFu, oka);
          if (!oka) {
            fail = true;
            *abort_flag = 1;
            break;
          }
          tc_fence_after();
          int32_t tok = 0;
          if (row_ok) {
            tok = __ldg(p.prev + static_cast<size_t>(b) * p.K + k + 1);
            if (tok < 0 || tok >= p.V) {
              record_error(p.status, kStatusDeviceOob);
              tok = 0;
            }
          }
          gather_operand(k + 1, row_ok, tok);
          store_operand();
          tmem_wait_st();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(a_full);
        }
        bool ok = mbar_wait(&acc_full[buf], (i / kNumAcc) & 1, p.timeout_ns, abort_flag);
        ok = __all_sync(0xFFFFFFFFu, ok);
        if (!ok) {
          fail = true;
          *abort_flag = 1;
          break;
        }
        tc_fence_after();
        if (first && etid == 0) trace_stamp(p, cta, k, 2);
        first = false;
#pragma unroll
        for (int s = 0; s < nsub; ++s) {
          if (fail) break;
          const int sub = sub_lo + s;
          const int jsub = 2 * i + sub;                   // sub-tile index in ring order
          const int vbase = tile * kTileN + sub * kSubV + 32 * g;  // this thread's first token
          // this sub-tile's 32 accumulator columns (the half-tile modes read them in two
          // 16-column pieces after the ring slots); after the last sub-tile of the tile the
          // buffer goes back
          const uint32_t acc_col = tmem_checked(
              lane_base + static_cast<uint32_t>(buf * kTileN + sub * kSubV + 32 * g), tmem_base,
              32, 0, kTmemA, q * 32, p.status);
          uint32_t acc[32];
          if (!kHalf) {
            if (nkk == 0) {
#pragma unroll
              for (int j = 0; j < 32; ++j) acc[j] = 0u;
            } else {
              tmem_ld_x32(acc_col, acc);
              tmem_wait_ld();
            }
            if (s == nsub - 1) {
              tc_fence_before();
              __syncwarp();
              if (lane == 0) mbar_arrive(&acc_empty[buf]);  // wait::ld returned the values
            }
          }
          float uval[32], pt[32];
          if (kHalf) {
            // half sub-tiles: fill 2 jsub + h holds U and the target for tokens
            // [32 h, 32 h + 32) of every row (row-pair boxes: 64 tokens of rows
            // [64 h, 64 h + 64)); this thread reads fill u_fill, every warp takes and releases
            // both, so each slot keeps one group of readers taking its fills in order
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              const int j = 2 * jsub + h, sh = j % nus;
              bool okh = mbar_wait(&u_full[sh], static_cast<uint32_t>(j / nus) & 1u,
                                   p.timeout_ns, abort_flag);
              okh = __all_sync(0xFFFFFFFFu, okh);
              if (!okh) {
                fail = true;
                *abort_flag = 1;
                break;
              }
              uint32_t dep = 0u;
              if (h == u_fill) {
                const uint8_t* row = sU + smem_checked(sh * 2 * ubox + row_off, ubox + 128,
                                                       kNumUStages * kUStageBytes, p.status);
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                  const uint32_t off = static_cast<uint32_t>(u ^ swz) << 4;
                  const float4 x = *reinterpret_cast<const float4*>(row + off);
                  const float4 z = *reinterpret_cast<const float4*>(row + ubox + off);
                  uval[4 * u + 0] = x.x;
                  uval[4 * u + 1] = x.y;
                  uval[4 * u + 2] = x.z;
                  uval[4 * u + 3] = x.w;
                  pt[4 * u + 0] = z.x;
                  pt[4 * u + 1] = z.y;
                  pt[4 * u + 2] = z.z;
                  pt[4 * u + 3] = z.w;
                  if (u == 0 || u == 7) dep ^= __float_as_uint(x.x) ^ __float_as_uint(z.w);
                }
              }
              arrive_after_reads(&u_empty[sh], dep, s_sink, lane);
            }
            if (fail) break;
          } else {
            const int su = jsub % nus;
            bool oku = mbar_wait(&u_full[su], static_cast<uint32_t>(jsub / nus) & 1u,
                                 p.timeout_ns, abort_flag);
            oku = __all_sync(0xFFFFFFFFu, oku);
            if (!oku) {
              fail = true;
              *abort_flag = 1;
              break;
            }
            const uint8_t* row = sU + smem_checked(su * 2 * ubox + row_off, 128,
                                                   kNumUStages * kUStageBytes, p.status);
            uint32_t dep = 0u;
#pragma unroll
            for (int u = 0; u < 8; ++u) {
              const float4 x =
                  *reinterpret_cast<const float4*>(row + (static_cast<uint32_t>(u ^ swz) << 4));
              uval[4 * u + 0] = x.x;
              uval[4 * u + 1] = x.y;
              uval[4 * u + 2] = x.z;
              uval[4 * u + 3] = x.w;
              if (u == 0 || u == 7) dep ^= __float_as_uint(x.x) ^ __float_as_uint(x.w);
            }
            arrive_after_reads(&u_empty[su], dep, s_sink, lane);
          }
          const bool full_chunk = vbase + 32 <= p.V;  // warp-uniform
          if (kHalf) {
            // two 16-token pieces (the residual draw's two blocks); every lane reads the
            // accumulator (a warp-wide load), a lane with no request only wastes its work
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
              uint32_t a16[16];
              if (nkk == 0) {
#pragma unroll
                for (int j = 0; j < 16; ++j) a16[j] = 0u;
              } else {
                tmem_ld_x16(acc_col + static_cast<uint32_t>(16 * hh), a16);
                tmem_wait_ld();
              }
              if (hh == 1 && s == nsub - 1) {
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&acc_empty[buf]);
              }
              const int v0 = vbase + 16 * hh;
              if (MODE == kModeLabel) {
                // sum of min(q, p) over the 16 tokens (past V the target is masked)
                const float2 sq = make_float2(scale2, scale2), oq = make_float2(offq2, offq2);
                const float2 sp = make_float2(p.target_scale2, p.target_scale2);
                const float2 op = make_float2(offp2, offp2);
                float2 acc2 = make_float2(0.f, 0.f);
#pragma unroll
                for (int j = 0; j < 16; j += 2) {
                  const float2 lj = __fadd2_rn(
                      make_float2(uval[16 * hh + j], uval[16 * hh + j + 1]),
                      make_float2(__uint_as_float(a16[j]), __uint_as_float(a16[j + 1])));
                  const float2 aq = __ffma2_rn(lj, sq, oq);
                  float2 pv = make_float2(pt[16 * hh + j], pt[16 * hh + j + 1]);
                  if (!full_chunk) {
                    if (v0 + j >= p.V) pv.x = -INFINITY;
                    if (v0 + j + 1 >= p.V) pv.y = -INFINITY;
                  }
                  const float2 ap = __ffma2_rn(pv, sp, op);
                  acc2 = __fadd2_rn(acc2, make_float2(ex2_approx(fminf(aq.x, ap.x)),
                                                      ex2_approx(fminf(aq.y, ap.y))));
                }
                sum += acc2.x + acc2.y;
              } else {
                // the verification draw: weights max(0, p - q) (p alone for a bonus draw),
                // relative to 2^0; stage 1 G = log2(block mass) - log2(E)
                float w[16];
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                  const float lj = uval[16 * hh + j] + __uint_as_float(a16[j]);
                  const float pj = ex2_approx(fmaf(pt[16 * hh + j], p.target_scale2, offp2));
                  const float qj = ex2_approx(fmaf(lj, scale2, offq2));  // 0 if offq2 = -inf
                  float wj = fmaxf(0.f, pj - qj);
                  if (v0 + j >= p.V || v0 + j == res_excl) wj = 0.f;
                  w[j] = wj;
                }
                const float bs = sum16(w);
                const float G = bs > 0.f ? lg2_approx(bs) - lE[2 * sub + hh] : -INFINITY;
                const uint32_t w2 = hh ? (sub ? nzb[3] : nzb[1]) : (sub ? nza[3] : nza[1]);
                keep_best(G, v0, w2, w, my_best, kEpiThreads, best, best_v, best_w);
              }
            }
            continue;
          }
          if (!row_ok) continue;
          // sample, greedy, teacher-forced: calibrated logits l = U + bias
          float l[32];
#pragma unroll
          for (int j = 0; j < 32; j += 2) {
            const float2 lj = __fadd2_rn(make_float2(uval[j], uval[j + 1]),
                                         make_float2(__uint_as_float(acc[j]),
                                                     __uint_as_float(acc[j + 1])));
            l[j] = lj.x;
            l[j + 1] = lj.y;
          }
          if (MODE == kModeTeacherForced) {
            float* dst = p.logits + (static_cast<size_t>(b) * p.K + k) * p.V + vbase;
            if (full_chunk) {
#pragma unroll
              for (int c = 0; c < 8; ++c)
                reinterpret_cast<float4*>(dst)[c] =
                    make_float4(l[4 * c], l[4 * c + 1], l[4 * c + 2], l[4 * c + 3]);
            } else {
#pragma unroll
              for (int j = 0; j < 32; ++j)
                if (vbase + j < p.V) dst[j] = l[j];
            }
          }
          if (!full_chunk) {
#pragma unroll
            for (int j = 0; j < 32; ++j)
              if (vbase + j >= p.V) l[j] = -INFINITY;
          }
          const float mb0 = max16(l), mb1 = max16(l + 16);
          const float lmax = fmaxf(mb0, mb1);
          if (lmax == -INFINITY) continue;  // nothing here can be drawn
          const float ymax = lmax * scale2;
          if (ymax > m2) {
            sum *= ex2_approx(m2 - ymax);
            m2 = ymax;
          }
          // w = 2^(l scale2 - m2): the tokens' weights relative to the running maximum
          float w[32];
          {
            const float2 s2 = make_float2(scale2, scale2), nm = make_float2(-m2, -m2);
#pragma unroll
            for (int j = 0; j < 32; j += 2) {
              const float2 d = __ffma2_rn(make_float2(l[j], l[j + 1]), s2, nm);
              w[j] = ex2_approx(d.x);
              w[j + 1] = ex2_approx(d.y);
            }
          }
          const float bs0 = sum16(w), bs1 = sum16(w + 16);
          sum += bs0 + bs1;
          if (MODE == kModeSample) {
            // stage 1: G = m2 + log2(block mass) - log2(E); stage 2 runs once, after the sweep
            const float G0 = bs0 > 0.f ? m2 + lg2_approx(bs0) - lE[2 * sub] : -INFINITY;
            const float G1 = bs1 > 0.f ? m2 + lg2_approx(bs1) - lE[2 * sub + 1] : -INFINITY;
            // (with the noise warps the best block's stage-2 word is drawn again after the
            // sweep, from best_v)
            keep_best(G0, vbase, kNoise ? 0u : (sub ? nza[3] : nza[1]), l, my_best, kEpiThreads,
                      best, best_v, best_w);
            keep_best(G1, vbase + 16, kNoise ? 0u : (sub ? nzb[3] : nzb[1]), l + 16, my_best,
                      kEpiThreads, best, best_v, best_w);
          } else if (MODE == kModeGreedy) {
            keep_best(mb0 * scale2, vbase, 0u, l, my_best, kEpiThreads, best, best_v, best_w);
            keep_best(mb1 * scale2, vbase + 16, 0u, l + 16, my_best, kEpiThreads, best, best_v,
                      best_w);
          }
        }
      }

      // ---- the thread's winner of the position: stage 2 of the race in its best block
      // (the greedy maximum's first token), from the values kept in shared memory
      float yb = -INFINITY, lb = 0.f;  // best score (G, or y when greedy) and its logit
      int vb = 0x7FFFFFFF;
      if ((kRace || MODE == kModeGreedy) && !fail && row_ok && best > -INFINITY) {
        float v16[16];
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const float4 x = my_best[c * kEpiThreads];
          v16[4 * c] = x.x;
          v16[4 * c + 1] = x.y;
          v16[4 * c + 2] = x.z;
          v16[4 * c + 3] = x.w;
        }
        int js;
        if (MODE == kModeResidual) {
          js = race_stage2(v16, best_w);  // the weights themselves
        } else {
          const float vmax = max16(v16);
          if (MODE == kModeSample) {
            if (kNoise) {
              // the stage-2 word of the best block (token best_v = 128 tile + 64 sub + 32 g +
              // 16 h): word 3 (sub-tile 1) or 1 (sub-tile 0) of the call for block half h
              const uint32_t tag = 1u + 2u * static_cast<uint32_t>(g);
              uint32_t za[4], zb[4];
              philox4x32_10_rk2(static_cast<uint32_t>(best_v >> 7), static_cast<uint32_t>(k),
                                b_global, tag, tag + 1u, p.round_key0, p.round_key1, za, zb);
              const bool s1 = ((best_v >> 6) & 1) != 0, h1 = ((best_v >> 4) & 1) != 0;
              best_w = h1 ? (s1 ? zb[3] : zb[1]) : (s1 ? za[3] : za[1]);
            }
            float w16[16];
#pragma unroll
            for (int j = 0; j < 16; ++j) w16[j] = ex2_approx((v16[j] - vmax) * scale2);
            js = race_stage2(w16, best_w);
          } else {
            js = 15;
#pragma unroll
            for (int j = 15; j >= 0; --j)
              if (v16[j] == vmax) js = j;
          }
        }
        float lj = 0.f;
#pragma unroll
        for (int j = 0; j < 16; ++j)
          if (j == js) lj = v16[j];
        yb = best;
        vb = best_v + js;
        lb = lj;
      }

      // ---- merge the column groups (and copies) of each request, publish the CTA's
      // partial; record slot sl = copy * 2 + g, rpc rows per record field
      if (etid == 0) trace_stamp(p, cta, k, 3);
      // the global key of this thread's row, read now so that the merge hides the load
      const unsigned long long gk_pre =
          (kKeys && !kTF && row_ok) ? __ldcg(p.keys + k * kRows + b) : 0ull;
      const float score = yb;
      const int slot = copy * 2 + g;
      // the record's five fields, rpc floats apart, inside the merge region
      const bool rec_ok = smem_range_ok(static_cast<uint32_t>((slot * 5 * rpc + b) * 4),
                                        static_cast<uint32_t>((4 * rpc + 1) * 4), kMergeBytes,
                                        p.status);
      if (!fail && rec_ok) {
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
        for (int ss = 1; ss < 2 * ncopy; ++ss) {
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
          // a CTA whose best is already beaten by the global key read at the start of the
          // merge leaves the key alone (keys only grow), which keeps the atomics on the 128
          // key words of the position from serialising behind every CTA's update
          if (key > gk_pre) atomicMax(p.keys + k * kRows + b, key);
          s_bound[b] = key;  // the CTA's best: the speculative gather's fallback
          if (!kTF && key > gk_pre && k + 1 < p.K) {
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

      // ---- arrive at the grid barrier (the wait comes after the speculative operand)
      if (etid == 0 && !fail) {
        const bool skip = (p.debug_skip_cta == cta) && (k == 0);
        // the release add orders every epilogue thread's partial and key writes
        // (synchronised by the named barrier above) before the arrival
        if (!skip) red_release_gpu_add(p.bar, 1u);
      }

      if (etid == 0) trace_stamp(p, cta, k, 7);
      // ---- speculative operand for the next position: the likely winner is the better of
      // the global key (read after this CTA's arrival) and this CTA's best; its embedding
      // loads are in flight while the grid barrier completes, and it is written to TMEM
      // (after a re-check of the key) at the start of the next position
      // (The operand registers are written on every path, even past the last position or
      // after a failure, so that they are plainly dead during the tile sweep.)
      {
        // (teacher-forced modes prepared the next operand in the last tile: nothing here, and
        // a_empty's phase is not waited for twice)
        const bool next = k + 1 < p.K && !kTF;
        bool ok = next && !fail;
        if (ok) ok = mbar_wait(a_empty, k & 1, p.timeout_ns, abort_flag);  // MMAs done with E
        ok = __all_sync(0xFFFFFFFFu, ok);
        if (next && !fail && !ok) {
          fail = true;
          *abort_flag = 1;
        }
        if (ok) tc_fence_after();
        const int knext = next ? k + 1 : k;
        const bool live = ok && row_ok;
        // the gated head's sampled operand: its gate rows load before the key read
        const bool gate_first = gated_op && !kTF;
        const bool rnn_first = rnn_op && !kTF;
        if (gate_first) {
          load_gate_packed(p, knext, b, live, 2 * g, wv0);
          load_gate_packed(p, knext, b, live, 2 * g + 1, wv1);
        } else if (rnn_first) {
          // the decayed state into this row's accumulator columns [128 g, 128 g + 128): every
          // MMA of the position is done (a_empty) and every accumulator read
          if (ok) {
#pragma unroll
            for (int half = 0; half < 2; ++half) {
              uint32_t sp[32];
              tmem_ld_x32(tmem_checked(lane_base + kTmemA + static_cast<uint32_t>(g * 64 + 32 * half),
                                       tmem_base, 32, kTmemA, kTmemCols, q * 32, p.status),
                          sp);
              tmem_wait_ld();
              rnn_decay_chunk(p, knext, b, live, 2 * g + half, sp,
                              tmem_checked(lane_base + static_cast<uint32_t>(g * 128 + 64 * half),
                                           tmem_base, 64, 0, kTmemA, q * 32, p.status),
                              half ? wv1 : wv0);
            }
            tmem_wait_st();
          } else {
#pragma unroll
            for (int j = 0; j < 32; ++j) wv0[j] = wv1[j] = 0u;
          }
        } else {
          prefetch_gates(knext, live);
        }
        int32_t tok = 0;
        if (live) {
          if (rnn_op) {
            // the RNN head's next state is made after the barrier: speculating on it costs
            // the state's read-back and both gates, and misses more often than it hits
            spec_key = ~0ull;
          } else {
            const unsigned long long gk = __ldcg(p.keys + k * kRows + b);
            const unsigned long long lk = s_bound[b];
            spec_key = (key_epoch(gk) == p.epoch && gk > lk) ? gk : lk;
            tok = key_token(spec_key);
            if (key_epoch(spec_key) != p.epoch || tok < 0 || tok >= p.V) {
              spec_key = ~0ull;  // never matches: gathered again after the barrier
              tok = 0;
            }
          }
        }
        if (gate_first) {
          gate_times_embedding(p, live, 2 * g, tok, wv0);
          gate_times_embedding(p, live, 2 * g + 1, tok, wv1);
        } else if (!kTF && !rnn_op) {
          gather_operand(knext, live, tok);
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
    tmem_wait_st();  // no operand write may be in flight when TMEM is released
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
int draft_threads(int mode, bool copies) {
  return mode == kModeResidual               ? threads_of<kModeResidual, false>()
         : (mode == kModeSample && !copies) ? threads_of<kModeSample, false>()
                                             : kThreads;
}

cudaError_t launch_draft(const DraftArgs& args, int mode, int grid, cudaStream_t stream,
                         uint32_t extra_smem, bool dependent) {
  const void* fn = nullptr;
  const bool copies = args.p.B <= 64;  // small batches fill the MMA rows with copies
  const bool gated = args.p.H != nullptr || args.p.A != nullptr;
  // plain and gated builds (the teacher-forced parity mode takes its gates at run time)
#define DSPARK_DRAFT_FN(M, C, G) reinterpret_cast<const void*>(&draft_kernel<M, C, G>)
  switch (mode) {
    case kModeSample:
      fn = copies ? (gated ? DSPARK_DRAFT_FN(kModeSample, true, true)
                           : DSPARK_DRAFT_FN(kModeSample, true, false))
                  : (gated ? DSPARK_DRAFT_FN(kModeSample, false, true)
                           : DSPARK_DRAFT_FN(kModeSample, false, false));
      break;
    case kModeGreedy:
      fn = copies ? (gated ? DSPARK_DRAFT_FN(kModeGreedy, true, true)
                           : DSPARK_DRAFT_FN(kModeGreedy, true, false))
                  : (gated ? DSPARK_DRAFT_FN(kModeGreedy, false, true)
                           : DSPARK_DRAFT_FN(kModeGreedy, false, false));
      break;
    case kModeTeacherForced:
      fn = copies ? DSPARK_DRAFT_FN(kModeTeacherForced, true, true)
                  : DSPARK_DRAFT_FN(kModeTeacherForced, false, true);
      break;
    case kModeLabel:  // half-sub-tile ring slots: always the 128-row instantiation
      fn = gated ? DSPARK_DRAFT_FN(kModeLabel, false, true)
                 : DSPARK_DRAFT_FN(kModeLabel, false, false);
      break;
    case kModeResidual:
      fn = gated ? DSPARK_DRAFT_FN(kModeResidual, false, true)
                 : DSPARK_DRAFT_FN(kModeResidual, false, false);
      break;
    default: return cudaErrorInvalidValue;
  }
#undef DSPARK_DRAFT_FN
  cudaError_t err = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(kSmemBytes));
  if (err != cudaSuccess) return err;
  void* kargs[] = {const_cast<DraftArgs*>(&args)};
  if (dependent && extra_smem == 0) {
    cudaLaunchAttribute attrs[2];
    attrs[0].id = cudaLaunchAttributeCooperative;
    attrs[0].val.cooperative = 1;
    attrs[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attrs[1].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(draft_threads(mode, copies));
    cfg.dynamicSmemBytes = kSmemBytes;
    cfg.stream = stream;
    cfg.attrs = attrs;
    cfg.numAttrs = 2;
    err = cudaLaunchKernelExC(&cfg, fn, kargs);
    if (err == cudaSuccess) return err;
    (void)cudaGetLastError();  // refused: the plain cooperative launch below
  }
  err = cudaLaunchCooperativeKernel(fn, dim3(grid), dim3(draft_threads(mode, copies)), kargs,
                                    kSmemBytes + extra_smem, stream);
  // a refused launch leaves its (non-sticky) error as the thread's last error: clear it, so
  // that the caller's next CUDA error check does not see it again
  if (err != cudaSuccess) (void)cudaGetLastError();
  return err;
}

}  // namespace dspark
