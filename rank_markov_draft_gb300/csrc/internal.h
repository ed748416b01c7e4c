// internal.h -- host/device interface between the C ABI (api.cu) and the
// kernels.  Not part of the public boundary.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "dspark.h"

namespace dspark {

constexpr int kMaxK = 64;           // block positions per call
constexpr int kMaxRank = 256;       // Markov rank
constexpr int kBatchChunk = 128;    // requests per draft launch (MMA M)
constexpr int kDraftTileN = 128;    // vocabulary entries per draft MMA tile (MMA N)
constexpr int kDraftBoxV = 64;      // W2 TMA box width: one 128-byte swizzled row of bf16
constexpr int kDraftSliceRows = 128;  // W2 rows (the contraction dimension) per ring slot
// rows of one W2 box (and ring slot): the whole rank when it fits, else 128
inline int draft_slice_rows(int r) { return r < kDraftSliceRows ? r : kDraftSliceRows; }
constexpr int kMaxTopk = 32;
constexpr int kTopkPartUnits = 4096;  // per-piece top-k lists the context can hold
constexpr int kTraceSlots = 8;      // timestamps per (CTA, step) in the draft trace
constexpr uint64_t kDefaultTimeoutNs = 2000ull * 1000ull * 1000ull;  // 2 s per wait

// Per-(step, request, CTA) record of the draft kernel's cross-CTA reduction.
struct DraftPartial {
  unsigned long long key;  // (epoch, race score, token) packed, see draft.cu
  float m2;                // running max of l * log2(e) / T'
  float sum;               // sum of 2^(y - m2)
  float lbest;             // calibrated logit of this CTA's best token
  float pad;
};

// Per-request inputs of the draft kernel's residual mode (the verification draw).
struct ResRow {
  float offq2;  // log2 q(v) = l(v) * log2(e) / Td + offq2; -inf: no draft mass subtracted
  float offp2;  // log2 p(v) = P(v) * log2(e) / Tt + offp2
  int pos;      // draw position (noise counter)
  int excl;     // token whose weight is zero (a greedy draft's rejected token), or -1
};

struct DraftParams {
  const uint16_t* W1;       // [V, r]
  const int32_t* anchors;   // [B] (chunk)
  const int32_t* prev;      // teacher-forced predecessors [B, K] (chunk), or null
  const uint16_t* H;        // gated: [B, K, r] (chunk) bf16, or null (RNN head: input gate)
  const uint16_t* A;        // RNN head: decay gate [B, K, r] (chunk) bf16, or null
  int B, K, V, r;
  int b_global0;            // index of the chunk's first request in the call (noise key)
  int n_tiles;              // ceil(V / 128)
  int box_rows;             // rows of the U TMA box (multiple of 8, >= B)
  // U boxes of row pairs: the map views U as [B][K][V / 32][32] and a box holds 64 tokens
  // (two 32-token chunks) of up to 64 rows, each row's 256 bytes read contiguously (needs
  // V % 32 == 0); otherwise boxes of 32 tokens of every row
  int u_rowpair;
  float inv_t;              // 1 / T' (T' = T, or 1 when greedy)
  uint32_t seed_lo, seed_hi;
  uint32_t round_key0[10];  // Philox key schedule (seed_lo + i * Weyl0), host-computed
  uint32_t round_key1[10];  // (seed_hi + i * Weyl1)
  int32_t* tokens;          // [B, K] (chunk)
  float* logprobs;          // [B, K] (chunk)
  float* logits;            // teacher-forced: [B, K, V] (chunk)
  float* lse;               // teacher-forced: [B, K] (chunk)
  // fused confidence head (conf == null: off)
  const uint16_t* conf_h;   // [B, K, d] (chunk)
  const uint16_t* conf_w;   // [d (+ r)]
  float conf_bias;
  int conf_d;
  int conf_with_markov;
  float conf_threshold;
  const float* conf_tau;    // [K] STS temperatures, or null (all 1)
  float* conf;              // [B, K] (chunk)
  float* cumprod;           // [B, K] (chunk)
  int32_t* verify_len;      // [B] (chunk)
  // context scratch
  unsigned long long* keys; // [kMaxK][128]
  DraftPartial* partials;   // [kMaxK][128][grid]
  uint32_t* bar;            // grid-barrier counter
  int* status;              // device status word
  uint32_t bar_base;        // counter value at launch
  uint32_t epoch;           // key epoch of this launch (1 .. 16383)
  int debug_skip_cta;       // fault injection: CTA skipping its step-0 arrival (-1: none)
  unsigned long long* trace;  // optional phase timestamps [grid][K][kTraceSlots] (null: off)
  uint64_t timeout_ns;      // per-wait limit
  // acceptance-label mode (null otherwise)
  const float* target;      // [B, K+1, V] (chunk) target logits (read through tm_p)
  const float* lse_t;       // [B, K+1] (chunk) log sum_v exp(target / Tt)
  const float* offq2;       // [B, K] (chunk) log2 q(v) = l(v) * log2(e) / Td + offq2
  float* label;             // [B, K] (chunk) 1 - TV(q, p)
  float target_scale2;      // log2(e) / Tt
  // residual mode (verification draw, K = 1): per-row constants; the draw rows of the
  // caller's U [B, res_K, V] and P [B, res_K + 1, V] gathered in place through tm_u, tm_p
  const ResRow* rows;       // [B] (chunk), or null
  int res_K;
};

struct DraftArgs {
  CUtensorMap tm_w2;  // W2 [r, V] bf16, box {64, min(r, 128)}, 128B swizzle
  CUtensorMap tm_u;   // U chunk [B, K, V] fp32, box {32, 1, box_rows}, 128B swizzle (or
                      // row-pair boxes); residual mode: U as rows [B K, V], box {32, 1}
                      // (gathered by four)
  CUtensorMap tm_p;   // label mode: target chunk [B, K+1, V] fp32, box {32, 1, box_rows},
                      // 128B swizzle (or row-pair boxes); residual mode: P as rows
                      // [B (K + 1), V], box {32, 1}
  DraftParams p;
};

enum DraftMode {
  kModeSample = 0,
  kModeGreedy = 1,
  kModeTeacherForced = 2,
  kModeLabel = 3,
  kModeResidual = 4,  // one position: block race over max(0, p - q) (the verification draw)
};

int draft_smem_bytes();
int draft_threads(int mode, bool copies);
// extra_smem > 0 asks for that much more dynamic shared memory than the kernel allows, which
// the runtime refuses (the refused-launch test); the refusal's error is cleared before return
// dependent: launched as a programmatic dependent of the preceding kernel of the stream (which
// may then overlap the prologue; the kernel waits for it before reading any input), falling
// back to a plain cooperative launch where the runtime refuses the combination
cudaError_t launch_draft(const DraftArgs& args, int mode, int grid, cudaStream_t stream,
                         uint32_t extra_smem = 0, bool dependent = false);

// Gate GEMM: partial[split][m][n] = sum_{j in split} h[m, j] * Wg[j, n].
struct GateArgs {
  CUtensorMap tm_h;   // h [M, d] bf16, box {64, 128}
  CUtensorMap tm_wg;  // Wg [d, r] bf16, box {64, 64}
  float* partial;     // [splits][M][r]
  int M, d, r, splits, chunks_per_split;
  int* status;
  uint64_t timeout_ns;
};
cudaError_t launch_gate_gemm(const GateArgs& args, cudaStream_t stream);
cudaError_t launch_gate_finalize(const float* partial, int splits, int64_t n, float* H,
                                 uint16_t* Hb, cudaStream_t stream);

// Top-k of each row of U [rows][V] (V a multiple of 4).  part_i / part_v: scratch
// for up to part_units per-piece lists of kMaxTopk entries (null: whole rows
// only).  *launches receives the number of kernels launched.
cudaError_t launch_topk(const float* U, int rows, int V, int topk, int32_t* cand, float* cval,
                        int32_t* part_i, float* part_v, int part_units, int* status,
                        uint64_t timeout_ns, int* launches, cudaStream_t stream);
cudaError_t launch_pair_scores(const int32_t* cand, const float* cval, const uint16_t* A,
                               const uint16_t* Bt, const int32_t* anchors, const float* H,
                               int B, int K, int V, int r, int topk, float* S, int* status,
                               uint64_t timeout_ns, cudaStream_t stream);
cudaError_t launch_walk(const int32_t* cand, const float* S, const int32_t* anchors,
                        const uint16_t* A, int B, int K, int V, int r, int topk, float inv_t,
                        int sample, uint32_t seed_lo, uint32_t seed_hi, int32_t* tokens,
                        float* logprobs, const dspark_conf_args* conf, int* status,
                        cudaStream_t stream);
// ---- speculative verification (verify.cu)
struct VerifyArgs {
  const float* P;             // [B, K+1, V] target logits
  const float* U;             // [B, K, V] base logits of the draft
  const uint16_t* W1;         // [V, r]
  const uint16_t* W2;         // [r, V]
  const float* H;             // [B, K, r] gate (null: ungated)
  const int32_t* tokens;      // [B, K] drafted tokens
  const float* logq;          // [B, K] the draft's log-probabilities of them (draft T > 0)
  const int32_t* anchors;     // [B]
  const int32_t* ell;         // [B] verified positions (null: K)
  int B, K, V, r;
  float draft_temperature, target_temperature;
  uint32_t seed_lo, seed_hi;
  int32_t* n_acc;             // [B]
  int32_t* next_token;        // [B]
  float* accept_prob;         // [B, K] or null
  int* status;
  // context scratch
  float* lse_t;               // [B, K+1]
  int32_t* argmax_t;          // [B, K+1]
  // the draw (sampled target): the residual mode's per-row constants, predecessors and
  // gate rows at the draw position; rows null: no draw (a greedy target's token is its
  // argmax)
  uint16_t* H_sel;            // [B, r] bf16
  int32_t* prev_sel;          // [B]
  ResRow* rows;               // [B]
  // per-request scratch, zero between calls (the request's last CTA clears it)
  unsigned long long* fail_mask;  // [B] bit k: the test of position k failed
  int* count;                     // [B] CTAs of the request done
};
// One kernel: the target-row scan with the acceptance tests and the draw's per-row
// constants (the draft kernel's residual mode then reads the draw rows of U and P in place).
cudaError_t launch_verify(const VerifyArgs& v, cudaStream_t stream, int* launches);

// ---- acceptance label (label.cu)
// One warp per drafted position: its predecessor, the offset that turns the
// draft head's logits into log2 q (draft T > 0), and the label itself where one
// side is greedy (the other cases are summed by the draft kernel's label mode).
struct LabelPrepArgs {
  const float* P;             // [B, K+1, V]
  const float* U;             // [B, K, V]
  const uint16_t* W1;         // [V, r]
  const uint16_t* W2;         // [r, V]
  const float* H;             // [B, K, r] or null
  const int32_t* anchors;     // [B]
  const int32_t* tokens;      // [B, K]
  const float* logq;          // [B, K] (draft T > 0)
  float* lse_t;               // [B, K+1] out, rows k < K (target T > 0)
  int32_t* argmax_t;          // [B, K+1] out, rows k < K (target T = 0)
  int B, K, V, r;
  float inv_td, inv_tt;       // 0: greedy
  int32_t* prev;              // [B, K] out
  float* offq2;               // [B, K] out (draft T > 0)
  float* label;               // [B, K] out where one side is greedy
  int* status;
};
// One kernel: the scan of each drafted position's target row, then that row's
// preparation (predecessor, log2 q offset, the label where one side is greedy).
cudaError_t launch_label_prep(const LabelPrepArgs& a, cudaStream_t stream);

// ---- load-aware prefix scheduler (schedule.cu)
constexpr int kScheduleMaxCandidates = 16384;  // R * K
cudaError_t launch_schedule(const float* a, int R, int K, const float* sps, int32_t* ell,
                            float* theta, cudaStream_t stream);

cudaError_t launch_confidence(const uint16_t* h, const uint16_t* W1, const int32_t* anchors,
                              const int32_t* tokens, const uint16_t* w, float bias,
                              int with_markov, int B, int K, int d, int r, int V,
                              float threshold, const float* tau, float* conf, float* cumprod,
                              int32_t* verify_len, int* status, cudaStream_t stream);

// ---- sequential temperature scaling (calibrate.cu)
cudaError_t launch_sts_fit(const float* conf, const float* label, int N, int K, float tau_lo,
                           float tau_hi, float* tau, float* loss, cudaStream_t stream);

}  // namespace dspark
