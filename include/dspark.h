/*
 * dspark.h -- C ABI of the DSpark Markov-head drafting hot path on GB300
 * (sm_103a).  Every entry point takes plain pointers and sizes; no C++ or
 * framework types cross this boundary.
 *
 * Conventions (all entry points)
 * ------------------------------
 * Memory.  Every tensor argument is a DEVICE pointer owned by the caller,
 *   contiguous and row-major, on the context's device; the library neither
 *   frees nor keeps them after the call's stream work finishes.  bf16 tensors
 *   are passed as uint16_t bit patterns, tokens as int32_t.  Pointers must be
 *   16-byte aligned.  The library allocates no device memory inside a hot
 *   call: the context (dspark_ctx_create) owns all scratch (grid-barrier
 *   counter, per-step argmax keys, cross-CTA partials, gate activations,
 *   status word), sized for the B_max / V_max / K_max given at creation.
 * Streams.  Work is enqueued on `stream` (a cudaStream_t; NULL = legacy
 *   default stream) and runs asynchronously; outputs are valid once the
 *   stream has been synchronised.  A context holds one scratch area, so calls
 *   on one context must not overlap: issue them on one stream.
 * Errors.  Every call returns a dspark_status.  Argument errors are detected
 *   on the host before anything is enqueued (argument checks come before the
 *   context check, so they can be exercised with ctx == NULL).  Errors found
 *   by kernels (a grid-barrier or pipeline wait that ran out of time, a token
 *   id out of range) are written to the context's device status word; read it
 *   with dspark_get_status after synchronising the stream.  After a device
 *   error the context is poisoned: further hot calls return
 *   DSPARK_ERR_CTX_POISONED until dspark_ctx_reset is called.
 * Temperature.  temperature > 0 draws from softmax(l / T) exactly, in two
 *   stages over blocks of 16 consecutive token ids (block beta = v >> 4):
 *   (1) the block maximising ln Z_beta - ln E_beta wins, Z_beta the block's
 *   sum of exp(l / T) and E_beta = -ln u1(beta) a unit exponential (a race
 *   won with probability Z_beta / Z); (2) inside it, the first token (by id)
 *   whose cumulative exp(l / T) exceeds u2(beta) * Z_beta.  temperature == 0
 *   is greedy.  Returned log-probabilities are those of the drawn token under
 *   softmax(l / T'), T' = T (T > 0) or 1 (T == 0).
 * Noise.  Philox4x32-10 (Salmon et al., SC'11) keyed by (seed low 32 bits,
 *   seed high 32 bits) with counter (beta >> 3, k, b, 1 + (beta & 3)); with
 *   h = (beta >> 2) & 1, word 2h gives u1(beta) and word 2h + 1 gives
 *   u2(beta), each as u = ((word & 0x7FFFFF) + 0.5) * 2^-23.  b is the
 *   request's index in the call's batch, k its 0-based block position.  The
 *   same (seed, b, k, beta) always yields the same noise.
 * Ties.  Argmax and top-k orders break ties to the smaller token id.
 */
#ifndef DSPARK_H
#define DSPARK_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define DSPARK_ABI_VERSION 2

typedef struct dspark_ctx dspark_ctx;
typedef struct CUstream_st* dspark_stream_t; /* same type as cudaStream_t */

typedef enum dspark_status {
  DSPARK_OK = 0,
  DSPARK_ERR_INVALID_ARG = 1,    /* null pointer, bad size, misaligned pointer */
  DSPARK_ERR_UNSUPPORTED = 2,    /* shape outside what the kernels implement */
  DSPARK_ERR_CUDA = 3,           /* a CUDA runtime or driver call failed */
  DSPARK_ERR_TIMEOUT = 4,        /* device: a bounded wait ran out (kernel exited cleanly) */
  DSPARK_ERR_DEVICE_OOB = 5,     /* device: a token id read on the device was out of range */
  DSPARK_ERR_NO_DEVICE = 6,      /* no usable sm_103 device */
  DSPARK_ERR_CTX_POISONED = 7,   /* a previous device error needs dspark_ctx_reset */
  DSPARK_ERR_CAPACITY = 8        /* B, K or V above the context's creation limits */
} dspark_status;

/* Optional confidence head, fused into the draft / walk epilogues, or run
 * standalone by dspark_confidence.
 * Source: DSpark explainer, "Confidence-scheduled verification":
 *   c_k = sigmoid(w^T [h_k ; W1[x_{k-1}]] + bias), survival a_j = prod_{i<=j} c_i;
 * vLLM speculators "DSpark" guide, "Confidence Head" (the Markov embedding is
 * concatenated only when with_markov is set).
 * verify_len[b] = longest prefix j with a_j >= threshold (0 if none). */
typedef struct dspark_conf_args {
  const uint16_t* h;     /* [B, K, d] bf16 backbone hidden states */
  const uint16_t* w;     /* [d + r] bf16 if with_markov, else [d] */
  float bias;            /* scalar bias (0 in the pages' equation) */
  int d;                 /* hidden size, > 0, multiple of 8 */
  int with_markov;       /* 1: concatenate the previous token's Markov embedding */
  float threshold;       /* survival threshold for verify_len */
  float* conf;           /* out [B, K] fp32 */
  float* cumprod;        /* out [B, K] fp32 */
  int32_t* verify_len;   /* out [B] int32 */
  const float* tau;      /* [K] per-position temperatures from sequential temperature
                            scaling (c_k = sigmoid(z_k / tau_k)), device; NULL: all 1 */
} dspark_conf_args;

/* --------------------------------------------------------------------- */
/* Context                                                                 */
/* --------------------------------------------------------------------- */

/* Create a context on `device` with scratch for up to B_max requests, K_max
 * block positions (<= 64) and V_max vocabulary entries.  Allocates device
 * memory (the only allocation the library makes).  *ctx receives the handle;
 * release it with dspark_ctx_destroy. */
int dspark_ctx_create(dspark_ctx** ctx, int device, int B_max, int V_max, int K_max);

/* Free the context's device memory.  The caller must have synchronised every
 * stream that used it. */
int dspark_ctx_destroy(dspark_ctx* ctx);

/* Clear the device status word, the barrier counter and the argmax keys on
 * `stream`, and un-poison the context. */
int dspark_ctx_reset(dspark_ctx* ctx, dspark_stream_t stream);

/* Read the device status word (a dspark_status) into *device_status.  Reads
 * with a blocking copy on the context's device; call after the work stream has
 * been synchronised.  A non-OK value poisons the context. */
int dspark_get_status(dspark_ctx* ctx, int* device_status);

/* Testing knob: make CTA `cta` skip its grid-barrier arrival at step 0 in the
 * next draft launch (so every CTA's bounded wait runs out and the kernel exits
 * with DSPARK_ERR_TIMEOUT), with waits limited to timeout_ms.  cta = -1 turns
 * the knob off and timeout_ms <= 0 restores the default limit (2000 ms). */
int dspark_debug_set(dspark_ctx* ctx, int cta, int timeout_ms);

/* Testing knob: the next draft-kernel launch through this context asks the
 * CUDA runtime for 1 KB more dynamic shared memory than the kernel allows, so
 * the runtime refuses it on the host: the call returns DSPARK_ERR_CUDA, that
 * launch enqueues nothing, the refusal's error is cleared from the CUDA
 * runtime's last-error state, and the context stays usable (no reset needed).
 * Covers one launch.  Source: none on the pages (a test aid for the host-side
 * error path of a refused launch configuration). */
int dspark_debug_refuse_next_launch(dspark_ctx* ctx);

/* Profiling knob: the next draft launch (its first 128-request chunk) writes
 * global-timer stamps (ns) of every CTA's step phases into device_buffer,
 * laid out [grid][K][8] as unsigned 64-bit values: slot 0 step start, 1
 * embeddings gathered, 2 first accumulator ready, 3 last tile done, 4 partial
 * published, 5 grid barrier passed, 6 (last step only) final reduction done.
 * Unused slots are left untouched.  capacity counts 64-bit entries; a launch
 * whose trace would not fit writes nothing.  device_buffer == NULL turns the
 * trace off.  Source: none on the pages (a measurement aid of this library). */
int dspark_debug_trace(dspark_ctx* ctx, unsigned long long* device_buffer, int64_t capacity);

/* Text of a status code (static storage). */
const char* dspark_strerror(int code);

/* DSPARK_ABI_VERSION of the loaded library. */
int dspark_abi_version(void);

/* Number of kernels the last hot call on `ctx` enqueued. */
int dspark_last_launch_count(dspark_ctx* ctx);

/* --------------------------------------------------------------------- */
/* Markov-head draft                                                        */
/* --------------------------------------------------------------------- */

/* Vanilla Markov head, sampled left to right over a block.
 * Source: "DFlash-2's Selector and DSpark's Markov Head: An Equivalence
 * Observation", section "What the two methods do" (logits_k = U_k +
 * W1[a]^T W2, W1 in R^{V x 256}, W2 in R^{256 x V}); DSpark explainer,
 * "Semi-autoregressive generation" (anchor is the first prediction position;
 * left-to-right sampling) and "The Markov head" (B(x_{k-1}, .) = W1[x_{k-1}]
 * W2); "DSpark: Repair the Joint, Meter the Verify", "Fix 1" and "Why the
 * normalization has to be local" (exact local softmax per position).
 *   U        [B, K, V] fp32 base logits of the parallel backbone
 *   W1       [V, r] bf16 (Markov embedding table), W2 [r, V] bf16
 *   anchors  [B] int32: x_0, the token that feeds position 0's bias
 *   r        rank: 0 (head disabled: logits = U) or a multiple of 16, <= 256
 *   V        multiple of 8; K in [1, K_max]; B in [1, B_max]
 *   tokens   out [B, K] int32: x_1 .. x_K
 *   logprobs out [B, K] fp32: log q(x_k) under the local softmax
 *   conf     optional fused confidence head (NULL = off); uses W1[x_{k-1}]
 * One persistent cooperative kernel per 128 requests (requests are split in
 * chunks of 128; the noise uses the request's index in the whole call). */
int dspark_markov_draft(dspark_ctx* ctx, const float* U, const uint16_t* W1,
                        const uint16_t* W2, const int32_t* anchors, int B, int K, int V, int r,
                        float temperature, uint64_t seed, int32_t* tokens, float* logprobs,
                        const dspark_conf_args* conf, dspark_stream_t stream);

/* Gated Markov head: logits_t = U_t + (W1[a] (.) H(h_t))^T W2 with
 * H(h_t) = sigmoid(h_t . Wg) (no bias).
 * Source: equivalence page, "The equivalence: remove the gate, recover the
 * Markov Head" (context-gated variant) and "What the two methods do" (gate
 * H(h_t) computed from the current hidden state); vLLM guide, "Markov Head"
 * (gated variant).  The gate's functional form is this library's reading.
 *   h [B, K, d] bf16, Wg [d, r] bf16, d a multiple of 64; r a multiple of 64.
 * The gated embedding W1[a] (.) H is rounded to bf16 as the MMA operand.
 * Other arguments as dspark_markov_draft.  Launches the gate GEMM, its
 * finaliser, then the draft kernel. */
int dspark_gated_draft(dspark_ctx* ctx, const float* U, const uint16_t* W1,
                       const uint16_t* W2, const int32_t* anchors, const uint16_t* h,
                       const uint16_t* Wg, int d, int B, int K, int V, int r,
                       float temperature, uint64_t seed, int32_t* tokens, float* logprobs,
                       const dspark_conf_args* conf, dspark_stream_t stream);

/* RNN head: a recurrent state carried across the block's positions.
 * Source: DSpark explainer, "The RNN head" (a recurrent state s_k inside the
 * block mixing the previous state, the previous token's embedding and the
 * current backbone hidden h_k); "DSpark: Repair the Joint, Meter the Verify",
 * "Fix 1" ("Two instantiations of B": the RNN head carries a recurrent state
 * through the block); vLLM guide, "Key Parameters" (--markov-head-type rnn).
 * The pages give no equations; this library's reading is
 *   s_k = a_k (.) s_{k-1} + g_k (.) W1[x_{k-1}],  s_{-1} = 0,
 *   a_k = sigmoid(h_k . Wa) (decay),  g_k = sigmoid(h_k . Wg) (input; 1 when
 *   Wg == NULL),  logits_k = U_k + s_k W2,
 * so a = 0 gives the gated head and a = 0, g = 1 the vanilla one.  The state
 * is carried as the bf16 MMA operand (rounded at every position).
 *   h [B, K, d] bf16, Wa [d, r] bf16, Wg [d, r] bf16 or NULL; d and r
 *   multiples of 64.  Other arguments as dspark_markov_draft; the fused
 *   confidence head uses W1[x_{k-1}] as its Markov embedding.
 * Launches one or two gate GEMMs with their finalisers, then the draft kernel. */
int dspark_rnn_draft(dspark_ctx* ctx, const float* U, const uint16_t* W1, const uint16_t* W2,
                     const int32_t* anchors, const uint16_t* h, const uint16_t* Wa,
                     const uint16_t* Wg, int d, int B, int K, int V, int r, float temperature,
                     uint64_t seed, int32_t* tokens, float* logprobs,
                     const dspark_conf_args* conf, dspark_stream_t stream);

/* The RNN head's teacher-forced logits and LSE (parity mode): the state driven by
 * the given predecessors prev_tokens [B, K] (x_0 .. x_{K-1}); outputs as
 * dspark_markov_logits.  Source and reading as dspark_rnn_draft. */
int dspark_rnn_logits(dspark_ctx* ctx, const float* U, const uint16_t* W1, const uint16_t* W2,
                      const int32_t* prev_tokens, const uint16_t* h, const uint16_t* Wa,
                      const uint16_t* Wg, int d, int B, int K, int V, int r, float temperature,
                      float* logits, float* lse, dspark_stream_t stream);

/* The gate alone: H[m, :] = sigmoid(h[m, :] . Wg) for m < M.
 * Source: equivalence page, "What the two methods do" (the gate H(h_t) is a
 * function of the current hidden state alone, so every (request, position)
 * is gated at once, ahead of the draft); its sigmoid(h . Wg) form is this
 * library's reading (the gated workload fixes it).
 * h [M, d] bf16, Wg [d, r] bf16, H out [M, r] fp32; d, r multiples of 64,
 * M <= B_max * K_max. */
int dspark_gate(dspark_ctx* ctx, const uint16_t* h, const uint16_t* Wg, int M, int d, int r,
                float* H, dspark_stream_t stream);

/* Context-free variant of dspark_markov_draft that allocates no device memory.
 * The pages have no counterpart: this is an integration aid of this library.
 * For callers that may not allocate device memory themselves (a library inside
 * a host framework that owns all device memory through its own pool, or a
 * serving loop that forbids cudaMalloc / cudaFree because they can synchronise
 * the device).  Inputs and outputs are the caller's, as in dspark_markov_draft
 * (no confidence head); the kernel's scratch is one fixed array of about 7.9 MB
 * compiled into the library, present on every GPU that loads it until the
 * process exits.
 *   Limits: K <= 16 and B <= 16383 * 128 (else DSPARK_ERR_CAPACITY), other
 *   shape rules as dspark_markov_draft; the current device must be sm_103
 *   and hold the pointers.
 *   device_status: optional device int that receives the launch's device
 *   status (a dspark_status) in stream order; NULL to skip.
 *   Set-up: the first call in a CUDA context (per device: its primary
 *   context) looks up the array's device address (cudaGetSymbolAddress) with
 *   that device current; make that first call before any stream capture.  A
 *   new context on the device (after cudaDeviceReset, say) triggers a new
 *   look-up at its first call, since the array may have moved.
 *   Sharing: every call on a device uses the same array and starts by clearing
 *   its counters and keys on `stream`; calls that overlap on the GPU (other
 *   streams or host threads) race and must be serialised by the caller. */
int dspark_markov_draft_noalloc(const float* U, const uint16_t* W1, const uint16_t* W2,
                                const int32_t* anchors, int B, int K, int V, int r,
                                float temperature, uint64_t seed, int32_t* tokens,
                                float* logprobs, int* device_status, dspark_stream_t stream);

/* --------------------------------------------------------------------- */
/* Selector-style top-k execution                                           */
/* --------------------------------------------------------------------- */

/* Top-k candidate sets and adjacent-pair score tables.
 * Source: equivalence page, "Where the parallelism comes from" (top-16 of the
 * base logits; all 16 x 16 predecessor/candidate calibrations in parallel),
 * "What the two methods do" (S_t(a, b) = U_t(b) + <A(a) (.) H(h_t), B(b)>)
 * and "Two implications" (the same truncation for a trained Markov head,
 * A = W1, B = W2^T).
 *   U [B, K, V] fp32; A, Bt [V, r] bf16 (Bt row b is B(b)); anchors [B]
 *   h, Wg: gate inputs as dspark_gated_draft, or both NULL (ungated, H = 1)
 *   topk in [1, 32], topk <= V; r a multiple of 16 (64 if gated), <= 256
 *   cand   out [B, K, topk] int32, ordered by (U desc, id asc)
 *   cand_U out [B, K, topk] fp32 (U of each candidate)
 *   scores out [B, K, topk, topk] fp32: scores[b,t,i,j] = S_t(p_i, c_j) with
 *          p = cand[b, t-1, :] for t >= 1 and p_i = anchors[b] for t = 0. */
int dspark_selector_scores(dspark_ctx* ctx, const float* U, const uint16_t* A,
                           const uint16_t* Bt, const int32_t* anchors, const uint16_t* h,
                           const uint16_t* Wg, int d, int B, int K, int V, int r, int topk,
                           int32_t* cand, float* cand_U, float* scores, dspark_stream_t stream);

/* The light sequential walk over the pair tables: per request, for t = 0..K-1
 * draw candidate j from row `slot` (slot = 0 at t = 0) by the head's own
 * two-stage block race (above) over scores/T, restricted to the candidates:
 * the candidates of one 16-token block race with their summed mass, tokens
 * outside the set have none (T = 0: greedy); then slot = j.  With topk = V
 * this is the full head's draw.  log-probabilities are under the topk-way
 * softmax.
 * Source: equivalence page, "Where the parallelism comes from" (a greedy walk,
 * or sampling, over the precomputed scores) and "Two implications", step 3.
 *   cand [B, K, topk], scores [B, K, topk, topk] as produced above
 *   A [V, r], anchors [B]: only read by the fused confidence head (which uses
 *   A[x_{t-1}] as the Markov embedding); may be NULL when conf == NULL. */
int dspark_selector_walk(dspark_ctx* ctx, const int32_t* cand, const float* scores,
                         const int32_t* anchors, const uint16_t* A, int B, int K, int V, int r,
                         int topk, float temperature, uint64_t seed, int32_t* tokens,
                         float* logprobs, const dspark_conf_args* conf, dspark_stream_t stream);

/* --------------------------------------------------------------------- */
/* Confidence head (standalone)                                             */
/* --------------------------------------------------------------------- */

/* c_k = sigmoid((w[:d] . h[b,k] + with_markov * w[d:] . W1[x_{k-1}] + bias) / tau_k),
 * cumprod a_k, verify_len = longest prefix with a_k >= threshold.
 * Source: as dspark_conf_args.  tokens [B, K] = x_1..x_K; x_0 = anchors[b].
 * W1 may be NULL when with_markov == 0; tau [K] device (NULL: all 1). */
int dspark_confidence(dspark_ctx* ctx, const uint16_t* h, const uint16_t* W1,
                      const int32_t* anchors, const int32_t* tokens, const uint16_t* w,
                      float bias, int with_markov, int B, int K, int d, int r, int V,
                      float threshold, const float* tau, float* conf, float* cumprod,
                      int32_t* verify_len, dspark_stream_t stream);

/* Sequential temperature scaling (STS) of the confidence head: one temperature
 * per position, fitted left to right against cumulative prefix survival.
 * Source: DSpark explainer, "Confidence-scheduled verification" (the raw head's
 * calibration error is brought down by fitting one temperature per position,
 * left to right, against cumulative prefix-survival probabilities; the
 * ranking is kept).  tau_k minimises, over the N calibration rows, the binary
 * cross-entropy between prod_{i<=k} sigmoid(z_i / tau_i) (tau_0 .. tau_{k-1}
 * already fitted) and prod_{i<=k} label_i, with z_i the logit of the raw
 * confidence (clamped to [2^-24, 1 - 2^-24]) and the survival clamped to
 * [1e-7, 1 - 1e-7] inside the logarithms.  The 1-D search over ln tau in
 * [ln tau_lo, ln tau_hi]: 32 evenly spaced points, keep the best (ties to the
 * smaller), narrow to the interval between its neighbours, 8 rounds.
 *   conf [N, K] fp32 raw confidences (the head with tau = 1)
 *   label [N, K] fp32 acceptance labels (dspark_accept_label) or 0/1 outcomes
 * Outputs tau [K] fp32 and loss [K] (mean cross-entropy at tau_k; may be
 * NULL).  Device pointers; one kernel, no host synchronisation.  0 < tau_lo <
 * tau_hi; K <= 64. */
int dspark_sts_fit(dspark_ctx* ctx, const float* conf, const float* label, int N, int K,
                   float tau_lo, float tau_hi, float* tau, float* loss, dspark_stream_t stream);

/* --------------------------------------------------------------------- */
/* Teacher-forced calibrated logits (parity / test mode)                    */
/* --------------------------------------------------------------------- */

/* logits[b, k, :] = U[b, k, :] + (W1[x_{k-1}] (.) H)^T W2 for given
 * predecessors prev_tokens[b, k] = x_{k-1} (x_0 = the anchor), and
 * lse[b, k] = log sum_v exp(logits[b, k, v] / T').
 * Source: equivalence page, per-candidate form logits_k(b | a) = U_k(b) +
 * W1[a]^T W2[:, b].  h, Wg: NULL (vanilla) or the gate inputs (gated).
 * Writes the full [B, K, V] fp32 logits: meant for checking, not speed. */
int dspark_markov_logits(dspark_ctx* ctx, const float* U, const uint16_t* W1,
                         const uint16_t* W2, const int32_t* prev_tokens, const uint16_t* h,
                         const uint16_t* Wg, int d, int B, int K, int V, int r,
                         float temperature, float* logits, float* lse, dspark_stream_t stream);

/* --------------------------------------------------------------------- */
/* Speculative verification of a drafted block                             */
/* --------------------------------------------------------------------- */

/* The target's accept-or-correct rule over each request's verify window.
 * Source: "DSpark: Repair the Joint, Meter the Verify", "Watch the Mass Land
 * Wrong" (accept a drafted token with probability min(1, p/q); on a rejection
 * the target resamples); DSpark explainer, "Confidence-scheduled
 * verification" (that probability is 1 - TV(p^d_k, p^t_k)), "Hardware-aware
 * prefix scheduling" (every retained token goes through this rule) and "Two
 * bottlenecks after you already have a parallel drafter" (a bonus token when
 * the whole draft survives).  For k = 0 .. ell[b]-1 in order, drafted token
 * x_k survives with probability min(1, p_k(x_k) / q_k(x_k)); at the first
 * rejection (position j) the next token is drawn from the normalised residual
 * max(0, p_j - q_j); if all ell[b] survive, it is drawn from p_{ell[b]}.
 *   P [B, K+1, V] fp32 target logits (row k: position k; row K: after a fully
 *     accepted block); p_k = softmax(P[b,k] / target_temperature), one-hot at
 *     the argmax (ties to the smaller id) when target_temperature == 0.
 *   U, W1, W2, anchors (and h, Wg, d when gated): the draft head's inputs, as
 *     given to the draft call; q_k = softmax(l_k / draft_temperature) of its
 *     calibrated logits given the drafted predecessor (one-hot at x_k when
 *     draft_temperature == 0).
 *   tokens [B, K] drafted tokens; draft_logprobs [B, K] their log q_k(x_k) as
 *     returned by the draft call (required when draft_temperature > 0).
 *   ell [B] verified positions per request in [0, K] (NULL: K; values outside
 *     are clamped), e.g. the confidence head's verify_len.
 * Outputs: n_acc [B] accepted prefix length; next_token [B] the target's token
 * after it; accept_prob [B, K] (NULL: not written) min(1, p/q) for k < ell[b],
 * -1 beyond.  Noise: Philox4x32-10 keyed by the seed; position k's acceptance
 * uniform from counter (k, 0, b, 13) word 0; the draw at position j uses the
 * block race of the draft (16-token blocks) on counter (beta >> 3, j, b,
 * 9 + (beta & 3)).  Sizes within the context's B_max, K_max, V_max; V % 8 == 0
 * and 16-byte aligned P and U.  Drafted tokens out of [0, V) are reported as
 * DSPARK_ERR_DEVICE_OOB.  Scratch: the context's per-request verification
 * buffers (allocated at creation); the draw reads the rows of U and P at each
 * request's draw position in place. */
int dspark_verify(dspark_ctx* ctx, const float* P, const float* U, const uint16_t* W1,
                  const uint16_t* W2, const int32_t* anchors, const uint16_t* h,
                  const uint16_t* Wg, int d, const int32_t* tokens, const float* draft_logprobs,
                  const int32_t* ell, int B, int K, int V, int r, float draft_temperature,
                  float target_temperature, uint64_t seed, int32_t* n_acc, int32_t* next_token,
                  float* accept_prob, dspark_stream_t stream);

/* --------------------------------------------------------------------- */
/* Acceptance label of each drafted position                               */
/* --------------------------------------------------------------------- */

/* c*_k = 1 - TV(p^d_k, p^t_k) = sum_v min(p^d_k(v), p^t_k(v)) for every
 * drafted position.  Source: DSpark explainer, "Confidence-scheduled
 * verification": the confidence head is trained on this label, the
 * probability that the target accepts position k under speculative decoding.
 *   P [B, K+1, V] fp32 target logits, laid out as for dspark_verify (row K is
 *     not read); p^t_k = softmax(P[b,k] / target_temperature), one-hot at the
 *     argmax (ties to the smaller id) when target_temperature == 0.
 *   U, W1, W2, anchors (and h, Wg, d when gated): the draft head's inputs;
 *     p^d_k = softmax(l_k / draft_temperature) of its calibrated logits given
 *     the drafted predecessor (one-hot at x_k when draft_temperature == 0).
 *   tokens [B, K] drafted tokens; draft_logprobs [B, K] their log p^d_k(x_k)
 *     as returned by the draft call at draft_temperature (required when it is
 *     > 0: they supply the draft's normaliser).
 * Output label [B, K] fp32 in [0, 1].  When both temperatures are positive
 * the sum over the vocabulary runs in the draft kernel (one pass over U, W2
 * and P); when either side is greedy the label is one probability.  Sizes
 * within the context's B_max, K_max, V_max; V % 8 == 0; 16-byte aligned P and
 * U.  Drafted tokens out of [0, V) are reported as DSPARK_ERR_DEVICE_OOB.
 * Device pointers; no host synchronisation. */
int dspark_accept_label(dspark_ctx* ctx, const float* P, const float* U, const uint16_t* W1,
                        const uint16_t* W2, const int32_t* anchors, const uint16_t* h,
                        const uint16_t* Wg, int d, const int32_t* tokens,
                        const float* draft_logprobs, int B, int K, int V, int r,
                        float draft_temperature, float target_temperature, float* label,
                        dspark_stream_t stream);

/* --------------------------------------------------------------------- */
/* Load-aware prefix scheduler                                              */
/* --------------------------------------------------------------------- */

/* Verify lengths that maximise the target's throughput by the greedy rule.
 * Source: DSpark explainer, "Hardware-aware prefix scheduling": with R
 * requests, request r verifying a prefix of length ell_r and the target batch
 * B = sum_r (1 + ell_r), the objective is Theta = (R + sum of the admitted
 * extensions' survival) * SPS(B); start at B = R, rank candidate extensions
 * globally by survival probability, admit them while Theta increases
 * (strictly) and stop at the first one that would not.  Candidates are ranked
 * by (survival desc, position asc, request asc), which keeps every prefix
 * whole because survival never grows along a request.
 *   a [R, K] survival of extension (r, k) (e.g. the confidence head's cumprod)
 *   sps [sps_len] SPS(B) for B = 0 .. sps_len - 1, sps_len >= R (K + 1) + 1
 * Outputs ell [R] (device) and theta (device scalar, may be NULL).  R * K <=
 * 16384; with K = 0 nothing is admitted (ell = 0, theta = R SPS(R)) and a may
 * be NULL.  All arrays are device pointers; one kernel, no host
 * synchronisation. */
int dspark_schedule(dspark_ctx* ctx, const float* a, int R, int K, const float* sps, int sps_len,
                    int32_t* ell, float* theta, dspark_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* DSPARK_H */
