/*
 * dspark_oracle.c -- plain, slow, fp64 CPU oracle of the DSpark Markov-head
 * drafting hot path.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test-suite, the smoke check and the
 * benchmark's CPU-baseline leg may load this file's library.  It shares no
 * code, header, table or constant generator with the CUDA path.
 *
 * Every floating-point step is carried out in double precision from the exact
 * widening of the bf16 weights and the fp32 base logits.  Loops follow the
 * pages' definitions in their order; the only parallelism is OpenMP over
 * independent vocabulary entries (or independent rows), which does not change
 * any sum's order.
 *
 * Sources (each function names the passage it follows):
 *  [EQV]  "DFlash-2's Selector and DSpark's Markov Head: An Equivalence
 *         Observation" (jialefu.github.io)
 *  [EXPL] "DSpark" explainer (himanshu-arora.com): sections "Semi-autoregressive
 *         generation", "The Markov head", "Confidence-scheduled verification"
 *  [FIX]  "DSpark: Repair the Joint, Meter the Verify" (stable-lab.github.io):
 *         "Fix 1: A First-Order Markov Head", "Why the normalization has to be
 *         local"
 *  [VLLM] "DSpark" (vLLM speculators user guide): "Markov Head", "Confidence
 *         Head", "Sample From Anchor", "Key Parameters"
 *
 * Readings where the pages are silent (the same readings the CUDA path takes):
 *  - x_0 is the anchor token, so every position k = 0..K-1 gets a bias
 *    ([EXPL] "Semi-autoregressive generation": the anchor is the first
 *    prediction position; [VLLM] "Sample From Anchor").
 *  - Temperature T > 0 draws from softmax(l / T) in two exact stages over
 *    blocks of 16 consecutive token ids (block beta = v >> 4):
 *      1. block race: beta* = argmax_beta  ln Z_beta - ln E_beta, where
 *         Z_beta = sum_{v in beta} exp(l_v / T) and E_beta = -ln u1(beta) is a
 *         unit exponential (the exponential race / Gumbel-max over blocks:
 *         P(beta* = beta) = Z_beta / Z);
 *      2. inverse CDF inside beta*: the smallest v in beta* whose cumulative
 *         mass (in token-id order) exceeds u2(beta*) * Z_beta*.
 *    So P(v) = (Z_beta / Z) (exp(l_v / T) / Z_beta) = softmax(l / T)_v.
 *    T == 0 is greedy argmax(l).  The returned log-probability is that of the
 *    drawn token under softmax(l / T') with T' = T (T > 0) or 1 (T == 0).
 *  - Ties in any argmax or top-k order go to the smaller token id (block id).
 *  - Noise: Philox4x32-10 (Salmon, Moraes, Dror, Shaw, "Parallel Random
 *    Numbers: As Easy as 1, 2, 3", SC'11), key = (seed low 32, seed high 32).
 *    A counter (c0, c1, c2, c3) and an output word w give
 *    u = ((word_w & 0x7FFFFF) + 0.5) * 2^-23 (the low 23 bits), exactly
 *    representable in fp32 and fp64 and strictly inside (0, 1).
 *      counter (beta >> 3, k, b, 1 + (beta & 3)), h = (beta >> 2) & 1:
 *      u1(beta) = word 2h, u2(beta) = word 2h + 1
 *    (so whoever owns every fourth block of a range draws both stages of two
 *    consecutive ones of its blocks from one Philox call).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* ------------------------------------------------------------------ */
/* helpers                                                             */
/* ------------------------------------------------------------------ */

static double bf16_to_double(uint16_t bits) {
  uint32_t u = ((uint32_t)bits) << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

static double sigmoid(double z) { return 1.0 / (1.0 + exp(-z)); }

void orc_set_threads(int n) {
#ifdef _OPENMP
  if (n > 0) omp_set_num_threads(n);
#else
  (void)n;
#endif
}

int orc_max_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

/* ------------------------------------------------------------------ */
/* Philox4x32-10, from its published definition (SC'11, section 3.2):  */
/* each round multiplies words 0 and 2 by fixed odd constants, takes   */
/* the high and low halves of the 64-bit products, and mixes the high  */
/* halves with words 1/3 and the round key; the key is bumped by the   */
/* Weyl constants (golden ratio, sqrt(3) - 1) between rounds.          */
/* ------------------------------------------------------------------ */

void orc_philox4x32_10(const uint32_t ctr[4], const uint32_t key[2], uint32_t out[4]) {
  const uint32_t mul0 = 0xD2511F53u, mul1 = 0xCD9E8D57u;
  const uint32_t weyl0 = 0x9E3779B9u, weyl1 = 0xBB67AE85u;
  uint32_t x0 = ctr[0], x1 = ctr[1], x2 = ctr[2], x3 = ctr[3];
  uint32_t k0 = key[0], k1 = key[1];
  for (int round = 0; round < 10; ++round) {
    if (round > 0) {
      k0 += weyl0;
      k1 += weyl1;
    }
    uint64_t p0 = (uint64_t)mul0 * (uint64_t)x0;
    uint64_t p1 = (uint64_t)mul1 * (uint64_t)x2;
    uint32_t hi0 = (uint32_t)(p0 >> 32), lo0 = (uint32_t)p0;
    uint32_t hi1 = (uint32_t)(p1 >> 32), lo1 = (uint32_t)p1;
    uint32_t y0 = hi1 ^ x1 ^ k0;
    uint32_t y1 = lo1;
    uint32_t y2 = hi0 ^ x3 ^ k1;
    uint32_t y3 = lo0;
    x0 = y0;
    x1 = y1;
    x2 = y2;
    x3 = y3;
  }
  out[0] = x0;
  out[1] = x1;
  out[2] = x2;
  out[3] = x3;
}

/* u in (0, 1) from word `w` of Philox4x32-10(counter (c0, c1, c2, c3), seed). */
double orc_uniform_ctr(uint64_t seed, uint32_t c0, uint32_t c1, uint32_t c2, uint32_t c3,
                       uint32_t w) {
  uint32_t ctr[4] = {c0, c1, c2, c3};
  uint32_t key[2] = {(uint32_t)(seed & 0xFFFFFFFFu), (uint32_t)(seed >> 32)};
  uint32_t out[4];
  orc_philox4x32_10(ctr, key, out);
  uint32_t word = out[w & 3u];
  return ((double)(word & 0x7FFFFFu) + 0.5) * (1.0 / 8388608.0); /* 2^-23 */
}

/* u(seed, b, k, v) with stream tag `tag`: counter (v >> 2, k, b, tag), word v & 3. */
double orc_uniform(uint64_t seed, uint32_t b, uint32_t k, uint32_t v, uint32_t tag) {
  return orc_uniform_ctr(seed, v >> 2, k, b, tag, v & 3u);
}

/* Stage-1 / stage-2 uniforms of block `blk` (request b, position k) on the race
   streams starting at tag `tag0` (1: the draft; 9: the verifier's resample). */
static double race_u1(uint64_t seed, uint32_t b, uint32_t k, uint32_t blk, uint32_t tag0) {
  return orc_uniform_ctr(seed, blk >> 3, k, b, tag0 + (blk & 3u), 2u * ((blk >> 2) & 1u));
}

static double race_u2(uint64_t seed, uint32_t b, uint32_t k, uint32_t blk, uint32_t tag0) {
  return orc_uniform_ctr(seed, blk >> 3, k, b, tag0 + (blk & 3u), 2u * ((blk >> 2) & 1u) + 1u);
}

/* Stage-1 uniform of block `blk` (request b, position k) of the draft. */
double orc_block_uniform(uint64_t seed, uint32_t b, uint32_t k, uint32_t blk) {
  return race_u1(seed, b, k, blk, 1u);
}

/* Stage-2 uniform of block `blk` (request b, position k) of the draft. */
double orc_within_uniform(uint64_t seed, uint32_t b, uint32_t k, uint32_t blk) {
  return race_u2(seed, b, k, blk, 1u);
}

/* The verifier's acceptance uniform of position k of request b:
   counter (k, 0, b, 13), word 0. */
double orc_accept_uniform(uint64_t seed, uint32_t b, uint32_t k) {
  return orc_uniform_ctr(seed, k, 0u, b, 13u, 0u);
}


/* ------------------------------------------------------------------ */
/* Gate H(h_t) = sigmoid(h_t . Wg) of the gated head.                   */
/* [EQV] "What the two methods do" (Selector score, gate H(h_t)) and   */
/* "The equivalence..." (gated Markov-head rule).  The pages leave the  */
/* gate's form open; this build reads it as a linear map of the current */
/* position's hidden state followed by a logistic sigmoid, no bias.     */
/* h [M, d] bf16, Wg [d, r] bf16 -> H [M, r] fp64.                       */
/* ------------------------------------------------------------------ */
void orc_gate(const uint16_t* h, const uint16_t* Wg, int64_t M, int d, int r, double* H) {
#pragma omp parallel for schedule(static)
  for (int64_t m = 0; m < M; ++m) {
    double* acc = H + m * (int64_t)r;
    for (int i = 0; i < r; ++i) acc[i] = 0.0;
    for (int j = 0; j < d; ++j) {
      double hj = bf16_to_double(h[m * (int64_t)d + j]);
      const uint16_t* wrow = Wg + (int64_t)j * r;
      for (int i = 0; i < r; ++i) acc[i] += hj * bf16_to_double(wrow[i]);
    }
    for (int i = 0; i < r; ++i) acc[i] = sigmoid(acc[i]);
  }
}

/* ------------------------------------------------------------------ */
/* One position of the Markov head.                                    */
/* [EQV] "What the two methods do": logits_k = U_k + W1[a]^T W2 with   */
/* a the previously sampled token; gated form logits_t = U_t +         */
/* (W1[a] (.) H(h_t))^T W2.  [EXPL] "The Markov head": B(x_{k-1}, .) = */
/* W1[x_{k-1}] W2.  [FIX] "Fix 1": the per-position distribution is    */
/* the local softmax exp(z_k(v) + B(t_{k-1}, v)) / sum_u exp(...).      */
/* Writes l[v] (calibrated logits) for v in [0, V).                     */
/* ------------------------------------------------------------------ */
/* l[v] = U[v] + sum_i e[i] * W2[i, v] for v in [0, V): the bias of a head  */
/* embedding e (length r) added to one row of base logits.                   */
static void bias_logits(const float* Urow, const uint16_t* W2, const double* e, int V, int r,
                        double* l) {
#pragma omp parallel
  {
#ifdef _OPENMP
    int nt = omp_get_num_threads(), tid = omp_get_thread_num();
#else
    int nt = 1, tid = 0;
#endif
    int64_t chunk = ((int64_t)V + nt - 1) / nt;
    int64_t v0 = (int64_t)tid * chunk, v1 = v0 + chunk;
    if (v1 > V) v1 = V;
    if (v0 < v1) {
      /* bias[v] = sum_i e[i] * W2[i, v], summed over i = 0..r-1 in order */
      for (int64_t v = v0; v < v1; ++v) l[v] = 0.0;
      for (int i = 0; i < r; ++i) {
        const uint16_t* w2row = W2 + (int64_t)i * V;
        double ei = e[i];
        for (int64_t v = v0; v < v1; ++v) l[v] += ei * bf16_to_double(w2row[v]);
      }
      for (int64_t v = v0; v < v1; ++v) l[v] = (double)Urow[v] + l[v];
    }
  }
}

static void calibrated_logits(const float* Urow, const uint16_t* W1, const uint16_t* W2,
                              const double* Hrow, int V, int r, int32_t prev, double* e,
                              double* l) {
  for (int i = 0; i < r; ++i) {
    double w1 = bf16_to_double(W1[(int64_t)prev * r + i]);
    e[i] = Hrow ? w1 * Hrow[i] : w1;
  }
  bias_logits(Urow, W2, e, V, r, l);
}

/* ------------------------------------------------------------------ */
/* RNN head: one step of the recurrent state.                          */
/* [EXPL] "The RNN head": a recurrent state s_k kept inside the block,  */
/* mixing the previous state, the previous token's embedding and the    */
/* current backbone hidden h_k; [FIX] "Fix 1" ("Two instantiations of   */
/* B": the RNN head carries a recurrent state through the block,        */
/* accumulating the in-block prefix); [VLLM] "Key Parameters"           */
/* (--markov-head-type rnn).  The pages give no equations; the reading  */
/* taken (the plainest gated linear recurrence that reduces to the      */
/* Markov heads) is                                                     */
/*   s_k = a_k (.) s_{k-1} + g_k (.) W1[x_{k-1}],   s_{-1} = 0,         */
/*   a_k = sigmoid(h_k . Wa) (decay),  g_k = sigmoid(h_k . Wg) (input), */
/*   bias_k = s_k W2,                                                   */
/* so a = 0 is the gated head and a = 0, g = 1 the vanilla one.  The    */
/* gates are inputs here (Arow, Grow: rows of orc_gate's output; Grow   */
/* NULL means g = 1).  Updates s in place.                              */
/* ------------------------------------------------------------------ */
static void rnn_state_step(const uint16_t* W1, int r, int32_t prev, const double* Arow,
                           const double* Grow, double* s) {
  for (int i = 0; i < r; ++i) {
    const double w1 = bf16_to_double(W1[(int64_t)prev * r + i]);
    s[i] = Arow[i] * s[i] + (Grow ? w1 * Grow[i] : w1);
  }
}

/* log sum_v exp(l[v] / Tp), max-shifted. */
static double log_sum_exp_scaled(const double* l, int V, double Tp) {
  double m = -INFINITY;
  for (int v = 0; v < V; ++v) {
    double z = l[v] / Tp;
    if (z > m) m = z;
  }
  if (m == -INFINITY) return -INFINITY;
  double s = 0.0;
  for (int v = 0; v < V; ++v) s += exp(l[v] / Tp - m);
  return m + log(s);
}

/* ------------------------------------------------------------------ */
/* One draw from softmax(z) over n items with token ids ids[0..n-1]    */
/* (ascending; NULL: ids are 0..n-1), by the two-stage block race of   */
/* the header.  w[0..n-1] is scratch.  Returns the index of the drawn   */
/* item (-1 if every z is -inf) and its decision margin: the smaller of */
/* the stage-1 gap (best block score - runner-up, in nats) and the      */
/* stage-2 distance of u2 * Z from the nearest cumulative boundary,     */
/* relative to Z (either is the relative error that would flip it).     */
/* ------------------------------------------------------------------ */
static int block_race_draw(const int32_t* ids, const double* z, double* w, int n, uint64_t seed,
                           uint32_t b, uint32_t k, uint32_t tag0, double* margin) {
  double m = -INFINITY;
  for (int i = 0; i < n; ++i)
    if (z[i] > m) m = z[i];
  if (m == -INFINITY) return -1;
#pragma omp parallel for schedule(static) if (n > 65536)
  for (int i = 0; i < n; ++i) w[i] = exp(z[i] - m);
  /* stage 1: one unit exponential per block, ln Z - ln E */
  double best = -INFINITY, second = -INFINITY, bestZ = 0.0;
  int bs = -1, be = -1;
  uint32_t bblk = 0;
  for (int i = 0; i < n;) {
    const uint32_t blk = (uint32_t)(ids ? ids[i] : i) >> 4;
    double Z = 0.0;
    int j = i;
    while (j < n && ((uint32_t)(ids ? ids[j] : j) >> 4) == blk) Z += w[j++];
    if (Z > 0.0) {
      const double E = -log(race_u1(seed, b, k, blk, tag0));
      const double score = log(Z) - log(E);
      if (score > best) {
        second = best;
        best = score;
        bs = i;
        be = j;
        bblk = blk;
        bestZ = Z;
      } else if (score > second) {
        second = score;
      }
    }
    i = j;
  }
  /* stage 2: inverse CDF inside the winning block, in token-id order */
  const double target = race_u2(seed, b, k, bblk, tag0) * bestZ;
  double C = 0.0, m2 = 0.0;
  int pick = -1, last = -1;
  for (int i = bs; i < be; ++i) {
    if (w[i] == 0.0) continue;
    const double prevC = C;
    C += w[i];
    last = i;
    if (target < C) {
      pick = i;
      m2 = fmin(target - prevC, C - target) / bestZ;
      break;
    }
  }
  if (pick < 0) pick = last; /* target at the very top (rounding): the last live item */
  *margin = fmin(best - second, m2);
  return pick;
}

/* ------------------------------------------------------------------ */
/* Markov-head draft over a block (vanilla, or gated when H != NULL).   */
/* [EXPL] "Semi-autoregressive generation" + "The Markov head": the    */
/* head samples left to right, x_0 = anchor, position k's logits get   */
/* the bias of x_{k-1}.  [FIX] "Why the normalization has to be local": */
/* the returned per-token log-probability is exact under the local     */
/* softmax.  [VLLM] "Key Parameters": rank 0 disables the head.         */
/*                                                                    */
/* Inputs are full arrays indexed by the global request b: U [B,K,V],   */
/* anchors [B], H [B,K,r] or NULL.  Requests b0 .. b0+nb-1 are run;     */
/* outputs are compact [nb, K]:                                         */
/*   tokens    oracle's own choice at each position                    */
/*   logprobs  log-probability of that choice                           */
/*   margins   s(best) - s(second best) of the perturbed scores        */
/* If `forced` ([nb, K]) is given, the path continues on forced tokens  */
/* (x_k = forced[k]) and forced_logprobs receives their log-probability. */
/* Returns 0, or -1 on bad arguments / allocation failure.              */
/* ------------------------------------------------------------------ */
/* One request of the draft; buffers l, s ([V]) and e ([r]) are the caller's. */
/* A != NULL: the RNN head (A the decay gates, H the input gates or NULL), */
/* with e carrying the recurrent state across positions.                   */
static int draft_one_request(const float* U, const uint16_t* W1, const uint16_t* W2,
                             const int32_t* anchors, const double* H, const double* A, int K,
                             int V, int r, double temperature, uint64_t seed, int b, int bi,
                             const int32_t* forced, int32_t* tokens, double* logprobs,
                             double* margins, double* forced_logprobs, double* l, double* s,
                             double* e) {
  const double Tp = temperature > 0.0 ? temperature : 1.0;
  int32_t prev = anchors[b];
  if (A)
    for (int i = 0; i < r; ++i) e[i] = 0.0; /* s_{-1} = 0 */
  for (int k = 0; k < K; ++k) {
    const float* Urow = U + ((int64_t)b * K + k) * V;
    const double* Hrow = H ? H + ((int64_t)b * K + k) * r : NULL;
    if (prev < 0 || prev >= V) return -1;
    if (A) {
      rnn_state_step(W1, r, prev, A + ((int64_t)b * K + k) * r, Hrow, e);
      bias_logits(Urow, W2, e, V, r, l);
    } else {
      calibrated_logits(Urow, W1, W2, Hrow, V, r, prev, e, l);
    }
    const int64_t o = (int64_t)bi * K + k;
    int best = 0;
    if (temperature > 0.0) {
      /* z = l / T, then the two-stage block race (header) */
      double* z = s;
      double* w = s + V;
      for (int v = 0; v < V; ++v) z[v] = l[v] / temperature;
      best = block_race_draw(NULL, z, w, V, seed, (uint32_t)b, (uint32_t)k, 1u, &margins[o]);
      if (best < 0) return -1;
    } else {
      /* argmax, ties to the smaller token id; runner-up for the margin */
      for (int v = 1; v < V; ++v)
        if (l[v] > l[best]) best = v;
      double second = -INFINITY;
      for (int v = 0; v < V; ++v)
        if (v != best && l[v] > second) second = l[v];
      margins[o] = l[best] - second;
    }
    const double lse = log_sum_exp_scaled(l, V, Tp);
    tokens[o] = best;
    logprobs[o] = l[best] / Tp - lse;
    if (forced) {
      const int32_t f = forced[o];
      if (f < 0 || f >= V) return -1;
      if (forced_logprobs) forced_logprobs[o] = l[f] / Tp - lse;
      prev = f;
    } else {
      prev = best;
    }
  }
  return 0;
}

static int run_draft(const float* U, const uint16_t* W1, const uint16_t* W2,
                     const int32_t* anchors, const double* H, const double* A, int B, int K,
                     int V, int r, double temperature, uint64_t seed, int b0, int nb,
                     const int32_t* forced, int32_t* tokens, double* logprobs, double* margins,
                     double* forced_logprobs) {
  if (B <= 0 || K <= 0 || V <= 0 || r < 0 || b0 < 0 || nb < 0 || b0 + nb > B) return -1;
  int bad = 0;
  /* Many small requests: one request per thread (the per-request vocabulary
     loops then run on that thread alone); otherwise requests run one after
     the other with the vocabulary loops shared by all threads. */
  const int per_request = nb >= 4 * orc_max_threads() && V <= 8192;
#pragma omp parallel if (per_request) reduction(| : bad)
  {
    double* l = (double*)malloc(sizeof(double) * (size_t)V);
    double* s = (double*)malloc(sizeof(double) * 2 * (size_t)V);
    double* e = (double*)malloc(sizeof(double) * (size_t)(r > 0 ? r : 1));
    if (!l || !s || !e) {
      bad = 1;
    } else {
#pragma omp for schedule(static)
      for (int bi = 0; bi < nb; ++bi) {
        if (draft_one_request(U, W1, W2, anchors, H, A, K, V, r, temperature, seed, b0 + bi, bi,
                              forced, tokens, logprobs, margins, forced_logprobs, l, s, e) != 0)
          bad = 1;
      }
    }
    free(l);
    free(s);
    free(e);
  }
  return bad ? -1 : 0;
}

int orc_markov_draft(const float* U, const uint16_t* W1, const uint16_t* W2,
                     const int32_t* anchors, const double* H, int B, int K, int V, int r,
                     double temperature, uint64_t seed, int b0, int nb, const int32_t* forced,
                     int32_t* tokens, double* logprobs, double* margins,
                     double* forced_logprobs) {
  return run_draft(U, W1, W2, anchors, H, NULL, B, K, V, r, temperature, seed, b0, nb, forced,
                   tokens, logprobs, margins, forced_logprobs);
}

/* The RNN head's draft (rnn_state_step above): A [B,K,r] decay gates     */
/* (required), G [B,K,r] input gates or NULL; otherwise as orc_markov_draft. */
int orc_rnn_draft(const float* U, const uint16_t* W1, const uint16_t* W2,
                  const int32_t* anchors, const double* A, const double* G, int B, int K, int V,
                  int r, double temperature, uint64_t seed, int b0, int nb, const int32_t* forced,
                  int32_t* tokens, double* logprobs, double* margins, double* forced_logprobs) {
  if (A == NULL || r <= 0) return -1;
  return run_draft(U, W1, W2, anchors, G, A, B, K, V, r, temperature, seed, b0, nb, forced,
                   tokens, logprobs, margins, forced_logprobs);
}

/* ------------------------------------------------------------------ */
/* Teacher-forced calibrated logits: the Markov-head rule with the      */
/* predecessor of every position given ([EQV] per-candidate form        */
/* logits_k(b | a) = U_k(b) + W1[a]^T W2[:, b]).                        */
/* prev [B, K] holds x_0 .. x_{K-1}.  Rows b0 .. b0+nb-1; outputs       */
/* compact: logits [nb, K, V] fp64, lse [nb, K] = log sum exp(l / T').  */
/* ------------------------------------------------------------------ */
int orc_markov_logits(const float* U, const uint16_t* W1, const uint16_t* W2,
                      const int32_t* prev, const double* H, int B, int K, int V, int r,
                      double temperature, int b0, int nb, double* logits, double* lse) {
  if (B <= 0 || K <= 0 || V <= 0 || r < 0 || b0 < 0 || nb < 0 || b0 + nb > B) return -1;
  double* e = (double*)malloc(sizeof(double) * (size_t)(r > 0 ? r : 1));
  if (!e) return -1;
  const double Tp = temperature > 0.0 ? temperature : 1.0;
  for (int bi = 0; bi < nb; ++bi) {
    const int b = b0 + bi;
    for (int k = 0; k < K; ++k) {
      const int32_t a = prev[(int64_t)b * K + k];
      if (a < 0 || a >= V) {
        free(e);
        return -1;
      }
      double* l = logits + ((int64_t)bi * K + k) * V;
      calibrated_logits(U + ((int64_t)b * K + k) * V, W1, W2,
                        H ? H + ((int64_t)b * K + k) * r : NULL, V, r, a, e, l);
      lse[(int64_t)bi * K + k] = log_sum_exp_scaled(l, V, Tp);
    }
  }
  free(e);
  return 0;
}

/* ------------------------------------------------------------------ */
/* RNN head, teacher-forced: the recurrent state driven by the given   */
/* predecessors prev [B, K] (x_0 .. x_{K-1}); A [B,K,r] decay gates, G  */
/* [B,K,r] input gates or NULL.  Rows b0 .. b0+nb-1; outputs compact    */
/* logits [nb, K, V] fp64, lse [nb, K] = log sum exp(l / T').           */
/* ------------------------------------------------------------------ */
int orc_rnn_logits(const float* U, const uint16_t* W1, const uint16_t* W2, const int32_t* prev,
                   const double* A, const double* G, int B, int K, int V, int r,
                   double temperature, int b0, int nb, double* logits, double* lse) {
  if (B <= 0 || K <= 0 || V <= 0 || r <= 0 || A == NULL || b0 < 0 || nb < 0 || b0 + nb > B)
    return -1;
  double* st = (double*)malloc(sizeof(double) * (size_t)r);
  if (!st) return -1;
  const double Tp = temperature > 0.0 ? temperature : 1.0;
  for (int bi = 0; bi < nb; ++bi) {
    const int b = b0 + bi;
    for (int i = 0; i < r; ++i) st[i] = 0.0;
    for (int k = 0; k < K; ++k) {
      const int32_t a = prev[(int64_t)b * K + k];
      if (a < 0 || a >= V) {
        free(st);
        return -1;
      }
      const int64_t o = (int64_t)b * K + k;
      rnn_state_step(W1, r, a, A + o * r, G ? G + o * r : NULL, st);
      double* l = logits + ((int64_t)bi * K + k) * V;
      bias_logits(U + o * V, W2, st, V, r, l);
      lse[(int64_t)bi * K + k] = log_sum_exp_scaled(l, V, Tp);
    }
  }
  free(st);
  return 0;
}

/* ------------------------------------------------------------------ */
/* Confidence head and prefix survival.                                 */
/* [EXPL] "Confidence-scheduled verification": c_k = sigmoid(w^T [h_k;  */
/* W1[x_{k-1}]]), prefix survival a_j = prod_{i<=j} c_i.  [VLLM]         */
/* "Confidence Head": a linear head on the hidden state, concatenated    */
/* with the previous-token Markov embedding when that option is set.    */
/* A scalar bias is added (0 in the pages' equation).  verify_len[b] is  */
/* the longest prefix whose survival stays >= threshold.                */
/* h [B,K,d], W1 [V,r], anchors [B], tokens [B,K] (x_1..x_K), w [d(+r)]. */
/* Outputs full [B,K] / [B].                                            */
/* ------------------------------------------------------------------ */
int orc_confidence(const uint16_t* h, const uint16_t* W1, const int32_t* anchors,
                   const int32_t* tokens, const uint16_t* w, double bias, int with_markov,
                   int B, int K, int d, int r, int V, double threshold, const double* tau,
                   double* conf, double* cumprod, int32_t* verify_len) {
  if (B <= 0 || K <= 0 || d < 0 || r < 0) return -1;
  int bad = 0;
#pragma omp parallel for schedule(static) reduction(| : bad)
  for (int b = 0; b < B; ++b) {
    double surv = 1.0;
    int len = 0, open = 1;
    for (int k = 0; k < K; ++k) {
      const int32_t prev = (k == 0) ? anchors[b] : tokens[(int64_t)b * K + k - 1];
      double z = bias;
      const uint16_t* hk = h + ((int64_t)b * K + k) * d;
      for (int j = 0; j < d; ++j) z += bf16_to_double(w[j]) * bf16_to_double(hk[j]);
      if (with_markov) {
        if (prev < 0 || prev >= V) {
          bad = 1;
          break;
        }
        for (int i = 0; i < r; ++i)
          z += bf16_to_double(w[d + i]) * bf16_to_double(W1[(int64_t)prev * r + i]);
      }
      const double c = sigmoid(tau ? z / tau[k] : z); /* STS: one temperature per position */
      surv *= c;
      conf[(int64_t)b * K + k] = c;
      cumprod[(int64_t)b * K + k] = surv;
      if (open && surv >= threshold) {
        len = k + 1;
      } else {
        open = 0;
      }
    }
    verify_len[b] = len;
  }
  return bad ? -1 : 0;
}

/* ------------------------------------------------------------------ */
/* Top-k candidate sets of the base logits.                             */
/* [EQV] "Where the parallelism comes from", choice 1: at each position */
/* keep the top-16 tokens under the base logits U; "Two implications",  */
/* 2: the same top-k truncation for a trained DSpark head.               */
/* Order: U descending, ties to the smaller token id.  margin =          */
/* U(k-th) - U((k+1)-th) (+inf when V == k).                             */
/* U [B,K,V] -> cand [B,K,topk] int32, cval [B,K,topk], margin [B,K].    */
/* ------------------------------------------------------------------ */
int orc_topk(const float* U, int B, int K, int V, int topk, int32_t* cand, double* cval,
             double* margin) {
  if (B <= 0 || K <= 0 || V <= 0 || topk <= 0 || topk > V || topk > 64) return -1;
#pragma omp parallel for schedule(dynamic)
  for (int64_t row = 0; row < (int64_t)B * K; ++row) {
    const float* u = U + row * V;
    /* insertion into a sorted list of the topk+1 best (value desc, id asc) */
    int32_t ids[65];
    double vals[65];
    int n = 0, cap = topk + 1;
    for (int v = 0; v < V; ++v) {
      double x = (double)u[v];
      if (n == cap && !(x > vals[n - 1])) continue; /* equal value: larger id loses */
      int p = (n < cap) ? n : cap - 1;
      while (p > 0 && x > vals[p - 1]) {
        if (p < cap) {
          vals[p] = vals[p - 1];
          ids[p] = ids[p - 1];
        }
        --p;
      }
      vals[p] = x;
      ids[p] = v;
      if (n < cap) ++n;
    }
    for (int j = 0; j < topk; ++j) {
      cand[row * topk + j] = ids[j];
      cval[row * topk + j] = vals[j];
    }
    margin[row] = (n > topk) ? vals[topk - 1] - vals[topk] : INFINITY;
  }
  return 0;
}

/* ------------------------------------------------------------------ */
/* Adjacent-pair score tables.                                          */
/* [EQV] "What the two methods do": S_t(a, b) = U_t(b) + <A(a) (.)     */
/* H(h_t), B(b)>; "Where the parallelism comes from", choice 2: all     */
/* k x k predecessor/candidate pairs of adjacent positions.  H == NULL  */
/* is the ungated form (H = 1).  Predecessor set of position 0 is the   */
/* anchor alone; its row is replicated over all k rows.                  */
/* S [B,K,topk,topk] fp64: S[b,t,i,j] = cval[b,t,j] + sum_q             */
/* A[p_i][q] * H[b,t,q] * Bt[c_j][q].                                    */
/* ------------------------------------------------------------------ */
int orc_pair_scores(const int32_t* cand, const double* cval, const uint16_t* A,
                    const uint16_t* Bt, const int32_t* anchors, const double* H, int B, int K,
                    int V, int r, int topk, double* S) {
  if (B <= 0 || K <= 0 || V <= 0 || r < 0 || topk <= 0) return -1;
  int bad = 0;
#pragma omp parallel for schedule(static) reduction(| : bad)
  for (int64_t bt = 0; bt < (int64_t)B * K; ++bt) {
    const int b = (int)(bt / K), t = (int)(bt % K);
    const double* Hrow = H ? H + bt * r : NULL;
    for (int i = 0; i < topk; ++i) {
      const int32_t p = (t == 0) ? anchors[b] : cand[(bt - 1) * topk + i];
      for (int j = 0; j < topk; ++j) {
        const int32_t c = cand[bt * topk + j];
        if (p < 0 || p >= V || c < 0 || c >= V) {
          bad = 1;
          continue;
        }
        double acc = 0.0;
        for (int q = 0; q < r; ++q) {
          double aq = bf16_to_double(A[(int64_t)p * r + q]);
          if (Hrow) aq *= Hrow[q];
          acc += aq * bf16_to_double(Bt[(int64_t)c * r + q]);
        }
        S[(bt * topk + i) * topk + j] = cval[bt * topk + j] + acc;
      }
    }
  }
  return bad ? -1 : 0;
}

/* ------------------------------------------------------------------ */
/* Light sequential walk over the pair tables.                          */
/* [EQV] "Where the parallelism comes from": a greedy walk, or sampling, */
/* over the precomputed scores; "Two implications", 2, step 3.  The     */
/* sampling rule is the Markov head's own restricted to the candidates: */
/* the block race over the candidates' token ids (noise keyed by block  */
/* id), so with k = V the walk is the full head and with k < V it is    */
/* the head with every other token masked; log-probabilities are under  */
/* the k-way softmax.                                                   */
/* cand [B,K,topk], S [B,K,topk,topk] -> compact outputs [nb, K].       */
/* forced ([nb,K], nullable): continue on these tokens (must be in the  */
/* candidate set); forced_logprobs receives their log-probability.      */
/* ------------------------------------------------------------------ */
int orc_walk(const int32_t* cand, const double* S, int B, int K, int topk, double temperature,
             uint64_t seed, int b0, int nb, const int32_t* forced, int32_t* tokens,
             double* logprobs, double* margins, double* forced_logprobs) {
  if (B <= 0 || K <= 0 || topk <= 0 || topk > 64 || b0 < 0 || nb < 0 || b0 + nb > B) return -1;
  const double Tp = temperature > 0.0 ? temperature : 1.0;
  int bad = 0;
#pragma omp parallel for schedule(static) reduction(| : bad)
  for (int bi = 0; bi < nb; ++bi) {
    const int b = b0 + bi;
    int slot = 0; /* predecessor slot; position 0's rows all hold the anchor */
    for (int t = 0; t < K; ++t) {
      const int64_t bt = (int64_t)b * K + t;
      const double* row = S + (bt * topk + slot) * topk;
      const int32_t* c = cand + bt * topk;
      int best = 0;
      double margin = 0.0;
      if (temperature > 0.0) {
        /* the head's block race restricted to the candidates: candidates in
           token-id order, z = S / T (tokens outside the set have mass 0) */
        int ord[64];
        int32_t ids[64];
        double z[64], w[64];
        for (int j = 0; j < topk; ++j) {
          int p = j;
          while (p > 0 && c[ord[p - 1]] > c[j]) {
            ord[p] = ord[p - 1];
            --p;
          }
          ord[p] = j;
        }
        for (int q = 0; q < topk; ++q) {
          ids[q] = c[ord[q]];
          z[q] = row[ord[q]] / temperature;
        }
        const int q = block_race_draw(ids, z, w, topk, seed, (uint32_t)b, (uint32_t)t, 1u, &margin);
        if (q < 0) {
          bad = 1;
          break;
        }
        best = ord[q];
      } else {
        for (int j = 1; j < topk; ++j)
          if (row[j] > row[best] || (row[j] == row[best] && c[j] < c[best])) best = j;
        double second = -INFINITY;
        for (int j = 0; j < topk; ++j)
          if (j != best && row[j] > second) second = row[j];
        margin = row[best] - second;
      }
      double m = -INFINITY;
      for (int j = 0; j < topk; ++j)
        if (row[j] / Tp > m) m = row[j] / Tp;
      double ssum = 0.0;
      for (int j = 0; j < topk; ++j) ssum += exp(row[j] / Tp - m);
      const double lse = m + log(ssum);
      const int64_t o = (int64_t)bi * K + t;
      tokens[o] = c[best];
      logprobs[o] = row[best] / Tp - lse;
      margins[o] = margin;
      int next = best;
      if (forced) {
        next = -1;
        for (int j = 0; j < topk; ++j)
          if (c[j] == forced[o]) next = j;
        if (next < 0) {
          bad = 1;
          break;
        }
        if (forced_logprobs) forced_logprobs[o] = row[next] / Tp - lse;
      }
      slot = next;
    }
  }
  return bad ? -1 : 0;
}

/* ------------------------------------------------------------------ */
/* Speculative verification of a drafted block.                        */
/* [FIX] "Watch the Mass Land Wrong": the target verifies a drafted     */
/* token by accepting it with probability min(1, p/q), and resamples    */
/* when it rejects.  [EXPL] "Confidence-scheduled verification": that   */
/* acceptance probability is 1 - TV(p^d_k, p^t_k); "Hardware-aware      */
/* prefix scheduling": every retained token goes through the target's   */
/* accept-or-correct rule, and truncating the verified prefix changes   */
/* the work, not the output distribution; "Two bottlenecks after you    */
/* already have a parallel drafter": the target adds a bonus token when */
/* the whole draft survives.  Reading (the pages say "resamples"): at   */
/* the first rejection, at position j, the token is drawn from the      */
/* normalised residual max(0, p_j - q_j), which makes the committed     */
/* tokens exactly the target's; when all ell verified tokens survive,   */
/* the bonus is drawn from p_ell.                                       */
/*                                                                    */
/* P [B, K+1, V] fp32 target logits (row k: the target's distribution   */
/* at position k; row K: after a fully accepted block); p_k =           */
/* softmax(P[b,k]/Tt) (Tt = 0: one-hot at the argmax, ties to the       */
/* smaller id).  q_k = the draft's distribution at position k given the */
/* drafted predecessor (x_{-1} = anchor): softmax(l_k/Td) with l_k the  */
/* calibrated logits (gated when H != NULL); Td = 0: one-hot at x_k.    */
/* ell [B] verified positions (NULL: K).  Position k's acceptance       */
/* uniform is orc_accept_uniform(seed, b, k); draws use the block race  */
/* on the verifier's streams (tag 9) at the position drawn for.         */
/* Outputs (compact [nb]): n_acc = accepted prefix length, next_token,  */
/* accept_prob [nb, K] = min(1, p_k(x_k)/q_k(x_k)) for k < ell (else    */
/* -1), margins [nb] = the smallest decision margin (|u - a| of every  */
/* acceptance test, and the draw's margin).                            */
/* ------------------------------------------------------------------ */
static void target_probs(const float* Prow, int V, double Tt, double* pv) {
  if (Tt > 0.0) {
    double m = -INFINITY;
    for (int v = 0; v < V; ++v)
      if ((double)Prow[v] / Tt > m) m = (double)Prow[v] / Tt;
    double sum = 0.0;
    for (int v = 0; v < V; ++v) sum += exp((double)Prow[v] / Tt - m);
    for (int v = 0; v < V; ++v) pv[v] = exp((double)Prow[v] / Tt - m) / sum;
  } else {
    int best = 0;
    for (int v = 1; v < V; ++v)
      if (Prow[v] > Prow[best]) best = v;
    for (int v = 0; v < V; ++v) pv[v] = (v == best) ? 1.0 : 0.0;
  }
}

static void draft_probs(const double* l, int V, double Td, int32_t x, double* qv) {
  if (Td > 0.0) {
    const double lse = log_sum_exp_scaled(l, V, Td);
    for (int v = 0; v < V; ++v) qv[v] = exp(l[v] / Td - lse);
  } else {
    for (int v = 0; v < V; ++v) qv[v] = (v == x) ? 1.0 : 0.0;
  }
}

int orc_verify(const float* P, const float* U, const uint16_t* W1, const uint16_t* W2,
               const int32_t* anchors, const double* H, const int32_t* tokens,
               const int32_t* ell, int B, int K, int V, int r, double Td, double Tt,
               uint64_t seed, int b0, int nb, int32_t* n_acc, int32_t* next_token,
               double* accept_prob, double* margins) {
  if (B <= 0 || K <= 0 || V <= 0 || r < 0 || b0 < 0 || nb < 0 || b0 + nb > B) return -1;
  double* l = (double*)malloc(sizeof(double) * (size_t)V);
  double* pv = (double*)malloc(sizeof(double) * (size_t)V);
  double* qv = (double*)malloc(sizeof(double) * (size_t)V);
  double* z = (double*)malloc(sizeof(double) * (size_t)V);
  double* w = (double*)malloc(sizeof(double) * (size_t)V);
  double* e = (double*)malloc(sizeof(double) * (size_t)(r > 0 ? r : 1));
  int bad = (!l || !pv || !qv || !z || !w || !e);
  for (int bi = 0; bi < nb && !bad; ++bi) {
    const int b = b0 + bi;
    const int L = ell ? ell[b] : K;
    if (L < 0 || L > K) {
      bad = 1;
      break;
    }
    double margin = INFINITY;
    int32_t prev = anchors[b];
    int n = 0, pos = L, rejected = 0;
    for (int k = 0; k < K; ++k) accept_prob[(int64_t)bi * K + k] = -1.0;
    for (int k = 0; k < L; ++k) {
      const int32_t x = tokens[(int64_t)b * K + k];
      if (prev < 0 || prev >= V || x < 0 || x >= V) {
        bad = 1;
        break;
      }
      calibrated_logits(U + ((int64_t)b * K + k) * V, W1, W2,
                        H ? H + ((int64_t)b * K + k) * r : NULL, V, r, prev, e, l);
      target_probs(P + ((int64_t)b * (K + 1) + k) * V, V, Tt, pv);
      draft_probs(l, V, Td, x, qv);
      const double a = (qv[x] > 0.0) ? fmin(1.0, pv[x] / qv[x]) : 1.0;
      accept_prob[(int64_t)bi * K + k] = a;
      const double u = orc_accept_uniform(seed, (uint32_t)b, (uint32_t)k);
      margin = fmin(margin, fabs(u - a));
      if (u < a) {
        ++n;
        prev = x;
        continue;
      }
      /* rejected: the residual max(0, p - q), as log-weights for the race */
      for (int v = 0; v < V; ++v) {
        const double d = pv[v] - qv[v];
        z[v] = d > 0.0 ? log(d) : -INFINITY;
      }
      pos = k;
      rejected = 1;
      break;
    }
    if (bad) break;
    if (!rejected) {
      /* bonus: the target's own draw at position ell */
      target_probs(P + ((int64_t)b * (K + 1) + L) * V, V, Tt, pv);
      for (int v = 0; v < V; ++v) z[v] = pv[v] > 0.0 ? log(pv[v]) : -INFINITY;
    }
    double dm = 0.0;
    const int y = block_race_draw(NULL, z, w, V, seed, (uint32_t)b, (uint32_t)pos, 9u, &dm);
    if (y < 0) {
      bad = 1;
      break;
    }
    n_acc[bi] = n;
    next_token[bi] = y;
    margins[bi] = fmin(margin, dm);
  }
  free(l);
  free(pv);
  free(qv);
  free(z);
  free(w);
  free(e);
  return bad ? -1 : 0;
}

/* ------------------------------------------------------------------ */
/* Load-aware prefix scheduler.                                         */
/* [EXPL] "Hardware-aware prefix scheduling": R requests, request r may  */
/* verify a prefix of length ell_r; the target batch is B = sum_r (1 +   */
/* ell_r) tokens; with survival a_{r,j} of extension (r, j) the          */
/* objective is Theta(S) = (R + sum_{(r,j) in S} a_{r,j}) SPS(B).  The    */
/* greedy: start at B = R, rank the candidate extensions globally by     */
/* survival probability, admit them while Theta increases and stop when  */
/* admitting the next one would not increase it; request r cannot admit  */
/* position j+1 without j.  Readings: candidates are ranked by (a desc,  */
/* position asc, request asc) -- a_{r,j} = prod_{i<=j} c_{r,i} never     */
/* increases along a request, so this order keeps every prefix whole;   */
/* "increases" is strict.                                                */
/* a [R, K] (position k = 0..K-1 is extension k of request r),          */
/* sps [R * (K + 1) + 1] = SPS(B) for B = 0 .. R (K + 1).               */
/* Outputs ell [R] and *theta = Theta of the admitted set; margin =     */
/* the smallest relative gap |Theta_next - Theta| / Theta over every    */
/* admission test made (the stopping one included).                     */
/* ------------------------------------------------------------------ */
typedef struct {
  double a;
  int k, r;
} sched_cand;

static int sched_before(const sched_cand* x, const sched_cand* y) {
  if (x->a != y->a) return x->a > y->a;
  if (x->k != y->k) return x->k < y->k;
  return x->r < y->r;
}

int orc_schedule(const double* a, int R, int K, const double* sps, int32_t* ell, double* theta,
                 double* margin) {
  if (R <= 0 || K < 0) return -1;
  const int n = R * K;
  sched_cand* c = (sched_cand*)malloc(sizeof(sched_cand) * (size_t)(n > 0 ? n : 1));
  if (!c) return -1;
  for (int r = 0; r < R; ++r)
    for (int k = 0; k < K; ++k) {
      c[r * K + k].a = a[(int64_t)r * K + k];
      c[r * K + k].k = k;
      c[r * K + k].r = r;
    }
  /* insertion sort: plain and obviously ordered */
  for (int i = 1; i < n; ++i) {
    sched_cand x = c[i];
    int p = i;
    while (p > 0 && sched_before(&x, &c[p - 1])) {
      c[p] = c[p - 1];
      --p;
    }
    c[p] = x;
  }
  for (int r = 0; r < R; ++r) ell[r] = 0;
  double sum = (double)R;
  double th = sum * sps[R];
  *margin = INFINITY;
  for (int i = 0; i < n; ++i) {
    const double next = (sum + c[i].a) * sps[R + i + 1];
    *margin = fmin(*margin, fabs(next - th) / (th > 0.0 ? th : 1.0));
    if (!(next > th)) break;
    sum += c[i].a;
    th = next;
    ell[c[i].r] += 1;
  }
  *theta = th;
  free(c);
  return 0;
}

/* ------------------------------------------------------------------ */
/* Acceptance label of each drafted position.                          */
/* [EXPL] "Confidence-scheduled verification": the confidence head's    */
/* training label is c*_k = 1 - TV(p^d_k, p^t_k) = 1 - 1/2 ||p^d_k -     */
/* p^t_k||_1, the per-step acceptance probability under speculative     */
/* decoding.  p^d_k: the draft head's softmax at position k given the   */
/* drafted predecessor (one-hot at x_k when drafted greedily, Td = 0);  */
/* p^t_k = softmax(P[b,k] / Tt) (one-hot at the argmax when Tt = 0).    */
/* Computed as sum_v min(p^d_k(v), p^t_k(v)), which equals 1 - TV.     */
/* P [B, K+1, V] (row K unused), tokens [B, K] -> label [B, K] (full).  */
/* ------------------------------------------------------------------ */
int orc_accept_label(const float* P, const float* U, const uint16_t* W1, const uint16_t* W2,
                     const int32_t* anchors, const double* H, const int32_t* tokens, int B, int K,
                     int V, int r, double Td, double Tt, double* label) {
  if (B <= 0 || K <= 0 || V <= 0 || r < 0) return -1;
  double* l = (double*)malloc(sizeof(double) * (size_t)V);
  double* pv = (double*)malloc(sizeof(double) * (size_t)V);
  double* qv = (double*)malloc(sizeof(double) * (size_t)V);
  double* e = (double*)malloc(sizeof(double) * (size_t)(r > 0 ? r : 1));
  int bad = (!l || !pv || !qv || !e);
  for (int b = 0; b < B && !bad; ++b) {
    int32_t prev = anchors[b];
    for (int k = 0; k < K; ++k) {
      const int32_t x = tokens[(int64_t)b * K + k];
      if (prev < 0 || prev >= V || x < 0 || x >= V) {
        bad = 1;
        break;
      }
      calibrated_logits(U + ((int64_t)b * K + k) * V, W1, W2,
                        H ? H + ((int64_t)b * K + k) * r : NULL, V, r, prev, e, l);
      target_probs(P + ((int64_t)b * (K + 1) + k) * V, V, Tt, pv);
      draft_probs(l, V, Td, x, qv);
      double s = 0.0;
      for (int v = 0; v < V; ++v) s += fmin(pv[v], qv[v]);
      label[(int64_t)b * K + k] = s;
      prev = x;
    }
  }
  free(l);
  free(pv);
  free(qv);
  free(e);
  return bad ? -1 : 0;
}

/* ------------------------------------------------------------------ */
/* Sequential temperature scaling (STS) of the confidence head.         */
/* [EXPL] "Confidence-scheduled verification": the raw head is          */
/* calibrated with one temperature per position, fitted left to right   */
/* against cumulative prefix-survival probabilities, which keeps the    */
/* ranking.  Reading: the calibrated confidence is c_k = sigmoid(z_k /   */
/* tau_k), z_k the head's logit; tau_k minimises, over the N             */
/* calibration rows, the binary cross-entropy between the model's        */
/* prefix survival a_k = prod_{i<=k} sigmoid(z_i / tau_i) (tau_0 ..      */
/* tau_{k-1} already fitted) and the target survival                     */
/* y_k = prod_{i<=k} label_i (acceptance labels c*_i, or 0/1 outcomes).  */
/* z_k = ln(c_k / (1 - c_k)) of the raw confidence clamped to            */
/* [2^-24, 1 - 2^-24]; the survival inside the cross-entropy is clamped  */
/* to [1e-7, 1 - 1e-7].  The 1-D minimisation over x = ln tau in         */
/* [ln lo, ln hi]: STS_G evenly spaced points, keep the best (ties to     */
/* the smaller), narrow to the interval between its neighbours, STS_R    */
/* rounds.                                                                */
/* conf, label [N, K] fp32 -> tau [K], loss [K] (mean cross-entropy).    */
/* ------------------------------------------------------------------ */
#define STS_G 32
#define STS_R 8

static double sts_loss(const double* z, const double* a, const double* y, int N, double inv_tau) {
  double L = 0.0;
  for (int n = 0; n < N; ++n) {
    double q = a[n] * sigmoid(z[n] * inv_tau);
    if (q < 1e-7) q = 1e-7;
    if (q > 1.0 - 1e-7) q = 1.0 - 1e-7;
    L -= y[n] * log(q) + (1.0 - y[n]) * log1p(-q);
  }
  return L;
}

int orc_sts_fit(const float* conf, const float* label, int N, int K, double lo, double hi,
                double* tau, double* loss) {
  if (N <= 0 || K <= 0 || !(lo > 0.0) || !(hi > lo)) return -1;
  double* z = (double*)malloc(sizeof(double) * (size_t)N);
  double* a = (double*)malloc(sizeof(double) * (size_t)N);
  double* y = (double*)malloc(sizeof(double) * (size_t)N);
  if (!z || !a || !y) {
    free(z);
    free(a);
    free(y);
    return -1;
  }
  for (int n = 0; n < N; ++n) a[n] = y[n] = 1.0;
  const double cmin = 1.0 / 16777216.0;
  for (int k = 0; k < K; ++k) {
    for (int n = 0; n < N; ++n) {
      double c = conf[(int64_t)n * K + k];
      if (c < cmin) c = cmin;
      if (c > 1.0 - cmin) c = 1.0 - cmin;
      z[n] = log(c / (1.0 - c));
      y[n] *= (double)label[(int64_t)n * K + k];
    }
    double x0 = log(lo), x1 = log(hi), xb = x0, Lb = 0.0;
    for (int round = 0; round < STS_R; ++round) {
      int best = -1;
      const double step = (x1 - x0) / (STS_G - 1);
      for (int g = 0; g < STS_G; ++g) {
        const double x = x0 + step * g;
        const double L = sts_loss(z, a, y, N, exp(-x));
        if (best < 0 || L < Lb) {
          best = g;
          Lb = L;
          xb = x;
        }
      }
      const double nx0 = x0 + step * (best > 0 ? best - 1 : 0);
      const double nx1 = x0 + step * (best < STS_G - 1 ? best + 1 : STS_G - 1);
      x0 = nx0;
      x1 = nx1;
    }
    tau[k] = exp(xb);
    if (loss) loss[k] = Lb / N;
    for (int n = 0; n < N; ++n) a[n] *= sigmoid(z[n] / tau[k]);
  }
  free(z);
  free(a);
  free(y);
  return 0;
}
