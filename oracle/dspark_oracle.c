/*
 * dspark_oracle.c -- the plain, slow, double-precision CPU oracle of the DSpark
 * per-round hot path.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the independent checker against which
 * the CUDA library is compared.  It shares no code, header, table or helper with
 * the CUDA path; only tests, the smoke check and the bench's CPU-baseline leg
 * load it.  Nothing in the product path may call it.
 *
 * Every function follows the plain definition of what it computes: naive loops
 * over the vocabulary, double accumulation, no pruning, no online tricks, no
 * blocking.  Citations name the web page and the section / equation they follow:
 *
 *   [blog]   "[DeepSeek-6] DSpark: From Draft Models to Serving-Aware Speculative
 *             Decoding" (xutianle.me), sections 1-7.
 *   [digest] "DSpark ... 10 key concepts" digest (aimsg.uk), items 2, 8, 9.
 *   [report] "DSpark: Confidence-Scheduled Speculative Decoding with
 *             Semi-Autoregressive Generation -- study report" (devpress.csdn),
 *             Key formulas: Eq.4, Eq.7, Eq.8 and the throughput objective.
 *
 * Readings of passages the pages leave open are stated where they are used.
 *
 * Parity pins (all in tests/test_oracle_*.py, CPU only):
 *   philox      -- published known-answer vectors + uniformity tests
 *   draft       -- the Markov-bias-free special case draws every position
 *                  independently from softmax(U_k) (chi-square on V = 5); the law
 *                  of a planted chain; p and lse of a one-hot construction
 *                  (W1 = I, so the bias is log A[prev, v]: a transposed W2 fails
 *                  it); uniform logits give p = 1/V; the two-level draw restated
 *                  from raw words
 *   confidence  -- closed form on hand-made cases; w = 0 gives 1/2; T -> inf gives 1/2
 *   schedule    -- exhaustive search over all verify lengths on tiny batches;
 *                  closed-form SPS cases
 *   verify      -- exact output law by enumeration at V = 8, gamma <= 3; Monte-Carlo
 *                  chi-square; Eq.8 identity for the first-position acceptance rate
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORACLE_OK 0
#define ORACLE_ERR_INVALID 1
#define ORACLE_ERR_NOMEM 2

/* Records an error from inside a parallel request loop. */
static void set_status(int* status, int value) {
#ifdef _OPENMP
#pragma omp critical(oracle_status)
#endif
  *status = value;
}

/* ------------------------------------------------------------------------- */
/* Counter-based generator: Philox4x32 with 10 rounds.                        */
/* J. K. Salmon, M. A. Moraes, R. O. Dror, D. E. Shaw, "Parallel Random       */
/* Numbers: As Easy as 1, 2, 3", SC'11, section 3 (the Philox S-box and its   */
/* 4x32 multipliers / Weyl key schedule).                                     */
/* ------------------------------------------------------------------------- */

void oracle_philox4x32_10(const uint32_t ctr_in[4], const uint32_t key_in[2],
                          uint32_t out[4]) {
  uint32_t x0 = ctr_in[0], x1 = ctr_in[1], x2 = ctr_in[2], x3 = ctr_in[3];
  uint32_t k0 = key_in[0], k1 = key_in[1];
  for (int round = 0; round < 10; ++round) {
    /* two 32x32 -> 64 bit products give the "hi" and "lo" halves */
    uint64_t prod_a = (uint64_t)0xD2511F53u * (uint64_t)x0;
    uint64_t prod_b = (uint64_t)0xCD9E8D57u * (uint64_t)x2;
    uint32_t hi_a = (uint32_t)(prod_a >> 32), lo_a = (uint32_t)prod_a;
    uint32_t hi_b = (uint32_t)(prod_b >> 32), lo_b = (uint32_t)prod_b;
    uint32_t y0 = hi_b ^ x1 ^ k0;
    uint32_t y1 = lo_b;
    uint32_t y2 = hi_a ^ x3 ^ k1;
    uint32_t y3 = lo_a;
    x0 = y0; x1 = y1; x2 = y2; x3 = y3;
    /* Weyl sequence key schedule: golden ratio and sqrt(3)-1 */
    k0 += 0x9E3779B9u;
    k1 += 0xBB67AE85u;
  }
  out[0] = x0; out[1] = x1; out[2] = x2; out[3] = x3;
}

/* One 32-bit word of Philox4x32-10 for key (seed mod 2^32, seed div 2^32) and
 * counter (c0, position k, request index, (round << 3) | stream). */
uint32_t oracle_philox_word(uint64_t seed, uint64_t round, uint32_t stream,
                            uint32_t req, uint32_t k, uint32_t c0, uint32_t word) {
  uint32_t ctr[4], key[2], out[4];
  ctr[0] = c0;
  ctr[1] = k;
  ctr[2] = req;
  ctr[3] = (uint32_t)((round << 3) | (uint64_t)(stream & 7u));
  key[0] = (uint32_t)(seed & 0xffffffffu);
  key[1] = (uint32_t)(seed >> 32);
  oracle_philox4x32_10(ctr, key, out);
  return out[word & 3u];
}

/* The random numbers of this library (a choice of this implementation: the
 * pages do not say how tokens are sampled).
 *
 * Word v of a stream: counter (v div 4, k, request, round<<3 | stream), word
 * v mod 4.  The accept uniform of position k (stream 1) uses word 0.  The
 * two-level draws (oracle_block_draw) use word j of stream s for block j's
 * Gumbel noise and word j of stream s + 4 for the entry inside the winning
 * block: s = 0 for the draft, 2 for the residual, 3 for the bonus token. */
uint32_t oracle_rng_word(uint64_t seed, uint64_t round, uint32_t stream,
                         uint32_t req, uint32_t k, uint32_t v) {
  return oracle_philox_word(seed, round, stream, req, k, v >> 2, v & 3u);
}

/* Uniform in the open interval (0, 1) from 23 bits m: (2m + 1) / 2^24.
 * Smallest 2^-24, largest 1 - 2^-24. */
double oracle_u01_bits(uint32_t m) {
  return ((double)(m & 0x7fffffu) + 0.5) * (1.0 / 8388608.0);
}

/* The accept uniform from a whole word: its top 23 bits. */
double oracle_u01(uint32_t w) { return oracle_u01_bits(w >> 9); }

/* Standard Gumbel variate by inversion of its CDF exp(-exp(-g)). */
double oracle_gumbel_from_bits(uint32_t m) {
  double u = oracle_u01_bits(m);
  return -log(-log(u));
}

/* ------------------------------------------------------------------------- */
/* Small helpers: element access for fp32 / bf16 storage.                     */
/* ------------------------------------------------------------------------- */

static double load_elem(const void* base, int dtype, size_t idx) {
  if (dtype == 0) return (double)((const float*)base)[idx];
  uint32_t bits = ((uint32_t)((const uint16_t*)base)[idx]) << 16;
  float f;
  memcpy(&f, &bits, sizeof f);
  return (double)f;
}

/* ------------------------------------------------------------------------- */
/* Building blocks                                                            */
/* ------------------------------------------------------------------------- */

/* Markov transition bias ([blog] section 4; [report] Eq.4):
 * B_k(v) = sum_i W1[prev, i] * W2[v, i].
 * W1 is the [V, r] embedding looked up by the previous token; W2 is the weight of
 * the bias-free linear layer r -> V, stored as a linear layer stores it, [V, r].
 * The fused draft logit of position k is l(v) = U_k(v) + B_k(v). */
void oracle_draft_logits(int V, int r, const float* U_row, const void* W1,
                         const void* W2, int wdt, int prev, double* l_out) {
  for (int v = 0; v < V; ++v) {
    double acc = 0.0;
    for (int i = 0; i < r; ++i)
      acc += load_elem(W1, wdt, (size_t)prev * r + i) *
             load_elem(W2, wdt, (size_t)v * r + i);
    l_out[v] = (double)U_row[v] + acc;
  }
}

/* log sum_v exp(l(v)), by the max-shifted two-pass definition. */
double oracle_logsumexp(int V, const double* l) {
  double m = -INFINITY;
  for (int v = 0; v < V; ++v)
    if (l[v] > m) m = l[v];
  double s = 0.0;
  for (int v = 0; v < V; ++v) s += exp(l[v] - m);
  return m + log(s);
}

/* p(v) = exp(l(v) - logsumexp(l)): the ordinary softmax ([blog] section 4). */
void oracle_softmax(int V, const double* l, double* p_out) {
  double lse = oracle_logsumexp(V, l);
  for (int v = 0; v < V; ++v) p_out[v] = exp(l[v] - lse);
}

/* The sampler of every draw (draft, residual, bonus): an exact draw from
 * non-negative weights w(v) in two levels.
 *
 * The entries are cut into blocks of 4 consecutive ones, block j holding
 * v = 4j .. 4j+3 (the last block may be shorter), with weight W_j = the sum of
 * its w(v).  A Gumbel-max over the blocks picks j* = argmax_j log W_j + G_j
 * (ties to the smallest j; blocks with W_j = 0 never win), where
 * G_j = -log(-log u_j) and u_j = ((w >> 9) + 1/2) / 2^23 from the word
 * w = word (j mod 4) of Philox call j / 4 of `stream`.  Inside j* the entry is
 * drawn by inverse CDF with u' from word (j* mod 4) of call j* / 4 of
 * stream + 4 (same map to (0, 1)): the first v of j* whose cumulative weight
 * exceeds u' times W_j*.  The block wins with probability W_j / sum W, the
 * entry then with w(v) / W_j: v is drawn with probability w(v) / sum w.
 * logscale is added to every log W_j (so that weights exp(l - m) race as
 * log sum exp l); it changes no decision, only the reported scores.
 * *margin is the smaller of the top-two gap of log W_j + G_j and the distance
 * of u' from the nearest inner boundary of the block's CDF (as a fraction of
 * W_j*).  Returns -1 when every weight is 0. */
int oracle_block_draw(int V, const double* w, double logscale, uint64_t seed,
                      uint64_t round, uint32_t stream, uint32_t req, uint32_t k,
                      double* margin) {
  double best = -INFINITY, second = -INFINITY;
  int jb = -1;
  for (int j = 0; 4 * j < V; ++j) {
    double s = 0.0;
    for (int v = 4 * j; v < V && v < 4 * j + 4; ++v) s += w[v];
    if (s <= 0.0) continue;
    uint32_t word = oracle_philox_word(seed, round, stream, req, k,
                                       (uint32_t)j >> 2, (uint32_t)j & 3u);
    double z = logscale + log(s) + oracle_gumbel_from_bits(word >> 9);
    if (z > best) {
      second = best;
      best = z;
      jb = j;
    } else if (z > second) {
      second = z;
    }
  }
  if (jb < 0) {
    if (margin) *margin = 0.0;
    return -1;
  }
  uint32_t wp = oracle_philox_word(seed, round, stream + 4u, req, k,
                                   (uint32_t)jb >> 2, (uint32_t)jb & 3u);
  double u = oracle_u01(wp);
  int v0 = 4 * jb, v1 = (4 * jb + 4 < V) ? 4 * jb + 4 : V;
  double S = 0.0;
  int last = -1;
  for (int v = v0; v < v1; ++v) {
    S += w[v];
    if (w[v] > 0.0) last = v;
  }
  double target = u * S, cum = 0.0, dmin = INFINITY;
  int x = -1;
  for (int v = v0; v < v1; ++v) {
    if (!(w[v] > 0.0)) continue;
    cum += w[v];
    if (x < 0 && target < cum) x = v;
    if (v != last) {
      double d = fabs(u - cum / S);
      if (d < dmin) dmin = d;
    }
  }
  if (x < 0) x = last;
  if (margin) *margin = fmin(best - second, dmin);
  return x;
}

/* A draw from softmax(score) (entries with score = -inf excluded) by
 * oracle_block_draw on the weights exp(score - max).  Returns -1 when every
 * score is -inf. */
int oracle_softmax_draw(int V, const double* score, uint64_t seed,
                        uint64_t round, uint32_t stream, uint32_t req,
                        uint32_t k, double* margin) {
  double m = -INFINITY;
  for (int v = 0; v < V; ++v)
    if (score[v] > m) m = score[v];
  if (m == -INFINITY) {
    if (margin) *margin = 0.0;
    return -1;
  }
  double* w = (double*)malloc(sizeof(double) * (size_t)V);
  if (!w) return -1;
  for (int v = 0; v < V; ++v) w[v] = exp(score[v] - m);
  int x = oracle_block_draw(V, w, m, seed, round, stream, req, k, margin);
  free(w);
  return x;
}

/* The draft's draw of x_k from softmax(l): streams 0 (blocks) and 4 (entry). */
int oracle_block_sample(int V, const double* l, uint64_t seed, uint64_t round,
                        uint32_t req, uint32_t k, double* margin) {
  return oracle_softmax_draw(V, l, seed, round, 0u, req, k, margin);
}

/* Residual of rejection sampling ([digest] item 2: resample at the first
 * divergence): rho(v) = max(0, p_t(v) - p_d(v)), unnormalised. */
void oracle_residual(int V, const double* p_t, const double* p_d, double* rho) {
  for (int v = 0; v < V; ++v) {
    double d = p_t[v] - p_d[v];
    rho[v] = d > 0.0 ? d : 0.0;
  }
}

/* Analytic acceptance label ([report] Eq.8; [blog] section 5):
 * c* = 1 - 0.5 * || p_d - p_t ||_1 . */
double oracle_acceptance_label(int V, const double* p_d, const double* p_t) {
  double l1 = 0.0;
  for (int v = 0; v < V; ++v) l1 += fabs(p_d[v] - p_t[v]);
  return 1.0 - 0.5 * l1;
}

/* The draft distribution of position k given the previous token. */
void oracle_draft_probs(int V, int r, const float* U_row, const void* W1,
                        const void* W2, int wdt, int prev, double* p_out) {
  oracle_draft_logits(V, r, U_row, W1, W2, wdt, prev, p_out);
  /* in place: logits -> probabilities */
  double lse = oracle_logsumexp(V, p_out);
  for (int v = 0; v < V; ++v) p_out[v] = exp(p_out[v] - lse);
}

/* ------------------------------------------------------------------------- */
/* The gated recurrent Markov head.  [blog] section 4 and [digest] item 8 name
 * a gated Markov head and an RNN head that keeps a state through the draft
 * block; neither page gives their equations.  This is the plainest head with
 * that description, and it keeps the Markov head's projection:
 *
 *   e_k = W1[x_{k-1}],   a_k = sigmoid(g .* e_k + c)   (g, c in R^r),
 *   s_0 = 0,             s_k = e_k + a_k .* s_{k-1},
 *   B_k(v) = sum_i s_k[i] * W2[v, i],
 *
 * so p_k(v) ~ exp(U_k(v) + B_k(v)) depends on the whole prefix x_0..x_{k-1}
 * ([report] Eq.4's B_k(x_0, x_<k, v)).  With a_k = 0 it is the Markov head.  */
/* ------------------------------------------------------------------------- */

/* x rounded to the nearest bf16 value (ties to even), by its float's bits. */
static double round_bf16(double x) {
  float f = (float)x;
  uint32_t u;
  memcpy(&u, &f, sizeof u);
  if ((u & 0x7f800000u) != 0x7f800000u) u = (u + 0x7fffu + ((u >> 16) & 1u)) & 0xffff0000u;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

/* s <- e + a .* s for the previous token prev (one step of the recurrence).
 * bf16_state: the new state is rounded to bf16 (the precision a tensor-core
 * operand holds it in); 0 keeps the exact definition. */
static void gated_step(int r, const void* W1, int wdt, const float* g,
                       const float* c, int prev, int bf16_state, double* s) {
  for (int i = 0; i < r; ++i) {
    const double e = load_elem(W1, wdt, (size_t)prev * r + i);
    const double a = 1.0 / (1.0 + exp(-((double)g[i] * e + (double)c[i])));
    s[i] = e + a * s[i];
    if (bf16_state) s[i] = round_bf16(s[i]);
  }
}

/* l(v) = U_row(v) + sum_i s[i] * W2[v, i]. */
static void state_logits(int V, int r, const float* U_row, const double* s,
                         const void* W2, int wdt, double* l_out) {
  for (int v = 0; v < V; ++v) {
    double acc = 0.0;
    for (int i = 0; i < r; ++i) acc += s[i] * load_elem(W2, wdt, (size_t)v * r + i);
    l_out[v] = (double)U_row[v] + acc;
  }
}

/* The states s_1..s_G of one request ([G][r]) for the prefix anchor, x[0..G-2]
 * (bf16_state: each rounded to bf16 as it is formed). */
int oracle_gated_states(int G, int V, int r, const void* W1, int wdt,
                        const float* g, const float* c, int anchor,
                        const int32_t* x, int bf16_state, double* s_out) {
  if (G <= 0 || V <= 0 || r <= 0 || !W1 || !g || !c || !s_out || (G > 1 && !x))
    return ORACLE_ERR_INVALID;
  double* s = (double*)calloc((size_t)r, sizeof(double));
  if (!s) return ORACLE_ERR_NOMEM;
  int status = ORACLE_OK;
  for (int k = 1; k <= G; ++k) {
    const int prev = (k == 1) ? anchor : x[k - 2];
    if (prev < 0 || prev >= V) {
      status = ORACLE_ERR_INVALID;
      break;
    }
    gated_step(r, W1, wdt, g, c, prev, bf16_state, s);
    memcpy(s_out + (size_t)(k - 1) * r, s, sizeof(double) * (size_t)r);
  }
  free(s);
  return status;
}

/* ------------------------------------------------------------------------- */
/* Step 1: semi-autoregressive Markov draft ([report] Eq.4; [blog] sections 3-4)
 *
 *   P(X | x0) = prod_k p_k(x_k | x0, x_<k),  p_k(v) ~ exp(U_k(v) + B_k(v)),
 *
 * with x0 the anchor token ([blog] section 3: the anchor is the first predicted
 * position's input).  For k = 1..gamma and every request b in [b0, b1):
 *   l = U[b, k-1, :] + B_k(x_{k-1});   lse = log sum exp l;
 *   x_k = the two-level softmax draw of oracle_block_sample (streams 0 and 4);
 *   p_k(x_k) = exp(l(x_k) - lse).
 * When x_force is given, the previous token of step k >= 2 is taken from it
 * (teacher forcing: each step is checked on the other side's upstream token);
 * otherwise from this oracle's own sample. */
/* (gate_g, gate_c non-NULL: the gated recurrent head, its state carried
 * along the prefix; NULL: the Markov head) */
static int draft_impl(int B, int G, int V, int r, const float* U, const void* W1,
                      const void* W2, int wdt, const float* gate_g,
                      const float* gate_c, int bf16_state, const int32_t* anchor,
                      const int32_t* x_force, uint64_t seed, uint64_t round,
                      int b0, int b1, int32_t* x_out, double* p_out,
                      double* lse_out, double* margin_out) {
  if (B <= 0 || G <= 0 || V <= 0 || r <= 0 || !U || !W1 || !W2 || !anchor ||
      !x_out || b0 < 0 || b1 > B || b0 > b1 || (wdt != 0 && wdt != 1) ||
      (!gate_g) != (!gate_c))
    return ORACLE_ERR_INVALID;
  int status = ORACLE_OK;
#pragma omp parallel for schedule(dynamic, 1)
  for (int b = b0; b < b1; ++b) {
    double* l = (double*)malloc(sizeof(double) * (size_t)V);
    double* s = (double*)calloc((size_t)r, sizeof(double));
    if (!l || !s) {
      set_status(&status, ORACLE_ERR_NOMEM);
      free(l);
      free(s);
      continue;
    }
    int prev = anchor[b];
    for (int k = 1; k <= G; ++k) {
      if (k > 1) prev = x_force ? x_force[(size_t)b * G + k - 2]
                                : x_out[(size_t)b * G + k - 2];
      if (prev < 0 || prev >= V) {
        set_status(&status, ORACLE_ERR_INVALID);
        break;
      }
      const float* U_row = U + ((size_t)b * G + (k - 1)) * (size_t)V;
      if (gate_g) {
        gated_step(r, W1, wdt, gate_g, gate_c, prev, bf16_state, s);
        state_logits(V, r, U_row, s, W2, wdt, l);
      } else {
        oracle_draft_logits(V, r, U_row, W1, W2, wdt, prev, l);
      }
      double lse = oracle_logsumexp(V, l);
      double margin = 0.0;
      int xk = oracle_block_sample(V, l, seed, round, (uint32_t)b, (uint32_t)k,
                                   &margin);
      size_t o = (size_t)b * G + (k - 1);
      x_out[o] = xk;
      if (p_out) p_out[o] = exp(l[xk] - lse);
      if (lse_out) lse_out[o] = lse;
      if (margin_out) margin_out[o] = margin;
    }
    free(l);
    free(s);
  }
  return status;
}

int oracle_draft(int B, int G, int V, int r, const float* U, const void* W1,
                 const void* W2, int wdt, const int32_t* anchor,
                 const int32_t* x_force, uint64_t seed, uint64_t round, int b0,
                 int b1, int32_t* x_out, double* p_out, double* lse_out,
                 double* margin_out) {
  return draft_impl(B, G, V, r, U, W1, W2, wdt, NULL, NULL, 0, anchor, x_force, seed,
                    round, b0, b1, x_out, p_out, lse_out, margin_out);
}

/* The draft with the gated recurrent head (gate_g, gate_c [r]; bf16_state as
 * for oracle_gated_states). */
int oracle_gated_draft(int B, int G, int V, int r, const float* U, const void* W1,
                       const void* W2, int wdt, const float* gate_g,
                       const float* gate_c, int bf16_state, const int32_t* anchor,
                       const int32_t* x_force, uint64_t seed, uint64_t round,
                       int b0, int b1, int32_t* x_out, double* p_out,
                       double* lse_out, double* margin_out) {
  if (!gate_g || !gate_c) return ORACLE_ERR_INVALID;
  return draft_impl(B, G, V, r, U, W1, W2, wdt, gate_g, gate_c, bf16_state, anchor,
                    x_force, seed, round, b0, b1, x_out, p_out, lse_out, margin_out);
}

/* ------------------------------------------------------------------------- */
/* Step 2: confidence head ([report] Eq.7; [blog] section 5)
 *
 *   c_k = sigma( w^T [h_k ; W1[x_{k-1}]] / T_k ),
 *
 * with x_0 the anchor.  T_k is the Sequential-Temperature-Scaling temperature of
 * position k ([blog] section 5); it is 1 when sts_T is NULL.  No bias term:
 * Eq.7 shows none. */
int oracle_confidence(int B, int G, int H, int r, const void* h, int hdt,
                      const void* W1, int wdt, const float* w,
                      const float* sts_T, const int32_t* anchor,
                      const int32_t* x, int V, double* c_out) {
  if (B <= 0 || G <= 0 || H < 0 || r <= 0 || (H > 0 && !h) || !W1 || !w ||
      !anchor || !x || !c_out)
    return ORACLE_ERR_INVALID;
  for (int b = 0; b < B; ++b) {
    for (int k = 1; k <= G; ++k) {
      int prev = (k == 1) ? anchor[b] : x[(size_t)b * G + k - 2];
      if (prev < 0 || prev >= V) return ORACLE_ERR_INVALID;
      double z = 0.0;
      for (int i = 0; i < H; ++i)
        z += (double)w[i] * load_elem(h, hdt, ((size_t)b * G + (k - 1)) * H + i);
      for (int i = 0; i < r; ++i)
        z += (double)w[H + i] * load_elem(W1, wdt, (size_t)prev * r + i);
      double T = sts_T ? (double)sts_T[k - 1] : 1.0;
      c_out[(size_t)b * G + (k - 1)] = 1.0 / (1.0 + exp(-z / T));
    }
  }
  return ORACLE_OK;
}

/* ------------------------------------------------------------------------- */
/* Step 3: hardware-aware prefix scheduler ([blog] section 6; [report] the
 * throughput objective Theta = tau * SPS(B)).
 *
 *   a_{r,j} = prod_{i<=j} c_{r,i}            (prefix survival probability)
 *   B      = sum_r (l_r + 1)                 (the 1 is the target's own token)
 *   tau    = sum_r (1 + sum_{j<=l_r} a_{r,j}) (expected emitted tokens)
 *   Theta  = tau * SPS(B)
 *
 * Greedy with early stop: visit the candidates (r, j) in the order a desc, then
 * r asc, then j asc; admitting one adds a to tau and 1 to B; stop at the first
 * candidate whose admission gives Theta <= Theta_best (a tie stops).  The early
 * stop keeps the admission of x_{r,j} independent of x_{r,j} and later tokens
 * ([blog] section 7, the non-anticipating property).
 *
 * mode 0: fixed, l_r = gamma for every request (no truncation);
 * mode 1: greedy as above;
 * mode 2: dynamic top-K ([blog] section 7): admit exactly the first K candidates
 *         of this round's order, K given by the caller (the greedy count of two
 *         rounds earlier); K is clamped to [0, R*gamma].
 * In every mode nstar_out receives this round's greedy count and theta_out the
 * objective of the admitted set.  The SPS table is indexed by batch size and must
 * cover B = R * (gamma + 1). */
typedef struct {
  double a;
  int r, j;
} oracle_cand;

static int cand_cmp(const void* pa, const void* pb) {
  const oracle_cand* x = (const oracle_cand*)pa;
  const oracle_cand* y = (const oracle_cand*)pb;
  if (x->a > y->a) return -1;
  if (x->a < y->a) return 1;
  if (x->r != y->r) return x->r < y->r ? -1 : 1;
  if (x->j != y->j) return x->j < y->j ? -1 : 1;
  return 0;
}

int oracle_schedule(int R, int G, const double* c, const float* sps, int n_sps,
                    int mode, int K, int32_t* ell_out, int32_t* nstar_out,
                    double* theta_out, int32_t* order_out) {
  if (R <= 0 || G <= 0 || !c || !ell_out || mode < 0 || mode > 2)
    return ORACLE_ERR_INVALID;
  if (mode != 0 && (!sps || n_sps <= R * (G + 1))) return ORACLE_ERR_INVALID;
  int N = R * G;
  oracle_cand* cand = (oracle_cand*)malloc(sizeof(oracle_cand) * (size_t)N);
  if (!cand) return ORACLE_ERR_NOMEM;
  for (int r = 0; r < R; ++r) {
    double a = 1.0;
    for (int j = 1; j <= G; ++j) {
      a *= c[(size_t)r * G + (j - 1)];
      cand[(size_t)r * G + (j - 1)].a = a;
      cand[(size_t)r * G + (j - 1)].r = r;
      cand[(size_t)r * G + (j - 1)].j = j;
    }
  }
  qsort(cand, (size_t)N, sizeof(oracle_cand), cand_cmp);
  if (order_out)
    for (int i = 0; i < N; ++i) order_out[i] = cand[i].r * G + (cand[i].j - 1);

  int nstar = N;
  double theta_greedy = 0.0;
  if (mode != 0) {
    double tau = (double)R;
    int batch = R;
    double theta_best = tau * (double)sps[batch];
    nstar = 0;
    for (int i = 0; i < N; ++i) {
      double tau_new = tau + cand[i].a;
      double theta = tau_new * (double)sps[batch + 1];
      if (theta <= theta_best) break;
      theta_best = theta;
      tau = tau_new;
      batch += 1;
      nstar += 1;
    }
    theta_greedy = theta_best;
  }
  int admitted = nstar;
  if (mode == 0) admitted = N;
  if (mode == 2) admitted = K < 0 ? 0 : (K > N ? N : K);
  for (int r = 0; r < R; ++r) ell_out[r] = 0;
  double tau = (double)R;
  for (int i = 0; i < admitted; ++i) {
    ell_out[cand[i].r] += 1;
    tau += cand[i].a;
  }
  if (nstar_out) *nstar_out = nstar;
  if (theta_out) {
    if (mode == 1)
      *theta_out = theta_greedy;
    else if (sps && n_sps > R + admitted)
      *theta_out = tau * (double)sps[R + admitted];
    else
      *theta_out = NAN;
  }
  free(cand);
  return ORACLE_OK;
}

/* ------------------------------------------------------------------------- */
/* Step 4: lossless rejection-sampling verification ([digest] item 2; [blog]
 * section 1: accept the longest valid prefix plus one bonus token).
 *
 * For request b with verify length L = ell[b], positions k = 1..L in order:
 *   p_t = softmax(T[b, k-1, :])  (the target's distribution of position k),
 *   p_d = the draft distribution of position k given x_{k-1} (step 1),
 *   accept x_k while u_k < p_t(x_k) / p_d(x_k),  u_k = U01(stream 1, b, k, 0);
 *   at the first rejection, n = k - 1 and the corrected token is drawn from
 *   normalize(max(0, p_t - p_d)) (oracle_block_draw, streams 2 and 6, b, k);
 *   if every rho is 0 in floating point (a measure-zero event in exact
 *   arithmetic) it is drawn from p_t instead, with the same streams.
 * If all L tokens are accepted, n = L and the bonus token is drawn from
 * softmax(T[b, L, :]) (streams 3 and 7, b, k = L + 1).
 *
 * Outputs per request: n (accepted count), y (the corrected or bonus token),
 * flags (1 = bonus, 2 = residual, 4 = residual fell back to p_t); per verified
 * position the ratio p_t/p_d and |u - ratio| (NaN where not evaluated); per
 * request the margin of the draw of y. */
static int verify_impl(int B, int G, int V, int r, const float* T, const float* U,
                       const void* W1, const void* W2, int wdt, const float* gate_g,
                       const float* gate_c, int bf16_state, const int32_t* anchor,
                       const int32_t* x,
                       const int32_t* ell, uint64_t seed, uint64_t round, int b0,
                       int b1, int32_t* n_out, int32_t* y_out, int32_t* flags_out,
                       double* ratio_out, double* umargin_out,
                       double* ymargin_out) {
  if (B <= 0 || G <= 0 || V <= 0 || r <= 0 || !T || !U || !W1 || !W2 ||
      !anchor || !x || !ell || !n_out || !y_out || b0 < 0 || b1 > B || b0 > b1 ||
      (!gate_g) != (!gate_c))
    return ORACLE_ERR_INVALID;
  int status = ORACLE_OK;
#pragma omp parallel for schedule(dynamic, 1)
  for (int b = b0; b < b1; ++b) {
    double* p_d = (double*)malloc(sizeof(double) * (size_t)V);
    double* p_t = (double*)malloc(sizeof(double) * (size_t)V);
    double* score = (double*)malloc(sizeof(double) * (size_t)V);
    double* s = (double*)calloc((size_t)r, sizeof(double));
    if (!p_d || !p_t || !score || !s) {
      set_status(&status, ORACLE_ERR_NOMEM);
      free(p_d); free(p_t); free(score); free(s);
      continue;
    }
    int L = ell[b];
    if (L < 0 || L > G) {
      set_status(&status, ORACLE_ERR_INVALID);
      free(p_d); free(p_t); free(score); free(s);
      continue;
    }
    for (int k = 1; k <= G; ++k) {
      if (ratio_out) ratio_out[(size_t)b * G + k - 1] = NAN;
      if (umargin_out) umargin_out[(size_t)b * G + k - 1] = NAN;
    }
    int n = L, y = -1, flags = 0;
    double ymargin = 0.0;
    for (int k = 1; k <= L; ++k) {
      int prev = (k == 1) ? anchor[b] : x[(size_t)b * G + k - 2];
      int xk = x[(size_t)b * G + k - 1];
      if (prev < 0 || prev >= V || xk < 0 || xk >= V) {
        set_status(&status, ORACLE_ERR_INVALID);
        n = -1;
        break;
      }
      const float* U_row = U + ((size_t)b * G + (k - 1)) * (size_t)V;
      const float* T_row = T + ((size_t)b * (G + 1) + (k - 1)) * (size_t)V;
      if (gate_g) {
        gated_step(r, W1, wdt, gate_g, gate_c, prev, bf16_state, s);
        state_logits(V, r, U_row, s, W2, wdt, p_d);
        const double lse = oracle_logsumexp(V, p_d);
        for (int v = 0; v < V; ++v) p_d[v] = exp(p_d[v] - lse);
      } else {
        oracle_draft_probs(V, r, U_row, W1, W2, wdt, prev, p_d);
      }
      for (int v = 0; v < V; ++v) score[v] = (double)T_row[v];
      oracle_softmax(V, score, p_t);
      double ratio = p_t[xk] / p_d[xk];
      double u = oracle_u01(oracle_rng_word(seed, round, 1u, (uint32_t)b,
                                            (uint32_t)k, 0u));
      if (ratio_out) ratio_out[(size_t)b * G + k - 1] = ratio;
      if (umargin_out) umargin_out[(size_t)b * G + k - 1] = fabs(u - ratio);
      if (u < ratio) continue;
      n = k - 1;
      flags = 2;
      /* y ~ rho / sum rho, rho = max(0, p_t - p_d) (stream 2); an empty
       * residual in floating point draws from p_t with the same streams */
      oracle_residual(V, p_t, p_d, score);
      y = oracle_block_draw(V, score, 0.0, seed, round, 2u, (uint32_t)b,
                            (uint32_t)k, &ymargin);
      if (y < 0) {
        flags |= 4;
        y = oracle_block_draw(V, p_t, 0.0, seed, round, 2u, (uint32_t)b,
                              (uint32_t)k, &ymargin);
      }
      break;
    }
    if (n < 0) {
      n_out[b] = -1;
      y_out[b] = -1;
      free(p_d); free(p_t); free(score); free(s);
      continue;
    }
    if (n == L) {
      const float* T_row = T + ((size_t)b * (G + 1) + L) * (size_t)V;
      for (int v = 0; v < V; ++v) score[v] = (double)T_row[v];
      y = oracle_softmax_draw(V, score, seed, round, 3u, (uint32_t)b,
                              (uint32_t)(L + 1), &ymargin);
      flags = 1;
    }
    n_out[b] = n;
    y_out[b] = y;
    if (flags_out) flags_out[b] = flags;
    if (ymargin_out) ymargin_out[b] = ymargin;
    free(p_d); free(p_t); free(score); free(s);
  }
  return status;
}

int oracle_verify(int B, int G, int V, int r, const float* T, const float* U,
                  const void* W1, const void* W2, int wdt,
                  const int32_t* anchor, const int32_t* x, const int32_t* ell,
                  uint64_t seed, uint64_t round, int b0, int b1,
                  int32_t* n_out, int32_t* y_out, int32_t* flags_out,
                  double* ratio_out, double* umargin_out, double* ymargin_out) {
  return verify_impl(B, G, V, r, T, U, W1, W2, wdt, NULL, NULL, 0, anchor, x, ell, seed,
                     round, b0, b1, n_out, y_out, flags_out, ratio_out,
                     umargin_out, ymargin_out);
}

/* Verification of a draft made with the gated recurrent head: p_d of
 * position k from the state s_k of the prefix anchor, x_1..x_{k-1}. */
int oracle_gated_verify(int B, int G, int V, int r, const float* T,
                        const float* U, const void* W1, const void* W2, int wdt,
                        const float* gate_g, const float* gate_c, int bf16_state,
                        const int32_t* anchor, const int32_t* x,
                        const int32_t* ell, uint64_t seed, uint64_t round, int b0,
                        int b1, int32_t* n_out, int32_t* y_out,
                        int32_t* flags_out, double* ratio_out,
                        double* umargin_out, double* ymargin_out) {
  if (!gate_g || !gate_c) return ORACLE_ERR_INVALID;
  return verify_impl(B, G, V, r, T, U, W1, W2, wdt, gate_g, gate_c, bf16_state, anchor, x, ell,
                     seed, round, b0, b1, n_out, y_out, flags_out, ratio_out,
                     umargin_out, ymargin_out);
}

/* Number of threads the parallel request loops use (1 without OpenMP). */
int oracle_num_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

/* Sets the number of threads of the parallel request loops (n >= 1; no effect
 * without OpenMP).  Used to time the oracle on one core beside all of them. */
void oracle_set_num_threads(int n) {
#ifdef _OPENMP
  if (n >= 1) omp_set_num_threads(n);
#else
  (void)n;
#endif
}
