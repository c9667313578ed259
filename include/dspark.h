/*
 * dspark.h -- C ABI of libdspark, the GB300 (sm_103a) per-round hot path of
 * DSpark speculative decoding: semi-autoregressive Markov-head draft sampling,
 * the confidence head, the confidence-scheduled prefix truncation and lossless
 * rejection-sampling verification.
 *
 * Sources, cited by page title and section:
 *   [blog]   "[DeepSeek-6] DSpark: From Draft Models to Serving-Aware Speculative
 *             Decoding" (xutianle.me), sections 1, 3-7.
 *   [digest] "DSpark ... 10 key concepts" (aimsg.uk), items 2, 8, 9.
 *   [report] "DSpark: Confidence-Scheduled Speculative Decoding with
 *             Semi-Autoregressive Generation -- study report" (devpress.csdn),
 *             Key formulas Eq.4, Eq.7, Eq.8 and Theta = tau * SPS(B).
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - All tensor pointers are DEVICE pointers of the current CUDA device, row-major
 *    and densely packed.  The caller owns every buffer; the library never
 *    allocates device memory.  Scratch space is the caller's `workspace` of at
 *    least dspark_workspace_size(B, gamma, V) bytes, 256-byte aligned; one
 *    workspace must not be used by two calls that run concurrently.
 *  - `stream` is a cudaStream_t (NULL = the legacy default stream).  Calls only
 *    enqueue work and never synchronise, except dspark_read_status.
 *  - Shapes: B requests (1..65535), gamma draft positions (1..32), V vocabulary entries
 *    (V % 8 == 0), r Markov rank (r % 16 == 0, 16..256), H hidden size.
 *    Position k = 1..gamma is row k-1 of the per-position tensors.
 *  - Weights: W1 [V, r] is the Markov embedding of the previous token; W2 [V, r]
 *    is the weight of the bias-free linear layer r -> V as a linear layer stores
 *    it, so the Markov bias of entry v is sum_i W1[prev, i] * W2[v, i]
 *    ([blog] section 4).  wdtype is DSPARK_BF16 or DSPARK_F32 for both.
 *  - Random numbers: Philox4x32-10 (Salmon et al., SC'11) keyed by
 *    (seed mod 2^32, seed / 2^32); a call at counter (c, position k, request b,
 *    (round << 3) | stream) gives four 32-bit words; word j of a stream is word
 *    (j mod 4) of call j / 4.  Accept uniform (stream 1): word 0,
 *    u = ((w >> 9) + 1/2) / 2^23.  Every categorical draw (draft x_k: stream 0;
 *    corrected token: stream 2; bonus token: stream 3) is one exact two-level
 *    draw from its weights: blocks of 4 consecutive entries race with the log
 *    of their summed weight plus -log(-log u_j), u_j from word j of the stream;
 *    inside the winning block the entry is drawn by inverse CDF with the
 *    uniform of word j of stream + 4.  `round` < 2^29.
 *  - Return value: a DSPARK_* status.  Argument errors are detected on the host
 *    before anything is enqueued.  Errors found by the kernels (a bounded wait
 *    that gave up, non-finite logits) are recorded in a status word inside the
 *    workspace and read with dspark_read_status.
 */
#ifndef DSPARK_H
#define DSPARK_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* status codes */
#define DSPARK_OK 0
#define DSPARK_ERR_INVALID 1      /* null pointer, bad size, table too short */
#define DSPARK_ERR_UNSUPPORTED 2  /* a size outside the supported range */
#define DSPARK_ERR_CUDA 3         /* a CUDA launch or runtime call failed */
#define DSPARK_ERR_TIMEOUT 4      /* a device-side bounded wait gave up */
#define DSPARK_ERR_WORKSPACE 5    /* workspace too small or misaligned */
#define DSPARK_ERR_NONFINITE 6    /* a NaN or infinite logit was met */

/* storage types */
#define DSPARK_F32 0
#define DSPARK_BF16 1

/* scheduler modes */
#define DSPARK_SCHED_FIXED 0   /* no truncation: l_r = gamma */
#define DSPARK_SCHED_GREEDY 1  /* greedy Theta maximisation with early stop */
#define DSPARK_SCHED_TOPK 2    /* dynamic top-K, K = greedy count of round - 2 */

/* flags of dspark_verify_ex, dspark_round_ex, dspark_draft_schedule_ex and
 * dspark_acceptance_label_ex */
#define DSPARK_EARLY_TARGET_STATS 1u  /* the draft took the target rows' softmax statistics */
#define DSPARK_ADVANCE_ROUND 2u       /* the call's last kernel adds 1 to *round_dev */
#define DSPARK_TARGET_STATS_FROM_VERIFY 4u  /* dspark_acceptance_label_ex: a verification left them */
#define DSPARK_SCRATCH_FROM_DRAFT 8u  /* dspark_verify_ex: dspark_draft_schedule cleared the scratch */
#define DSPARK_GATED_STATES 16u       /* dspark_verify_ex: the draft used the gated recurrent head */
#define DSPARK_ALL_ROW_STATS 32u      /* verification takes the statistics of every row j < ell */
#define DSPARK_CHAIN_TARGET_STATS 64u /* the draft takes the statistics of the rows the accept chains reach */

/* Bytes of device scratch the entry points below need for these sizes; 0 when
 * a size is not positive. */
size_t dspark_workspace_size(int B, int gamma, int V);

/*
 * Semi-autoregressive Markov draft ([report] Eq.4; [blog] sections 3-4).
 * For k = 1..gamma (x_0 = anchor, [blog] section 3):
 *   l_k(v) = U[b, k-1, v] + sum_i W1[x_{k-1}, i] * W2[v, i]
 *   x_k    ~ softmax(l_k), the two-level draw on streams 0 and 4 (b, k)
 *   lse_k  = log sum_v exp l_k(v);   p_k(x_k) = exp(l_k(x_k) - lse_k)
 * In:  U [B, gamma, V] f32, W1/W2 [V, r] (wdtype), anchor [B] i32 in [0, V).
 * Out: x_out [B, gamma] i32, p_out [B, gamma] f32, lse_out [B, gamma] f32.
 * Ties of the perturbed block log-mass go to the smallest block.
 */
int dspark_markov_draft(const float* U, const void* W1, const void* W2, int wdtype,
                        const int32_t* anchor, int B, int gamma, int V, int r,
                        uint64_t seed, uint64_t round,
                        int32_t* x_out, float* p_out, float* lse_out,
                        void* workspace, size_t workspace_bytes, void* stream);

/*
 * dspark_markov_draft with two additions (both may be NULL, which gives
 * dspark_markov_draft exactly).
 *  - T_early [B, gamma+1, V] f32, 16-byte aligned: target logits that the
 *    caller already holds when the draft starts.  The softmax statistics of
 *    its rows j < gamma of every request -- the rows verification tests when
 *    every position is verified ([digest] item 2; [blog] section 1) -- are
 *    taken while the draft runs, by warps that stream T in the memory time
 *    the draft leaves idle, and left in the workspace for
 *    dspark_verify_ex(..., DSPARK_EARLY_TARGET_STATS).  This reads 4 * V bytes
 *    per row even for rows that the schedule later leaves unverified, so it
 *    pays when the schedule verifies most positions.  In a serving engine
 *    the target's logits of a round usually exist only after its draft; the
 *    flag serves callers that hold them earlier (one micro-batch's verify
 *    overlapping another's draft, or a replayed round).
 *  - round_dev: device pointer to the round index (a uint64 < 2^29).  When
 *    given, the kernels read the round from it when they start and `round` is
 *    ignored, so that one captured CUDA graph serves consecutive rounds.
 */
int dspark_markov_draft_ex(const float* U, const float* T_early, const void* W1, const void* W2,
                           int wdtype, const int32_t* anchor, int B, int gamma, int V, int r,
                           uint64_t seed, uint64_t round, const uint64_t* round_dev,
                           int32_t* x_out, float* p_out, float* lse_out,
                           void* workspace, size_t workspace_bytes, void* stream);

/*
 * Confidence head ([report] Eq.7; [blog] section 5):
 *   c_k = sigmoid( (sum_i w[i] h[b,k-1,i] + sum_i w[H+i] W1[x_{k-1}, i]) / T_k )
 * with x_0 = anchor and T_k = sts_T[k-1] (Sequential Temperature Scaling,
 * [blog] section 5), or 1 when sts_T is NULL.  No bias term (Eq.7 has none).
 * In:  h [B, gamma, H] (hdtype), W1 [V, r] (wdtype), w [H + r] f32,
 *      sts_T [gamma] f32 or NULL, anchor [B], x [B, gamma] i32.
 * Out: c_out [B, gamma] f32.  A previous token outside [0, V) gives c = 0
 * (this call has no workspace to report it in; dspark_round also records
 * DSPARK_ERR_INVALID in its status word).
 */
int dspark_confidence(const void* h, int hdtype, const void* W1, int wdtype,
                      const float* w, const float* sts_T, const int32_t* anchor,
                      const int32_t* x, int B, int gamma, int H, int r, int V,
                      float* c_out, void* stream);

/*
 * Hardware-aware prefix scheduler ([blog] sections 6-7; [report] Theta).
 *   a_{b,j} = prod_{i<=j} c_{b,i};  B' = sum_b (l_b + 1);
 *   tau = sum_b (1 + sum_{j<=l_b} a_{b,j});  Theta = tau * SPS(B').
 * Candidates (b, j) are ordered by a desc, then b asc, then j asc.
 * GREEDY: admit in that order while Theta strictly rises; the first candidate
 *   that does not raise it stops the scan (non-anticipating, [blog] section 7).
 * TOPK:   admit exactly the first K candidates, K = khist[round % 2], the greedy
 *   count this call wrote two rounds earlier ([blog] section 7); rounds 0 and 1
 *   run the greedy.  Every mode writes this round's greedy count to
 *   khist[round % 2] after reading it (khist: device [2] i32, caller-owned).
 * FIXED:  l_b = gamma.
 * In:  c [B, gamma] f32 in [0, 1]; sps [n_sps] f32 indexed by batch size,
 *      n_sps > B * (gamma + 1) (not read in FIXED mode).  B * gamma <= 8192
 *      (GREEDY and TOPK; FIXED has no limit).
 * Out: ell_out [B] i32, nstar_out [1] i32 (greedy count), theta_out [1] f64
 *      (Theta of the admitted set; 0 in FIXED mode).
 */
int dspark_schedule(const float* c, int B, int gamma, const float* sps, int n_sps,
                    int mode, uint64_t round, int32_t* khist,
                    int32_t* ell_out, int32_t* nstar_out, double* theta_out,
                    void* workspace, size_t workspace_bytes, void* stream);

/* dspark_schedule with the round index read from the device word *round_dev
 * when round_dev is not NULL (see dspark_markov_draft_ex). */
int dspark_schedule_ex(const float* c, int B, int gamma, const float* sps, int n_sps,
                       int mode, uint64_t round, const uint64_t* round_dev, int32_t* khist,
                       int32_t* ell_out, int32_t* nstar_out, double* theta_out,
                       void* workspace, size_t workspace_bytes, void* stream);

/*
 * Lossless rejection-sampling verification ([digest] item 2; [blog] section 1).
 * For request b and k = 1..ell[b]: p_t = softmax(T[b, k-1, :]); accept x_k
 * while u < p_t(x_k) / p_d(x_k), u = uniform(stream 1, b, k).  At the first
 * rejection the corrected token is drawn from normalize(max(0, p_t - p_d))
 * (the two-level draw on streams 2 and 6, b, k), p_d = softmax(U[b,k-1,:] +
 * bias(x_{k-1})) recomputed from lse_d; if that residual is empty in floating
 * point, from p_t with the same streams.  If all ell[b] tokens are accepted,
 * the bonus token is drawn from softmax(T[b, ell[b], :]) (streams 3 and 7,
 * k = ell[b]+1).
 * In:  T [B, gamma+1, V] f32 (row k-1 scores position k); U, W1, W2, anchor as
 *      for the draft; x, p_d, lse_d [B, gamma] from the draft; ell [B] i32 in
 *      [0, gamma].
 * Out: n_out [B] i32 accepted count; tok_out [B] i32 corrected or bonus token.
 * Rows read: the accept tests run along each request's prefix and stop at its
 * first rejection, so row k-1 is read only once positions 1..k-1 were
 * accepted (every row 0), plus row ell[b] of a request that accepted all of
 * its positions (the bonus draw).  The result is the same as reading every
 * row j < ell[b]; DSPARK_ALL_ROW_STATS (dspark_verify_ex) reads them all.
 */
int dspark_verify(const float* T, const float* U, const void* W1, const void* W2,
                  int wdtype, const int32_t* anchor, const int32_t* x,
                  const float* p_d, const float* lse_d, const int32_t* ell,
                  int B, int gamma, int V, int r, uint64_t seed, uint64_t round,
                  int32_t* n_out, int32_t* tok_out,
                  void* workspace, size_t workspace_bytes, void* stream);

/*
 * dspark_verify with options (flags 0 and round_dev NULL give dspark_verify):
 *  - DSPARK_EARLY_TARGET_STATS: the workspace already holds the softmax
 *    statistics of the rows j < gamma of this T, left by
 *    dspark_markov_draft_ex(T_early = T) on the same workspace earlier in
 *    stream order (or those of the rows the accept tests reach, left by
 *    dspark_draft_schedule_ex with DSPARK_CHAIN_TARGET_STATS); the call skips
 *    its own pass over those rows.  If no such draft preceded it, the kernels
 *    record DSPARK_ERR_INVALID.  A row the tests use that holds a NaN or +inf
 *    is reported as DSPARK_ERR_NONFINITE.
 *  - round_dev: the round index as a device word (see dspark_markov_draft_ex).
 *  - DSPARK_ADVANCE_ROUND (needs round_dev): the call's last kernel adds 1 to
 *    *round_dev after every kernel of the call has read it.
 *  - DSPARK_GATED_STATES: x, p_d and lse_d come from dspark_gated_markov_draft
 *    on the same workspace, earlier in stream order; the residual's bias
 *    operand is the state it left there (tensor-core path only, else
 *    DSPARK_ERR_UNSUPPORTED).
 *  - DSPARK_SCRATCH_FROM_DRAFT: a dspark_draft_schedule on the same workspace,
 *    earlier in stream order, cleared this call's scratch (its argmax keys and
 *    bonus list; the tensor-core path does, others ignore the flag), so the
 *    call skips its memset and its kernels run as one chain of dependent
 *    launches.
 *  - DSPARK_ALL_ROW_STATS: take the softmax statistics of every row j < ell[b]
 *    before the accept tests, as dspark_acceptance_label_ex with
 *    DSPARK_TARGET_STATS_FROM_VERIFY needs them; without it (and without
 *    DSPARK_EARLY_TARGET_STATS) only the rows the accept tests reach are
 *    read.  Together with DSPARK_EARLY_TARGET_STATS: DSPARK_ERR_INVALID.
 * Other flag bits return DSPARK_ERR_INVALID.
 */
int dspark_verify_ex(const float* T, const float* U, const void* W1, const void* W2,
                     int wdtype, const int32_t* anchor, const int32_t* x,
                     const float* p_d, const float* lse_d, const int32_t* ell,
                     int B, int gamma, int V, int r, uint64_t seed, uint64_t round,
                     uint64_t* round_dev, unsigned flags,
                     int32_t* n_out, int32_t* tok_out,
                     void* workspace, size_t workspace_bytes, void* stream);

/*
 * Acceptance labels of the verified positions (the study report's label for
 * training the confidence head: the probability that rejection sampling
 * accepts position k, Eq.8, the mass p_d and p_t share).  For request b and
 * k = 1..ell[b]:  label[b, k-1] = sum_v min(p_d(v), p_t(v)), p_d =
 * softmax(U[b,k-1,:] + bias(x_{k-1})) from lse_d, p_t = softmax(T[b, k-1, :]);
 * positions k > ell[b] get 0.  Arguments as for dspark_verify (the same
 * workspace layout: it overwrites the target-row statistics there).  One
 * persistent launch runs every position; U and T rows stream in by TMA.
 * Tensor-core path only (bf16 W1/W2, r = 256, V >= 192); other weights
 * return DSPARK_ERR_UNSUPPORTED.
 * Out: label_out [B, gamma] f32, caller-owned.
 */
int dspark_acceptance_label(const float* T, const float* U, const void* W1, const void* W2,
                            int wdtype, const int32_t* anchor, const int32_t* x,
                            const float* lse_d, const int32_t* ell, int B, int gamma,
                            int V, int r, float* label_out, void* workspace,
                            size_t workspace_bytes, void* stream);

/*
 * dspark_acceptance_label reading the target rows' softmax statistics that
 * the round already took, so that each U and T row is read once (flags 0
 * gives dspark_acceptance_label, which streams the rows for them first):
 *  - DSPARK_EARLY_TARGET_STATS: left by dspark_markov_draft_ex(T_early = T)
 *    on the same workspace (rows j < gamma), with or without the verification
 *    that used them; after a draft with DSPARK_CHAIN_TARGET_STATS, which
 *    leaves only some rows, the kernel records DSPARK_ERR_INVALID;
 *  - DSPARK_TARGET_STATS_FROM_VERIFY: left by a dspark_verify_ex with
 *    DSPARK_ALL_ROW_STATS on the same workspace and T (rows j < ell[b]), with
 *    no draft on the workspace since; otherwise the kernel records
 *    DSPARK_ERR_INVALID;
 * either earlier in stream order.  Both flags at once, or other bits, return
 * DSPARK_ERR_INVALID.
 */
int dspark_acceptance_label_ex(const float* T, const float* U, const void* W1, const void* W2,
                               int wdtype, const int32_t* anchor, const int32_t* x,
                               const float* lse_d, const int32_t* ell, int B, int gamma,
                               int V, int r, unsigned flags, float* label_out, void* workspace,
                               size_t workspace_bytes, void* stream);

/*
 * Sequential temperature scaling of the confidence head ([blog] section 5; the
 * study report's answer on calibration), a post-hoc fit on held-out samples.
 * Sample n: confidence logits z[n, :] (c = sigmoid(z / T_k)), verified length
 * ell[n] in [0, gamma] and accepted count acc[n] <= ell[n].  Position k of
 * sample n is observed when k <= ell[n], with outcome 1 if acc[n] >= k.  For
 * k = 1..gamma in order, T_k is the grid value that minimises the expected
 * calibration error (15 equal-width bins on [0, 1]: sum over bins of
 * |sum(P - outcome)| / observed samples) of P = prod_{i<k} sigmoid(z_i / T_i)
 * * sigmoid(z_k / T_k) over the observed samples; the first grid value wins
 * ties; a position no sample observes gets T = 1 and ECE 0.  fp64 throughout.
 * In:  z [N, gamma] f32, ell [N] i32, acc [N] i32, grid [ngrid] f32 (> 0), all
 *      device; gamma <= 32, ngrid <= 256.
 * Out: T_out [gamma] f32 (usable as sts_T of dspark_confidence), ece_out
 *      [gamma] f32.  Workspace: dspark_sts_workspace_size bytes, 256-byte
 *      aligned (that size is 0 when a size is not positive).
 */
size_t dspark_sts_workspace_size(int N, int gamma, int ngrid);
int dspark_sts_fit(const float* z, const int32_t* ell, const int32_t* acc, int N, int gamma,
                   const float* grid, int ngrid, float* T_out, float* ece_out,
                   void* workspace, size_t workspace_bytes, void* stream);

/*
 * The Markov draft with a gated recurrent head.  [blog] section 4 and
 * [digest] item 8 name a gated Markov head and an RNN head whose state runs
 * through the draft block, without equations; this library's plain form
 * keeps the Markov head's rank-r space and projection:
 *   e_k = W1[x_{k-1}],  a_k = sigmoid(gate_g * e_k + gate_c)  (elementwise),
 *   s_0 = 0,  s_k = e_k + a_k * s_{k-1}  (kept in bf16, as the tensor cores read it),
 *   l_k(v) = U[b, k-1, v] + sum_i s_k[i] * W2[v, i],
 * so the draft distribution depends on the whole prefix x_0 .. x_{k-1}; with
 * a_k = 0 it is dspark_markov_draft.  Sampling, outputs, T_early and round_dev
 * as for dspark_markov_draft_ex.  gate_g, gate_c: float32 [r], 16-byte
 * aligned.  The states are left in the workspace for dspark_verify_ex
 * (DSPARK_GATED_STATES).  Tensor-core path only (bf16, r = 256, V >= 192);
 * otherwise DSPARK_ERR_UNSUPPORTED.
 */
int dspark_gated_markov_draft(const float* U, const float* T_early, const void* W1, const void* W2,
                              int wdtype, const float* gate_g, const float* gate_c,
                              const int32_t* anchor, int B, int gamma, int V, int r,
                              uint64_t seed, uint64_t round, const uint64_t* round_dev,
                              int32_t* x_out, float* p_out, float* lse_out,
                              void* workspace, size_t workspace_bytes, void* stream);

/*
 * The first stage of a round: the Markov draft, the confidence head of every
 * drafted position and the schedule (blog sections 4-7; study report Eq.7),
 * with the arguments of dspark_markov_draft_ex, dspark_confidence and
 * dspark_schedule_ex.  T_early (may be NULL) is taken along as in
 * dspark_markov_draft_ex.  On the tensor-core path (bf16, r = 256) this is
 * one persistent launch: its finalize computes the confidences and the last
 * CTA to finish it runs the schedule (up to 4096 candidates; beyond, a
 * schedule kernel follows) while the others stream the target-row
 * statistics; it also clears the verification's scratch
 * (DSPARK_SCRATCH_FROM_DRAFT).  Other paths run the three kernels in turn.
 * Errors as for those three calls.
 */
int dspark_draft_schedule(const float* U, const float* T_early, const void* W1, const void* W2,
                          int wdtype, const void* h, int hdtype, const float* w,
                          const float* sts_T, const int32_t* anchor,
                          int B, int gamma, int V, int r, int H,
                          const float* sps, int n_sps, int mode, int32_t* khist,
                          uint64_t seed, uint64_t round, uint64_t* round_dev,
                          int32_t* x_out, float* p_out, float* lse_out, float* c_out,
                          int32_t* ell_out, int32_t* nstar_out, double* theta_out,
                          void* workspace, size_t workspace_bytes, void* stream);

/*
 * dspark_draft_schedule with flags (0 gives it exactly):
 *  - DSPARK_CHAIN_TARGET_STATS (needs T_early): take the statistics only of
 *    the target rows the accept tests can reach ([blog] section 1: the tests
 *    run along the prefix and stop at the first rejection).  The warps that
 *    stream T go position by position; before row j of request b they run
 *    the accept tests of b's positions 1..j that are decidable from what the
 *    draft has published (x_k once every CTA is past position k, lse_t of row
 *    k-1 once all its segments are out), and skip the row once a test fails
 *    by a margin of 2^-8 relative.  A position not yet decidable counts as
 *    accepted, so a row is skipped only when verification is certain to stop
 *    before it; some rows past a rejection may still be read.  At the engine
 *    point about a quarter of the rows j < gamma are read.  Verification then
 *    takes DSPARK_EARLY_TARGET_STATS; dspark_acceptance_label_ex refuses
 *    these statistics.  Other paths than the tensor-core persistent draft
 *    take every row j < gamma.
 * Other bits return DSPARK_ERR_INVALID.
 */
int dspark_draft_schedule_ex(const float* U, const float* T_early, const void* W1, const void* W2,
                             int wdtype, const void* h, int hdtype, const float* w,
                             const float* sts_T, const int32_t* anchor,
                             int B, int gamma, int V, int r, int H,
                             const float* sps, int n_sps, int mode, int32_t* khist,
                             uint64_t seed, uint64_t round, uint64_t* round_dev, unsigned flags,
                             int32_t* x_out, float* p_out, float* lse_out, float* c_out,
                             int32_t* ell_out, int32_t* nstar_out, double* theta_out,
                             void* workspace, size_t workspace_bytes, void* stream);

/*
 * One whole round: dspark_draft_schedule, then dspark_verify_ex, enqueued in
 * that order on one stream with no host synchronisation.  Arguments as above.  A round
 * can be captured into a CUDA graph (the draft's cooperative launch
 * included); a replay repeats the captured seed and round (dspark_round_ex
 * with a device round index advances it).
 */
int dspark_round(const float* U, const float* T, const void* W1, const void* W2,
                 int wdtype, const void* h, int hdtype, const float* w,
                 const float* sts_T, const int32_t* anchor,
                 int B, int gamma, int V, int r, int H,
                 const float* sps, int n_sps, int mode, int32_t* khist,
                 uint64_t seed, uint64_t round,
                 int32_t* x_out, float* p_out, float* lse_out, float* c_out,
                 int32_t* ell_out, int32_t* nstar_out, double* theta_out,
                 int32_t* n_out, int32_t* tok_out,
                 void* workspace, size_t workspace_bytes, void* stream);

/*
 * dspark_round with the options of the _ex calls: with
 * DSPARK_EARLY_TARGET_STATS the draft takes the statistics of T's rows
 * j < gamma while it runs (T is an input of the round) and verification
 * skips its own pass over them; with DSPARK_CHAIN_TARGET_STATS the draft
 * takes only the rows the accept tests reach (see dspark_draft_schedule_ex)
 * and verification decides on them; with DSPARK_ALL_ROW_STATS verification
 * takes the statistics of every row j < ell[b] (see dspark_verify_ex); at
 * most one of the three (else DSPARK_ERR_INVALID); with round_dev the round index is the device
 * word *round_dev (`round` ignored), and DSPARK_ADVANCE_ROUND makes the
 * round's last kernel add 1 to it, so that replaying one captured graph runs
 * consecutive rounds (the caller refreshes U, T, h and the anchors in place
 * between replays).
 */
int dspark_round_ex(const float* U, const float* T, const void* W1, const void* W2,
                    int wdtype, const void* h, int hdtype, const float* w,
                    const float* sts_T, const int32_t* anchor,
                    int B, int gamma, int V, int r, int H,
                    const float* sps, int n_sps, int mode, int32_t* khist,
                    uint64_t seed, uint64_t round, uint64_t* round_dev, unsigned flags,
                    int32_t* x_out, float* p_out, float* lse_out, float* c_out,
                    int32_t* ell_out, int32_t* nstar_out, double* theta_out,
                    int32_t* n_out, int32_t* tok_out,
                    void* workspace, size_t workspace_bytes, void* stream);

/*
 * The Markov draft without a caller workspace.  The method has no counterpart:
 * this entry serves callers that cannot allocate device memory at the time of
 * the call (an engine whose pool owns all of HBM, a plugin given no allocator,
 * a decode loop that must not call cudaMalloc).  It computes exactly what
 * dspark_markov_draft computes, with its scratch in a fixed array of
 * DSPARK_NOALLOC_SCRATCH_BYTES inside the library's device memory, which every
 * GPU that loads the library holds until the process exits.  Inputs and outputs
 * are the caller's, as above.  It allocates nothing.
 *  - With CUDA's lazy module loading the array is loaded, and so takes device
 *    memory, when its device address is first looked up on a device.  Call
 *    dspark_noalloc_init once per device at start-up, with that device
 *    current, before the caller's pool reserves HBM and before any stream
 *    capture; otherwise the first draft call on the device does the lookup.
 *  - All calls share the one array: calls whose work overlaps on the GPU race.
 *    Each call clears what must start at zero, the status word included.
 *    Errors that the kernels detect (a bounded wait that gave up, a
 *    non-finite logit, an anchor outside [0, V)) are recorded in the array's
 *    status word; dspark_noalloc_read_status returns and clears it.
 *  - Sizes whose draft scratch (about 8 * gamma * B bytes per vocabulary slice
 *    of the draft kernel) exceeds the array return DSPARK_ERR_WORKSPACE before
 *    anything is enqueued.
 */
#define DSPARK_NOALLOC_SCRATCH_BYTES (4u << 20)
int dspark_markov_draft_noalloc(const float* U, const void* W1, const void* W2, int wdtype,
                                const int32_t* anchor, int B, int gamma, int V, int r,
                                uint64_t seed, uint64_t round,
                                int32_t* x_out, float* p_out, float* lse_out, void* stream);

/* Looks up the no-allocation draft's scratch array on the current device (and
 * so loads it there); DSPARK_OK or DSPARK_ERR_CUDA.  No counterpart on the
 * pages: it lets a caller that cannot allocate later place this one-time cost
 * at start-up. */
int dspark_noalloc_init(void);

/* Waits for `stream`, then copies the status word of the no-allocation draft's
 * scratch array (what the kernels of the latest dspark_markov_draft_noalloc
 * call recorded, a DSPARK_* code) to *host_status and clears it.  Returns
 * DSPARK_OK, DSPARK_ERR_INVALID (null host_status) or DSPARK_ERR_CUDA. */
int dspark_noalloc_read_status(int* host_status, void* stream);

/*
 * Self-test of the device-side bounded waits (no counterpart on the pages).
 * Enqueues one small kernel whose wait can never be satisfied -- mode 0 an
 * mbarrier that no thread arrives on, mode 1 a grid barrier that expects two
 * CTAs in a one-CTA grid.  The wait gives up after the library's limit (1 s),
 * records DSPARK_ERR_TIMEOUT in the status word and the kernel returns; the
 * CUDA context stays usable.  Read the result with dspark_read_status.
 * Uses (and overwrites) the first 256 bytes of `workspace` (256-byte aligned,
 * workspace_bytes >= 256).  Returns DSPARK_ERR_INVALID for another mode.
 */
int dspark_selftest_wait_timeout(int mode, void* workspace, size_t workspace_bytes, void* stream);

/* Waits for `stream`, then copies the workspace status word (a DSPARK_* code,
 * the first error any kernel recorded since the last clear) to *host_status and
 * clears it.  Returns DSPARK_OK or DSPARK_ERR_CUDA. */
int dspark_read_status(void* workspace, int* host_status, void* stream);

/* Static text for a status code. */
const char* dspark_strerror(int status);

#ifdef __cplusplus
}
#endif

#endif /* DSPARK_H */
