// The C ABI of libdspark: host-side argument checks, workspace checks and the
// enqueueing of the per-round kernels.  Every entry point validates its sizes
// and pointers before it enqueues anything and never synchronises the stream.
#include <stdint.h>

#include "kernels.h"

using namespace dspark;

namespace {

bool aligned(const void* p, size_t a) { return ((uintptr_t)p % a) == 0; }

int check_ws(void* ws, size_t ws_bytes, int B, int gamma, int V) {
  if (!ws || !aligned(ws, 256)) return DSPARK_ERR_WORKSPACE;
  if (ws_bytes < ws_layout(B, gamma, V).total) return DSPARK_ERR_WORKSPACE;
  return DSPARK_OK;
}

int cuda_status(cudaError_t e) { return e == cudaSuccess ? DSPARK_OK : DSPARK_ERR_CUDA; }

#define DSPARK_TRY(expr)            \
  do {                              \
    const int _st = (expr);         \
    if (_st != DSPARK_OK) return _st; \
  } while (0)

int draft_checks(const float* U, const void* W1, const void* W2, int wdtype, const int32_t* anchor, int B,
                 int gamma, int V, int r, int32_t* x_out, float* p_out, float* lse_out, void* ws,
                 size_t ws_bytes) {
  DSPARK_TRY(draft_arg_checks(U, W1, W2, wdtype, anchor, B, gamma, V, r, x_out, p_out, lse_out));
  return check_ws(ws, ws_bytes, B, gamma, V);
}

int confidence_checks(const void* h, int hdtype, const void* W1, int wdtype, const float* w,
                      const int32_t* anchor, const int32_t* x, int B, int gamma, int H, int r, int V,
                      float* c_out) {
  DSPARK_TRY(check_dtype(hdtype));
  DSPARK_TRY(check_dtype(wdtype));
  if (B <= 0 || gamma <= 0 || H < 0 || r <= 0 || V <= 0) return DSPARK_ERR_INVALID;
  if (gamma > kMaxGamma || B > 65535) return DSPARK_ERR_UNSUPPORTED;
  if ((H > 0 && !h) || !W1 || !w || !anchor || !x || !c_out) return DSPARK_ERR_INVALID;
  return DSPARK_OK;
}

int schedule_checks(const float* c, int B, int gamma, const float* sps, int n_sps, int mode,
                    const int32_t* khist, const int32_t* ell_out, const int32_t* nstar_out,
                    const double* theta_out) {
  if (B <= 0 || gamma <= 0) return DSPARK_ERR_INVALID;
  if (mode < DSPARK_SCHED_FIXED || mode > DSPARK_SCHED_TOPK) return DSPARK_ERR_INVALID;
  // the candidate sort holds B * gamma keys in one CTA's shared memory; the
  // fixed mode sorts nothing
  if (gamma > kMaxGamma || (mode != DSPARK_SCHED_FIXED && (long long)B * gamma > kMaxCandidates))
    return DSPARK_ERR_UNSUPPORTED;
  if (!c || !ell_out || !nstar_out || !theta_out) return DSPARK_ERR_INVALID;
  if (mode != DSPARK_SCHED_FIXED && (!sps || (long long)n_sps <= (long long)B * (gamma + 1)))
    return DSPARK_ERR_INVALID;
  if (mode == DSPARK_SCHED_TOPK && !khist) return DSPARK_ERR_INVALID;
  return DSPARK_OK;
}

int verify_checks(const float* T, const float* U, const void* W1, const void* W2, int wdtype,
                  const int32_t* anchor, const int32_t* x, const float* p_d, const float* lse_d,
                  const int32_t* ell, int B, int gamma, int V, int r, int32_t* n_out, int32_t* tok_out,
                  void* ws, size_t ws_bytes) {
  DSPARK_TRY(check_shapes(B, gamma, V, r));
  DSPARK_TRY(check_dtype(wdtype));
  if (!T || !U || !W1 || !W2 || !anchor || !x || !p_d || !lse_d || !ell || !n_out || !tok_out)
    return DSPARK_ERR_INVALID;
  if (!aligned(T, 16) || !aligned(U, 16)) return DSPARK_ERR_INVALID;
  return check_ws(ws, ws_bytes, B, gamma, V);
}

}  // namespace

extern "C" {

size_t dspark_workspace_size(int B, int gamma, int V) {
  if (B <= 0 || gamma <= 0 || V <= 0) return 0;
  return ws_layout(B, gamma, V).total;
}

int dspark_markov_draft_ex(const float* U, const float* T_early, const void* W1, const void* W2, int wdtype,
                           const int32_t* anchor, int B, int gamma, int V, int r, uint64_t seed, uint64_t round,
                           const uint64_t* round_dev, int32_t* x_out, float* p_out, float* lse_out,
                           void* workspace, size_t workspace_bytes, void* stream) {
  DSPARK_TRY(draft_checks(U, W1, W2, wdtype, anchor, B, gamma, V, r, x_out, p_out, lse_out, workspace,
                          workspace_bytes));
  if (round >= (1ull << 29)) return DSPARK_ERR_INVALID;
  if (T_early && !aligned(T_early, 16)) return DSPARK_ERR_INVALID;
  DraftArgs a{U, W1, W2, wdtype, anchor, B, gamma, V, r,
              make_rng_key(seed, round, reinterpret_cast<const unsigned long long*>(round_dev)), x_out, p_out,
              lse_out, workspace, T_early};
  return cuda_status(launch_markov_draft(a, (cudaStream_t)stream));
}

int dspark_gated_markov_draft(const float* U, const float* T_early, const void* W1, const void* W2, int wdtype,
                              const float* gate_g, const float* gate_c, const int32_t* anchor, int B, int gamma,
                              int V, int r, uint64_t seed, uint64_t round, const uint64_t* round_dev,
                              int32_t* x_out, float* p_out, float* lse_out, void* workspace, size_t workspace_bytes,
                              void* stream) {
  DSPARK_TRY(draft_checks(U, W1, W2, wdtype, anchor, B, gamma, V, r, x_out, p_out, lse_out, workspace,
                          workspace_bytes));
  if (round >= (1ull << 29)) return DSPARK_ERR_INVALID;
  if (T_early && !aligned(T_early, 16)) return DSPARK_ERR_INVALID;
  if (!gate_g || !gate_c || !aligned(gate_g, 16) || !aligned(gate_c, 16)) return DSPARK_ERR_INVALID;
  if (!draft_tc_supported(wdtype, r, V)) return DSPARK_ERR_UNSUPPORTED;
  DraftArgs a{U, W1, W2, wdtype, anchor, B, gamma, V, r,
              make_rng_key(seed, round, reinterpret_cast<const unsigned long long*>(round_dev)), x_out, p_out,
              lse_out, workspace, T_early};
  a.gate_g = gate_g;
  a.gate_c = gate_c;
  return cuda_status(launch_markov_draft(a, (cudaStream_t)stream));
}

int dspark_markov_draft(const float* U, const void* W1, const void* W2, int wdtype, const int32_t* anchor,
                        int B, int gamma, int V, int r, uint64_t seed, uint64_t round, int32_t* x_out,
                        float* p_out, float* lse_out, void* workspace, size_t workspace_bytes,
                        void* stream) {
  return dspark_markov_draft_ex(U, nullptr, W1, W2, wdtype, anchor, B, gamma, V, r, seed, round, nullptr, x_out,
                                p_out, lse_out, workspace, workspace_bytes, stream);
}

int dspark_confidence(const void* h, int hdtype, const void* W1, int wdtype, const float* w,
                      const float* sts_T, const int32_t* anchor, const int32_t* x, int B, int gamma, int H,
                      int r, int V, float* c_out, void* stream) {
  DSPARK_TRY(confidence_checks(h, hdtype, W1, wdtype, w, anchor, x, B, gamma, H, r, V, c_out));
  // The confidence call has no workspace: its kernel reports range errors by
  // writing 0 confidences; the status word is only used by the round entry.
  return cuda_status(launch_confidence(h, hdtype, W1, wdtype, w, sts_T, anchor, x, B, gamma, H, r, V, c_out,
                                       nullptr, (cudaStream_t)stream));
}

int dspark_schedule_ex(const float* c, int B, int gamma, const float* sps, int n_sps, int mode, uint64_t round,
                       const uint64_t* round_dev, int32_t* khist, int32_t* ell_out, int32_t* nstar_out,
                       double* theta_out, void* workspace, size_t workspace_bytes, void* stream) {
  DSPARK_TRY(schedule_checks(c, B, gamma, sps, n_sps, mode, khist, ell_out, nstar_out, theta_out));
  if (!workspace || !aligned(workspace, 256) || workspace_bytes < 256) return DSPARK_ERR_WORKSPACE;
  int* status = ws_ptr<int>(workspace, 0);
  return cuda_status(launch_schedule(c, B, gamma, sps, mode, round,
                                     reinterpret_cast<const unsigned long long*>(round_dev), khist, ell_out,
                                     nstar_out, theta_out, status, (cudaStream_t)stream));
}

int dspark_schedule(const float* c, int B, int gamma, const float* sps, int n_sps, int mode, uint64_t round,
                    int32_t* khist, int32_t* ell_out, int32_t* nstar_out, double* theta_out, void* workspace,
                    size_t workspace_bytes, void* stream) {
  return dspark_schedule_ex(c, B, gamma, sps, n_sps, mode, round, nullptr, khist, ell_out, nstar_out, theta_out,
                            workspace, workspace_bytes, stream);
}

int dspark_verify_ex(const float* T, const float* U, const void* W1, const void* W2, int wdtype,
                     const int32_t* anchor, const int32_t* x, const float* p_d, const float* lse_d,
                     const int32_t* ell, int B, int gamma, int V, int r, uint64_t seed, uint64_t round,
                     uint64_t* round_dev, unsigned flags, int32_t* n_out, int32_t* tok_out, void* workspace,
                     size_t workspace_bytes, void* stream) {
  DSPARK_TRY(verify_checks(T, U, W1, W2, wdtype, anchor, x, p_d, lse_d, ell, B, gamma, V, r, n_out, tok_out,
                           workspace, workspace_bytes));
  if (round >= (1ull << 29)) return DSPARK_ERR_INVALID;
  if (flags & ~(unsigned)(DSPARK_EARLY_TARGET_STATS | DSPARK_ADVANCE_ROUND | DSPARK_SCRATCH_FROM_DRAFT |
                          DSPARK_GATED_STATES | DSPARK_ALL_ROW_STATS))
    return DSPARK_ERR_INVALID;
  if ((flags & DSPARK_EARLY_TARGET_STATS) && (flags & DSPARK_ALL_ROW_STATS)) return DSPARK_ERR_INVALID;
  if ((flags & DSPARK_GATED_STATES) && !draft_tc_supported(wdtype, r, V)) return DSPARK_ERR_UNSUPPORTED;
  if ((flags & DSPARK_ADVANCE_ROUND) && !round_dev) return DSPARK_ERR_INVALID;
  unsigned long long* rd = reinterpret_cast<unsigned long long*>(round_dev);
  // only the tensor-core draft of dspark_draft_schedule clears the scratch
  const bool zeroed = (flags & DSPARK_SCRATCH_FROM_DRAFT) && draft_tc_supported(wdtype, r, V);
  VerifyArgs a{T, U, W1, W2, wdtype, anchor, x, p_d, lse_d, ell, B, gamma, V, r, make_rng_key(seed, round, rd),
               n_out, tok_out, workspace, (flags & DSPARK_EARLY_TARGET_STATS) != 0,
               (flags & DSPARK_ADVANCE_ROUND) ? rd : nullptr, zeroed, (flags & DSPARK_GATED_STATES) != 0,
               (flags & DSPARK_ALL_ROW_STATS) != 0};
  return cuda_status(launch_verify(a, (cudaStream_t)stream));
}

int dspark_verify(const float* T, const float* U, const void* W1, const void* W2, int wdtype,
                  const int32_t* anchor, const int32_t* x, const float* p_d, const float* lse_d,
                  const int32_t* ell, int B, int gamma, int V, int r, uint64_t seed, uint64_t round,
                  int32_t* n_out, int32_t* tok_out, void* workspace, size_t workspace_bytes, void* stream) {
  return dspark_verify_ex(T, U, W1, W2, wdtype, anchor, x, p_d, lse_d, ell, B, gamma, V, r, seed, round, nullptr,
                          0u, n_out, tok_out, workspace, workspace_bytes, stream);
}

size_t dspark_sts_workspace_size(int N, int gamma, int ngrid) {
  if (N <= 0 || gamma <= 0 || ngrid <= 0) return 0;
  return sts_workspace_bytes(N, ngrid);
}

int dspark_sts_fit(const float* z, const int32_t* ell, const int32_t* acc, int N, int gamma, const float* grid,
                   int ngrid, float* T_out, float* ece_out, void* workspace, size_t workspace_bytes, void* stream) {
  if (!z || !ell || !acc || !grid || !T_out || !ece_out) return DSPARK_ERR_INVALID;
  if (N <= 0 || gamma <= 0 || ngrid <= 0) return DSPARK_ERR_INVALID;
  if (gamma > kMaxGamma || ngrid > kMaxStsGrid) return DSPARK_ERR_UNSUPPORTED;
  if (!workspace || !aligned(workspace, 256) || workspace_bytes < sts_workspace_bytes(N, ngrid))
    return DSPARK_ERR_WORKSPACE;
  return cuda_status(launch_sts_fit(z, ell, acc, N, gamma, grid, ngrid, T_out, ece_out, workspace,
                                    (cudaStream_t)stream));
}

int dspark_acceptance_label_ex(const float* T, const float* U, const void* W1, const void* W2, int wdtype,
                               const int32_t* anchor, const int32_t* x, const float* lse_d, const int32_t* ell, int B,
                               int gamma, int V, int r, unsigned flags, float* label_out, void* workspace,
                               size_t workspace_bytes, void* stream) {
  DSPARK_TRY(check_shapes(B, gamma, V, r));
  DSPARK_TRY(check_dtype(wdtype));
  if (!T || !U || !W1 || !W2 || !anchor || !x || !lse_d || !ell || !label_out) return DSPARK_ERR_INVALID;
  if (!aligned(T, 16) || !aligned(U, 16)) return DSPARK_ERR_INVALID;
  DSPARK_TRY(check_ws(workspace, workspace_bytes, B, gamma, V));
  if (flags & ~(unsigned)(DSPARK_EARLY_TARGET_STATS | DSPARK_TARGET_STATS_FROM_VERIFY)) return DSPARK_ERR_INVALID;
  if ((flags & DSPARK_EARLY_TARGET_STATS) && (flags & DSPARK_TARGET_STATS_FROM_VERIFY)) return DSPARK_ERR_INVALID;
  if (!draft_tc_supported(wdtype, r, V)) return DSPARK_ERR_UNSUPPORTED;
  cudaStream_t s = (cudaStream_t)stream;
  const WsLayout L = ws_layout(B, gamma, V);
  DSPARK_TRY(cuda_status(cudaMemsetAsync(label_out, 0, sizeof(float) * (size_t)B * gamma, s)));
  // the target rows' softmax partials: taken along by a draft (rows j < gamma,
  // kStatsSeg segments), left by a verification (rows j < ell, kVerifySeg
  // segments), or taken here
  int nsegs = verify_num_segs(V);
  if (flags & DSPARK_EARLY_TARGET_STATS) nsegs = stats_num_segs(V);
  else if (!(flags & DSPARK_TARGET_STATS_FROM_VERIFY))
    DSPARK_TRY(cuda_status(launch_row_stats(T, ell, B, gamma, V, workspace, s)));
  int* counters = ws_ptr<int>(workspace, L.counters);
  return cuda_status(launch_acceptance_label_tc(T, U, W1, W2, anchor, x, lse_d, ell,
                                                ws_ptr<float2>(workspace, L.row_part), nsegs,
                                                (flags & DSPARK_EARLY_TARGET_STATS) ? counters + 2 : nullptr,
                                                (flags & DSPARK_TARGET_STATS_FROM_VERIFY) ? counters + 4 : nullptr,
                                                label_out, B, gamma, V, ws_ptr<int>(workspace, L.status), s));
}

int dspark_acceptance_label(const float* T, const float* U, const void* W1, const void* W2, int wdtype,
                            const int32_t* anchor, const int32_t* x, const float* lse_d, const int32_t* ell, int B,
                            int gamma, int V, int r, float* label_out, void* workspace, size_t workspace_bytes,
                            void* stream) {
  return dspark_acceptance_label_ex(T, U, W1, W2, wdtype, anchor, x, lse_d, ell, B, gamma, V, r, 0u, label_out,
                                    workspace, workspace_bytes, stream);
}

int dspark_draft_schedule_ex(const float* U, const float* T_early, const void* W1, const void* W2, int wdtype,
                             const void* h, int hdtype, const float* w, const float* sts_T, const int32_t* anchor,
                             int B, int gamma, int V, int r, int H, const float* sps, int n_sps, int mode,
                             int32_t* khist, uint64_t seed, uint64_t round, uint64_t* round_dev, unsigned flags,
                             int32_t* x_out, float* p_out, float* lse_out, float* c_out, int32_t* ell_out,
                             int32_t* nstar_out, double* theta_out, void* workspace, size_t workspace_bytes,
                             void* stream) {
  DSPARK_TRY(draft_checks(U, W1, W2, wdtype, anchor, B, gamma, V, r, x_out, p_out, lse_out, workspace,
                          workspace_bytes));
  if (flags & ~(unsigned)DSPARK_CHAIN_TARGET_STATS) return DSPARK_ERR_INVALID;
  if ((flags & DSPARK_CHAIN_TARGET_STATS) && !T_early) return DSPARK_ERR_INVALID;
  DSPARK_TRY(confidence_checks(h, hdtype, W1, wdtype, w, anchor, x_out, B, gamma, H, r, V, c_out));
  DSPARK_TRY(schedule_checks(c_out, B, gamma, sps, n_sps, mode, khist, ell_out, nstar_out, theta_out));
  if (round >= (1ull << 29)) return DSPARK_ERR_INVALID;
  if (T_early && !aligned(T_early, 16)) return DSPARK_ERR_INVALID;
  cudaStream_t s = (cudaStream_t)stream;
  unsigned long long* rd = reinterpret_cast<unsigned long long*>(round_dev);
  const RngKey key = make_rng_key(seed, round, rd);
  int* status = ws_ptr<int>(workspace, ws_layout(B, gamma, V).status);
  // The tensor-core draft computes the confidence head in its finalize, runs
  // the schedule in its last CTA and clears the verification's scratch on its
  // way; the CUDA-core draft is followed by the confidence and schedule kernels.
  const bool tc = draft_tc_supported(wdtype, r, V);
  DraftArgs da{U, W1, W2, wdtype, anchor, B, gamma, V, r, key, x_out, p_out, lse_out, workspace, T_early, tc,
               h, hdtype, w, sts_T, H, tc ? c_out : nullptr, sps, mode, khist, tc ? ell_out : nullptr, nstar_out,
               theta_out};
  da.chain_stats = (flags & DSPARK_CHAIN_TARGET_STATS) != 0;
  DSPARK_TRY(cuda_status(launch_markov_draft(da, s)));
  if (!tc) {
    DSPARK_TRY(cuda_status(launch_confidence(h, hdtype, W1, wdtype, w, sts_T, anchor, x_out, B, gamma, H, r, V,
                                             c_out, status, s)));
    DSPARK_TRY(cuda_status(launch_schedule(c_out, B, gamma, sps, mode, round, rd, khist, ell_out, nstar_out,
                                           theta_out, status, s)));
  }
  return DSPARK_OK;
}

int dspark_draft_schedule(const float* U, const float* T_early, const void* W1, const void* W2, int wdtype,
                          const void* h, int hdtype, const float* w, const float* sts_T, const int32_t* anchor, int B,
                          int gamma, int V, int r, int H, const float* sps, int n_sps, int mode, int32_t* khist,
                          uint64_t seed, uint64_t round, uint64_t* round_dev, int32_t* x_out, float* p_out,
                          float* lse_out, float* c_out, int32_t* ell_out, int32_t* nstar_out, double* theta_out,
                          void* workspace, size_t workspace_bytes, void* stream) {
  return dspark_draft_schedule_ex(U, T_early, W1, W2, wdtype, h, hdtype, w, sts_T, anchor, B, gamma, V, r, H, sps,
                                  n_sps, mode, khist, seed, round, round_dev, 0u, x_out, p_out, lse_out, c_out, ell_out,
                                  nstar_out, theta_out, workspace, workspace_bytes, stream);
}

int dspark_round_ex(const float* U, const float* T, const void* W1, const void* W2, int wdtype, const void* h,
                    int hdtype, const float* w, const float* sts_T, const int32_t* anchor, int B, int gamma, int V,
                    int r, int H, const float* sps, int n_sps, int mode, int32_t* khist, uint64_t seed,
                    uint64_t round, uint64_t* round_dev, unsigned flags, int32_t* x_out, float* p_out,
                    float* lse_out, float* c_out, int32_t* ell_out, int32_t* nstar_out, double* theta_out,
                    int32_t* n_out, int32_t* tok_out, void* workspace, size_t workspace_bytes, void* stream) {
  DSPARK_TRY(verify_checks(T, U, W1, W2, wdtype, anchor, x_out, p_out, lse_out, ell_out, B, gamma, V, r, n_out,
                           tok_out, workspace, workspace_bytes));
  if (flags & ~(unsigned)(DSPARK_EARLY_TARGET_STATS | DSPARK_ADVANCE_ROUND | DSPARK_ALL_ROW_STATS |
                          DSPARK_CHAIN_TARGET_STATS))
    return DSPARK_ERR_INVALID;
  const unsigned forms = flags & (DSPARK_EARLY_TARGET_STATS | DSPARK_ALL_ROW_STATS | DSPARK_CHAIN_TARGET_STATS);
  if (forms & (forms - 1)) return DSPARK_ERR_INVALID;   // at most one of the three
  if ((flags & DSPARK_ADVANCE_ROUND) && !round_dev) return DSPARK_ERR_INVALID;
  // the draft takes the target rows' statistics (every row j < gamma, or the
  // rows the accept chains reach) and verification decides on them
  const bool early = (flags & (DSPARK_EARLY_TARGET_STATS | DSPARK_CHAIN_TARGET_STATS)) != 0;
  DSPARK_TRY(dspark_draft_schedule_ex(U, early ? T : nullptr, W1, W2, wdtype, h, hdtype, w, sts_T, anchor, B, gamma,
                                      V, r, H, sps, n_sps, mode, khist, seed, round, round_dev,
                                      flags & DSPARK_CHAIN_TARGET_STATS, x_out, p_out, lse_out, c_out, ell_out,
                                      nstar_out, theta_out, workspace, workspace_bytes, stream));
  unsigned vflags = (flags & ~(unsigned)DSPARK_CHAIN_TARGET_STATS) | DSPARK_SCRATCH_FROM_DRAFT;
  if (early) vflags |= DSPARK_EARLY_TARGET_STATS;
  return dspark_verify_ex(T, U, W1, W2, wdtype, anchor, x_out, p_out, lse_out, ell_out, B, gamma, V, r, seed, round,
                          round_dev, vflags, n_out, tok_out, workspace, workspace_bytes, stream);
}

int dspark_round(const float* U, const float* T, const void* W1, const void* W2, int wdtype, const void* h,
                 int hdtype, const float* w, const float* sts_T, const int32_t* anchor, int B, int gamma, int V,
                 int r, int H, const float* sps, int n_sps, int mode, int32_t* khist, uint64_t seed,
                 uint64_t round, int32_t* x_out, float* p_out, float* lse_out, float* c_out, int32_t* ell_out,
                 int32_t* nstar_out, double* theta_out, int32_t* n_out, int32_t* tok_out, void* workspace,
                 size_t workspace_bytes, void* stream) {
  return dspark_round_ex(U, T, W1, W2, wdtype, h, hdtype, w, sts_T, anchor, B, gamma, V, r, H, sps, n_sps, mode,
                         khist, seed, round, nullptr, 0u, x_out, p_out, lse_out, c_out, ell_out, nstar_out,
                         theta_out, n_out, tok_out, workspace, workspace_bytes, stream);
}

int dspark_selftest_wait_timeout(int mode, void* workspace, size_t workspace_bytes, void* stream) {
  if (mode != 0 && mode != 1) return DSPARK_ERR_INVALID;
  if (!workspace || !aligned(workspace, 256) || workspace_bytes < 256) return DSPARK_ERR_WORKSPACE;
  return cuda_status(launch_selftest_wait(mode, workspace, (cudaStream_t)stream));
}

int dspark_read_status(void* workspace, int* host_status, void* stream) {
  if (!workspace || !host_status) return DSPARK_ERR_INVALID;
  cudaStream_t s = (cudaStream_t)stream;
  int* status = ws_ptr<int>(workspace, 0);
  int value = 0;
  if (cudaMemcpyAsync(&value, status, sizeof(int), cudaMemcpyDeviceToHost, s) != cudaSuccess) return DSPARK_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return DSPARK_ERR_CUDA;
  if (cudaMemsetAsync(status, 0, sizeof(int), s) != cudaSuccess) return DSPARK_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return DSPARK_ERR_CUDA;
  *host_status = value;
  return DSPARK_OK;
}

const char* dspark_strerror(int status) {
  switch (status) {
    case DSPARK_OK: return "ok";
    case DSPARK_ERR_INVALID: return "invalid argument (null pointer, size or table length)";
    case DSPARK_ERR_UNSUPPORTED: return "unsupported size (B > 65535, gamma > 32, V % 8, r % 16 or r > 256, B*gamma > 8192 for a sorting schedule)";
    case DSPARK_ERR_CUDA: return "a CUDA launch or runtime call failed";
    case DSPARK_ERR_TIMEOUT: return "a device-side bounded wait gave up";
    case DSPARK_ERR_WORKSPACE: return "workspace missing, misaligned (256 B) or smaller than dspark_workspace_size";
    case DSPARK_ERR_NONFINITE: return "a NaN or infinite logit or confidence was met";
    default: return "unknown status";
  }
}

}  // extern "C"
