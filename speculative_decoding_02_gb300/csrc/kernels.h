// Internal launch functions of libdspark (host side).  Each enqueues its
// kernels on `stream` and returns the cudaError_t of the launch.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <utility>

#include "common.cuh"

namespace dspark {

// Launches kern with the programmatic stream-serialization attribute: it may
// start while the previous kernel in the stream runs, and it calls pdl_wait()
// before it touches anything an earlier kernel writes or reads.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                              Args&&... args) {
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

struct DraftArgs {
  const float* U;
  const void* W1;
  const void* W2;
  int wdtype;
  const int32_t* anchor;
  int B, gamma, V, r;
  RngKey key;
  int32_t* x_out;
  float* p_out;
  float* lse_out;
  void* ws;
  // optional: target logits [B, gamma+1, V] whose rows j < gamma get their
  // softmax statistics into the workspace during (or right after) the draft
  const float* T_stats;
  // the tensor-core draft clears the verification's scratch (its argmax keys
  // and bonus list) at its start, so that the verification that follows in
  // the same round needs no memset of its own
  bool zero_verify_scratch;
  // optional (c_out not null): the confidence head of every position, computed
  // by the tensor-core draft's finalize (draft_tc_supported); the CUDA-core
  // draft ignores it and the caller runs launch_confidence instead
  const void* h;
  int hdtype;
  const float* w;
  const float* sts_T;
  int H;
  float* c_out;
  // optional (ell_out not null, with c_out, tensor-core path): the round's
  // schedule right after the finalize, run by the persistent draft's last CTA
  // while the others stream statistics (up to 4096 candidates), else by the
  // schedule kernel launched after the draft; the CUDA-core draft ignores it
  const float* sps;
  int mode;
  int32_t* khist;
  int32_t* ell_out;
  int32_t* nstar_out;
  double* theta_out;
  // optional: the gated recurrent head's gates g, c [r] (null: the Markov
  // head); tensor-core path only, its states go to the workspace
  const float* gate_g;
  const float* gate_c;
  // with T_stats, tensor-core persistent path: only the rows the accept
  // chains can reach (a row is skipped once its request is known to reject
  // at an earlier position); workspace counter [5] then reads 1
  bool chain_stats;
};

struct VerifyArgs {
  const float* T;
  const float* U;
  const void* W1;
  const void* W2;
  int wdtype;
  const int32_t* anchor;
  const int32_t* x;
  const float* p_d;
  const float* lse_d;
  const int32_t* ell;
  int B, gamma, V, r;
  RngKey key;
  int32_t* n_out;
  int32_t* tok_out;
  void* ws;
  // the draft already left the statistics of the target rows j < gamma in the
  // workspace (DraftArgs::T_stats): skip the row pass
  bool stats_ready;
  // when not null, the round's last kernel adds 1 to this device round index
  unsigned long long* advance_round;
  // the draft of this round cleared the scratch (DraftArgs::zero_verify_scratch)
  bool scratch_zeroed;
  // the draft used the gated recurrent head: its states in the workspace are
  // the residual's bias operand (tensor-core path)
  bool gated_states;
  // without stats_ready: take the statistics of every row j < ell (the classic
  // pass, reusable by the acceptance labels) instead of only the rows each
  // request's accept chain reaches
  bool all_row_stats;
};

// Host-side argument checks shared by every entry point that takes these
// sizes (api.cu and noalloc.cu), so that a limit changed in one place holds
// for all of them.
inline int check_dtype(int dt) { return (dt == DSPARK_F32 || dt == DSPARK_BF16) ? DSPARK_OK : DSPARK_ERR_INVALID; }

// Shapes shared by the draft and verify calls.
inline int check_shapes(int B, int gamma, int V, int r) {
  if (B <= 0 || gamma <= 0 || V <= 0 || r <= 0) return DSPARK_ERR_INVALID;
  if (gamma > kMaxGamma) return DSPARK_ERR_UNSUPPORTED;
  if (V % 8 != 0 || r % 16 != 0 || r > 256) return DSPARK_ERR_UNSUPPORTED;
  if (B > 65535) return DSPARK_ERR_UNSUPPORTED;
  if ((long long)B * (gamma + 1) * (long long)V >= (1ll << 40)) return DSPARK_ERR_UNSUPPORTED;
  return DSPARK_OK;
}

// The pointer and alignment checks of a draft call (everything but the
// workspace).
inline int draft_arg_checks(const float* U, const void* W1, const void* W2, int wdtype, const int32_t* anchor,
                            int B, int gamma, int V, int r, const int32_t* x_out, const float* p_out,
                            const float* lse_out) {
  int st = check_shapes(B, gamma, V, r);
  if (st != DSPARK_OK) return st;
  if ((st = check_dtype(wdtype)) != DSPARK_OK) return st;
  if (!U || !W1 || !W2 || !anchor || !x_out || !p_out || !lse_out) return DSPARK_ERR_INVALID;
  if (((uintptr_t)U | (uintptr_t)W1 | (uintptr_t)W2) % 16 != 0) return DSPARK_ERR_INVALID;
  return DSPARK_OK;
}

cudaError_t launch_markov_draft(const DraftArgs& a, cudaStream_t stream);

// Tensor-core draft (bf16 weights, r = 256, V >= 192); the dispatcher above picks it.
bool draft_tc_supported(int wdtype, int r, int V);

// One small kernel whose wait never completes (mode 0: an mbarrier, mode 1: a
// grid barrier); it gives up after the library's wait limit and records
// DSPARK_ERR_TIMEOUT in the workspace status word.  Uses the workspace's first
// 256 bytes.
cudaError_t launch_selftest_wait(int mode, void* ws, cudaStream_t stream);
cudaError_t launch_markov_draft_tc(const DraftArgs& a, cudaStream_t stream);

// Tensor maps of the tensor-core kernels: W2 [V, 256] bf16 in 64 x `rows` boxes
// (128-byte swizzle, rows <= 256); a [B, G, V] fp32 tensor in [R rows x 1 x 32 columns]
// boxes (128-byte swizzle); the same tensor as [B, G, V / 32, 32] in boxes of
// R rows x 64 columns (make_u_tile_map, 128-byte swizzle, V >= 32), which land
// in shared memory as [row][half][32 columns].
cudaError_t make_w2_tensor_map(const void* W2, int V, CUtensorMap* map, int rows = 192);
cudaError_t make_u_tensor_map(const float* U, int B, int G, int V, int R, CUtensorMap* map);
cudaError_t make_u_tile_map(const float* U, int B, int G, int V, int R, CUtensorMap* map);
cudaError_t launch_residual_tc(const float* T, const float* U, const void* W1, const void* W2,
                               const int32_t* resid_prev, const float* lse_d, const int32_t* resid_k,
                               const float* resid_lse, unsigned long long* resid_key, int B, int G, int V,
                               RngKey key, const void* gstate, unsigned int* fin, int32_t* tok_out, int* status,
                               cudaStream_t stream);

// Acceptance labels (tensor-core path, one persistent launch over the
// positions): sum_v min(p_d, p_t) per verified position into label [B][G]
// (zeroed by the caller), from target-row partials already in the workspace
// (row_part, nsegs per row).
cudaError_t launch_acceptance_label_tc(const float* T, const float* U, const void* W1, const void* W2,
                                       const int32_t* anchor, const int32_t* x, const float* lse_d,
                                       const int32_t* ell, const float2* row_part, int nsegs,
                                       const int* stats_done, const int* full_rows, float* label, int B, int G,
                                       int V, int* status,
                                       cudaStream_t stream);

// The softmax partials of the target rows j < ell_b of every request into the
// workspace (verify's first two kernels); ell == nullptr takes every row
// j < gamma and marks the statistics as complete for a later verify.
cudaError_t launch_row_stats(const float* T, const int32_t* ell, int B, int gamma, int V, void* ws,
                             cudaStream_t stream);

// Sequential temperature scaling (per-position grid search on the prefix
// product, fp64); the workspace holds per-block ECE bin sums.
constexpr int kStsBins = 15;       // ECE bins
constexpr int kStsChunk = 2048;    // samples per block
constexpr int kMaxStsGrid = 256;   // grid values
size_t sts_workspace_bytes(int N, int ngrid);
cudaError_t launch_sts_fit(const float* z, const int32_t* ell, const int32_t* acc, int N, int gamma,
                           const float* grid, int ngrid, float* T_out, float* ece_out, void* ws,
                           cudaStream_t stream);

cudaError_t launch_confidence(const void* h, int hdtype, const void* W1, int wdtype,
                              const float* w, const float* sts_T, const int32_t* anchor,
                              const int32_t* x, int B, int gamma, int H, int r, int V,
                              float* c_out, int* status, cudaStream_t stream);

// `round` is the round index unless round_dev (a device word) is given.
cudaError_t launch_schedule(const float* c, int B, int gamma, const float* sps, int mode,
                            unsigned long long round, const unsigned long long* round_dev, int32_t* khist,
                            int32_t* ell_out, int32_t* nstar_out, double* theta_out, int* status,
                            cudaStream_t stream);

cudaError_t launch_verify(const VerifyArgs& a, cudaStream_t stream);

}  // namespace dspark
