// Semi-autoregressive Markov draft ("[DeepSeek-6] DSpark" blog, sections 3-4;
// study report Eq.4): for each position k the Markov bias of the previous token
// is added to the backbone logits, and the token is drawn from their softmax
// (a Gumbel race over blocks of 4 tokens on their log-mass, then the inverse
// CDF inside the winning block) while an online softmax accumulates the
// normaliser.
//
// CUDA-core path: one launch per position.  A CTA owns 32 requests and one
// kDraftSlice-wide slice of the vocabulary; it gathers the 32 embedding rows
// W1[x_{k-1}] into shared memory once and walks its slice in 64-column tiles of
// W2, computing the bias with fp32 FMAs.  Every (request, slice) pair leaves an
// online-softmax partial (m, s) and pushes its best perturbed block log-mass
// (with the token drawn inside that block) into a per-request 64-bit argmax
// key (atomicMax).  A per-position finalize kernel
// merges the partials into lse_k, decodes x_k and recomputes l_k(x_k) to give
// p_k(x_k).
#include "kernels.h"

namespace dspark {
namespace {

constexpr int kRowsPerCta = 32;
constexpr int kColsPerTile = 64;
constexpr int kThreads = 256;

template <int WDT>
__global__ void __launch_bounds__(kThreads)
draft_step_cuda_core(const float* __restrict__ U, const void* __restrict__ W1,
                     const void* __restrict__ W2, const int32_t* __restrict__ prev_tok,
                     int prev_stride, int B, int G, int V, int r, int k, RngKey key_arg,
                     float2* __restrict__ part, unsigned long long* __restrict__ keys,
                     int* __restrict__ status) {
  const RngKey key = live_key(key_arg);
  extern __shared__ float smem[];
  float* Es = smem;                          // [kRowsPerCta][r]
  float* Ws = Es + kRowsPerCta * r;          // [kColsPerTile][r + 1]
  const int ldw = r + 1;
  const int slice = blockIdx.x;
  const int b0 = blockIdx.y * kRowsPerCta;
  const int v_begin = slice * kDraftSlice;
  const int v_end = min(V, v_begin + kDraftSlice);
  const int tid = threadIdx.x;

  for (int idx = tid; idx < kRowsPerCta * r; idx += kThreads) {
    const int m = idx / r, i = idx - (idx / r) * r;
    const int b = b0 + m;
    float e = 0.f;
    if (b < B) {
      const int p = checked_token(prev_tok[(size_t)b * prev_stride], V, status);
      e = load_weight<WDT>(W1, (size_t)p * r + i);
    }
    Es[idx] = e;
  }

  const int m = tid >> 3;              // request row inside the CTA
  const int cg = (tid & 7) * 8;        // first of this thread's 8 columns in a tile
  const int b = b0 + m;
  const bool row_ok = b < B;
  const float* Urow = U + ((size_t)(row_ok ? b : 0) * G + (k - 1)) * (size_t)V;
  float run_m = -INFINITY, run_s = 0.f;
  unsigned long long best = 0ull;
  bool bad = false;

  for (int vt = v_begin; vt < v_end; vt += kColsPerTile) {
    __syncthreads();
    for (int idx = tid; idx < kColsPerTile * r; idx += kThreads) {
      const int c = idx / r, i = idx - (idx / r) * r;
      const int v = vt + c;
      Ws[c * ldw + i] = (v < v_end) ? load_weight<WDT>(W2, (size_t)v * r + i) : 0.f;
    }
    __syncthreads();
    float acc[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) acc[j] = 0.f;
    for (int i = 0; i < r; ++i) {
      const float e = Es[m * r + i];
#pragma unroll
      for (int j = 0; j < 8; ++j) acc[j] = fmaf(e, Ws[(cg + j) * ldw + i], acc[j]);
    }
    if (!row_ok) continue;
#pragma unroll
    for (int q = 0; q < 2; ++q) {
      // one block of 4 tokens (blocks never straddle v_end: V % 8 == 0)
      const int v4 = vt + cg + 4 * q;
      if (v4 >= v_end) continue;
      float l[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        l[j] = Urow[v4 + j] + acc[4 * q + j];
        bad |= !isfinite(l[j]);
      }
      // online softmax over the block's terms, and the block's own log-mass
      const float m4 = fmaxf(fmaxf(l[0], l[1]), fmaxf(l[2], l[3]));
      if (m4 == -INFINITY) continue;   // no mass in this block
      float e[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) e[j] = expf(l[j] - m4);
      const float s4 = ((e[0] + e[1]) + e[2]) + e[3];
      if (m4 > run_m) {
        run_s = (run_m == -INFINITY ? 0.f : run_s * expf(run_m - m4)) + s4;
        run_m = m4;
      } else {
        run_s += s4 * expf(m4 - run_m);
      }
      // the block's perturbed log-mass; the token inside it only when it
      // could still win this thread's race
      const uint32_t jb = (uint32_t)v4 >> 2;
      const uint32_t w = word_of(rng_call(key, kStreamDraft, (uint32_t)b, (uint32_t)k, jb >> 2), jb & 3u);
      const float z = m4 + logf(s4) + gumbel_from_bits(w >> 9);
      if (argmax_key(z, v4) > best) {
        const int v = block_pick(key, kStreamDraft, (uint32_t)b, (uint32_t)k, jb, e[0], e[1], e[2], e[3]);
        const unsigned long long kz = argmax_key(z, v);
        best = kz > best ? kz : best;
      }
    }
  }
  // the 8 threads of a request row are 8 consecutive lanes
  warp_softmax_reduce(run_m, run_s, 0xffffffffu, 8);
  best = warp_max_u64(best, 0xffffffffu, 8);
  if (row_ok && (tid & 7) == 0) {
    part[(size_t)b * gridDim.x + slice] = make_float2(run_m, run_s);
    atomicMax(&keys[(size_t)b * kKeyStride], best);
  }
  if (bad) record_status(status, DSPARK_ERR_NONFINITE);
}

// One warp per request: merge the slice partials into lse_k, decode x_k and
// recompute the fused logit of x_k for p_k(x_k).
template <int WDT>
__global__ void draft_finalize(const float* __restrict__ U, const void* __restrict__ W1,
                               const void* __restrict__ W2, const int32_t* __restrict__ prev_tok,
                               int prev_stride, int B, int G, int V, int r, int k, int nslices,
                               const float2* __restrict__ part,
                               const unsigned long long* __restrict__ keys,
                               int32_t* __restrict__ x_out, float* __restrict__ p_out,
                               float* __restrict__ lse_out, int* __restrict__ status) {
  const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (warp >= B) return;
  const int b = warp;
  float m = -INFINITY, s = 0.f;
  for (int i = lane; i < nslices; i += 32) {
    const float2 pr = part[(size_t)b * nslices + i];
    softmax_merge(m, s, pr.x, pr.y);
  }
  warp_softmax_reduce(m, s, 0xffffffffu, 32);
  const float lse = m + logf(s);
  const unsigned long long kk = keys[(size_t)b * kKeyStride];
  int x = argmax_key_index(kk);
  if (kk == 0ull || x < 0 || x >= V) {
    if (lane == 0) record_status(status, DSPARK_ERR_NONFINITE);
    x = 0;
  }
  const int prev = checked_token(prev_tok[(size_t)b * prev_stride], V, status);
  float dot = 0.f;
  for (int i = lane; i < r; i += 32)
    dot = fmaf(load_weight<WDT>(W1, (size_t)prev * r + i), load_weight<WDT>(W2, (size_t)x * r + i), dot);
  for (int off = 16; off > 0; off >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, off);
  if (lane == 0) {
    const size_t o = (size_t)b * G + (k - 1);
    const float l = U[o * (size_t)V + x] + dot;
    x_out[o] = x;
    p_out[o] = expf(l - lse);
    lse_out[o] = lse;
  }
}

template <int WDT>
cudaError_t run_draft(const DraftArgs& a, cudaStream_t stream) {
  const WsLayout L = ws_layout(a.B, a.gamma, a.V);
  int* status = ws_ptr<int>(a.ws, L.status);
  unsigned long long* keys = ws_ptr<unsigned long long>(a.ws, L.draft_keys);
  float2* part = ws_ptr<float2>(a.ws, L.draft_part);
  const int nslices = draft_num_slices(a.V);
  cudaError_t e = cudaMemsetAsync(keys, 0, sizeof(unsigned long long) * kKeyStride * (size_t)a.gamma * a.B, stream);
  if (e != cudaSuccess) return e;
  const size_t smem = sizeof(float) * ((size_t)kRowsPerCta * a.r + (size_t)kColsPerTile * (a.r + 1));
  e = cudaFuncSetAttribute(draft_step_cuda_core<WDT>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  const dim3 grid(nslices, div_up(a.B, kRowsPerCta));
  for (int k = 1; k <= a.gamma; ++k) {
    const int32_t* prev = (k == 1) ? a.anchor : a.x_out + (k - 2);
    const int stride = (k == 1) ? 1 : a.gamma;
    unsigned long long* kk = keys + (size_t)(k - 1) * a.B * kKeyStride;
    float2* pp = part + (size_t)(k - 1) * nslices * a.B;
    draft_step_cuda_core<WDT><<<grid, kThreads, smem, stream>>>(
        a.U, a.W1, a.W2, prev, stride, a.B, a.gamma, a.V, a.r, k, a.key, pp, kk, status);
    draft_finalize<WDT><<<div_up(a.B * 32, 256), 256, 0, stream>>>(
        a.U, a.W1, a.W2, prev, stride, a.B, a.gamma, a.V, a.r, k, nslices, pp, kk, a.x_out,
        a.p_out, a.lse_out, status);
  }
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_markov_draft(const DraftArgs& a, cudaStream_t stream) {
  if (draft_tc_supported(a.wdtype, a.r, a.V)) return launch_markov_draft_tc(a, stream);
  // the target-statistics marker (set again below when this call takes the
  // statistics), the marker of verification's full row pass and the marker of
  // statistics taken along the accept chains only (this path takes every row)
  // are cleared by every draft
  const WsLayout L = ws_layout(a.B, a.gamma, a.V);
  cudaError_t e = cudaMemsetAsync(ws_ptr<unsigned int>(a.ws, L.counters) + 2, 0, 4 * sizeof(unsigned int), stream);
  if (e != cudaSuccess) return e;
  e = a.wdtype == DSPARK_BF16 ? run_draft<DSPARK_BF16>(a, stream) : run_draft<DSPARK_F32>(a, stream);
  if (e == cudaSuccess && a.T_stats != nullptr) e = launch_row_stats(a.T_stats, nullptr, a.B, a.gamma, a.V, a.ws, stream);
  return e;
}

}  // namespace dspark
