// Lossless rejection-sampling verification (the "10 key concepts" digest, item
// 2: accept the longest valid prefix, resample at the first divergence; the
// "[DeepSeek-6] DSpark" blog, section 1: plus one bonus token).
//
// 1. verify_prep       one CTA lists the target rows whose softmax statistics
//                      the accept tests need (rows 0..ell_b - 1 of T[b]) as a
//                      flat, ragged-free task list.
// 2. verify_row_stats  the streaming pass: every (row, segment) task reads one
//                      kVerifySeg-long piece of a listed row with 16-byte
//                      loads and leaves an online-softmax partial.
// 3. verify_decide     one warp per request, one lane per position: merge the
//                      partials into lse_t, form p_t(x_k) / p_d(x_k), compare
//                      it with the accept uniform; the first failing lane is
//                      the rejection.
// 4. verify_bonus_race only for requests that accepted their whole prefix: the
//                      race of the bonus token over row j = ell_b (the other
//                      requests never need that row).
// 5. residual          only for rejecting requests: recompute the draft logits
//                      of the rejected position (bias of x_{k-1} + U row) and
//                      run the two-level block race over max(0, p_t - p_d)
//                      (the tensor-core draft kernel in residual mode, or its
//                      CUDA-core form).
// 6. verify_residual_finalize  one CTA per request: the bonus token, or the
//                      corrected token from the residual race's key, or, when
//                      the residual was empty in floating point, a draw from
//                      p_t itself.
// Steps 1-2 are skipped when the draft already took the statistics of every
// row j < gamma (the caller held T when the draft started).  Otherwise, unless
// the caller asks for the statistics of every row j < ell (to reuse them for
// the acceptance labels), steps 1-3 are one kernel, verify_chain, that reads
// only the rows the accept tests reach: row j of a request once its positions
// 1..j were accepted.
#include <algorithm>
#include <mutex>

#include <cooperative_groups.h>

#include "kernels.h"
#include "tc_common.cuh"

namespace cg = cooperative_groups;

namespace dspark {
namespace {

constexpr int kRowThreads = 256;
constexpr float kLog2eF = 1.4426950408889634f;

__device__ __forceinline__ float exp2_fast(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// ell == nullptr lists every row j < G and marks the statistics of those
// rows as complete (counters[2] = the number of row segments), the state a
// draft that took them along leaves behind.
__global__ void __launch_bounds__(1024)
verify_prep(const int32_t* __restrict__ ell, int B, int G, int nsegs, int32_t* __restrict__ rows,
            int* __restrict__ counters, int* __restrict__ status) {
  __shared__ int warp_tot[32];
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  const int chunk = div_up(B, 1024);
  const int lo = tid * chunk, hi = min(B, lo + chunk);
  int run = 0;
  for (int b = lo; b < hi; ++b) {
    int L = ell ? ell[b] : G;
    if (L < 0 || L > G) {
      record_status(status, DSPARK_ERR_INVALID);
      L = L < 0 ? 0 : G;
    }
    run += L;
  }
  int incl = run;
  for (int off = 1; off < 32; off <<= 1) {
    const int o = __shfl_up_sync(0xffffffffu, incl, off);
    if (lane >= off) incl += o;
  }
  if (lane == 31) warp_tot[wid] = incl;
  __syncthreads();
  if (wid == 0) {
    int wt = warp_tot[lane];
    for (int off = 1; off < 32; off <<= 1) {
      const int o = __shfl_up_sync(0xffffffffu, wt, off);
      if (lane >= off) wt += o;
    }
    warp_tot[lane] = wt;
  }
  __syncthreads();
  int pos = (incl - run) + (wid > 0 ? warp_tot[wid - 1] : 0);
  for (int b = lo; b < hi; ++b) {
    const int L = ell ? min(max(ell[b], 0), G) : G;
    for (int j = 0; j < L; ++j) rows[pos++] = b * (G + 1) + j;
  }
  if (tid == 1023) {
    counters[0] = pos;
    if (!ell) counters[2] = B * G * nsegs;
    else counters[4] = 1;   // the row pass that follows takes every row j < ell
  }
}

// Block-wide (max, sum) of per-thread online-softmax states: the maximum
// first, then every thread rescales its own sum once, then one sum.
__device__ __forceinline__ float2 block_softmax(float m, float s, float* s_red) {
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  float mx = m;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
  if (lane == 0) s_red[wid] = mx;
  __syncthreads();
  mx = s_red[0];
#pragma unroll
  for (int w = 1; w < kRowThreads / 32; ++w) mx = fmaxf(mx, s_red[w]);
  float t = (m == -INFINITY) ? 0.f : s * exp2_fast((m - mx) * kLog2eF);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) t += __shfl_xor_sync(0xffffffffu, t, off);
  __syncthreads();
  if (lane == 0) s_red[wid] = t;
  __syncthreads();
  float S = 0.f;
#pragma unroll
  for (int w = 0; w < kRowThreads / 32; ++w) S += s_red[w];
  return make_float2(mx, S);
}

// Softmax statistics of the target rows the accept tests need (rows j < ell[b]
// of every request, listed by verify_prep).  One (row, segment) task per
// iteration: seg_len entries of a row (kVerifySeg, or kStatsSeg for the
// layout a draft leaves when it takes the statistics along; a multiple of
// 8 * 4 * kRowThreads), read as batches of eight 16-byte
// loads per thread (all issued before any arithmetic), folded into an online
// softmax.  Few registers, so that many CTAs per SM keep enough loads in
// flight to stream T at the HBM rate.
__global__ void __launch_bounds__(kRowThreads)
verify_row_stats(const float* __restrict__ T, int V, int nsegs, int seg_len, const int32_t* __restrict__ rows,
                 const int* __restrict__ counters, float2* __restrict__ row_part, int* __restrict__ status) {
  __shared__ float s_red[kRowThreads / 32];
  constexpr int kBatch = 8;                                     // float4 loads per batch
  constexpr int kStride = 4 * kRowThreads;                      // entries between a thread's loads
  const int nbatches = seg_len / (kBatch * kStride);
  const int nrows = counters[0];
  const int tid = threadIdx.x;
  const int ntasks = nrows * nsegs;
  bool bad = false;
  for (int t = blockIdx.x; t < ntasks; t += gridDim.x) {
    const int ri = t / nsegs, seg = t - ri * nsegs;
    const int rowid = rows[ri];
    const float* Trow = T + (size_t)rowid * V;
    const int v0 = seg * seg_len, v1 = min(V, v0 + seg_len);
    float m = -INFINITY, s = 0.f;
#pragma unroll 1
    for (int bt = 0; bt < nbatches; ++bt) {
      const int vb = v0 + bt * kBatch * kStride + 4 * tid;
      if (vb >= v1) break;
      float4 t4[kBatch];
#pragma unroll
      for (int j = 0; j < kBatch; ++j) {
        const int v = vb + kStride * j;
        t4[j] = v < v1 ? __ldcs(reinterpret_cast<const float4*>(Trow + v))
                       : make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
      }
      float bm = -INFINITY;
#pragma unroll
      for (int j = 0; j < kBatch; ++j) bm = fmaxf(fmaxf(bm, fmaxf(t4[j].x, t4[j].y)), fmaxf(t4[j].z, t4[j].w));
      bad |= !(bm < INFINITY);
      if (bm > m) {
        s = (m == -INFINITY) ? 0.f : s * exp2_fast((m - bm) * kLog2eF);
        m = bm;
      }
      if (m == -INFINITY) continue;
      const float mb = m * kLog2eF;
#pragma unroll
      for (int j = 0; j < kBatch; ++j)
        s += (exp2_fast(fmaf(t4[j].x, kLog2eF, -mb)) + exp2_fast(fmaf(t4[j].y, kLog2eF, -mb))) +
             (exp2_fast(fmaf(t4[j].z, kLog2eF, -mb)) + exp2_fast(fmaf(t4[j].w, kLog2eF, -mb)));
    }
    const float2 ms = block_softmax(m, s, s_red);
    if (tid == 0) row_part[(size_t)rowid * nsegs + seg] = ms;
    __syncthreads();
  }
  if (bad) record_status(status, DSPARK_ERR_NONFINITE);
}

// Block screen value 2^23 + h from a word's high 16 bits h (one byte permutation).
__device__ __forceinline__ float block_hf_v(uint32_t w) {
  return __uint_as_float(__byte_perm(w, 0x4B000000u, 0x7632));
}
constexpr float kScreenThrV = 8454142.0f;   // 2^23 + 65534 (see the draft race)

// The bonus draw of every request that accepted its whole prefix (listed by
// verify_decide in bonus_rows), from its row j = ell[b] ([blog] section 1):
// the two-level draw from softmax(T[b, j, :]) on streams 3 and 7, one
// (listed request, kBonusSeg-long segment) task per iteration.  A thread takes 16 consecutive tokens at a time (four blocks, one
// Philox call): the block weights exp(T - m) against the running maximum m,
// a screen of each block on its 16 high random bits, exact values for the
// rare candidates and the token inside a block that takes the lead.
// Entries vc .. vc+15 of a row (-inf past v1), four 16-byte streaming loads.
__device__ __forceinline__ void load_chunk16(const float* __restrict__ row, int vc, int v1, float4 (&t)[4]) {
#pragma unroll
  for (int i = 0; i < 4; ++i)
    t[i] = (vc + 4 * i < v1) ? __ldcs(reinterpret_cast<const float4*>(row + vc + 4 * i))
                             : make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
}

constexpr int kBonusSeg = 8192;   // vocabulary entries per bonus-race task
// Two warps per CTA: the race runs beside the residual resample (another
// stream), whose CTAs leave about 10 K registers per SM free.
constexpr int kBonusThreads = 64;

__global__ void __launch_bounds__(kBonusThreads)
verify_bonus_race(const float* __restrict__ T, const int32_t* __restrict__ ell,
                  const int32_t* __restrict__ bonus_rows, int B, int G, int V, int nsegs, RngKey key_arg,
                  unsigned long long* __restrict__ bonus_key, unsigned int* __restrict__ fin,
                  int32_t* __restrict__ tok_out, int* __restrict__ status) {
  pdl_wait();   // the bonus list from verify_decide (a no-op on the side stream)
  const int nrows = min(bonus_rows[0], B);
  const RngKey key = live_key(key_arg);
  __shared__ unsigned long long s_k[kBonusThreads / 32];
  constexpr int kChunks = kBonusSeg / (16 * kBonusThreads);
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  const int ntasks = nrows * nsegs;
  bool bad = false;
  for (int t = blockIdx.x; t < ntasks; t += gridDim.x) {
    const int b = bonus_rows[1 + t / nsegs], seg = t - (t / nsegs) * nsegs;
    const int jrow = min(max(ell[b], 0), G);
    const int rowid = b * (G + 1) + jrow;
    const uint32_t pos = (uint32_t)(jrow + 1);
    const float* Trow = T + (size_t)rowid * V;
    const int v0 = seg * kBonusSeg, v1 = min(V, v0 + kBonusSeg);
    // zbest: this thread's best perturbed log-mass (bestv its token); zthr:
    // the best known in the warp, a value some lane has reached, which the
    // screen compares against (bound = exp(m - zthr), 2^-10 over)
    float m = -INFINITY, zbest = -INFINITY, zthr = -INFINITY, bound = INFINITY;
    int bestv = -1;
    // a thread's 16 entries of chunk ch+1 are loaded while chunk ch is raced
    float4 nx[4];
    load_chunk16(Trow, v0 + 16 * tid, v1, nx);
    for (int ch = 0; ch < kChunks; ++ch) {
      const int vc = v0 + 16 * (ch * kBonusThreads + tid);
      float tv[16];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        tv[4 * i] = nx[i].x; tv[4 * i + 1] = nx[i].y; tv[4 * i + 2] = nx[i].z; tv[4 * i + 3] = nx[i].w;
      }
      if (ch + 1 < kChunks) load_chunk16(Trow, vc + 16 * kBonusThreads, v1, nx);
      if (vc < v1) {
        float cm = tv[0];
#pragma unroll
        for (int c = 1; c < 16; ++c) cm = fmaxf(cm, tv[c]);
        bad |= !(cm < INFINITY);
        if (cm > m) {
          m = cm;
          if (zthr > -INFINITY) bound = exp2_fast((m - zthr) * kLog2eF) * (1.0f + 0x1p-10f);
        }
        if (m > -INFINITY) {
          const float mb = m * kLog2eF;
          float e[16];
#pragma unroll
          for (int c = 0; c < 16; ++c) e[c] = exp2_fast(fmaf(tv[c], kLog2eF, -mb));
          float W[4];
#pragma unroll
          for (int q = 0; q < 4; ++q) W[q] = ((e[4 * q] + e[4 * q + 1]) + e[4 * q + 2]) + e[4 * q + 3];
          const uint4 ra = rng_call(key, kStreamBonus, (uint32_t)b, pos, (uint32_t)vc >> 4);
          const uint32_t wq[4] = {ra.x, ra.y, ra.z, ra.w};
          if (zbest == -INFINITY) {
            // open this thread's race with its block most likely to win
            float bw = 0.f, bd = 1.f;
            int bq = 0;
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              const float d = 8454144.0f - block_hf_v(wq[q]);
              if (W[q] * bd > bw * d) { bw = W[q]; bd = d; bq = q; }
            }
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              if (q == bq) {
                zbest = m + logf(W[q]) + gumbel_from_bits(wq[q] >> 9);
                bestv = block_pick(key, kStreamBonus, (uint32_t)b, pos, ((uint32_t)vc >> 2) + q, e[4 * q],
                                   e[4 * q + 1], e[4 * q + 2], e[4 * q + 3]);
                W[q] = 0.f;
              }
            }
            if (zbest > zthr) {
              zthr = zbest;
              bound = exp2_fast((m - zthr) * kLog2eF) * (1.0f + 0x1p-10f);
            }
          }
          const float b16 = bound * 65536.0f;
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            if (W[q] > 0.f && fmaf(W[q], b16, block_hf_v(wq[q])) > kScreenThrV) {
              const float z = m + logf(W[q]) + gumbel_from_bits(wq[q] >> 9);
              if (z > zbest) {
                zbest = z;
                bestv = block_pick(key, kStreamBonus, (uint32_t)b, pos, ((uint32_t)vc >> 2) + q, e[4 * q],
                                   e[4 * q + 1], e[4 * q + 2], e[4 * q + 3]);
                if (z > zthr) {
                  zthr = z;
                  bound = exp2_fast((m - zthr) * kLog2eF) * (1.0f + 0x1p-10f);
                }
              }
            }
          }
        }
      }
      // the lanes pool their thresholds after every chunk, so that a block
      // is screened against the warp's best, not only the thread's own
      float zw = zthr;
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) zw = fmaxf(zw, __shfl_xor_sync(0xffffffffu, zw, off));
      if (zw > zthr) {
        zthr = zw;
        bound = m > -INFINITY ? exp2_fast((m - zthr) * kLog2eF) * (1.0f + 0x1p-10f) : INFINITY;
      }
    }
    unsigned long long best = bestv >= 0 ? argmax_key(zbest, bestv) : 0ull;
    best = warp_max_u64(best, 0xffffffffu, 32);
    if (lane == 0) s_k[wid] = best;
    __syncthreads();
    if (tid == 0) {
      for (int w = 1; w < kBonusThreads / 32; ++w) best = s_k[w] > best ? s_k[w] : best;
      if (best) atomicMax(&bonus_key[b], best);
    }
    __syncthreads();
  }
  if (bad) record_status(status, DSPARK_ERR_NONFINITE);
  // fin given: the last CTA to finish writes the bonus tokens (every task's
  // key is final then)
  if (fin != nullptr) {
    __shared__ int s_last;
    __syncthreads();
    if (tid == 0) {
      __threadfence();
      s_last = atomicAdd(fin, 1u) == gridDim.x - 1u;
    }
    __syncthreads();
    if (s_last) {
      __threadfence();
      for (int i = tid; i < nrows; i += kBonusThreads) {
        const int b = bonus_rows[1 + i];
        const unsigned long long kb = __ldcg(bonus_key + b);
        if (kb == 0ull) record_status(status, DSPARK_ERR_NONFINITE);
        tok_out[b] = kb ? argmax_key_index(kb) : 0;
      }
    }
  }
}

__global__ void verify_decide(const float* __restrict__ T, const int32_t* __restrict__ x,
                              const float* __restrict__ p_d, const int32_t* __restrict__ ell,
                              const int32_t* __restrict__ anchor, int B, int G, int V, int nsegs, RngKey key_arg,
                              const float2* __restrict__ row_part, const float* __restrict__ tx,
                              int32_t* __restrict__ resid_k, float* __restrict__ resid_lse,
                              int32_t* __restrict__ resid_prev,
                              int32_t* __restrict__ n_out, int32_t* __restrict__ bonus_rows,
                              const int* __restrict__ stats_done, int* __restrict__ status) {
  pdl_wait();   // ell from the schedule
  const RngKey key = live_key(key_arg);
  const int b = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  // statistics taken by the draft: they must cover every row j < G
  if (stats_done && b == 0 && lane == 0 && *stats_done < B * G * nsegs) record_status(status, DSPARK_ERR_INVALID);
  if (b >= B) return;
  const int L = min(max(ell[b], 0), G);
  bool reject = false;
  float lse_t = 0.f;
  int xraw = 0;
  if (lane < L) {
    // every load that does not depend on another is issued first: the token,
    // p_d, T at the token when the draft gathered it (tx) and the row's
    // partials; else T at the token after them
    const int rowid = b * (G + 1) + lane;
    xraw = x[(size_t)b * G + lane];
    const float pd = p_d[(size_t)b * G + lane];
    float t = tx ? __ldcg(tx + (size_t)b * G + lane) : 0.f;
    float m = -INFINITY, s = 0.f;
    merge_partials(row_part + (size_t)rowid * nsegs, nsegs, m, s);
    const int xk = checked_token(xraw, V, status);
    if (!tx) t = T[(size_t)rowid * V + xk];
    lse_t = m + logf(s);
    const float q = expf(t - lse_t);
    const float ratio = q / pd;
    const uint4 rw = rng4(key, kStreamAccept, (uint32_t)b, (uint32_t)(lane + 1), 0u);
    reject = !(uniform01(rw.x) < ratio);
  }
  const unsigned ballot = __ballot_sync(0xffffffffu, reject);
  const int n = ballot ? (__ffs(ballot) - 1) : L;
  // the rows the tests used (rows 0..n, row n only when position n + 1 was
  // tested) must be finite; rows past them may never have been read (a draft
  // that took only the rows the accept chains reach)
  const unsigned used = n < L ? (n >= 31 ? 0xffffffffu : (2u << n) - 1u) : (L >= 32 ? 0xffffffffu : (1u << L) - 1u);
  if ((__ballot_sync(0xffffffffu, lane < L && !(lse_t < INFINITY)) & used) && lane == 0)
    record_status(status, DSPARK_ERR_NONFINITE);
  const float lse_n = __shfl_sync(0xffffffffu, lse_t, n & 31);
  const int x_prev = __shfl_sync(0xffffffffu, xraw, (n + 31) & 31);   // x_n (lane n - 1)
  if (lane == 0) {
    n_out[b] = n;
    resid_k[b] = n < L ? n + 1 : 0;
    if (n < L) {
      resid_lse[b] = lse_n;
      resid_prev[b] = n == 0 ? anchor[b] : x_prev;
    } else {
      // the bonus race takes it (a list of at most B: a count past it means
      // the list did not start empty)
      const int slot = atomicAdd(bonus_rows, 1);
      if (slot < B) bonus_rows[1 + slot] = b;
      else record_status(status, DSPARK_ERR_INVALID);
    }
  }
}

// ---------------------------------------------------------------------------
// Verification along each request's accept chain.  The accept test of
// position k needs the softmax normaliser of target row k - 1, and once a
// position is rejected no later row can change the round's result.  So the
// rows are read in the order of the chains: row j of request b only once
// positions 1..j of b were accepted.  At the engine point about 2.9 of 16
// positions are accepted, so about 4 of the 16 rows a request submits are
// read.
//
// A cluster of kChainCluster CTAs owns one request at a time.  Each CTA copies
// its eighth of row j into shared memory (1-D bulk copies, two stages of
// kChainChunk floats), folds it into a (max, sum of exp) partial and leaves it
// in its shared memory; after a cluster barrier every CTA reads the eight
// partials (distributed shared memory) and reduces them by the same tree, so
// all of them take the same decision and go on to row j + 1 or to the next
// request together.  T at the drafted token comes with the partial of the CTA
// whose eighth holds it.  Requests come from a counter, one atomic per
// request, taken by rank 0 when the cluster is free: a cluster busy with a
// long chain holds no other request, and one that starts late (not resident
// at first) takes only what is left.  Once every request has been handed out
// HBM has room, and a step folds the next kChainTailRows rows of the chain
// at once, ahead of their decisions (taken in order after one barrier; rows
// past a rejection are read for nothing): the long chains left at the end
// then move several positions per barrier.  Nothing else is shared between
// clusters.
// ---------------------------------------------------------------------------
constexpr int kChainCluster = 8;            // CTAs reading one row together
constexpr int kChainThreads = 512;
constexpr int kChainChunk = 12288;          // floats per bulk copy (48 KB)
constexpr int kChainStages = 2;
constexpr int kChainTailRows = 4;           // rows per step once every request is handed out
constexpr int kChainSmemBytes = kChainStages * kChainChunk * 4;
constexpr int kChainVec = kChainChunk / 4 / kChainThreads;   // float4 per thread per chunk
constexpr int kChainWarps = kChainThreads / 32;
static_assert(kChainVec * 4 * kChainThreads == kChainChunk, "a chunk is whole float4 per thread");
static_assert(kChainTailRows <= kChainWarps, "one warp per row decides");

struct ChainShared {
  uint64_t full[kChainStages];   // bulk copy of a chunk landed
  // this CTA's partial of each row of the step, by step parity: (max, sum of
  // exp, T at the drafted token when this CTA's share holds it, rank 0: every
  // request handed out)
  float4 part[2][kChainTailRows];
  float2 red[kChainTailRows][kChainWarps];
  float txv[kChainTailRows];     // T at the drafted token (the thread holding it)
  int sx[32];                    // the request's drafted tokens (checked), ...
  float spd[32], su[32];         // ... their draft probabilities and accept uniforms
  int req[2];                    // rank 0: the request the cluster takes next, by hand-off parity
  float lse[kChainTailRows];
  int acc[kChainTailRows];
  int out;                       // every request handed out (rank 0's word at the last barrier)
  int bnext;
};

// 1-D bulk copy global -> this CTA's shared memory, completing on `bar`
// (16-byte aligned addresses, size % 16 == 0).
__device__ __forceinline__ void chain_copy(float* dst, const float* src, uint32_t bytes, uint64_t* bar) {
  tc::mbar_arrive_expect_tx(bar, bytes);
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                   tc::smem_u32(dst)),
               "l"(src), "r"(bytes), "r"(tc::smem_u32(bar))
               : "memory");
}

// (max, sum of exp) reduction over a warp: the maximum first, then each lane
// rescales its sum once to it, then one sum.  A fixed shuffle tree with the
// fast base-2 exponential: every CTA of a cluster runs the same sequence on
// the same values, so all of them get the same bits.
__device__ __forceinline__ void chain_warp_reduce(float& m, float& s, int width) {
  float M = m;
  for (int off = width / 2; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
  float t = m == -INFINITY ? 0.f : s * exp2_fast((m - M) * kLog2eF);
  for (int off = width / 2; off > 0; off >>= 1) t += __shfl_xor_sync(0xffffffffu, t, off);
  m = M;
  s = t;
}

__global__ void __cluster_dims__(kChainCluster, 1, 1) __launch_bounds__(kChainThreads, 2)
verify_chain(const float* __restrict__ T, const int32_t* __restrict__ x, const float* __restrict__ p_d,
             const int32_t* __restrict__ ell, const int32_t* __restrict__ anchor, int B, int G, int V,
             RngKey key_arg, unsigned int* __restrict__ req_next, int32_t* __restrict__ resid_k,
             float* __restrict__ resid_lse, int32_t* __restrict__ resid_prev, int32_t* __restrict__ n_out,
             int32_t* __restrict__ bonus_rows, int* __restrict__ full_stats, int* __restrict__ status) {
  extern __shared__ __align__(128) float buf[];   // kChainStages x kChainChunk
  __shared__ ChainShared sh;
  cg::cluster_group cl = cg::this_cluster();
  const int rank = (int)cl.block_rank();
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  if (tid == 0) {
    for (int s = 0; s < kChainStages; ++s) tc::mbar_init(&sh.full[s], 1);
    tc::fence_mbar_init();
  }
  __syncthreads();
  pdl_wait();   // ell from the schedule, x and p_d from the draft, the request counter cleared
  if (blockIdx.x == 0 && tid == 0) *full_stats = 0;   // the row partials no longer cover every row j < ell
  // this CTA's share of a row: floats [c0, c1), in chunks of kChainChunk
  const int share = div_up(div_up(V, kChainCluster), 4) * 4;
  const int c0 = min(V, rank * share), c1 = min(V, c0 + share);
  const int nch = div_up(c1 - c0, kChainChunk);
  // The chunk stream: chunk g of the kernel goes to stage g % kChainStages
  // and completes phase (g / kChainStages) & 1 of its barrier.  Thread 0
  // counts the chunks it issued (n_iss); every thread counts those used
  // (n_use), in step.
  uint32_t n_iss = 0, n_use = 0;
  bool dead = false;   // a copy wait gave up: this CTA copies nothing more
  bool bad = false;
  bool all_out = false;   // every request handed out (the same in every CTA of the cluster)
  uint32_t nb = 0;     // steps (parity of the partial slots)
  uint32_t hand = 0;   // hand-offs (parity of the request slots)
  if (rank == 0 && tid == 0) sh.req[0] = (int)atomicAdd(req_next, 1u);
  cl.sync();
  if (tid == 0) sh.bnext = *cl.map_shared_rank(&sh.req[0], 0);
  __syncthreads();
  int b = sh.bnext;
  while (b < B) {
    const int Lraw = ell[b];
    const int L = min(max(Lraw, 0), G);
    if (rank == 0 && tid == 0 && (Lraw < 0 || Lraw > G)) record_status(status, DSPARK_ERR_INVALID);
    const float* rows = T + (size_t)b * (G + 1) * V;   // row j at rows + j * V
    // the drafted tokens, their draft probabilities and the accept uniforms
    // of every position, one load each
    if (wid == 0 && lane < L) {
      const size_t it = (size_t)b * G + lane;
      sh.sx[lane] = checked_token(x[it], V, status);
      sh.spd[lane] = p_d[it];
      sh.su[lane] = uniform01(rng4(live_key(key_arg), kStreamAccept, (uint32_t)b, (uint32_t)(lane + 1), 0u).x);
    }
    __syncthreads();
    int j = 0;       // next undecided position - 1 (= next row)
    int n = L;       // accepted positions (L: all of them)
    float lse_rej = 0.f;
    for (;;) {
      // ---- the step's rows: j, and once every request is out, the rows after it
      const int nr = L > 0 ? (all_out ? min(kChainTailRows, L - j) : 1) : 0;
      const uint32_t total = (uint32_t)(nr * nch);   // chunks of this step
      uint32_t s_iss = 0;                            // issued of them (thread 0)
      auto top_up = [&]() {
        while (!dead && s_iss < total && n_iss - n_use < (uint32_t)kChainStages) {
          const int r = (int)(s_iss / (uint32_t)nch), c = (int)(s_iss % (uint32_t)nch);
          const int a = c0 + c * kChainChunk;
          const int st = (int)(n_iss % kChainStages);
          chain_copy(buf + st * kChainChunk, rows + (size_t)(j + r) * V + a,
                     4u * (uint32_t)(min(c1, a + kChainChunk) - a), &sh.full[st]);
          ++n_iss;
          ++s_iss;
        }
      };
      if (tid == 0) top_up();
      int bad_rows = 0;
      for (int r = 0; r < nr; ++r) {
        const int xj = sh.sx[j + r];
        float m = -INFINITY, s = 0.f;
        bool br = false;
        for (int c = 0; c < nch; ++c) {
          const int st = (int)(n_use % kChainStages);
          if (!dead && !tc::mbar_wait_bounded(&sh.full[st], (n_use / kChainStages) & 1u, status)) dead = true;
          const int n4 = (min(c1, c0 + (c + 1) * kChainChunk) - (c0 + c * kChainChunk)) >> 2;
          const float4* b4 = reinterpret_cast<const float4*>(buf + st * kChainChunk);
          float4 q[kChainVec];
#pragma unroll
          for (int k = 0; k < kChainVec; ++k) {
            const int i = tid + k * kChainThreads;
            q[k] = i < n4 ? b4[i] : make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
          }
          // T at the drafted token, by the thread that holds it
          const int e = xj - (c0 + c * kChainChunk);
          if (e >= 0 && e < 4 * n4 && ((e >> 2) % kChainThreads) == tid) {
            const float4 qe = b4[e >> 2];
            sh.txv[r] = (e & 3) == 0 ? qe.x : ((e & 3) == 1 ? qe.y : ((e & 3) == 2 ? qe.z : qe.w));
          }
          float bm = -INFINITY;
#pragma unroll
          for (int k = 0; k < kChainVec; ++k) bm = fmaxf(fmaxf(bm, fmaxf(q[k].x, q[k].y)), fmaxf(q[k].z, q[k].w));
          br |= !(bm < INFINITY);
          if (bm > m) {
            s = (m == -INFINITY) ? 0.f : s * exp2_fast((m - bm) * kLog2eF);
            m = bm;
          }
          if (m > -INFINITY) {
            const float mb = m * kLog2eF;
#pragma unroll
            for (int k = 0; k < kChainVec; ++k)
              s += (exp2_fast(fmaf(q[k].x, kLog2eF, -mb)) + exp2_fast(fmaf(q[k].y, kLog2eF, -mb))) +
                   (exp2_fast(fmaf(q[k].z, kLog2eF, -mb)) + exp2_fast(fmaf(q[k].w, kLog2eF, -mb)));
          }
          // every thread is done with this stage before it is refilled
          dead = __syncthreads_or(dead) != 0;
          ++n_use;
          if (tid == 0) top_up();
        }
        bad_rows |= (int)br << r;
        // the row's partial over this warp's lanes
        chain_warp_reduce(m, s, 32);
        if (lane == 0) sh.red[r][wid] = make_float2(m, s);
      }
      // ---- one partial per row of the step: warp r reduces row r over the warps
      __syncthreads();
      if (wid < nr) {
        const int r = wid;
        float2 pr = lane < kChainWarps ? sh.red[r][lane] : make_float2(-INFINITY, 0.f);
        chain_warp_reduce(pr.x, pr.y, kChainWarps);
        const int xj = sh.sx[j + r];
        if (lane == 0)
          sh.part[nb & 1][r] =
              make_float4(pr.x, pr.y, (xj >= c0 && xj < c1) ? sh.txv[r] : 0.f,
                          rank == 0 && *reinterpret_cast<volatile unsigned int*>(req_next) >= (unsigned int)B ? 1.f
                                                                                                             : 0.f);
      } else if (nr == 0 && tid == 0) {
        sh.part[nb & 1][0] = make_float4(-INFINITY, 0.f, 0.f, 0.f);
      }
      // every peer has read the slots of step nb - 2 (it arrived at the
      // barrier of step nb - 1 after reading them)
      cl.sync();
      // ---- the decisions, warp r for row r, from the cluster's partials
      // (one lane per rank, the same reduction tree in every CTA; T at the
      // token from the rank whose share holds it)
      if (wid < nr) {
        const int r = wid;
        const float4 pr = lane < kChainCluster ? *cl.map_shared_rank(&sh.part[nb & 1][r], lane)
                                               : make_float4(-INFINITY, 0.f, 0.f, 0.f);
        float pm2 = pr.x, ps2 = pr.y;
        chain_warp_reduce(pm2, ps2, kChainCluster);
        const int pos = j + r;
        const float t = __shfl_sync(0xffffffffu, pr.z, min(sh.sx[pos] / share, kChainCluster - 1));
        const float out = __shfl_sync(0xffffffffu, pr.w, 0);   // rank 0's word
        if (lane == 0) {
          const float lse_t = pm2 + logf(ps2);
          sh.acc[r] = sh.su[pos] < expf(t - lse_t) / sh.spd[pos];
          sh.lse[r] = lse_t;
          if (r == 0) sh.out = out != 0.f;
        }
      }
      ++nb;
      __syncthreads();
      if (nr > 0) all_out = all_out || sh.out != 0;
      // ---- the chain goes on past every accepted row of the step, up to the
      // first rejection (rows after it count for nothing, their values too)
      bool ended = nr == 0;
      for (int r = 0; r < nr; ++r) {
        bad |= (bad_rows >> r) & 1;
        if (!sh.acc[r]) {
          n = j + r;
          lse_rej = sh.lse[r];
          ended = true;
          break;
        }
      }
      if (!ended) {
        j += nr;
        ended = j == L;
      }
      if (ended) break;
    }
    // rank 0 writes the request's results
    if (rank == 0 && tid == 0) {
      if (n < L) {
        n_out[b] = n;
        resid_k[b] = n + 1;
        resid_lse[b] = lse_rej;
        resid_prev[b] = n == 0 ? anchor[b] : sh.sx[n - 1];
      } else {
        // every verified position accepted (or none to verify): the bonus race
        n_out[b] = L;
        resid_k[b] = 0;
        const int slot = atomicAdd(bonus_rows, 1);
        if (slot < B) bonus_rows[1 + slot] = b;
        else record_status(status, DSPARK_ERR_INVALID);
      }
    }
    // the next request (two hand-off slots: rank 0 rewrites one only after a
    // cluster barrier that every peer reached after reading it)
    ++hand;
    if (rank == 0 && tid == 0) sh.req[hand & 1] = (int)atomicAdd(req_next, 1u);
    cl.sync();
    if (tid == 0) sh.bnext = *cl.map_shared_rank(&sh.req[hand & 1], 0);
    __syncthreads();
    b = sh.bnext;
  }
  if (bad) record_status(status, DSPARK_ERR_NONFINITE);
  // no CTA leaves while a peer may still read its shared memory; every chunk
  // this CTA issued was used (or given up on) in its step
  cl.sync();
  if (tid == 0 && dead)
    for (uint32_t g = n_iss > (uint32_t)kChainStages ? n_iss - kChainStages : 0u; g < n_iss; ++g)
      tc::mbar_drain(&sh.full[g % kChainStages], (g / kChainStages) & 1u);
}

template <int WDT>
__global__ void __launch_bounds__(kRowThreads)
verify_residual_cuda_core(const float* __restrict__ T, const float* __restrict__ U,
                          const void* __restrict__ W1, const void* __restrict__ W2,
                          const int32_t* __restrict__ anchor, const int32_t* __restrict__ x,
                          const float* __restrict__ lse_d, int B, int G, int V, int r, RngKey key_arg,
                          const int32_t* __restrict__ resid_k, const float* __restrict__ resid_lse,
                          unsigned long long* __restrict__ resid_key, int* __restrict__ status) {
  extern __shared__ float Es[];   // [r]
  __shared__ unsigned long long s_k1[kRowThreads / 32];
  const int b = blockIdx.y;
  const int ks = resid_k[b];
  if (ks <= 0) return;
  const RngKey key = live_key(key_arg);
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  const int prev = checked_token((ks == 1) ? anchor[b] : x[(size_t)b * G + ks - 2], V, status);
  for (int i = tid; i < r; i += kRowThreads) Es[i] = load_weight<WDT>(W1, (size_t)prev * r + i);
  __syncthreads();
  const float* Urow = U + ((size_t)b * G + (ks - 1)) * (size_t)V;
  const float* Trow = T + ((size_t)b * (G + 1) + (ks - 1)) * (size_t)V;
  const float ld = lse_d[(size_t)b * G + ks - 1];
  const float lt = resid_lse[b];
  const int v_begin = blockIdx.x * kDraftSlice, v_end = min(V, v_begin + kDraftSlice);
  unsigned long long k1 = 0ull;
  for (int v4 = v_begin + 4 * tid; v4 < v_end; v4 += 4 * kRowThreads) {
    // one block of 4 entries of the residual draw (streams 2 and 6)
    float rho[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int v = v4 + q;
      float bias = 0.f;
      for (int i = 0; i < r; ++i) bias = fmaf(Es[i], load_weight<WDT>(W2, (size_t)v * r + i), bias);
      const float pd = expf(Urow[v] + bias - ld);
      const float pt = expf(Trow[v] - lt);
      rho[q] = fmaxf(pt - pd, 0.f);
    }
    const float W = ((rho[0] + rho[1]) + rho[2]) + rho[3];
    if (W > 0.f) {
      const uint32_t j = (uint32_t)v4 >> 2;
      const uint32_t w = word_of(rng_call(key, kStreamResidual, (uint32_t)b, (uint32_t)ks, j >> 2), j & 3u);
      const float z = logf(W) + gumbel_from_bits(w >> 9);
      if (argmax_key(z, v4) > k1) {
        const int v = block_pick(key, kStreamResidual, (uint32_t)b, (uint32_t)ks, j, rho[0], rho[1], rho[2], rho[3]);
        const unsigned long long kz = argmax_key(z, v);
        k1 = kz > k1 ? kz : k1;
      }
    }
  }
  k1 = warp_max_u64(k1, 0xffffffffu, 32);
  if (lane == 0) s_k1[wid] = k1;
  __syncthreads();
  if (tid == 0) {
    for (int w = 1; w < kRowThreads / 32; ++w) k1 = s_k1[w] > k1 ? s_k1[w] : k1;
    if (k1) atomicMax(&resid_key[(size_t)b * kKeyStride], k1);
  }
}

// One block per request.  A request that accepted its whole prefix takes the
// bonus race's winner.  A rejecting request takes the winner of the residual
// draw; if the residual had no positive entry in floating point (a measure-zero
// event in exact arithmetic) it draws from p_t instead, with the same streams.
__global__ void __launch_bounds__(kRowThreads)
verify_residual_finalize(const float* __restrict__ T, int B, int G, int V, RngKey key_arg,
                         const int32_t* __restrict__ resid_k, const unsigned long long* __restrict__ resid_key,
                         const unsigned long long* __restrict__ bonus_key, int32_t* __restrict__ tok_out,
                         int* __restrict__ status) {
  __shared__ unsigned long long s_k[kRowThreads / 32];
  pdl_wait();   // the residual and bonus keys
  const int b = blockIdx.x;
  const int ks = resid_k[b];
  if (ks <= 0) {
    if (threadIdx.x == 0) {
      const unsigned long long kb = bonus_key[b];
      if (kb == 0ull) record_status(status, DSPARK_ERR_NONFINITE);
      tok_out[b] = kb ? argmax_key_index(kb) : 0;
    }
    return;
  }
  const unsigned long long k1 = resid_key[(size_t)b * kKeyStride];
  if (k1) {
    if (threadIdx.x == 0) tok_out[b] = argmax_key_index(k1);
    return;
  }
  const RngKey key = live_key(key_arg);
  const float* Trow = T + ((size_t)b * (G + 1) + (ks - 1)) * (size_t)V;
  // the row's maximum, then the two-level draw of softmax(T row) (streams 2
  // and 6) with weights exp(T - max)
  __shared__ float s_m[kRowThreads / 32];
  float mx = -INFINITY;
  for (int v = 4 * threadIdx.x; v < V; v += 4 * kRowThreads) {
    const float4 t4 = *reinterpret_cast<const float4*>(Trow + v);
    mx = fmaxf(mx, fmaxf(fmaxf(t4.x, t4.y), fmaxf(t4.z, t4.w)));
  }
  for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
  if ((threadIdx.x & 31) == 0) s_m[threadIdx.x >> 5] = mx;
  __syncthreads();
  mx = s_m[0];
  for (int w = 1; w < kRowThreads / 32; ++w) mx = fmaxf(mx, s_m[w]);
  unsigned long long best = 0ull;
  for (int v = 4 * threadIdx.x; v < V; v += 4 * kRowThreads) {
    const float4 t4 = *reinterpret_cast<const float4*>(Trow + v);
    const float e0 = expf(t4.x - mx), e1 = expf(t4.y - mx), e2 = expf(t4.z - mx), e3 = expf(t4.w - mx);
    const float W = ((e0 + e1) + e2) + e3;
    if (!(W > 0.f)) continue;
    const uint32_t j = (uint32_t)v >> 2;
    const uint32_t w = word_of(rng_call(key, kStreamResidual, (uint32_t)b, (uint32_t)ks, j >> 2), j & 3u);
    const float z = mx + logf(W) + gumbel_from_bits(w >> 9);
    if (argmax_key(z, v) > best) {
      const int vv = block_pick(key, kStreamResidual, (uint32_t)b, (uint32_t)ks, j, e0, e1, e2, e3);
      const unsigned long long kz = argmax_key(z, vv);
      best = kz > best ? kz : best;
    }
  }
  best = warp_max_u64(best, 0xffffffffu, 32);
  if ((threadIdx.x & 31) == 0) s_k[threadIdx.x >> 5] = best;
  __syncthreads();
  if (threadIdx.x == 0) {
    for (int w = 1; w < kRowThreads / 32; ++w) best = s_k[w] > best ? s_k[w] : best;
    if (!best) record_status(status, DSPARK_ERR_NONFINITE);
    tok_out[b] = best ? argmax_key_index(best) : 0;
  }
}

// The last kernel of a round whose index lives in device memory: the next
// round reads index + 1.
__global__ void advance_round(unsigned long long* round_dev) {
  pdl_wait();   // every kernel of the round has read the index
  if (threadIdx.x == 0) *round_dev += 1ull;
}

// verify_prep, then verify_row_stats on a grid sized by the occupancy query.
cudaError_t row_stats(const float* T, const int32_t* ell, int B, int gamma, int V, void* ws, cudaStream_t stream) {
  const WsLayout L = ws_layout(B, gamma, V);
  int* status = ws_ptr<int>(ws, L.status);
  int* counters = ws_ptr<int>(ws, L.counters);
  int32_t* rows = ws_ptr<int32_t>(ws, L.rows);
  float2* row_part = ws_ptr<float2>(ws, L.row_part);
  // every row j < gamma: the segment layout of the statistics a draft takes along
  const int seg_len = ell ? kVerifySeg : kStatsSeg;
  const int nsegs = div_up(V, seg_len);
  verify_prep<<<1, 1024, 0, stream>>>(ell, B, gamma, nsegs, rows, counters, status);
  int dev = 0, sms = 0, per_sm = 0;
  cudaError_t e;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
  if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
  if ((e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, verify_row_stats, kRowThreads, 0)) != cudaSuccess)
    return e;
  const long long stat_tasks = (long long)B * gamma * nsegs;
  const int grid_stats = (int)std::max<long long>(1, std::min<long long>(stat_tasks, (long long)sms * std::max(1, per_sm)));
  verify_row_stats<<<grid_stats, kRowThreads, 0, stream>>>(T, V, nsegs, seg_len, rows, counters, row_part, status);
  return cudaGetLastError();
}

// A second stream per device on which the bonus race runs beside the
// residual resample (the two read different rows and write different keys;
// the residual finalize needs both).  Created on first use; one mutex per
// device keeps each fork and join of its two events in one piece when host
// threads share the device.
struct SideStream {
  std::mutex mu;
  cudaStream_t s = nullptr;
  cudaEvent_t fork = nullptr, join = nullptr;
};
constexpr int kMaxSideDevices = 64;
SideStream g_side[kMaxSideDevices];
std::mutex g_side_init;

cudaError_t side_stream(SideStream** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxSideDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_side_init);
  SideStream& ss = g_side[dev];
  if (ss.s == nullptr) {
    if ((e = cudaStreamCreateWithFlags(&ss.s, cudaStreamNonBlocking)) != cudaSuccess) return e;
    if ((e = cudaEventCreateWithFlags(&ss.fork, cudaEventDisableTiming)) != cudaSuccess) return e;
    if ((e = cudaEventCreateWithFlags(&ss.join, cudaEventDisableTiming)) != cudaSuccess) return e;
  }
  *out = &ss;
  return cudaSuccess;
}

template <int WDT>
cudaError_t run_verify(const VerifyArgs& a, cudaStream_t stream) {
  const WsLayout L = ws_layout(a.B, a.gamma, a.V);
  int* status = ws_ptr<int>(a.ws, L.status);
  float2* row_part = ws_ptr<float2>(a.ws, L.row_part);
  unsigned long long* bonus_key = ws_ptr<unsigned long long>(a.ws, L.bonus_key);
  unsigned long long* resid_key = ws_ptr<unsigned long long>(a.ws, L.resid_key);
  int32_t* resid_k = ws_ptr<int32_t>(a.ws, L.resid_k);
  float* resid_lse = ws_ptr<float>(a.ws, L.resid_lse);
  int32_t* bonus_rows = ws_ptr<int32_t>(a.ws, L.bonus_rows);
  int32_t* resid_prev = ws_ptr<int32_t>(a.ws, L.resid_prev);
  const int nsegs = a.stats_ready ? stats_num_segs(a.V) : verify_num_segs(a.V);
  // the scratch that must start at zero: the bonus and residual keys, the
  // bonus list and the finish counters (not what a draft left after them:
  // resid_prev, tx, the gated states)
  cudaError_t e = cudaSuccess;
  if (!a.scratch_zeroed &&
      (e = cudaMemsetAsync(ws_ptr<char>(a.ws, L.bonus_key), 0, L.resid_k - L.bonus_key, stream)) != cudaSuccess)
    return e;
  // statistics of every row j < ell first (the classic pass), or none: the
  // chain reads the rows its accept tests reach
  const bool chain = !a.stats_ready && !a.all_row_stats;
  if (!a.stats_ready && !chain && (e = row_stats(a.T, a.ell, a.B, a.gamma, a.V, a.ws, stream)) != cudaSuccess)
    return e;
  int dev = 0, sms = 0;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
  if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
  // a tensor-core draft that took T along also gathered T at its tokens (tx)
  const bool tc = draft_tc_supported(a.wdtype, a.r, a.V);
  // the kernels from here on are chained by programmatic dependent launch
  // (each starts while the one before it ends; see pdl_wait)
  if (chain) {
    if ((e = cudaFuncSetAttribute(verify_chain, cudaFuncAttributeMaxDynamicSharedMemorySize, kChainSmemBytes)) !=
        cudaSuccess)
      return e;
    // as many clusters as can be resident at once, no more than requests
    int resident = 0;
    {
      cudaLaunchConfig_t cfg{};
      cfg.gridDim = dim3(sms * 2);
      cfg.blockDim = dim3(kChainThreads);
      cfg.dynamicSmemBytes = kChainSmemBytes;
      cfg.stream = stream;
      if (cudaOccupancyMaxActiveClusters(&resident, verify_chain, &cfg) != cudaSuccess) {
        (void)cudaGetLastError();
        resident = sms * 2 / kChainCluster;
      }
    }
    const int clusters = std::max(1, std::min(a.B, resident));
    e = launch_pdl(verify_chain, dim3(clusters * kChainCluster), dim3(kChainThreads), kChainSmemBytes, stream, a.T,
                   a.x, a.p_d, a.ell, a.anchor, a.B, a.gamma, a.V, a.key, ws_ptr<unsigned int>(a.ws, L.chain_next),
                   resid_k, resid_lse, resid_prev, a.n_out, bonus_rows, ws_ptr<int>(a.ws, L.counters) + 4, status);
  } else {
    e = launch_pdl(verify_decide, dim3(div_up(a.B * 32, 256)), dim3(256), 0, stream, a.T, a.x, a.p_d, a.ell,
                   a.anchor, a.B, a.gamma, a.V, nsegs, a.key, (const float2*)row_part,
                   (const float*)(a.stats_ready && tc ? ws_ptr<float>(a.ws, L.tx) : nullptr), resid_k, resid_lse,
                   resid_prev, a.n_out, bonus_rows,
                   (const int*)(a.stats_ready ? ws_ptr<int>(a.ws, L.counters) + 2 : nullptr), status);
  }
  if (e != cudaSuccess) return e;
  // the bonus race on the side stream (forked after verify_decide), the
  // residual on this one, joined before the finalize
  SideStream* ss = nullptr;
  if ((e = side_stream(&ss)) != cudaSuccess) return e;
  {
    std::lock_guard<std::mutex> lock(ss->mu);
    if ((e = cudaEventRecord(ss->fork, stream)) != cudaSuccess) return e;
    if ((e = cudaStreamWaitEvent(ss->s, ss->fork, 0)) != cudaSuccess) return e;
    const int bonus_segs = div_up(a.V, kBonusSeg);
    const int grid_bonus = std::min(a.B * bonus_segs, sms * 4);
    // the tensor-core path writes every token from the two kernels' last
    // CTAs; the CUDA-core path leaves them to verify_residual_finalize
    unsigned int* fin = ws_ptr<unsigned int>(a.ws, L.fin_count);
    verify_bonus_race<<<grid_bonus, kBonusThreads, 0, ss->s>>>(a.T, a.ell, bonus_rows, a.B, a.gamma, a.V, bonus_segs,
                                                              a.key, bonus_key, tc ? fin : nullptr, a.tok_out,
                                                              status);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    if ((e = cudaEventRecord(ss->join, ss->s)) != cudaSuccess) return e;
    if (tc) {
      e = launch_residual_tc(a.T, a.U, a.W1, a.W2, resid_prev, a.lse_d, resid_k, resid_lse, resid_key, a.B,
                             a.gamma, a.V, a.key, a.gated_states ? ws_ptr<void>(a.ws, L.gstate) : nullptr, fin + 1,
                             a.tok_out, status, stream);
      if (e != cudaSuccess) return e;
    } else {
      const dim3 grid_res(draft_num_slices(a.V), a.B);
      verify_residual_cuda_core<WDT><<<grid_res, kRowThreads, sizeof(float) * a.r, stream>>>(
          a.T, a.U, a.W1, a.W2, a.anchor, a.x, a.lse_d, a.B, a.gamma, a.V, a.r, a.key, resid_k, resid_lse,
          resid_key, status);
    }
    if ((e = cudaStreamWaitEvent(stream, ss->join, 0)) != cudaSuccess) return e;
  }
  if (!tc) {
    e = launch_pdl(verify_residual_finalize, dim3(a.B), dim3(kRowThreads), 0, stream, a.T, a.B, a.gamma, a.V, a.key,
                   (const int32_t*)resid_k, (const unsigned long long*)resid_key, (const unsigned long long*)bonus_key,
                   a.tok_out, status);
    if (e != cudaSuccess) return e;
  }
  if (a.advance_round != nullptr && (e = launch_pdl(advance_round, dim3(1), dim3(32), 0, stream, a.advance_round)) !=
                                        cudaSuccess)
    return e;
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_row_stats(const float* T, const int32_t* ell, int B, int gamma, int V, void* ws,
                             cudaStream_t stream) {
  return row_stats(T, ell, B, gamma, V, ws, stream);
}

cudaError_t launch_verify(const VerifyArgs& a, cudaStream_t stream) {
  return a.wdtype == DSPARK_BF16 ? run_verify<DSPARK_BF16>(a, stream) : run_verify<DSPARK_F32>(a, stream);
}

}  // namespace dspark
