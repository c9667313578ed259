// Device-side helpers shared by the libdspark kernels: the counter-based
// generator, the uniform / Gumbel maps, argmax keys, status reporting and the
// workspace layout.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/dspark.h"

namespace dspark {

// ---------------------------------------------------------------------------
// Philox4x32-10 (Salmon, Moraes, Dror, Shaw, "Parallel Random Numbers: As Easy
// as 1, 2, 3", SC'11): ten rounds of two 32x32->64 multiplications whose high
// halves are xored with the other two words and the round key; the key walks a
// Weyl sequence.
// ---------------------------------------------------------------------------
constexpr uint32_t kPhiloxMulA = 0xD2511F53u;
constexpr uint32_t kPhiloxMulB = 0xCD9E8D57u;
constexpr uint32_t kPhiloxWeylA = 0x9E3779B9u;
constexpr uint32_t kPhiloxWeylB = 0xBB67AE85u;

// Random-number streams of one round (the fourth counter word is
// (round << 3) | stream).  Every draw races blocks of 4 entries on stream s and
// picks the entry inside the winning block from stream s + 4.
enum Stream : uint32_t { kStreamDraft = 0, kStreamAccept = 1, kStreamResidual = 2, kStreamBonus = 3 };
constexpr uint32_t kPickStreamOffset = 4;

// The key of one round with its ten round keys precomputed on the host, so
// that kernels read them as constant operands instead of recomputing the
// Weyl sequence per call.
struct RngKey {
  uint32_t rk0[10], rk1[10];   // round i uses (seed_lo + i A, seed_hi + i B)
  uint32_t round3;             // round << 3
  // when not null the round index is read from this device word when a kernel
  // starts (round3 is then ignored), so that one captured CUDA graph can serve
  // consecutive rounds
  const unsigned long long* round_dev;
};

__host__ __device__ inline RngKey make_rng_key(uint64_t seed, uint64_t round,
                                               const unsigned long long* round_dev = nullptr) {
  RngKey k;
  uint32_t k0 = (uint32_t)(seed & 0xffffffffu), k1 = (uint32_t)(seed >> 32);
  for (int i = 0; i < 10; ++i) {
    k.rk0[i] = k0;
    k.rk1[i] = k1;
    k0 += kPhiloxWeylA;
    k1 += kPhiloxWeylB;
  }
  k.round3 = (uint32_t)(round << 3);
  k.round_dev = round_dev;
  return k;
}

// The key of the round that runs: round3 from the device word when the caller
// keeps the round index in device memory.
__device__ __forceinline__ RngKey live_key(const RngKey& k) {
  RngKey r = k;
  if (k.round_dev != nullptr) r.round3 = (uint32_t)(__ldcg(k.round_dev) << 3);
  return r;
}

// Programmatic dependent launch.  A kernel launched with the programmatic
// stream-serialization attribute (launch_pdl) may begin while the kernel before
// it in the stream is still running.  pdl_wait() returns once that kernel has
// completed and its memory writes are visible (at once for a kernel launched
// without the attribute), so every read of an earlier kernel's output, and
// every write that an earlier kernel might still read, comes after it.  A
// kernel whose every thread waits this way completes after its predecessor,
// so the guarantee carries down the chain.  pdl_trigger() lets the next kernel
// in the stream start launching; it releases no data.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// The round index a kernel runs (device word or host argument).
__device__ __forceinline__ unsigned long long live_round(const RngKey& k) {
  return k.round_dev != nullptr ? __ldcg(k.round_dev) : (unsigned long long)(k.round3 >> 3);
}

__device__ __forceinline__ uint4 philox4x32_10(uint4 c, const RngKey& key) {
#pragma unroll
  for (int i = 0; i < 10; ++i) {
    // one 32x32 -> 64-bit product gives both halves
    const uint64_t pa = (uint64_t)kPhiloxMulA * c.x;
    const uint64_t pb = (uint64_t)kPhiloxMulB * c.z;
    c = make_uint4((uint32_t)(pb >> 32) ^ c.y ^ key.rk0[i], (uint32_t)pb, (uint32_t)(pa >> 32) ^ c.w ^ key.rk1[i],
                   (uint32_t)pa);
  }
  return c;
}

// One Philox call of (stream, request, position) with first counter word c0.
__device__ __forceinline__ uint4 rng_call(const RngKey& key, uint32_t stream, uint32_t req, uint32_t pos,
                                          uint32_t c0) {
  return philox4x32_10(make_uint4(c0, pos, req, key.round3 | stream), key);
}

// The four words for vocabulary entries 4q .. 4q+3 of (stream, request, position).
__device__ __forceinline__ uint4 rng4(const RngKey& key, uint32_t stream, uint32_t req,
                                      uint32_t pos, uint32_t q) {
  return rng_call(key, stream, req, pos, q);
}

__device__ __forceinline__ uint32_t word_of(const uint4& w, uint32_t j) {
  return j == 0 ? w.x : (j == 1 ? w.y : (j == 2 ? w.z : w.w));
}

// Uniform (2m + 1) / 2^24 from 23 random bits m: exact in float32.
__device__ __forceinline__ float uniform_bits(uint32_t m) {
  return __uint2float_rn(m) * 0x1p-23f + 0x1p-24f;
}

// The accept uniform of a position: the top 23 bits of a word.
__device__ __forceinline__ float uniform01(uint32_t w) { return uniform_bits(w >> 9); }

// The sampler of every draw: blocks of 4 consecutive entries race with the log
// of their summed weight plus Gumbel noise from one 32-bit word each (word j of
// the stream's call sequence: word j mod 4 of call j / 4); the entry inside the
// winning block is drawn by inverse CDF with the uniform of word j of stream +
// kPickStreamOffset.  Both levels together draw exactly from the weights.

// Entry of block j of `stream` from the block's four weights e0..e3 (any common
// scale): the first whose cumulative weight exceeds u times the block's, or the
// last with weight when rounding leaves none.
__device__ __forceinline__ int block_pick(const RngKey& key, uint32_t stream, uint32_t req, uint32_t pos, uint32_t j,
                                          float e0, float e1, float e2, float e3) {
  const float u = uniform01(word_of(rng_call(key, stream + kPickStreamOffset, req, pos, j >> 2), j & 3u));
  const float t = u * (((e0 + e1) + e2) + e3);
  float cum = e0;
  int c;
  if (t < cum) {
    c = 0;
  } else if (t < (cum += e1)) {
    c = 1;
  } else if (t < (cum += e2)) {
    c = 2;
  } else {
    c = e3 > 0.f ? 3 : (e2 > 0.f ? 2 : (e1 > 0.f ? 1 : 0));
  }
  return (int)(4u * j) + c;
}

// Standard Gumbel variate by inversion.  The inner logarithm uses the
// full-accuracy logf: near u = 1 its result is tiny and a fast approximation
// with absolute error would distort the largest noise values.
__device__ __forceinline__ float gumbel_from_bits(uint32_t m) {
  return -logf(-logf(uniform_bits(m)));
}

// ---------------------------------------------------------------------------
// Argmax keys: a 64-bit integer whose order is (value asc, index desc), so
// atomicMax picks the largest value and, on exact ties, the smallest index.
// 0 means "no candidate".
// ---------------------------------------------------------------------------
__device__ __forceinline__ unsigned long long argmax_key(float z, int v) {
  uint32_t b = __float_as_uint(z);
  b = (b & 0x80000000u) ? ~b : (b | 0x80000000u);
  return ((unsigned long long)b << 32) | (unsigned long long)(0xFFFFFFFFu - (uint32_t)v);
}
__device__ __forceinline__ int argmax_key_index(unsigned long long key) {
  return (int)(0xFFFFFFFFu - (uint32_t)(key & 0xFFFFFFFFull));
}
__device__ __forceinline__ float argmax_key_value(unsigned long long key) {
  uint32_t b = (uint32_t)(key >> 32);
  b = (b & 0x80000000u) ? (b & 0x7FFFFFFFu) : ~b;
  return __uint_as_float(b);
}

// ---------------------------------------------------------------------------
// Online softmax state: running max m and sum s of exp(l - m).
// ---------------------------------------------------------------------------
__device__ __forceinline__ void softmax_merge(float& m, float& s, float m2, float s2) {
  if (m2 == -INFINITY) return;
  if (m == -INFINITY) { m = m2; s = s2; return; }
  if (m2 > m) { s = s * expf(m - m2) + s2; m = m2; }
  else { s = s + s2 * expf(m2 - m); }
}

// Merges n softmax partials (max, sum) from p into (m, s), eight loads in
// flight at a time (a row's segment partials, read before the merge starts).
__device__ __forceinline__ void merge_partials(const float2* __restrict__ p, int n, float& m, float& s) {
  for (int i0 = 0; i0 < n; i0 += 8) {
    float2 q[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) q[j] = i0 + j < n ? __ldcg(p + i0 + j) : make_float2(-INFINITY, 0.f);
#pragma unroll
    for (int j = 0; j < 8; ++j) softmax_merge(m, s, q[j].x, q[j].y);
  }
}

__device__ __forceinline__ void warp_softmax_reduce(float& m, float& s, unsigned mask, int width) {
  for (int off = width / 2; off > 0; off >>= 1) {
    float m2 = __shfl_xor_sync(mask, m, off, width);
    float s2 = __shfl_xor_sync(mask, s, off, width);
    softmax_merge(m, s, m2, s2);
  }
}

__device__ __forceinline__ unsigned long long warp_max_u64(unsigned long long k, unsigned mask, int width) {
  for (int off = width / 2; off > 0; off >>= 1) {
    unsigned long long o = __shfl_xor_sync(mask, k, off, width);
    k = o > k ? o : k;
  }
  return k;
}

// First error wins; later errors do not overwrite it.
__device__ __forceinline__ void record_status(int* status, int code) {
  atomicCAS(status, 0, code);
}

// A token id read from memory, checked before it indexes a [V, r] table: an id
// outside [0, V) records DSPARK_ERR_INVALID and is replaced by 0.
__device__ __forceinline__ int checked_token(int t, int V, int* status) {
  if (t < 0 || t >= V) {
    if (status) record_status(status, DSPARK_ERR_INVALID);
    return 0;
  }
  return t;
}

template <int WDT>
__device__ __forceinline__ float load_weight(const void* base, size_t idx) {
  if (WDT == DSPARK_F32) return static_cast<const float*>(base)[idx];
  const uint16_t bits = static_cast<const uint16_t*>(base)[idx];
  return __uint_as_float(((uint32_t)bits) << 16);
}

// ---------------------------------------------------------------------------
// Tiling constants and the workspace layout (shared by host and device code).
// ---------------------------------------------------------------------------
constexpr int kDraftSlice = 1024;   // vocabulary columns per draft CTA (CUDA-core path)
constexpr int kVerifySeg = 32768;   // vocabulary entries per verify task
constexpr int kMaxGamma = 32;
constexpr int kMaxCandidates = 8192;

__host__ __device__ inline int div_up(int a, int b) { return (a + b - 1) / b; }

__host__ __device__ inline int draft_num_slices(int V) { return div_up(V, kDraftSlice); }
// Slices reserved per position in the draft partial buffer: enough for the
// CUDA-core grid and for one tensor-core CTA per SM (up to 160 SMs).
constexpr int kMaxDraftCtas = 160;
__host__ __device__ inline int draft_part_slices(int V) {
  return draft_num_slices(V) > kMaxDraftCtas ? draft_num_slices(V) : kMaxDraftCtas;
}
__host__ __device__ inline int verify_num_segs(int V) { return div_up(V, kVerifySeg); }

// The statistics a draft takes along (one warp per task) use shorter segments,
// so that the last tasks finish soon after the draft; the partial buffer is
// sized for the larger count.
constexpr int kStatsSeg = 16384;
__host__ __device__ inline int stats_num_segs(int V) { return div_up(V, kStatsSeg); }

// Each argmax key that many CTAs read and raise during a pass sits in its own
// 128-byte line, so that the traffic of different rows spreads over L2.
constexpr int kKeyStride = 16;   // u64 slots per key

struct WsLayout {
  size_t status;      // int32 status word
  size_t counters;    // int32 [8]: [0] verify row count, [1] unused, [2] target-row
                      // statistics: tasks taken (>= B*gamma*nsegs once rows j < gamma are done),
                      // [3] draft CTAs past the finalize, [4] 1 while the row partials hold
                      // verification's statistics of every row j < ell (cleared by every draft),
                      // [5] 1 when a draft took only the rows the accept chains can reach; word
                      // 32 (its own 128-byte line, away from the task counter's atomics): the
                      // draft's grid-barrier counter
  size_t draft_keys;  // u64 [gamma][B], kKeyStride apart
  size_t draft_part;  // float2 [gamma][B][nslices]
  size_t rows;        // int32 [B*gamma] row ids b*(gamma+1)+j (j < ell_b) of the rows whose stats verify needs
  size_t row_part;    // float2 [B*(gamma+1)][nsegs]: softmax partials of target-row segments
                      // (kVerifySeg long after verify's own pass, kStatsSeg after a draft's)
  size_t bonus_key;   // u64 [B]
  size_t resid_key;   // u64 [B] residual key, kKeyStride apart
  size_t resid_k;     // int32 [B] rejected position k* (0 = none)
  size_t resid_lse;   // float [B] lse of the target row at k*
  size_t resid_prev;  // int32 [B] x_{k*-1} as stored (the anchor when k* = 1)
  size_t tx;          // float [B*gamma] T[b, k-1, x_k], gathered by a draft that takes T along
  size_t gstate;      // bf16 [B][gamma][256] the gated head's states s_k (tensor-core path)
  size_t chain_stats; // int32 [B] first position known to reject (0: none), int32 [B] positions
                      // known not to reject, u32 [B*(gamma+1)] segments of each row written: a
                      // draft that takes the statistics of the rows the accept chains reach
  size_t bonus_rows;  // int32 [1 + B]: count, then the requests that accepted their whole prefix
  size_t fin_count;   // u32 [2]: CTAs of the bonus race and of the residual that are done
  size_t chain_next;  // u32: requests verify_chain's clusters have taken
  size_t total;
};

__host__ __device__ inline size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

__host__ __device__ inline WsLayout ws_layout(int B, int gamma, int V) {
  WsLayout L;
  size_t off = 0;
  const size_t rows = (size_t)B * (gamma + 1);
  L.status = off;      off = align256(off + 4);
  L.counters = off;    off = align256(off + 4 * 33);
  L.draft_keys = off;  off = align256(off + 8ull * kKeyStride * gamma * B);
  L.draft_part = off;  off = align256(off + 8ull * gamma * draft_part_slices(V) * B);
  L.rows = off;        off = align256(off + 4ull * rows);
  L.row_part = off;    off = align256(off + 8ull * rows * stats_num_segs(V));
  // [bonus_key, resid_k): the verification scratch that must start at zero
  L.bonus_key = off;   off = align256(off + 8ull * B);
  L.resid_key = off;   off = align256(off + 8ull * kKeyStride * B);
  L.bonus_rows = off;  off = align256(off + 4ull * (B + 1));
  L.fin_count = off;   off = align256(off + 8);
  L.chain_next = off;  off = align256(off + 4);
  // then what verification writes before it reads, and what a draft leaves
  L.resid_k = off;     off = align256(off + 4ull * B);
  L.resid_lse = off;   off = align256(off + 4ull * B);
  L.resid_prev = off;  off = align256(off + 4ull * B);
  L.tx = off;          off = align256(off + 4ull * B * gamma);
  L.gstate = off;      off = align256(off + 2ull * 256 * B * gamma);
  L.chain_stats = off; off = align256(off + 4ull * (2 * B + rows));
  L.total = off;
  return L;
}

template <typename T>
__host__ __device__ inline T* ws_ptr(void* ws, size_t off) {
  return reinterpret_cast<T*>(static_cast<char*>(ws) + off);
}

// One warp's draw from softmax(Trow) on the residual's streams (2 and 6) for
// request b at position ks: the fallback of a residual that had no positive
// entry in floating point (a measure-zero event).  Two passes over the row,
// the maximum and then the two-level race of blocks of 4 with weights
// exp(T - max), as verify_residual_finalize draws it with a whole CTA.
// Returns the token on every lane, -1 if no block had weight.
static __device__ __forceinline__ int warp_softmax_draw(const float* __restrict__ Trow, int V, uint32_t b, uint32_t ks,
                                                        const RngKey& key, int lane) {
  float mx = -INFINITY;
  for (int v = 4 * lane; v < V; v += 128) {
    const float4 t4 = *reinterpret_cast<const float4*>(Trow + v);
    mx = fmaxf(mx, fmaxf(fmaxf(t4.x, t4.y), fmaxf(t4.z, t4.w)));
  }
  for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
  unsigned long long best = 0ull;
  for (int v = 4 * lane; v < V; v += 128) {
    const float4 t4 = *reinterpret_cast<const float4*>(Trow + v);
    const float e0 = expf(t4.x - mx), e1 = expf(t4.y - mx), e2 = expf(t4.z - mx), e3 = expf(t4.w - mx);
    const float W = ((e0 + e1) + e2) + e3;
    if (!(W > 0.f)) continue;
    const uint32_t j = (uint32_t)v >> 2;
    const uint32_t w = word_of(rng_call(key, kStreamResidual, b, ks, j >> 2), j & 3u);
    const float z = mx + logf(W) + gumbel_from_bits(w >> 9);
    if (argmax_key(z, v) > best) {
      const int vv = block_pick(key, kStreamResidual, b, ks, j, e0, e1, e2, e3);
      const unsigned long long kz = argmax_key(z, vv);
      best = kz > best ? kz : best;
    }
  }
  best = warp_max_u64(best, 0xffffffffu, 32);
  return best ? argmax_key_index(best) : -1;
}

}  // namespace dspark
