// Markov draft on the 5th-generation tensor cores ("[DeepSeek-6] DSpark" blog,
// sections 3-4; study report Eq.4), and the residual resample of verification
// (the "10 key concepts" digest, item 2), which needs the same fused logits.
//
// Draft: one persistent, cooperative launch runs every position k; 152 CTAs,
// each owning a 128-request M tile (128 / R replicas of R rows for small
// batches) and a contiguous range of 64-column vocabulary tiles.  Per CTA:
//
//   warp 0      TMA producer: W2 in atoms of 192 rows x 64 K (bf16, 128-byte
//               swizzled, evict_last so W2 stays in L2 across positions) and
//               U in [R rows x 32 columns] fp32 boxes (evict_first); it runs
//               ahead across positions, so the next position's first tiles
//               load while the grid barrier resolves.
//   warp 1      TMEM allocation (512 columns) and the single-thread MMA
//               issuer: bias[128 x 64j] = E[128 x 256] * W2_rows^T, j <= 3
//               tiles per tcgen05.mma (kind::f16, fp32 accumulate; the first
//               group of a position is one tile), A = E in TMEM columns
//               384-511, two accumulators of 192 columns.
//   warps 2-17  epilogue, four per TMEM lane quarter (thread = request row,
//               16 columns per tile): tcgen05.ld of the accumulator, + U, the
//               online softmax and the block race of the sampler (blocks of
//               4 tokens, screened on 16 random bits, exact only for the rare
//               candidates).  A row's parts pool their first seeds in shared
//               memory; every part publishes its best to the row's argmax key
//               (atomicMax) whenever it reaches the row's threshold, and each
//               tile copies the key back asynchronously (one copy per row,
//               read without waiting) to raise the threshold from the other
//               CTAs' progress.  At a position's end the CTA arrives at the
//               grid barrier, merges its parts into one (m, s) partial per
//               row, gathers E = W1[x_k] speculatively and, after the
//               barrier, reloads the rows whose final token differs.
//
// Residual (MODE kResidual): the same pipeline for one position per request
// (the rejected k*), with U and T row segments staged by the epilogue's own
// coalesced asynchronous copies, racing blocks of max(0, p_t - p_d).
//
// Every wait is bounded; on a timeout the CTA records DSPARK_ERR_TIMEOUT,
// drains the copies and MMAs it issued, frees its TMEM and returns.
#include <cuda_bf16.h>

#include <algorithm>
#include <mutex>

#include "conf.cuh"
#include "kernels.h"
#include "sched.cuh"
#include "tc_common.cuh"

namespace dspark {
namespace {

using namespace tc;

constexpr int BM = 128;             // requests per M tile (TMEM lanes)
constexpr int BN = 64;              // vocabulary columns per tile (epilogue and U unit)
constexpr int kGroup = 3;           // tiles per MMA: N = 64 x (up to 3)
constexpr int kAccCols = kGroup * BN;  // 192 TMEM columns per accumulator
// Tiles of the MMA group that starts at tile g of a position: the first group
// is one tile, so that the epilogue starts after 16 narrow MMAs instead of 16
// wide ones; the rest take kGroup tiles.
__device__ __forceinline__ int group_tiles(int g) { return g == 0 ? 1 : kGroup; }
constexpr int KR = 256;             // Markov rank handled by this kernel
constexpr int kAtoms = KR / 64;     // 64-wide K atoms (128 bytes of bf16)
constexpr int kWStages = 4;         // W2 atom ring (one MMA's worth)
constexpr int kUStages = 3;         // U tile ring
constexpr int kUBox = 32;           // fp32 columns per U box (128 bytes, swizzled)
constexpr int kEpiWarps = 16;       // four warps per TMEM lane quarter
constexpr int kStatsWarps = 2;      // draft mode: warps that stream target-row statistics
constexpr int kThreads = 64 + 32 * kEpiWarps;                 // residual mode
constexpr int kDraftThreads = kThreads + 32 * kStatsWarps;    // draft mode (640 x 96 registers fit)
constexpr uint32_t kTmemCols = 512;  // two accumulators, then E
constexpr uint32_t kTmemE = 2 * kAccCols;   // first TMEM column of E (128 x 256 bf16)

constexpr int kWStageBytes = kAccCols * 128;     // 24576: 192 W2 rows x 64 K (bf16), swizzled
constexpr int kUStageBytes = BN * BM * 4;        // 32768: two [rows x 32] boxes
constexpr int kXBytes = 4 * BM * (4 + 4 + 8);     // combine scratch: 4 parts x 128 rows
constexpr int kBarBytes = 512;                   // mbarriers and flags
// Residual mode: a shallower W2 ring, and two stages of the U and T row
// segments of one tile (R rows x 64 columns each, 256-byte rows).
constexpr int kWStagesRes = 2;
constexpr int kResStageBytes = 2 * BM * 256;      // U then T
constexpr int kGkBytes = 2 * BM * 16;   // row-key copies: [position parity][row], 16 bytes each
// the rings: draft mode W2 and U; residual mode W2 and the U/T row stages, in
// the same space
constexpr int kDraftRingBytes = kWStages * kWStageBytes + kUStages * kUStageBytes;
constexpr int kResRingBytes = kWStagesRes * kWStageBytes + 2 * kResStageBytes;
constexpr int kRingBytes = kDraftRingBytes > kResRingBytes ? kDraftRingBytes : kResRingBytes;
constexpr int kSmemBytes = 1024 /*align*/ + kRingBytes + kBarBytes + kXBytes + kGkBytes;

struct __align__(8) Barriers {
  uint64_t full_w[kWStages], empty_w[kWStages];
  uint64_t full_u[kUStages], empty_u[kUStages];
  uint64_t acc_full[2], acc_empty[2];
  uint64_t e_full, drain;
  uint32_t tmem_base;
  int abort;
  int stop;   // epilogue-wide decision to leave the position loop
  int last;   // this CTA's arrival completed the current grid barrier
  int sched;  // this CTA finished the finalize last: it runs the schedule
};
static_assert(sizeof(Barriers) <= kBarBytes, "barrier block overflows its shared-memory slot");
static_assert(sizeof(SchedShared) <= kXBytes, "the schedule's scratch overflows the combine scratch");
static_assert(kSmemBytes <= 232448, "more dynamic shared memory than one CTA may use");

enum Mode { kDraft = 0, kResidual = 1 };

template <int MODE>
__host__ __device__ constexpr int threads_of() { return MODE == kDraft ? kDraftThreads : kThreads; }

// The confidence head computed by the draft's finalize (c_out null: not).
struct ConfArgs {
  const void* h;
  const float* w;
  const float* sts_T;
  float* c_out;
  int hdtype;
  int H;
  bool vec;
};

// The round's schedule run by the draft's last CTA to finish the finalize
// (ell_out null: not; the caller launches the schedule kernel instead).
struct SchedArgs {
  const float* c;                       // the confidences the finalize wrote
  const float* sps;
  int mode;
  int32_t* khist;
  int32_t* ell_out;
  int32_t* nstar_out;
  double* theta_out;
  unsigned int* done;                   // CTAs past the finalize (zeroed before the launch)
};

struct StepParams {
  const float* U;
  const __nv_bfloat16* W1;
  const __nv_bfloat16* W2;              // for the fused finalize
  const int32_t* anchor;
  // draft outputs written by the fused finalize (null: a separate kernel does it)
  int32_t* x_out;
  float* p_out;
  float* lse_out;
  // residual mode: rejected position k* of each request (0 = none), the
  // token before it, the draft lse of every position, the target lse of row
  // k*-1
  const float* T;
  const int32_t* resid_prev;            // x_{k*-1} (the anchor when k* = 1)
  const int32_t* resid_k;
  const float* lse_d;
  const float* resid_lse;
  unsigned long long* resid_key;
  // residual mode (fin not null): the last CTA to finish writes the tokens of
  // the rejecting requests (fin counts finished CTAs, zeroed before)
  unsigned int* fin;
  int32_t* tok_out;
  int nsegs;                            // draft mode: target-statistics segments per row
  // draft mode: softmax partials of the target rows j < G of every request,
  // taken while the draft runs (T_stats null: none); stats_part is the
  // [B*(G+1)][nsegs] partial buffer of verification, stats_next a task counter
  // zeroed before the launch
  const float* T_stats;
  float* tx;                            // [B][G] T[b, k-1, x_k] from the finalize (with T_stats)
  float2* stats_part;
  unsigned int* stats_next;
  // with T_stats: only the rows the accept chains can reach (chain_rej null:
  // every row j < G); chain_mark is set to 1 when so
  int* chain_rej;                       // [B] first position known to reject (0: none yet)
  int* chain_pass;                      // [B] positions 1..chain_pass[b] known not to reject
  unsigned int* rows_done;              // [B*(G+1)] segments of each row's partials written
  int* chain_mark;
  unsigned long long* keys;             // [G][B] argmax keys of every position, kKeyStride apart
  float2* part;                         // [G][part_slices][B] softmax partials
  unsigned int* gbar;                   // grid-barrier counter (zeroed before launch)
  int* status;
  int B, G, V;
  int k_first, k_last;                  // draft positions of this launch
  int part_slices;
  int nctas;                            // CTAs of the grid
  int ctas_per_mtile;
  int ntiles;                           // vocabulary tiles of width BN
  RngKey key;
  ConfArgs conf;                        // draft mode: the confidence head in the finalize
  // the gated recurrent head (gate_g null: the Markov head): its gates [KR]
  // and the states S [B][G][KR] (bf16) the draft writes and the finalize and
  // the residual read as their E rows
  const float* gate_g;
  const float* gate_c;
  __nv_bfloat16* S;
  SchedArgs sched;                      // draft mode: the schedule after the finalize
  // draft mode: the verification's scratch to clear at the start (null: none)
  unsigned long long* vz;               // [bonus_key, resid_k): keys, bonus list, finish counters
  int vz_words;
};

__device__ __forceinline__ int tile_begin(int slice, int nslices, int ntiles) {
  return (int)(((long long)ntiles * slice) / nslices);
}

// Block race of one request row inside one thread's column range (the
// two-level sampler: blocks of 4 tokens race with log of their softmax mass
// plus Gumbel noise; the token inside a leading block is drawn by inverse CDF).
//
// Block q's perturbed log-mass is z_q = run_m + log s_q + G_q, G_q = -log E_q,
// E_q = -log u_q, s_q = sum of exp(l - run_m) over the block.  It can beat zthr
// only if E_q < s_q exp(run_m - zthr); since E_q >= 1 - u_q this needs
// 1 - u_q < s_q * bound.  s_q comes from the softmax terms already computed
// for the normaliser, so the test costs one FMA and one max per block on the
// word's 16 high bits; only blocks that pass it (a few per thousand once zthr
// has settled) get the exact logarithms.
struct RowRace {
  float run_m, run_s;   // online softmax: running max and sum of exp(l - run_m)
  float zbest;          // best perturbed block log-mass of this thread's blocks
  int best_v;           // the token drawn inside that block
  float zthr;           // best perturbed log-mass known anywhere in the row (>= zbest)
  float zpub;           // zbest as last published to the row's global key
  float bound;          // exp(run_m - zthr) with a 2^-10 safety margin
};

constexpr float kLog2e = 1.4426950408889634f;

// Two fp32 values in one 64-bit register, and the two-wide fp32 add and fma
// of sm_100 and later (each lane rounded as the scalar operation rounds).
__device__ __forceinline__ uint64_t f2(float a, float b) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
  return r;
}
__device__ __forceinline__ void f2split(uint64_t r, float& a, float& b) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(r));
}
__device__ __forceinline__ uint64_t f2add(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ uint64_t f2fma(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}

// A block's softmax mass from its four terms: (e0 + e2) + (e1 + e3), the same
// sum wherever a block's mass is formed.
__device__ __forceinline__ float block_sum(float e0, float e1, float e2, float e3) {
  float a, b;
  f2split(f2add(f2(e0, e1), f2(e2, e3)), a, b);
  return a + b;
}

// The four softmax terms e_c = 2^(l_c log2 e - mb) of a block (l2e2 = (log2 e,
// log2 e), nmb2 = (-mb, -mb)) and their sum.
__device__ __forceinline__ float block_terms(float l0, float l1, float l2, float l3, uint64_t l2e2, uint64_t nmb2,
                                             float (&e)[4]) {
  float t0, t1, t2, t3;
  f2split(f2fma(f2(l0, l1), l2e2, nmb2), t0, t1);
  f2split(f2fma(f2(l2, l3), l2e2, nmb2), t2, t3);
  e[0] = ex2_approx(t0);
  e[1] = ex2_approx(t1);
  e[2] = ex2_approx(t2);
  e[3] = ex2_approx(t3);
  return block_sum(e[0], e[1], e[2], e[3]);
}

__device__ __forceinline__ float race_bound(float run_m, float zbest) {
  return exp2f((run_m - zbest) * kLog2e) * (1.0f + 0x1p-10f);
}

// The block race (draft: stream 0; residual: stream 2).  Block j (entries
// 4j .. 4j+3) takes word j of the stream's call sequence (word j mod 4 of
// call j / 4).  A thread's CPP / 4 blocks start at block v0 / 4, a multiple
// of CPP / 4, so one call covers them.
template <int CPP>
__device__ __forceinline__ void block_words(uint32_t (&wb)[CPP / 4], const RngKey& key, uint32_t stream,
                                            uint32_t req, uint32_t pos, int v0) {
  const uint32_t j0 = (uint32_t)v0 >> 2;
  const uint4 ra = rng_call(key, stream, req, pos, j0 >> 2);
  if constexpr (CPP == 16) {
    wb[0] = ra.x; wb[1] = ra.y; wb[2] = ra.z; wb[3] = ra.w;
  } else if constexpr (CPP == 8) {
    const bool up = (j0 & 2u) != 0;
    wb[0] = up ? ra.z : ra.x;
    wb[1] = up ? ra.w : ra.y;
  } else {
    static_assert(CPP == 4, "4, 8 or 16 columns per thread");
    wb[0] = word_of(ra, j0 & 3u);
  }
}

// 2^23 + h from a word's high 16 bits h, exactly, by one byte permutation.
__device__ __forceinline__ float block_hf(uint32_t w) { return __uint_as_float(__byte_perm(w, 0x4B000000u, 0x7632)); }

// wb[q] for a run-time q by explicit selects (no indexed local array).
template <int NB>
__device__ __forceinline__ uint32_t pick_word(const uint32_t (&wb)[NB], int q) {
  uint32_t w = wb[0];
#pragma unroll
  for (int i = 1; i < NB; ++i) w = (q == i) ? wb[i] : w;
  return w;
}

// Screen threshold on fmaf(mass, 65536 bound, 2^23 + h): an entry (a block of
// the draft, a token of the residual) can only win when h > 65535 - 65536 *
// mass * exp(-zthr), i.e. when the exact sum exceeds 2^23 + 65535.  Floats
// there are integers; one unit of slack absorbs the rounding of the fused
// product.
constexpr float kScreenThr = 8454142.0f;   // 2^23 + 65534

// Opens the online softmax state of a row part at its first tile: the running
// maximum is this tile's largest fused logit.  Later tiles keep it unless the
// rare path of the screen finds it exceeded.  Columns past the vocabulary hold
// -inf.
template <int CPP>
__device__ __forceinline__ void race_prep(RowRace& st, const float (&l)[CPP]) {
  float tm = l[0];
#pragma unroll
  for (int c = 1; c < CPP; ++c) tm = fmaxf(tm, l[c]);
  st.run_s = 0.f;
  st.run_m = tm;
  st.bound = race_bound(st.run_m, st.zthr);
}

// Opens the race of a row part: of this tile's blocks, the one most likely to
// win -- largest s_q / (1 - u_q), with its mass s_q and u_q from the 16 high
// bits, a monotone stand-in for L_q + G_q -- is resolved exactly (with its
// token drawn inside it) and becomes the part's best.  Its softmax mass is
// added here and its logits set to -inf, so the screen that follows does not
// meet it again.
template <int CPP>
__device__ __forceinline__ void race_seed(RowRace& st, float (&l)[CPP], const uint32_t (&wb)[CPP / 4], int v0,
                                          const RngKey& key, uint32_t req, uint32_t pos) {
  constexpr int NB = CPP / 4;
  const float mb = st.run_m * kLog2e;
  const uint64_t l2e2 = f2(kLog2e, kLog2e), nmb2 = f2(-mb, -mb);
  float bs = 0.f, bd = 1.f, e0 = 0.f, e1 = 0.f, e2 = 0.f, e3 = 0.f;
  uint32_t bw = 0u;
  int bq = -1;
#pragma unroll
  for (int q = 0; q < NB; ++q) {
    float e[4];
    const float sq = block_terms(l[4 * q], l[4 * q + 1], l[4 * q + 2], l[4 * q + 3], l2e2, nmb2, e);
    const float d = 8454144.0f - block_hf(wb[q]);   // 65536 - h, exactly
    if (sq * bd > bs * d || bq < 0) {
      bs = sq; bd = d; bw = wb[q]; bq = q;
      e0 = e[0]; e1 = e[1]; e2 = e[2]; e3 = e[3];
    }
  }
  const uint32_t j = ((uint32_t)v0 >> 2) + (uint32_t)bq;
  st.zbest = st.run_m + logf(bs) + gumbel_from_bits(bw >> 9);
  st.best_v = block_pick(key, kStreamDraft, req, pos, j, e0, e1, e2, e3);
  st.zthr = fmaxf(st.zthr, st.zbest);
  st.bound = race_bound(st.run_m, st.zthr);
  st.run_s += bs;
#pragma unroll
  for (int q = 0; q < NB; ++q)
#pragma unroll
    for (int c = 0; c < 4; ++c)
      if (q == bq) l[4 * q + c] = -INFINITY;
}

// Rare path of the screen.  When the screen's sum of the tile's softmax terms
// overflowed (`raise`), moves the running maximum up to this tile's and
// recomputes the terms against it; otherwise the terms are the screen's own,
// so that the softmax state depends on the logits alone and not on when
// another CTA's threshold arrived.  Rebuilds the block candidate mask, parks
// the terms in `spill` (block q in 16-byte chunk j0 + q, swizzled) and
// resolves the candidates one by one with the full 23-bit uniforms; a block
// that wins draws its token and tightens the bound for the rest.  Returns the
// tile's softmax sum.
template <int CPP>
__device__ __forceinline__ float race_resolve(RowRace& st, const float (&l)[CPP], const uint32_t (&wb)[CPP / 4],
                                              int v0, unsigned char* spill, int j0, int sw, const RngKey& key,
                                              uint32_t req, uint32_t pos, int* status, bool raise) {
  constexpr int NB = CPP / 4;
  float tm = l[0];
#pragma unroll
  for (int c = 1; c < CPP; ++c) tm = fmaxf(tm, l[c]);
  if (raise && tm > st.run_m) {
    st.run_s *= exp2f((st.run_m - tm) * kLog2e);
    st.run_m = tm;
    st.bound = race_bound(st.run_m, st.zthr);
  }
  const float mb = st.run_m * kLog2e;
  const uint64_t l2e2 = f2(kLog2e, kLog2e), nmb2 = f2(-mb, -mb);
  const float b16 = st.bound * 65536.0f;
  float s = 0.f;
  uint32_t cand = 0;
#pragma unroll
  for (int q = 0; q < NB; ++q) {
    float e[4];
    const float sq = block_terms(l[4 * q], l[4 * q + 1], l[4 * q + 2], l[4 * q + 3], l2e2, nmb2, e);
    s += sq;
    if (fmaf(sq, b16, block_hf(wb[q])) > kScreenThr) cand |= 1u << q;
    *reinterpret_cast<float4*>(spill + (((j0 + q) ^ sw) << 4)) = make_float4(e[0], e[1], e[2], e[3]);
  }
  if (!(s <= 3.0e38f)) record_status(status, DSPARK_ERR_NONFINITE);   // a NaN or infinite logit
#pragma unroll 1
  while (cand) {
    const int q = __ffs(cand) - 1;
    cand &= cand - 1;
    const float4 e = *reinterpret_cast<const float4*>(spill + (((j0 + q) ^ sw) << 4));
    const float sq = block_sum(e.x, e.y, e.z, e.w);
    const float z = st.run_m + logf(sq) + gumbel_from_bits(pick_word<NB>(wb, q) >> 9);
    if (z > st.zbest) {
      st.zbest = z;
      st.best_v = block_pick(key, kStreamDraft, req, pos, ((uint32_t)v0 >> 2) + (uint32_t)q, e.x, e.y, e.z, e.w);
      if (z > st.zthr) {
        st.zthr = z;
        st.bound = race_bound(st.run_m, st.zthr);
      }
    }
  }
  return s;
}

// Screens this tile's blocks against the best perturbed log-mass known for the
// row (zthr) and adds their softmax terms e_v = exp(l_v - run_m) (run_m may lag
// the true maximum: the terms are then above 1, which the merge of the
// partials allows; it is raised only when they overflow).  With the block's mass s_q and the high 16 bits h of its
// uniform: E_q = -log u_q > (65535 - h) / 65536, so the block can only win
// when h + 65536 s_q bound > 65535, with bound = exp(run_m - zthr) (2^-10
// over).  Only the largest left-hand side is kept; a tile that may hold a
// winner, or whose sum is not finite (a logit far above run_m), goes to
// race_resolve.
template <int CPP>
__device__ __forceinline__ void race_screen(RowRace& st, const float (&l)[CPP], const uint32_t (&wb)[CPP / 4],
                                            int v0, unsigned char* spill, int j0, int sw, const RngKey& key,
                                            uint32_t req, uint32_t pos, int* status) {
  constexpr int NB = CPP / 4;
  const float mb = st.run_m * kLog2e;
  const uint64_t l2e2 = f2(kLog2e, kLog2e), nmb2 = f2(-mb, -mb);
  const float b16 = st.bound * 65536.0f;
  float smax = 0.f, s = 0.f;
#pragma unroll
  for (int q = 0; q < NB; ++q) {
    float e[4];
    const float sq = block_terms(l[4 * q], l[4 * q + 1], l[4 * q + 2], l[4 * q + 3], l2e2, nmb2, e);
    s += sq;
    smax = fmaxf(smax, fmaf(sq, b16, block_hf(wb[q])));
  }
  const bool overflow = !(s <= 3.0e38f);
  if (smax > kScreenThr || overflow)
    s = race_resolve<CPP>(st, l, wb, v0, spill, j0, sw, key, req, pos, status, overflow);
  st.run_s += s;
}

// Race of the residual resample: the two-level draw from rho = max(0, p_t -
// p_d) on streams 2 and 6.  Blocks of 4 race with log W_q + G_q, W_q the
// block's summed rho.  A block can beat zthr only if E_q < W_q exp(-zthr), so
// the draft's screen applies with W_q in place of the softmax mass and
// bound = exp(-zthr).
struct ResRace {
  float zbest;   // best perturbed log-weight of this thread's blocks
  int best_v;    // the entry drawn inside that block
  float zthr;    // best known anywhere in the row (>= zbest)
  float zpub;    // zbest as last published to the row's key
  float bound;   // exp(-zthr) with a 2^-10 safety margin
};

__device__ __forceinline__ void resid_raise(ResRace& st, float z) {
  if (z > st.zthr) {
    st.zthr = z;
    st.bound = expf(-st.zthr) * (1.0f + 0x1p-10f);
  }
}

// One tile of the residual race.  rho[c] is this thread's entry v0 + c (any
// value; non-positive ones and those past the vocabulary weigh nothing).
// spill is the thread's row in shared memory (block q in 16-byte chunk
// j0 + q, swizzled by sw).
template <int CPP>
__device__ __forceinline__ void resid_tile(ResRace& st, float (&rho)[CPP], int nv, int v0, unsigned char* spill,
                                           int j0, int sw, const RngKey& key, uint32_t req, uint32_t pos) {
  constexpr int NB = CPP / 4;
#pragma unroll
  for (int c = 0; c < CPP; ++c) rho[c] = (c < nv) ? fmaxf(rho[c], 0.f) : 0.f;
  uint32_t wb[NB];
  block_words<CPP>(wb, key, kStreamResidual, req, pos, v0);
  float W[NB];
#pragma unroll
  for (int q = 0; q < NB; ++q) W[q] = block_sum(rho[4 * q], rho[4 * q + 1], rho[4 * q + 2], rho[4 * q + 3]);
  if (st.zbest == -INFINITY) {
    // open the race with the block most likely to win: largest W_q / (1 - u_q)
    float bw = 0.f, bd = 1.f;
    int bq = -1;
#pragma unroll
    for (int q = 0; q < NB; ++q) {
      const float d = 8454144.0f - block_hf(wb[q]);   // 65536 - h
      if (W[q] > 0.f && (bq < 0 || W[q] * bd > bw * d)) { bw = W[q]; bd = d; bq = q; }
    }
    if (bq < 0) return;   // no residual weight seen yet
    float r0 = 0.f, r1 = 0.f, r2 = 0.f, r3 = 0.f;
    uint32_t wq = 0u;
#pragma unroll
    for (int q = 0; q < NB; ++q)
      if (q == bq) { r0 = rho[4 * q]; r1 = rho[4 * q + 1]; r2 = rho[4 * q + 2]; r3 = rho[4 * q + 3]; wq = wb[q]; W[q] = 0.f; }
    st.zbest = logf(bw) + gumbel_from_bits(wq >> 9);
    st.best_v = block_pick(key, kStreamResidual, req, pos, ((uint32_t)v0 >> 2) + (uint32_t)bq, r0, r1, r2, r3);
    resid_raise(st, st.zbest);
  }
  const float b16 = st.bound * 65536.0f;
  float smax = 0.f;
#pragma unroll
  for (int q = 0; q < NB; ++q) smax = fmaxf(smax, fmaf(W[q], b16, block_hf(wb[q])));
  if (smax > kScreenThr) {
    uint32_t cand = 0;
#pragma unroll
    for (int q = 0; q < NB; ++q) {
      if (W[q] > 0.f && fmaf(W[q], b16, block_hf(wb[q])) > kScreenThr) cand |= 1u << q;
      *reinterpret_cast<float4*>(spill + (((j0 + q) ^ sw) << 4)) =
          make_float4(rho[4 * q], rho[4 * q + 1], rho[4 * q + 2], rho[4 * q + 3]);
    }
#pragma unroll 1
    while (cand) {
      const int q = __ffs(cand) - 1;
      cand &= cand - 1;
      const float4 e = *reinterpret_cast<const float4*>(spill + (((j0 + q) ^ sw) << 4));
      const float z = logf(block_sum(e.x, e.y, e.z, e.w)) + gumbel_from_bits(pick_word<NB>(wb, q) >> 9);
      if (z > st.zbest) {
        st.zbest = z;
        st.best_v = block_pick(key, kStreamResidual, req, pos, ((uint32_t)v0 >> 2) + (uint32_t)q, e.x, e.y, e.z, e.w);
        resid_raise(st, z);
      }
    }
  }
}

// E[m, 64h .. 64h+63] = W1[tok] (K atom h of the token's embedding) into this
// warp's TMEM lanes, columns kTmemE + 32h .. (two bf16 per column, lower k in
// the low half); zeros for rows without a request.
__device__ __forceinline__ void gather_e(const __nv_bfloat16* W1, int tok, bool active, int h, uint32_t taddr) {
  const uint4* wrow = reinterpret_cast<const uint4*>(W1 + (size_t)tok * KR);
  uint32_t ev[32];
#pragma unroll
  for (int c = 0; c < 8; ++c) {
    const uint4 val = active ? __ldg(wrow + h * 8 + c) : make_uint4(0, 0, 0, 0);
    ev[4 * c] = val.x; ev[4 * c + 1] = val.y; ev[4 * c + 2] = val.z; ev[4 * c + 3] = val.w;
  }
  tmem_store_32cols(taddr, ev);
}

// The gated recurrent head: this warp's part of E becomes the state of
// position k, s_k = e_k + a_k * s_{k-1} with e_k = W1[tok] and a_k =
// sigmoid(g * e_k + c) elementwise (K elements 64h .. 64h+63 of the row, two
// bf16 per TMEM column, lower k in the low half), rounded to bf16 as the
// tensor cores read it.  s_{k-1} is this E as it stands (prev_from_tmem), the
// row of S written one position earlier (prev_row, when a launch starts at
// k > 1), or zero.  The new state also goes to s_row (unless null).
__device__ __forceinline__ void gated_update_e(const __nv_bfloat16* W1, int tok, bool active, int h, uint32_t taddr,
                                               const float* __restrict__ gate_g, const float* __restrict__ gate_c,
                                               bool prev_from_tmem, const __nv_bfloat16* prev_row,
                                               __nv_bfloat16* s_row) {
  const uint4* wrow = reinterpret_cast<const uint4*>(W1 + (size_t)tok * KR);
#pragma unroll 1
  for (int q8 = 0; q8 < 4; ++q8) {   // 8 columns (16 K elements) at a time
    uint32_t sp[8], out[8];
    if (prev_from_tmem) {
      float f[8];
      tmem_load_cols<8>(taddr + q8 * 8, f);
#pragma unroll
      for (int i = 0; i < 8; ++i) sp[i] = __float_as_uint(f[i]);
    } else if (prev_row != nullptr && active) {
      const uint4 a0 = __ldcg(reinterpret_cast<const uint4*>(prev_row + 64 * h + 16 * q8));
      const uint4 a1 = __ldcg(reinterpret_cast<const uint4*>(prev_row + 64 * h + 16 * q8) + 1);
      sp[0] = a0.x; sp[1] = a0.y; sp[2] = a0.z; sp[3] = a0.w; sp[4] = a1.x; sp[5] = a1.y; sp[6] = a1.z; sp[7] = a1.w;
    } else {
#pragma unroll
      for (int i = 0; i < 8; ++i) sp[i] = 0u;
    }
    const uint4 w0 = active ? __ldg(wrow + h * 8 + 2 * q8) : make_uint4(0, 0, 0, 0);
    const uint4 w1 = active ? __ldg(wrow + h * 8 + 2 * q8 + 1) : make_uint4(0, 0, 0, 0);
    const uint32_t ew[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int kk = 64 * h + 16 * q8 + 2 * i;   // K element of the low half
      const float2 g2 = __ldg(reinterpret_cast<const float2*>(gate_g + kk));
      const float2 c2 = __ldg(reinterpret_cast<const float2*>(gate_c + kk));
      const float e0 = __uint_as_float(ew[i] << 16), e1 = __uint_as_float(ew[i] & 0xFFFF0000u);
      const float s0 = __uint_as_float(sp[i] << 16), s1 = __uint_as_float(sp[i] & 0xFFFF0000u);
      const float a0 = 1.f / (1.f + expf(-fmaf(g2.x, e0, c2.x)));
      const float a1 = 1.f / (1.f + expf(-fmaf(g2.y, e1, c2.y)));
      const __nv_bfloat162 n2 = __floats2bfloat162_rn(fmaf(a0, s0, e0), fmaf(a1, s1, e1));
      out[i] = active ? *reinterpret_cast<const uint32_t*>(&n2) : 0u;
    }
    tmem_store_8cols(taddr + q8 * 8, out);
    if (s_row != nullptr && active) {
      uint4* dst = reinterpret_cast<uint4*>(s_row + 64 * h + 16 * q8);
      dst[0] = make_uint4(out[0], out[1], out[2], out[3]);
      dst[1] = make_uint4(out[4], out[5], out[6], out[7]);
    }
  }
}

// Residual mode: copies the U and T row segments of one 64-column tile
// starting at column vt into a shared-memory stage, 16 threads to a 256-byte
// segment (coalesced).  Chunk c of row rr lands at rr * 256 + ((c ^ (rr & 15))
// << 4) (U), R * 256 further (T), so that row-per-lane reads spread over the
// banks.  off[rr] / off[BM + rr] are the element offsets of row rr's U / T
// rows, -1 for a request that did not reject.  Called by every epilogue thread.
template <int R>
__device__ __forceinline__ void resid_copy(unsigned char* stage, const long long* off, const float* U,
                                           const float* T, int vt, int V) {
  // 2 tensors x R rows x 16 chunks = R / 16 copies for each of the 512
  // epilogue threads: copy j of thread tid is tensor j / (R / 32), row
  // (j % (R / 32)) * 32 + tid / 16, chunk tid % 16.  The chunk, the row's low
  // bits (and so the swizzle) are the thread's own; with the loop unrolled
  // only the row offset lookup and the addresses remain per copy.
  constexpr int kPer = R / 16, kHalf = kPer / 2;
  const int tid = threadIdx.x - 64;
  const int c16 = tid & 15, r16 = tid >> 4;
  const int v = vt + c16 * 4;
  if (v < V) {
    unsigned char* dst0 = stage + r16 * 256 + ((c16 ^ (r16 & 15)) << 4);
#pragma unroll
    for (int j = 0; j < kPer; ++j) {
      const int tensor = j / kHalf, rr = (j % kHalf) * 32 + r16;
      const long long o = off[tensor * BM + rr];
      if (o >= 0) cp_async16(dst0 + tensor * (R * 256) + (j % kHalf) * 32 * 256, (tensor ? T : U) + o + v);
    }
  }
  cp_async_commit();
}

// R = rows of one request replica (32, 64 or 128).  With B <= 64 the M tile
// holds 128 / R copies of the requests so that every TMEM lane quarter -- and
// so every epilogue warp -- has rows to work on; each copy takes its own share
// of the tile's columns.
// Grid-wide barrier between draft positions.  Every CTA adds 1 to a counter in
// global memory after publishing its position-k results; the CTA then waits,
// bounded in time, until all `nctas` CTAs have arrived for this position.
__device__ __forceinline__ uint32_t ld_acquire_u32(const unsigned int* p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// Returns the counter's value before this arrival.  The add is an
// acquire-release atomic at GPU scope: its release covers this thread's
// writes and, through the CTA barrier that precedes every arrival, the other
// threads' writes and key atomics; its acquire lets the last CTA to arrive
// read what the others published without waiting in grid_wait.
__device__ __forceinline__ unsigned int grid_arrive(unsigned int* counter) {
  unsigned int old;
  asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], 1;" : "=r"(old) : "l"(counter) : "memory");
  return old;
}

__device__ __forceinline__ bool grid_wait(unsigned int* counter, uint32_t target, volatile int* abort, int* status) {
  const uint64_t t0 = globaltimer();
  while (ld_acquire_u32(counter) < target) {
    if (*abort) return false;
    if (globaltimer() - t0 > kWaitLimitNs) {
      *abort = 1;
      record_status(status, DSPARK_ERR_TIMEOUT);
      return false;
    }
  }
  return true;
}

__device__ __forceinline__ bool grid_barrier(unsigned int* counter, uint32_t target, volatile int* abort,
                                             int* status) {
  grid_arrive(counter);
  return grid_wait(counter, target, abort, status);
}

// Target-row statistics riding along the draft.  Verification needs the
// softmax normaliser of every target row it tests; those rows depend only on
// T, so when the caller already holds T they can be streamed while the draft
// runs, in the HBM time the draft leaves idle.  Each warp takes (row,
// segment) tasks from a shared counter -- rows j < G of every request,
// kStatsSeg entries per segment -- and leaves the segment's (max, sum of exp)
// in part[row][seg].  A segment is read in pieces of 2048 entries (16 float4
// per lane, all in flight before any arithmetic), with loads marked for early
// eviction from L2: W2, which every draft position re-reads from L2, must not
// be pushed out by a stream that is read once.
constexpr int kStatsLoadsWarp = 16;   // float4 per lane per piece of a warp that loads for itself
constexpr int kStatsPiece = 32 * 4 * kStatsLoadsWarp;   // entries per piece (8 KB)

// The (max, sum of exp) of one piece of a row, folded into a lane's running
// state (x: this lane's entries, -inf past the row's end).
template <int N>
__device__ __forceinline__ void stats_fold(float& m, float& s, const float4 (&x)[N], bool& bad) {
  float bm = -INFINITY;
#pragma unroll
  for (int i = 0; i < N; ++i) bm = fmaxf(fmaxf(bm, fmaxf(x[i].x, x[i].y)), fmaxf(x[i].z, x[i].w));
  bad |= !(bm < INFINITY);
  if (bm > m) {
    s = (m == -INFINITY) ? 0.f : s * ex2_approx((m - bm) * kLog2e);
    m = bm;
  }
  if (m == -INFINITY) return;
  const float mb = m * kLog2e;
  float acc = 0.f;
#pragma unroll
  for (int i = 0; i < N; ++i)
    acc += (ex2_approx(fmaf(x[i].x, kLog2e, -mb)) + ex2_approx(fmaf(x[i].y, kLog2e, -mb))) +
           (ex2_approx(fmaf(x[i].z, kLog2e, -mb)) + ex2_approx(fmaf(x[i].w, kLog2e, -mb)));
  s += acc;
}

// Row and segment of statistics task t.
__device__ __forceinline__ void stats_task_at(int t, int G, int nsegs, size_t& rowid, int& seg) {
  const int ri = t / nsegs;
  seg = t - ri * nsegs;
  const int b = ri / G, j = ri - b * G;
  rowid = (size_t)b * (G + 1) + j;
}

// (max, sum of exp) partial merge with one 2^x on the special-function unit,
// kept small: the accept tests below run beside the draft's epilogue warps,
// and every instruction they bring in competes with the epilogue's own for
// the SM's instruction cache.
__device__ __forceinline__ void chain_merge(float& m, float& s, float m2, float s2) {
  if (m2 > m) {
    const float tm = m, ts = s;
    m = m2; s = s2; m2 = tm; s2 = ts;
  }
  if (m2 > -INFINITY) s += s2 * ex2_approx((m2 - m) * kLog2e);
}

// The accept test of position m of request b, run by one warp on what the
// draft has published so far ([blog] section 1: accept x_m when u < p_t(x_m)
// / p_d(x_m), u the verification's uniform of stream 1 at (b, m)).  Returns
// -1 while an input is not out yet (lse_d of position m needs every CTA's
// softmax partial of m, which a CTA writes after its arrival at the grid
// barrier of m and before its next arrival -- at the barrier of m + 1, or
// the finalize's after the last position; lse_t of row m-1 needs every
// segment of that row), -2 when the test cannot be run (a non-finite ratio
// or a bad token: verification sees to it), 1 when the test fails with a
// margin of 2^-8 relative, 0 otherwise.
// p_d comes from the draft's partials and the fused logit of x_m as the
// finalize forms them, p_t from the row's partials as verify_decide merges
// them; the margin covers the rounding of the two and of the special-function
// unit's 2^x and log2, so that a position called rejected here is rejected
// there too.  Lane 0 reads the readiness with plain loads, acquires once it
// sees it, and takes the decision for the warp (the lanes' reductions may
// differ in their last bit).
__device__ __forceinline__ int chain_test(const StepParams* __restrict__ p, const RngKey& key, int b, int m,
                                          int lane) {
  const int B = p->B, G = p->G, V = p->V, nsegs = p->nsegs;
  const size_t rowid = (size_t)b * (G + 1) + (m - 1);
  int ready = 0;
  if (lane == 0) {
    ready = *reinterpret_cast<const volatile unsigned int*>(p->gbar) >=
                (uint32_t)p->nctas * (uint32_t)min(m + 1, G) &&
            *reinterpret_cast<const volatile unsigned int*>(p->rows_done + rowid) >= (uint32_t)nsegs;
    if (ready) {
      // acquire what the arrivals and the segment counts released
      (void)ld_acquire_u32(p->gbar);
      (void)ld_acquire_u32(p->rows_done + rowid);
    }
  }
  ready = __shfl_sync(0xffffffffu, ready, 0);
  __syncwarp();
  if (!ready) return -1;
  const float2* pp = p->part + (size_t)(m - 1) * p->part_slices * B + (size_t)b * p->part_slices;
  float md = -INFINITY, sd = 0.f;
#pragma unroll 1
  for (int i = lane; i < p->ctas_per_mtile; i += 32) {
    const float2 pr = __ldcg(pp + i);
    chain_merge(md, sd, pr.x, pr.y);
  }
#pragma unroll 1
  for (int off = 16; off > 0; off >>= 1) {
    const float m2 = __shfl_xor_sync(0xffffffffu, md, off), s2 = __shfl_xor_sync(0xffffffffu, sd, off);
    chain_merge(md, sd, m2, s2);
  }
  const unsigned long long kk = __ldcg(p->keys + ((size_t)(m - 1) * B + b) * kKeyStride);
  const int x = kk ? argmax_key_index(kk) : -1;
  int prev = p->anchor[b];
  if (m > 1) {
    const unsigned long long kp = __ldcg(p->keys + ((size_t)(m - 2) * B + b) * kKeyStride);
    prev = kp ? argmax_key_index(kp) : -1;
  }
  if (x < 0 || x >= V || prev < 0 || prev >= V) return -2;   // (the same on every lane)
  const __nv_bfloat16* erow =
      p->gate_g != nullptr ? p->S + ((size_t)b * G + (m - 1)) * KR : p->W1 + (size_t)prev * KR;
  // this lane's 8 of the 256 products (one 16-byte load per row)
  const uint4 e8 = __ldcg(reinterpret_cast<const uint4*>(erow) + lane);
  const uint4 w8 = __ldg(reinterpret_cast<const uint4*>(p->W2 + (size_t)x * KR) + lane);
  const __nv_bfloat162* ea = reinterpret_cast<const __nv_bfloat162*>(&e8);
  const __nv_bfloat162* wa = reinterpret_cast<const __nv_bfloat162*>(&w8);
  float dot = 0.f;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 ef = __bfloat1622float2(ea[i]), wf = __bfloat1622float2(wa[i]);
    dot = fmaf(ef.x, wf.x, fmaf(ef.y, wf.y, dot));
  }
#pragma unroll 1
  for (int off = 16; off > 0; off >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, off);
  int res = -2;
  if (lane == 0) {
    float mt = -INFINITY, st = 0.f;
#pragma unroll 1
    for (int i = 0; i < nsegs; ++i) {
      const float2 q2 = __ldcg(p->stats_part + rowid * nsegs + i);
      chain_merge(mt, st, q2.x, q2.y);
    }
    // p_t / p_d in base 2 on the special-function unit (within the margin)
    const float l2d = (p->U[((size_t)b * G + (m - 1)) * V + x] + dot - md) * kLog2e - lg2_approx(sd);
    const float l2t = (p->T_stats[rowid * V + x] - mt) * kLog2e - lg2_approx(st);
    const float ratio = ex2_approx(l2t - l2d);
    if (sd > 0.f && st > 0.f && ratio >= 0.f) {   // (sums that a row can have; not NaN)
      const uint4 rw = rng4(key, kStreamAccept, (uint32_t)b, (uint32_t)m, 0u);
      res = uniform01(rw.x) >= ratio * (1.0f + 0x1p-8f) ? 1 : 0;
    }
  }
  return __shfl_sync(0xffffffffu, res, 0);
}

// Whether row j of request b can be reached by the accept tests: no position
// 1..j is known to reject.  Positions are tested in order and the outcome is
// kept per request.  A test whose inputs are not out yet, or that cannot be
// run, counts as reachable: the row is taken ahead of its decision (waiting
// for the draft's barriers instead left the rows of the long chains for
// after the draft), so a row is skipped only once verification is certain to
// stop before it.  Inline: an out-of-line call here cost the draft ~10 us per
// launch in every form, lazy or not (the calling convention's hold on the
// kernel's registers).  Warp-uniform.
__device__ __forceinline__ bool chain_row_needed(const StepParams* __restrict__ p, const RngKey& key, int b, int j,
                                                 int lane) {
#pragma unroll 1
  for (int guard = 0; guard <= j; ++guard) {
    int rej = 0, pass = 0;
    if (lane == 0) {
      rej = *reinterpret_cast<volatile int*>(p->chain_rej + b);
      pass = *reinterpret_cast<volatile int*>(p->chain_pass + b);
    }
    rej = __shfl_sync(0xffffffffu, rej, 0);
    pass = __shfl_sync(0xffffffffu, pass, 0);
    if (rej != 0 && rej <= j) return false;
    if (pass >= j) return true;
    const int m = pass + 1;
    const int res = chain_test(p, key, b, m, lane);
    if (res < 0) return true;
    if (res == 1) {
      if (lane == 0) atomicCAS(p->chain_rej + b, 0, m);
      return false;
    }
    if (lane == 0) atomicMax(p->chain_pass + b, m);
  }
  return true;
}

// One warp, whole tasks with its own loads: kStatsLoadsWarp float4 per lane
// per piece, all in flight before any arithmetic, marked for early eviction
// from L2 (W2, which every draft position re-reads from L2, must not be
// pushed out by a stream read once).  The next task index is fetched while a
// task runs.  With chain_rej the tasks go position by position (every
// request's row 0, then row 1, ...), rows no accept test will reach are
// skipped, each finished segment is counted in rows_done, and non-finite
// entries are left to verification, which checks the rows its tests use (a
// row read here ahead of its request's rejection is not one of them).
template <bool kChain>
__device__ __forceinline__ void stats_tasks(const StepParams* __restrict__ p, const RngKey& key,
                                            volatile int* abort) {
  const float* __restrict__ T = p->T_stats;
  const int B = p->B, G = p->G, V = p->V, nsegs = p->nsegs;
  float2* __restrict__ part = p->stats_part;
  unsigned int* next = p->stats_next;
  const int lane = threadIdx.x & 31;
  const int ntasks = B * G * nsegs;
  // kChain false: the chain code is compiled out (its mere presence in the
  // loop cost the drafts that take every row, or none, ~5 us per launch);
  // kChain true keeps both paths behind the run-time test, which measured
  // ~6 us faster for the chains' draft than a loop with the chain path alone
  const bool chain = kChain && p->chain_rej != nullptr;
  const uint64_t pol = policy_evict_first();
  bool bad = false;
  unsigned int t = 0;
  if (lane == 0) t = atomicAdd(next, 1u);
  t = __shfl_sync(0xffffffffu, t, 0);
  while ((int)t < ntasks && !*abort) {
    unsigned int t_next = 0;
    if (lane == 0) t_next = atomicAdd(next, 1u);   // its reply is needed only at the next task
    size_t rowid;
    int seg;
    if (chain) {
      const int ri = (int)t / nsegs;
      seg = (int)t - ri * nsegs;
      const int j = ri / B, b = ri - j * B;
      rowid = (size_t)b * (G + 1) + j;
      if (j > 0) {
        // the request's known outcome first, here in the loop's own code; the
        // out-of-line tests only when a position must be tested
        int known = 0;   // 1: needed, -1: not needed, 0: test
        if (lane == 0) {
          const int rej = *reinterpret_cast<volatile int*>(p->chain_rej + b);
          const int pass = *reinterpret_cast<volatile int*>(p->chain_pass + b);
          known = (rej != 0 && rej <= j) ? -1 : (pass >= j ? 1 : 0);
        }
        known = __shfl_sync(0xffffffffu, known, 0);
        if (known < 0 || (known == 0 && !chain_row_needed(p, key, b, j, lane))) {
          t = __shfl_sync(0xffffffffu, t_next, 0);
          continue;
        }
      }
    } else {
      stats_task_at((int)t, G, nsegs, rowid, seg);
    }
    const float* row = T + rowid * V;
    const int v0 = seg * kStatsSeg, v1 = min(V, v0 + kStatsSeg);
    float m = -INFINITY, s = 0.f;
#pragma unroll 1
    for (int vp = v0; vp < v1; vp += kStatsPiece) {
      float4 x[kStatsLoadsWarp];
#pragma unroll
      for (int i = 0; i < kStatsLoadsWarp; ++i) {
        const int v = vp + 4 * (lane + 32 * i);
        x[i] = v < v1 ? ld_stream_f4(row + v, pol) : make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
      }
      stats_fold(m, s, x, bad);
    }
    warp_softmax_reduce(m, s, 0xffffffffu, 32);
    if (lane == 0) {
      part[rowid * nsegs + seg] = make_float2(m, s);
      // the segment count is a release add: the partial above is visible to
      // whoever acquires the count
      if (chain) asm volatile("red.release.gpu.global.add.u32 [%0], 1;" ::"l"(p->rows_done + rowid) : "memory");
    }
    t = __shfl_sync(0xffffffffu, t_next, 0);
  }
  if (bad && !chain) record_status(p->status, DSPARK_ERR_NONFINITE);
}

// The draft outputs of one (request, position), by one warp: merge the slice
// partials into lse_k, decode x_k from its argmax key and recompute the fused
// logit of x_k for p_k(x_k).
// The confidence head of one finalize item, kept out of line so that its
// loads in flight do not raise the draft loop's register count.
__device__ __noinline__ void finalize_conf(const ConfArgs& ca, const __nv_bfloat16* __restrict__ W1, int item,
                                           int k, int prev_x, int V, int lane, int* __restrict__ status) {
  if (ca.hdtype == DSPARK_BF16)
    conf_item<DSPARK_BF16, DSPARK_BF16>(ca.h, W1, ca.w, ca.sts_T, item, k, prev_x, ca.H, KR, V, ca.vec, lane,
                                        ca.c_out, status);
  else
    conf_item<DSPARK_F32, DSPARK_BF16>(ca.h, W1, ca.w, ca.sts_T, item, k, prev_x, ca.H, KR, V, ca.vec, lane,
                                       ca.c_out, status);
}

__device__ __forceinline__ void finalize_item(int item, int lane, const float* __restrict__ U,
                                              const __nv_bfloat16* __restrict__ W1,
                                              const __nv_bfloat16* __restrict__ W2, const int32_t* __restrict__ anchor,
                                              const unsigned long long* __restrict__ keys,
                                              const float2* __restrict__ part, int B, int G, int V, int nslices,
                                              int part_slices, int32_t* __restrict__ x_out, float* __restrict__ p_out,
                                              float* __restrict__ lse_out, const ConfArgs& ca,
                                              const float* __restrict__ T_early, float* __restrict__ tx,
                                              const __nv_bfloat16* __restrict__ S, int* __restrict__ status) {
  const int b = item / G, k = item - (item / G) * G + 1;
  const float2* pp = part + (size_t)(k - 1) * part_slices * B;
  float m = -INFINITY, s = 0.f;
  for (int i = lane; i < nslices; i += 32) {
    const float2 pr = __ldcg(pp + (size_t)b * part_slices + i);   // written by other CTAs of this launch
    softmax_merge(m, s, pr.x, pr.y);
  }
  warp_softmax_reduce(m, s, 0xffffffffu, 32);
  const float lse = m + logf(s);
  const unsigned long long kk = __ldcg(keys + ((size_t)(k - 1) * B + b) * kKeyStride);
  int x = kk ? argmax_key_index(kk) : -1;
  if (x < 0 || x >= V) {
    if (lane == 0) record_status(status, DSPARK_ERR_NONFINITE);
    x = 0;
  }
  // x_{k-1} as the output holds it (the anchor at k = 1)
  int prev_x = anchor[b];
  if (k > 1) {
    const unsigned long long kp = __ldcg(keys + ((size_t)(k - 2) * B + b) * kKeyStride);
    prev_x = kp ? argmax_key_index(kp) : -1;
    if (prev_x < 0 || prev_x >= V) prev_x = 0;
  }
  const int prev = checked_token(prev_x, V, status);
  // the bias operand: W1[x_{k-1}], or the gated head's state s_k
  const __nv_bfloat16* erow = S != nullptr ? S + ((size_t)b * G + (k - 1)) * KR : W1 + (size_t)prev * KR;
  float dot = 0.f;
  for (int i = lane; i < KR; i += 32)
    dot = fmaf(__bfloat162float(erow[i]), __bfloat162float(W2[(size_t)x * KR + i]), dot);
  for (int off = 16; off > 0; off >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, off);
  if (lane == 0) {
    const size_t o = (size_t)b * G + (k - 1);
    x_out[o] = x;
    p_out[o] = expf(U[o * (size_t)V + x] + dot - lse);
    lse_out[o] = lse;
    // the target logit of the drafted token, for the accept test (T taken along)
    if (T_early != nullptr) tx[o] = T_early[((size_t)b * (G + 1) + (k - 1)) * V + x];
  }
  if (ca.c_out != nullptr) finalize_conf(ca, W1, item, k, prev_x, V, lane, status);
}

// MODE kDraft: draft positions k_first..k_last for every request (U rows by
// TMA).  With more than one position the CTAs of the grid must be co-resident
// (cooperative launch): after each position they meet at a grid barrier so
// that the next position can read x_k from the argmax keys.  The producer and
// the MMA pipelines run on across positions, so the U and W2 tiles of the next
// position are already loading while the barrier resolves.
// MODE kResidual: for every request that rejected at position k*, the fused
// draft logits of k* again, raced over log max(0, p_t - p_d) (U and T rows
// read directly by the epilogue threads).
template <int R, int MODE, bool kChain = false>
__global__ void __launch_bounds__(threads_of<MODE>(), 1)
draft_step_tc(const __grid_constant__ CUtensorMap w2_map, const __grid_constant__ CUtensorMap u_map,
              const __grid_constant__ StepParams p) {
  constexpr int kRepl = BM / R;            // copies of each request row
  constexpr int kParts = 4 * kRepl;        // column parts of a tile
  constexpr int CPP = BN / kParts;         // columns per thread per tile
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
  constexpr int kWSt = MODE == kDraft ? kWStages : kWStagesRes;   // W2 ring depth of this mode
  unsigned char* W_s = smem;
  unsigned char* U_s = W_s + kWSt * kWStageBytes;      // draft: U ring; residual: U/T row stages
  Barriers* bars = reinterpret_cast<Barriers*>(smem + kRingBytes);
  unsigned char* X_s = reinterpret_cast<unsigned char*>(bars) + kBarBytes;   // combine scratch

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int mtile = blockIdx.x / p.ctas_per_mtile;
  const int slice = blockIdx.x - mtile * p.ctas_per_mtile;
  const int m0 = mtile * R;
  const int rows_valid = min(R, p.B - m0);
  const int t0 = tile_begin(slice, p.ctas_per_mtile, p.ntiles);
  const int t1 = tile_begin(slice + 1, p.ctas_per_mtile, p.ntiles);
  const int ntl = t1 - t0;
  const int kf = p.k_first, kl = p.k_last;
  volatile int* abort = &bars->abort;
  const RngKey key = live_key(p.key);
  if constexpr (MODE == kDraft) {
    if (p.chain_mark != nullptr && blockIdx.x == 0 && threadIdx.x == 0) *p.chain_mark = 1;
    if (p.vz != nullptr) {
      for (int i = blockIdx.x * threads_of<MODE>() + threadIdx.x; i < p.vz_words; i += gridDim.x * threads_of<MODE>())
        p.vz[i] = 0ull;
    }
  }
  // (no early trigger in either mode: the next kernel's CTAs, resident and
  // waiting on the SMs this grid leaves, were measured to slow the kernels
  // that follow)

  if (threadIdx.x == 0) {
    for (int s = 0; s < kWStages; ++s) { mbar_init(&bars->full_w[s], 1); mbar_init(&bars->empty_w[s], 1); }
    for (int s = 0; s < kUStages; ++s) { mbar_init(&bars->full_u[s], 1); mbar_init(&bars->empty_u[s], kEpiWarps); }
    for (int s = 0; s < 2; ++s) { mbar_init(&bars->acc_full[s], 1); mbar_init(&bars->acc_empty[s], kEpiWarps); }
    mbar_init(&bars->e_full, kEpiWarps);
    mbar_init(&bars->drain, 1);
    bars->abort = 0;
    bars->last = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tensormap(&w2_map);
    if (MODE == kDraft) prefetch_tensormap(&u_map);
  }
  if (warp == 1) tmem_alloc(&bars->tmem_base, kTmemCols);
  for (int idx = threadIdx.x; idx < kGkBytes / 16; idx += threads_of<MODE>())
    reinterpret_cast<uint4*>(X_s + kXBytes)[idx] = make_uint4(0u, 0u, 0u, 0u);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem_base;
  // residual mode: the set-up above overlapped the kernel before this one; its
  // outputs (the rejected positions, the keys to raise) are read by the
  // epilogue warps from here on.  The producer (W2 only) and the MMA issuer
  // read nothing an earlier kernel writes, so the W2 atoms start loading now.
  if (warp >= 2) pdl_wait();

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    const uint64_t pol_w = policy_evict_last(), pol_u = policy_evict_first();
    uint32_t wcount = 0, ucount = 0;
    bool ok = true;
    for (int k = kf; k <= kl && ok; ++k) {
      for (int g = 0; g < ntl && ok; g += group_tiles(g)) {
        // the W2 rows of an MMA group's tiles, one K atom at a time (rows past
        // the CTA's range or past V are loaded or zero-filled but not used)
        const int v0 = (t0 + g) * BN;
        for (int a = 0; a < kAtoms && ok; ++a, ++wcount) {
          const int s = wcount % kWSt;
          ok = mbar_wait(&bars->empty_w[s], ((wcount / kWSt) & 1) ^ 1, abort, p.status);
          if (ok && lane == 0) {
            mbar_arrive_expect_tx(&bars->full_w[s], kWStageBytes);
            tma_g2s_2d(W_s + s * kWStageBytes, &w2_map, a * 64, v0, &bars->full_w[s], pol_w);
          }
        }
        if (!ok) break;
        if constexpr (MODE != kDraft) continue;
        const int nsub = min(group_tiles(g), ntl - g);
        for (int j = 0; j < nsub && ok; ++j) {
          const int su = ucount % kUStages;
          ok = mbar_wait(&bars->empty_u[su], ((ucount / kUStages) & 1) ^ 1, abort, p.status);
          if (!ok) break;
          if (lane == 0) {
            // two [R rows x 32 columns] boxes of U[m0.., k-1, v..]; rows past B and
            // columns past V are filled with zeros by the copy engine
            const int v = v0 + j * BN;
            mbar_arrive_expect_tx(&bars->full_u[su], (uint32_t)(2 * kUBox * R * 4));
            unsigned char* dst = U_s + su * kUStageBytes;
            tma_g2s_3d(dst, &u_map, v, k - 1, m0, &bars->full_u[su], pol_u);
            tma_g2s_3d(dst + R * 128, &u_map, v + kUBox, k - 1, m0, &bars->full_u[su], pol_u);
          }
          ++ucount;
        }
      }
    }
    // drain: every copy this warp issued has landed before the CTA exits
    if (lane == 0 && *abort) {
      for (uint32_t c = (wcount > (uint32_t)kWSt ? wcount - kWSt : 0); c < wcount; ++c)
        mbar_drain(&bars->full_w[c % kWSt], (c / kWSt) & 1);
      for (uint32_t c = (ucount > kUStages ? ucount - kUStages : 0); c < ucount; ++c)
        mbar_drain(&bars->full_u[c % kUStages], (c / kUStages) & 1);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      uint32_t wcount = 0, gcount = 0;
      bool ok = true;
      for (int k = kf; k <= kl && ok; ++k) {
        ok = mbar_wait(&bars->e_full, (uint32_t)(k - kf) & 1, abort, p.status);
        tc_fence_after();
        for (int g = 0; g < ntl && ok; g += group_tiles(g), ++gcount) {
          // one MMA tile: up to kGroup vocabulary tiles, N = 64 per tile
          const int acc = gcount & 1;
          ok = mbar_wait(&bars->acc_empty[acc], ((gcount >> 1) & 1) ^ 1, abort, p.status);
          if (!ok) break;
          tc_fence_after();
          const uint32_t idesc = idesc_bf16_f32(BM, BN * min(group_tiles(g), ntl - g));
          const uint32_t d_tmem = tmem + acc * kAccCols;
          for (int a = 0; a < kAtoms && ok; ++a, ++wcount) {
            const int s = wcount % kWSt;
            ok = mbar_wait(&bars->full_w[s], (wcount / kWSt) & 1, abort, p.status);
            if (!ok) break;
            tc_fence_after();
            // A = E in TMEM: K elements 64a + 16kk .. are columns 32a + 8kk ..;
            // B = the atom's W2 rows, advanced 32 bytes per K step of 16
            const uint64_t bd0 = sw128_kmajor_desc(smem_u32(W_s + s * kWStageBytes));
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
              umma_bf16_tmem_a(d_tmem, tmem + kTmemE + a * 32 + kk * 8, bd0 + (uint64_t)(kk * 2), idesc,
                               (a | kk) != 0);
            umma_commit(&bars->empty_w[s]);
          }
          if (ok) umma_commit(&bars->acc_full[acc]);
        }
      }
      // all MMAs this thread issued are complete before TMEM is released
      umma_commit(&bars->drain);
      mbar_drain(&bars->drain, 0);
    }
    __syncwarp();
  } else if (warp < 2 + kEpiWarps) {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;               // TMEM lane quarter of this warp
    const int h = (warp - 2) >> 2;        // which of the four warps of the quarter
    const int m = q * 32 + lane;          // TMEM lane = row of the M tile
    const int rep = m / R, r = m - rep * R;
    const int part = rep * 4 + h;         // column part of every tile
    const int b = m0 + r;
    float* xm = reinterpret_cast<float*>(X_s);
    float* xs = xm + 4 * BM;
    unsigned long long* xk = reinterpret_cast<unsigned long long*>(xs + 4 * BM);
    // draft: shared-memory copies of the row keys, one region per position
    // parity (filled by the first warp of each lane quarter, read by all)
    ulonglong2* gk_rows = reinterpret_cast<ulonglong2*>(X_s + kXBytes);
    uint32_t it = 0, gcount = 0;
    int spec_prev = -1;   // token whose W1 row is in TMEM E from the speculative gather
    int spec_raw = 0;     // the key's token as read for that gather
    bool spec_final = false;   // that read came after every CTA had arrived
    for (int k = kf; k <= kl; ++k) {
      bool active = r < rows_valid;
      int ks = k;                           // position of this row
      int res_prev = 0;
      if constexpr (MODE == kResidual) {
        if (active) {
          ks = p.resid_k[b];
          res_prev = p.resid_prev[b];       // (loaded with ks; read only if ks > 0)
        } else {
          ks = 0;
        }
        active = ks > 0;
      }

      // E = W1[x_{k-1}] into TMEM (gather_e).  From the second position on, E
      // was already gathered speculatively from the row keys as they stood when
      // this CTA reached the grid barrier; a warp reloads only if one of its
      // rows' final x_{k-1} differs.
      int prev = 0;
      if (active) {
        int raw;
        if constexpr (MODE == kDraft)
          raw = (k == 1) ? p.anchor[b]
                : spec_final ? spec_raw
                             : argmax_key_index(__ldcg(p.keys + ((size_t)(k - 2) * p.B + b) * kKeyStride));
        else
          raw = res_prev;
        prev = checked_token(raw, p.V, p.status);
      }
      const uint32_t e_taddr = tmem + ((uint32_t)(q * 32) << 16) + kTmemE + h * 32;
      if (MODE == kDraft && p.gate_g != nullptr) {
        // the gated head: E becomes s_k (from s_{k-1}, which is E as it stands
        // within a launch); slice 0 of the M tile records it for the finalize
        // and the residual
        const size_t srow = (size_t)b * p.G;
        gated_update_e(p.W1, prev, active, h, e_taddr, p.gate_g, p.gate_c, k > kf,
                       (k == kf && k > 1) ? p.S + (srow + k - 2) * KR : nullptr,
                       (slice == 0 && rep == 0) ? p.S + (srow + k - 1) * KR : nullptr);
      } else if (MODE == kResidual && p.S != nullptr) {
        // residual of a gated-head draft: E is the state of position k*
        gather_e(p.S, active ? b * p.G + ks - 1 : 0, active, h, e_taddr);
      } else if (MODE != kDraft || k == kf) {
        gather_e(p.W1, prev, active, h, e_taddr);
      } else if (__any_sync(0xffffffffu, prev != spec_prev)) {
        // only the rows whose token changed are read again
        float ef[32];
        tmem_load_cols<32>(e_taddr, ef);
        uint32_t ev[32];
#pragma unroll
        for (int c = 0; c < 32; ++c) ev[c] = __float_as_uint(ef[c]);
        if (prev != spec_prev) {
          const uint4* wrow = reinterpret_cast<const uint4*>(p.W1 + (size_t)prev * KR);
#pragma unroll
          for (int c = 0; c < 8; ++c) {
            const uint4 val = active ? __ldg(wrow + h * 8 + c) : make_uint4(0, 0, 0, 0);
            ev[4 * c] = val.x; ev[4 * c + 1] = val.y; ev[4 * c + 2] = val.z; ev[4 * c + 3] = val.w;
          }
        }
        tmem_store_32cols(e_taddr, ev);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars->e_full);

      RowRace st{-INFINITY, 0.f, -INFINITY, -1, -INFINITY, -INFINITY, INFINITY};
      // every row's best is shared across CTAs (draft and residual)
      constexpr bool kShare = (MODE == kDraft);
      unsigned long long* row_key = (kShare && active) ? p.keys + ((size_t)(k - 1) * p.B + b) * kKeyStride : nullptr;
      ResRace rs{-INFINITY, -1, -INFINITY, -INFINITY, INFINITY};
      constexpr bool kShareRes = (MODE == kResidual);
      unsigned long long* res_key = (kShareRes && active) ? p.resid_key + (size_t)b * kKeyStride : nullptr;
      float ld2 = 0.f, lt2 = 0.f;
      if constexpr (MODE == kResidual) {
        if (active) {
          ld2 = p.lse_d[(size_t)b * p.G + ks - 1] * kLog2e;
          lt2 = p.resid_lse[b] * kLog2e;
        }
      }
      bool ok = true;
      // residual mode: the U and T row segments of each tile are copied into
      // shared memory one tile ahead by all epilogue threads (resid_copy)
      long long* off_u = reinterpret_cast<long long*>(X_s);   // element offset of row rr's U row, or -1
      long long* off_t = off_u + BM;
      if constexpr (MODE != kDraft) {
        const int tid = threadIdx.x - 64;
        if (tid < R) {
          const int bb = m0 + tid;
          int kk = 0;
          if (bb < p.B) kk = p.resid_k[bb];
          off_u[tid] = kk > 0 ? ((long long)bb * p.G + (kk - 1)) * p.V : -1;
          off_t[tid] = kk > 0 ? ((long long)bb * (p.G + 1) + (kk - 1)) * p.V : -1;
        }
        named_bar_sync(1, kEpiWarps * 32);
        if (ntl > 0) resid_copy<R>(U_s, off_u, p.U, p.T, t0 * BN, p.V);
      }
      for (int i = 0; i < ntl; ++i, ++it) {
        // the tiles of an MMA group (group_tiles) share an accumulator: wait
        // for it at the first, hand it back after reading the last
        const int sub = i == 0 ? 0 : (i - 1) % kGroup;   // tile's place in its MMA group
        const bool last_sub = i == 0 || sub == kGroup - 1 || i == ntl - 1;
        const int acc_i = gcount & 1;
        const int v0 = (t0 + i) * BN + part * CPP;
        const int nv = min(CPP, p.V - v0);
        if constexpr (MODE != kDraft) {
          // this tile's rows have landed (own copies, then everyone's); the
          // barrier also frees the other stage for the next tile's copies.
          // Every epilogue thread passes here each tile, failed or not.  The
          // row-key copy of the previous tile (the newest group of the first
          // warp of each quarter) may stay in flight.
          if (kShareRes && h == 0 && i > 0) cp_async_wait_one();
          else cp_async_wait_all();
          named_bar_sync(1, kEpiWarps * 32);
          if (i + 1 < ntl) resid_copy<R>(U_s + ((i + 1) & 1) * kResStageBytes, off_u, p.U, p.T, (t0 + i + 1) * BN, p.V);
        }
        // (warp-uniform: the TMEM load below is warp-wide)
        const bool got_acc =
            sub != 0 || __all_sync(0xffffffffu, mbar_wait(&bars->acc_full[acc_i], (gcount >> 1) & 1, abort, p.status));
        if (MODE != kDraft && !got_acc) ok = false;
        float v[CPP];
        if (got_acc) {
          tc_fence_after();
          tmem_load_cols<CPP>(tmem + ((uint32_t)(q * 32) << 16) + acc_i * kAccCols + sub * BN + part * CPP, v);
          if (last_sub) {
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars->acc_empty[acc_i]);
            ++gcount;
          }
        }
        if constexpr (MODE == kDraft) {
          const int su = it % kUStages;
          const bool got_u = got_acc && mbar_wait(&bars->full_u[su], (it / kUStages) & 1, abort, p.status);
          // this thread's columns: box (part*CPP)/32, 16-byte chunks j0.. of row r,
          // stored at chunk j ^ (r & 7) (128-byte swizzle)
          unsigned char* urow = U_s + su * kUStageBytes + ((part * CPP) / kUBox) * (R * 128) + r * 128;
          const int j0 = ((part * CPP) % kUBox) / 4;
          const bool live = got_u && active && nv > 0;
          uint32_t wb[CPP / 4];
          if (live) {
#pragma unroll
            for (int c = 0; c < CPP; c += 4) {
              const float4 u4 = *reinterpret_cast<const float4*>(urow + (((j0 + c / 4) ^ (r & 7)) << 4));
              f2split(f2add(f2(v[c + 0], v[c + 1]), f2(u4.x, u4.y)), v[c + 0], v[c + 1]);
              f2split(f2add(f2(v[c + 2], v[c + 3]), f2(u4.z, u4.w)), v[c + 2], v[c + 3]);
            }
            if (nv < CPP) {
              // past the end of the vocabulary: out of the softmax and the race
#pragma unroll
              for (int c = 0; c < CPP; ++c)
                if (c >= nv) v[c] = -INFINITY;
            }
            block_words<CPP>(wb, key, kStreamDraft, (uint32_t)b, (uint32_t)k, v0);
            if (st.run_m == -INFINITY) race_prep<CPP>(st, v);
            if (st.zbest == -INFINITY) race_seed<CPP>(st, v, wb, v0, key, (uint32_t)b, (uint32_t)k);
          }
          if (i == 0) {
            // the parts of a row pool their seeds before the first screen
            xm[part * R + r] = live ? st.zthr : -INFINITY;
            named_bar_sync(1, kEpiWarps * 32);
            if (live) {
              float zm = st.zthr;
#pragma unroll
              for (int j = 0; j < kParts; ++j) zm = fmaxf(zm, xm[j * R + r]);
              if (zm > st.zthr) {
                st.zthr = zm;
                st.bound = race_bound(st.run_m, st.zthr);
              }
            }
          }
          if (live) {
            // the row's best perturbed log-mass published by any CTA, from
            // the latest copy of its key that has landed in shared memory (0
            // while none has this position); nothing waits for the copies
            if (kShare && i >= 1) {
              const unsigned long long gkd =
                  *reinterpret_cast<volatile unsigned long long*>(&gk_rows[(k & 1) * BM + r].x);
              if (gkd) {
                const float zg = argmax_key_value(gkd);
                if (zg > st.zthr) {
                  st.zthr = zg;
                  st.bound = race_bound(st.run_m, st.zthr);
                }
              }
            }
            race_screen<CPP>(st, v, wb, v0, urow, j0, r & 7, key, (uint32_t)b, (uint32_t)k, p.status);
            // share this thread's progress with the other CTAs of the row
            if (kShare && st.best_v >= 0 && st.zbest > st.zpub && st.zbest >= st.zthr) {
              atomicMax(row_key, argmax_key(st.zbest, st.best_v));
              st.zpub = st.zbest;
            }
            if (kShare && h == 0 && rep == 0) {
              cp_async16(gk_rows + (k & 1) * BM + r, row_key);
              cp_async_commit();
            }
          }
          __syncwarp();
          if (!got_u) { ok = false; break; }
          if (lane == 0) mbar_arrive(&bars->empty_u[su]);
        } else {
          if (ok && got_acc && active && nv > 0) {
            // this thread's columns of its row: chunks j0.. of the staged U and
            // T segments; rho = max(0, p_t - p_d) goes back into the U slots
            // (non-positive entries are outside the residual's support and
            // never race)
            unsigned char* urow = U_s + (i & 1) * kResStageBytes + r * 256;
            const unsigned char* trow = urow + R * 256;
            const int j0 = (part * CPP) / 4, sw = r & 15;
            float uu[CPP];
            const uint64_t l2e2 = f2(kLog2e, kLog2e), nld2 = f2(-ld2, -ld2), nlt2 = f2(-lt2, -lt2);
#pragma unroll
            for (int c = 0; c < CPP; c += 4) {
              const float4 u4 = *reinterpret_cast<const float4*>(urow + (((j0 + c / 4) ^ sw) << 4));
              const float4 t4 = *reinterpret_cast<const float4*>(trow + (((j0 + c / 4) ^ sw) << 4));
              // exponents of p_d (fused logit) and p_t, two lanes at a time
              float ad[4], at[4];
              f2split(f2fma(f2add(f2(v[c], v[c + 1]), f2(u4.x, u4.y)), l2e2, nld2), ad[0], ad[1]);
              f2split(f2fma(f2add(f2(v[c + 2], v[c + 3]), f2(u4.z, u4.w)), l2e2, nld2), ad[2], ad[3]);
              f2split(f2fma(f2(t4.x, t4.y), l2e2, nlt2), at[0], at[1]);
              f2split(f2fma(f2(t4.z, t4.w), l2e2, nlt2), at[2], at[3]);
#pragma unroll
              for (int e = 0; e < 4; ++e) uu[c + e] = ex2_approx(at[e]) - ex2_approx(ad[e]);
            }
            // the row's best from other CTAs: the latest copy of its key that
            // has landed in shared memory (nothing waits for it)
            if (kShareRes && i >= 1) {
              const unsigned long long gkr = *reinterpret_cast<volatile unsigned long long*>(&gk_rows[r].x);
              if (gkr) resid_raise(rs, argmax_key_value(gkr));
            }
            resid_tile<CPP>(rs, uu, nv, v0, urow, j0, sw, key, (uint32_t)b, (uint32_t)ks);
            if (kShareRes && rs.best_v >= 0 && rs.zbest > rs.zpub && rs.zbest >= rs.zthr) {
              atomicMax(res_key, argmax_key(rs.zbest, rs.best_v));
              rs.zpub = rs.zbest;
            }
          }
          if (kShareRes && h == 0) {
            // one copy group per tile (empty when the row is idle or held by
            // another replica), so that the wait above always leaves exactly
            // this copy in flight
            if (ok && active && rep == 0) cp_async16(gk_rows + r, res_key);
            cp_async_commit();
          }
        }
      }
      if (MODE == kDraft && (st.run_m != st.run_m || st.run_m == INFINITY))
        record_status(p.status, DSPARK_ERR_NONFINITE);

      // combine the parts of each request row, then publish one partial per row
      unsigned long long key = 0ull;
      if constexpr (MODE == kDraft) key = st.best_v >= 0 ? argmax_key(st.zbest, st.best_v) : 0ull;
      else key = rs.best_v >= 0 ? argmax_key(rs.zbest, rs.best_v) : 0ull;
      named_bar_sync(1, kEpiWarps * 32);
      // Every key publish of this position was issued before the barrier
      // above, so the CTA arrives at the grid barrier now (the softmax
      // partials below are read only after the last barrier).
      if (kShare && k < kl && warp == 2 && lane == 0) {
        // the last CTA to arrive knows that every key is final already
        const uint32_t target = (uint32_t)(p.nctas * (k - kf + 1));
        bars->last = (!*abort && grid_arrive(p.gbar) + 1u == target) ? 1 : 0;
      }
      const int slot = part * R + r;               // parts of row r at r, R + r, ...
      xm[slot] = st.run_m;
      xs[slot] = st.run_s;
      xk[slot] = key;
      named_bar_sync(1, kEpiWarps * 32);
      if (part == 0 && active && ok) {
        float M = -INFINITY, S = 0.f;
        unsigned long long K = 0ull;
#pragma unroll
        for (int j = 0; j < kParts; ++j) {
          softmax_merge(M, S, xm[j * R + r], xs[j * R + r]);
          K = xk[j * R + r] > K ? xk[j * R + r] : K;
        }
        if constexpr (MODE == kDraft) {
          // No key update here: the CTA's best is already in the row key.
          // Each part published its best whenever it reached the part's
          // threshold, and a threshold is always a value some part has
          // published.
          p.part[((size_t)(k - 1) * p.B + b) * p.part_slices + slice] = make_float2(M, S);
        } else {
          if (K) atomicMax(&p.resid_key[(size_t)b * kKeyStride], K);
        }
      }
      (void)ok;
      if (k < kl) {
        // Speculative gather while the barrier resolves: this CTA's MMAs of
        // position k are complete (its last accumulator was read), so TMEM E
        // is free; load W1[x_k] for the row keys as they stand now.  After the
        // barrier the final keys are compared and only changed rows reload.
        if (MODE == kDraft && p.gate_g == nullptr) {
          int sp = 0;
          spec_final = kShare && bars->last;
          if (active) {
            spec_raw = argmax_key_index(__ldcg(p.keys + ((size_t)(k - 1) * p.B + b) * kKeyStride));
            sp = (spec_raw >= 0 && spec_raw < p.V) ? spec_raw : 0;
          }
          gather_e(p.W1, sp, active, h, tmem + ((uint32_t)(q * 32) << 16) + kTmemE + h * 32);
          spec_prev = active ? sp : 0;
        }
        if constexpr (kShare) {
          // this position's key copies have landed; the next position's
          // region starts empty (its copies, two positions back, have long
          // landed, and every warp passes the barrier below before it reads
          // the region again)
          if (h == 0 && rep == 0) {
            cp_async_wait_all();
            gk_rows[((k + 1) & 1) * BM + r] = make_ulonglong2(0ull, 0ull);
          }
        }
        // one thread takes the decision to go on, all epilogue warps read it
        // after the same barrier, so they all leave the loop together.  The
        // last CTA to arrive saw the count complete in its own arrival (an
        // acquire), so it does not wait.
        if (warp == 2 && lane == 0) {
          bool go = !*abort;
          if (go && !(kShare && bars->last))
            go = grid_wait(p.gbar, (uint32_t)(p.nctas * (k - kf + 1)), abort, p.status);
          bars->stop = go ? 0 : 1;
        }
        named_bar_sync(1, kEpiWarps * 32);
        if (bars->stop) break;
      }
    }
    cp_async_wait_all();   // no copy outlives the CTA's shared memory
    if constexpr (MODE == kResidual) {
      if (p.fin != nullptr) {
        // every residual key this CTA raises was raised before this barrier;
        // the CTA whose count completes the grid's writes the tokens: the
        // winner of each rejecting request's race, or (a residual with no
        // positive entry in floating point) a draw from its T row
        named_bar_sync(1, kEpiWarps * 32);
        if (warp == 2 && lane == 0) {
          __threadfence();
          bars->sched = atomicAdd(p.fin, 1u) == (unsigned int)p.nctas - 1u ? 1 : 0;
        }
        named_bar_sync(1, kEpiWarps * 32);
        if (bars->sched) {
          __threadfence();
          // one request per thread; the rare draws from a T row by the warp
          for (int base = 0; base < p.B; base += kEpiWarps * 32) {
            const int bb = base + (int)threadIdx.x - 64;
            int ks = 0;
            unsigned long long k1 = 0ull;
            if (bb < p.B) {
              ks = p.resid_k[bb];
              k1 = __ldcg(p.resid_key + (size_t)bb * kKeyStride);
            }
            if (bb < p.B && ks > 0 && k1) p.tok_out[bb] = argmax_key_index(k1);
            unsigned int fb = __ballot_sync(0xffffffffu, bb < p.B && ks > 0 && !k1);
            while (fb) {
              const int src = __ffs(fb) - 1;
              fb &= fb - 1;
              const int b2 = __shfl_sync(0xffffffffu, bb, src), k2 = __shfl_sync(0xffffffffu, ks, src);
              int tok = warp_softmax_draw(p.T + ((size_t)b2 * (p.G + 1) + (k2 - 1)) * p.V, p.V, (uint32_t)b2,
                                          (uint32_t)k2, key, lane);
              if (tok < 0) {
                if (lane == 0) record_status(p.status, DSPARK_ERR_NONFINITE);
                tok = 0;
              }
              if (lane == 0) p.tok_out[b2] = tok;
            }
          }
        }
      }
    }
    if constexpr (MODE == kDraft) {
      if (p.x_out != nullptr) {
        // Fused finalize (persistent launch over every position): once every
        // CTA's partials of the last position are out, the epilogue warps of
        // the grid finish the (request, position) items, one warp each.
        named_bar_sync(1, kEpiWarps * 32);
        if (warp == 2 && lane == 0) {
          bool go = !*abort;
          if (go) {
            grid_arrive(p.gbar);
            go = grid_wait(p.gbar, (uint32_t)(p.nctas * (kl - kf + 1)), abort, p.status);
          }
          bars->stop = go ? 0 : 1;
        }
        named_bar_sync(1, kEpiWarps * 32);
        if (!bars->stop) {
          for (int item = blockIdx.x * kEpiWarps + (warp - 2); item < p.B * p.G; item += p.nctas * kEpiWarps)
            finalize_item(item, lane, p.U, p.W1, p.W2, p.anchor, p.keys, p.part, p.B, p.G, p.V, p.ctas_per_mtile,
                          p.part_slices, p.x_out, p.p_out, p.lse_out, p.conf, p.T_stats, p.tx,
                          p.gate_g != nullptr ? p.S : nullptr, p.status);
          if (p.sched.ell_out != nullptr) {
            // The last CTA to finish its finalize items (every confidence is
            // written then) runs the round's schedule in its shared memory
            // (the rings are idle now) while the other CTAs go on to the
            // target-row statistics.
            named_bar_sync(1, kEpiWarps * 32);
            if (warp == 2 && lane == 0) {
              __threadfence();
              bars->sched = atomicAdd(p.sched.done, 1u) == (unsigned int)p.nctas - 1u ? 1 : 0;
            }
            named_bar_sync(1, kEpiWarps * 32);
            if (bars->sched) {
              __threadfence();
              SchedShared* sh = reinterpret_cast<SchedShared*>(X_s);
              schedule_block<kEpiWarps * 32>(p.sched.c, p.B, p.G, p.sched.sps, p.sched.mode, live_round(p.key),
                                             p.sched.khist, p.sched.ell_out, p.sched.nstar_out, p.sched.theta_out,
                                             p.status, smem, *sh, (int)threadIdx.x - 64,
                                             NamedSync<kEpiWarps * 32>{});
            }
          }
        }
      }
      // the draft is done: the epilogue warps help with whatever target-row
      // statistics are left
      if (p.T_stats != nullptr)
        stats_tasks<kChain>(&p, key, abort);
    }
  } else {
    // ------------------------------------------------------------ statistics
    // (draft mode only: the warps past the epilogue).  Their loads bypass the
    // SM's bulk-copy engine, which the draft's U and W2 tiles keep busy.
    if (p.T_stats != nullptr)
      stats_tasks<kChain>(&p, key, abort);
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, kTmemCols);
}

// One warp per (request, position): merge the slice partials into lse_k,
// decode x_k from its argmax key and recompute the fused logit of x_k.
__global__ void draft_finalize_tc(const float* __restrict__ U, const __nv_bfloat16* __restrict__ W1,
                                  const __nv_bfloat16* __restrict__ W2, const int32_t* __restrict__ anchor,
                                  const unsigned long long* __restrict__ keys, const float2* __restrict__ part,
                                  int B, int G, int V, int nslices, int part_slices, int32_t* __restrict__ x_out,
                                  float* __restrict__ p_out, float* __restrict__ lse_out, const ConfArgs ca,
                                  const float* __restrict__ T_early, float* __restrict__ tx,
                                  const __nv_bfloat16* __restrict__ S, int* __restrict__ status) {
  const int item = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  if (item >= B * G) return;
  finalize_item(item, threadIdx.x & 31, U, W1, W2, anchor, keys, part, B, G, V, nslices, part_slices, x_out, p_out,
                lse_out, ca, T_early, tx, S, status);
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  });
  return fn;
}

}  // namespace

// W2 [V, 256] bf16 viewed as a 2-D tensor (K innermost) with 64 x 64 boxes,
// 128-byte swizzled: one box is one K atom of a 64-column vocabulary tile.
cudaError_t make_w2_tensor_map(const void* W2, int V, CUtensorMap* map, int rows) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = encode_fn();
  if (!enc) return cudaErrorNotSupported;
  if (rows <= 0 || rows > 256) return cudaErrorInvalidValue;
  cuuint64_t dims[2] = {(cuuint64_t)KR, (cuuint64_t)V};
  cuuint64_t strides[1] = {(cuuint64_t)KR * 2};
  cuuint32_t box[2] = {64, (cuuint32_t)rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(W2), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

// U [B, G, V] fp32 viewed as a 3-D tensor (V innermost) with [R x 1 x 32]
// boxes, 128-byte swizzled: one box is 32 columns of R request rows at one
// position.
cudaError_t make_u_tensor_map(const float* U, int B, int G, int V, int R, CUtensorMap* map) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = encode_fn();
  if (!enc) return cudaErrorNotSupported;
  cuuint64_t dims[3] = {(cuuint64_t)V, (cuuint64_t)G, (cuuint64_t)B};
  cuuint64_t strides[2] = {(cuuint64_t)V * 4, (cuuint64_t)G * V * 4};
  cuuint32_t box[3] = {(cuuint32_t)kUBox, 1, (cuuint32_t)R};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<float*>(U), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

// U [B, G, V] fp32 viewed as a 4-D tensor {32 columns, V / 32 column blocks,
// G, B} with {32, 2, 1, R} boxes, 128-byte swizzled: one box is the 64
// columns of one vocabulary tile for R request rows at one position, fetched
// as 256 contiguous bytes per row (a [R x 1 x 32] box fetches 128 bytes per
// row, and a stream of those runs reaches about two thirds of the copy rate
// of 256-byte runs on GB300).  In shared memory row r's half h is the
// 128-byte line 2r + h.  Only whole 32-column blocks are in the view: with V
// % 32 != 0 the vocabulary's last tile must come from make_u_tensor_map's
// boxes; blocks past the view (and rows past B) are zero-filled.
cudaError_t make_u_tile_map(const float* U, int B, int G, int V, int R, CUtensorMap* map) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = encode_fn();
  if (!enc) return cudaErrorNotSupported;
  if (V < 32) return cudaErrorInvalidValue;
  cuuint64_t dims[4] = {32, (cuuint64_t)(V / 32), (cuuint64_t)G, (cuuint64_t)B};
  cuuint64_t strides[3] = {128, (cuuint64_t)V * 4, (cuuint64_t)G * V * 4};
  cuuint32_t box[4] = {32, 2, 1, (cuuint32_t)R};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, const_cast<float*>(U), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

namespace {

// Self-test of the bounded waits: mode 0 waits on an mbarrier that no thread
// arrives on, mode 1 at a grid barrier that expects two CTAs in a one-CTA
// grid.  Either wait gives up after kWaitLimitNs, records DSPARK_ERR_TIMEOUT in
// `status` and the kernel returns.
__global__ void selftest_wait_kernel(int mode, unsigned int* counter, int* status) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    volatile int* abort = &abort_flag;
    if (mode == 0)
      mbar_wait(&bar, 0, abort, status);
    else
      grid_barrier(counter, 2u, abort, status);
  }
  __syncthreads();
}

}  // namespace

cudaError_t launch_selftest_wait(int mode, void* ws, cudaStream_t stream) {
  unsigned int* counter = ws_ptr<unsigned int>(ws, 64);
  cudaError_t e = cudaMemsetAsync(counter, 0, sizeof(unsigned int), stream);
  if (e != cudaSuccess) return e;
  selftest_wait_kernel<<<1, 32, 0, stream>>>(mode, counter, ws_ptr<int>(ws, 0));
  return cudaGetLastError();
}

bool draft_tc_supported(int wdtype, int r, int V) { return wdtype == DSPARK_BF16 && r == KR && V >= kAccCols; }

cudaError_t launch_markov_draft_tc(const DraftArgs& a, cudaStream_t stream) {
  const WsLayout L = ws_layout(a.B, a.gamma, a.V);
  int* status = ws_ptr<int>(a.ws, L.status);
  unsigned int* ctr = ws_ptr<unsigned int>(a.ws, L.counters);
  unsigned int* gbar = ctr + 32;   // the grid-barrier counter, on a line of its own
  unsigned long long* keys = ws_ptr<unsigned long long>(a.ws, L.draft_keys);
  float2* part = ws_ptr<float2>(a.ws, L.draft_part);
  const int part_slices = draft_part_slices(a.V);

  CUtensorMap map;
  cudaError_t e = make_w2_tensor_map(a.W2, a.V, &map);
  if (e != cudaSuccess) return e;
  int dev = 0, sms = 0, coop = 0;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
  if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
  if ((e = cudaDeviceGetAttribute(&coop, cudaDevAttrCooperativeLaunch, dev)) != cudaSuccess) return e;
  const int R = a.B <= 32 ? 32 : (a.B <= 64 ? 64 : BM);
  CUtensorMap umap;
  if ((e = make_u_tensor_map(a.U, a.B, a.gamma, a.V, R, &umap)) != cudaSuccess) return e;
  auto kern = R == 32 ? draft_step_tc<32, kDraft> : (R == 64 ? draft_step_tc<64, kDraft> : draft_step_tc<BM, kDraft>);
  // the persistent launch taking the chains' target rows runs a kernel of its own
  auto kern_chain = R == 32 ? draft_step_tc<32, kDraft, true>
                            : (R == 64 ? draft_step_tc<64, kDraft, true> : draft_step_tc<BM, kDraft, true>);
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
  if (e != cudaSuccess) return e;
  if (a.T_stats != nullptr && a.chain_stats &&
      (e = cudaFuncSetAttribute(kern_chain, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes)) != cudaSuccess)
    return e;
  e = cudaMemsetAsync(keys, 0, sizeof(unsigned long long) * kKeyStride * (size_t)a.gamma * a.B, stream);
  if (e != cudaSuccess) return e;
  // the target-statistics task counter, the count of CTAs past the
  // finalize, the marker of verification's full row pass, the marker of
  // statistics taken along the accept chains only and the grid-barrier
  // counter (words 1..32)
  if ((e = cudaMemsetAsync(ctr + 1, 0, 32 * sizeof(unsigned int), stream)) != cudaSuccess) return e;

  const int mtiles = div_up(a.B, R);
  const int ntiles = div_up(a.V, BN);
  int per = std::max(1, sms / mtiles);
  per = std::min(per, std::min(ntiles, part_slices));
  const int nctas = mtiles * per;
  StepParams sp{};
  sp.U = a.U;
  sp.W1 = static_cast<const __nv_bfloat16*>(a.W1);
  sp.W2 = static_cast<const __nv_bfloat16*>(a.W2);
  sp.anchor = a.anchor;
  sp.keys = keys;
  sp.part = part;
  sp.gbar = gbar;
  sp.status = status;
  sp.B = a.B; sp.G = a.gamma; sp.V = a.V;
  sp.part_slices = part_slices;
  sp.nctas = nctas;
  sp.ctas_per_mtile = per;
  sp.ntiles = ntiles;
  sp.key = a.key;
  sp.nsegs = stats_num_segs(a.V);
  sp.stats_part = ws_ptr<float2>(a.ws, L.row_part);
  sp.stats_next = ctr + 2;
  sp.tx = ws_ptr<float>(a.ws, L.tx);
  if (a.gate_g != nullptr) {
    sp.gate_g = a.gate_g;
    sp.gate_c = a.gate_c;
    sp.S = ws_ptr<__nv_bfloat16>(a.ws, L.gstate);
  }
  if (a.c_out != nullptr)
    sp.conf = ConfArgs{a.h, a.w, a.sts_T, a.c_out, a.hdtype, a.H, conf_vec(a.h, a.W1, a.w, a.H, a.r)};
  if (a.zero_verify_scratch) {
    sp.vz = ws_ptr<unsigned long long>(a.ws, L.bonus_key);
    sp.vz_words = (int)((L.resid_k - L.bonus_key) / sizeof(unsigned long long));
  }

  // One persistent launch over all positions when every CTA can be resident
  // at once (one CTA per SM); otherwise one launch per position.
  int resident = 0;
  if ((e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&resident, kern, kDraftThreads, kSmemBytes)) !=
      cudaSuccess)
    return e;
  const bool want_sched = a.ell_out != nullptr && a.c_out != nullptr;
  bool sched_fused = false;
  if (coop && nctas <= resident * sms) {
    sp.k_first = 1;
    sp.k_last = a.gamma;
    // the schedule in the last CTA when its scan fits 512 threads (8
    // candidates each) and its keys and values fit the idle rings
    if (want_sched && (long long)a.B * a.gamma <= 8 * kEpiWarps * 32 &&
        schedule_smem_bytes(a.B, a.gamma) <= (size_t)kRingBytes) {
      sp.sched = SchedArgs{a.c_out, a.sps, a.mode, a.khist, a.ell_out, a.nstar_out, a.theta_out, ctr + 3};
      sched_fused = true;
    }
    // the target-row statistics ride along in the statistics warps, of every
    // row j < gamma or of the rows the accept chains can reach
    sp.T_stats = a.T_stats;
    if (a.T_stats != nullptr && a.chain_stats) {
      int* cst = ws_ptr<int>(a.ws, L.chain_stats);
      if ((e = cudaMemsetAsync(cst, 0, sizeof(int) * (2 * (size_t)a.B + (size_t)a.B * (a.gamma + 1)), stream)) !=
          cudaSuccess)
        return e;
      sp.chain_rej = cst;
      sp.chain_pass = cst + a.B;
      sp.rows_done = reinterpret_cast<unsigned int*>(cst + 2 * a.B);
      sp.chain_mark = reinterpret_cast<int*>(ctr) + 5;
    }
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(nctas);
    cfg.blockDim = dim3(kDraftThreads);
    cfg.dynamicSmemBytes = kSmemBytes;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    // the persistent launch also finishes the outputs (x, p, lse)
    sp.x_out = a.x_out;
    sp.p_out = a.p_out;
    sp.lse_out = a.lse_out;
    if ((e = cudaLaunchKernelEx(&cfg, sp.chain_rej != nullptr ? kern_chain : kern, map, umap, sp)) != cudaSuccess)
      return e;
  } else {
    for (int k = 1; k <= a.gamma; ++k) {
      sp.k_first = sp.k_last = k;
      kern<<<nctas, kDraftThreads, kSmemBytes, stream>>>(map, umap, sp);
    }
    draft_finalize_tc<<<div_up(a.B * a.gamma * 32, 256), 256, 0, stream>>>(
        a.U, static_cast<const __nv_bfloat16*>(a.W1), static_cast<const __nv_bfloat16*>(a.W2), a.anchor, keys,
        part, a.B, a.gamma, a.V, per, part_slices, a.x_out, a.p_out, a.lse_out, sp.conf, a.T_stats, sp.tx,
        sp.gate_g != nullptr ? sp.S : nullptr, status);
    // one launch per position: the target-row statistics follow the draft
    if (a.T_stats != nullptr && (e = cudaGetLastError()) == cudaSuccess)
      e = launch_row_stats(a.T_stats, nullptr, a.B, a.gamma, a.V, a.ws, stream);
    if (e != cudaSuccess) return e;
  }
  if (want_sched && !sched_fused) {
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    e = launch_schedule(a.c_out, a.B, a.gamma, a.sps, a.mode, (unsigned long long)(a.key.round3 >> 3),
                        a.key.round_dev, a.khist, a.ell_out, a.nstar_out, a.theta_out, status, stream);
    if (e != cudaSuccess) return e;
  }
  return cudaGetLastError();
}

// The residual resample of every rejecting request on the tensor cores: the
// bias of W1[x_{k*-1}] against all of W2 again (one GEMM, as for a draft
// position), p_d = exp(U + bias - lse_d), p_t = exp(T - lse_t), and a Gumbel
// race over log max(0, p_t - p_d) into resid_key (atomicMax).
cudaError_t launch_residual_tc(const float* T, const float* U, const void* W1, const void* W2,
                               const int32_t* resid_prev, const float* lse_d, const int32_t* resid_k,
                               const float* resid_lse, unsigned long long* resid_key, int B, int G, int V,
                               RngKey key, const void* gstate, unsigned int* fin, int32_t* tok_out, int* status,
                               cudaStream_t stream) {
  CUtensorMap map;
  cudaError_t e = make_w2_tensor_map(W2, V, &map);
  if (e != cudaSuccess) return e;
  int dev = 0, sms = 0;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
  if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
  const int R = B <= 32 ? 32 : (B <= 64 ? 64 : BM);
  auto kern = R == 32 ? draft_step_tc<32, kResidual>
                      : (R == 64 ? draft_step_tc<64, kResidual> : draft_step_tc<BM, kResidual>);
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
  if (e != cudaSuccess) return e;
  const int mtiles = div_up(B, R);
  const int ntiles = div_up(V, BN);
  int per = std::max(1, sms / mtiles);
  per = std::min(per, ntiles);
  StepParams sp{};
  sp.U = U;
  sp.W1 = static_cast<const __nv_bfloat16*>(W1);
  sp.T = T;
  sp.resid_prev = resid_prev;
  // a gated-head draft's states: the residual's E rows (null: W1 rows)
  sp.S = const_cast<__nv_bfloat16*>(static_cast<const __nv_bfloat16*>(gstate));
  sp.resid_k = resid_k;
  sp.lse_d = lse_d;
  sp.resid_lse = resid_lse;
  sp.resid_key = resid_key;
  sp.fin = fin;
  sp.tok_out = tok_out;
  sp.status = status;
  sp.B = B; sp.G = G; sp.V = V;
  sp.k_first = sp.k_last = 0;
  sp.nctas = mtiles * per;
  sp.ctas_per_mtile = per;
  sp.ntiles = ntiles;
  sp.key = key;
  // the U map is not read in this mode; any valid map will do
  e = launch_pdl(kern, dim3(mtiles * per), dim3(kThreads), kSmemBytes, stream, map, map, sp);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace dspark
