// Acceptance labels on the tensor cores (the study report's Eq.8: the
// probability that rejection sampling accepts position k is the mass the
// draft and target distributions share, sum_v min(p_d(v), p_t(v)); it is the
// confidence head's training label, "[DeepSeek-6] DSpark" blog, section 5).
//
// One persistent launch runs every position k = 1..G; 152 CTAs, each owning a
// 128-request M tile (128 / R replicas of R rows for small batches) and a
// contiguous range of 64-column vocabulary tiles, as the draft does.  For a
// fixed position every request's U and T rows form one box of the [V, G, B]
// and [V, G + 1, B] tensors, so both stream in by TMA like the draft's U:
//
//   warp 0      TMA producer: W2 atoms of 192 rows x 64 K (bf16, 128-byte
//               swizzled, evict_last) and, per 64-column tile, one box of
//               U[., k-1, .] and one of T[., k-1, .] (R rows x 64 columns,
//               256 contiguous bytes per row, evict_first) into a ring of two
//               stages; it runs ahead across positions.  With V % 32 != 0 the
//               vocabulary's last tile comes as two [R x 32] boxes per tensor.
//   warp 1      TMEM allocation and the single-thread MMA issuer: the bias
//               E * W2_rows^T of up to two tiles per tcgen05.mma (fp32 in
//               TMEM columns 0-255, two accumulators), E = W1[x_{k-1}] in
//               TMEM columns 256-383 or 384-511 by the parity of k, so that
//               the E of position k + 2 is gathered while position k + 1's
//               MMAs run and the issuer never waits for a gather at a
//               position boundary.
//   warps 2-17  epilogue (thread = request row, 16 columns per tile):
//               p_d = exp(acc + U - lse_d), p_t = exp(T - lse_t), sum of
//               min(p_d, p_t) over the row's columns; at a position's end the
//               parts of a row are added and each CTA adds its share into
//               label[b][k-1] (one atomicAdd per CTA and row).  When a
//               position's last accumulator is read (its MMAs are then
//               complete) the epilogue gathers E of position k + 2 into the
//               buffer position k used; the loads of position k + 1's lse_d and
//               target-row partials go out first, so that their latency
//               overlaps the row sums' barriers.
//
// lse_d comes from the draft; lse_t from target-row partials already in the
// workspace, so that each U and T row is read once.  Rows of positions past a
// request's verify length stream in with the box and are not used.  Every
// wait is bounded; on a timeout the CTA records DSPARK_ERR_TIMEOUT, drains the
// copies and MMAs it issued, frees its TMEM and returns.
#include <cuda_bf16.h>

#include <algorithm>

#include "kernels.h"
#include "tc_common.cuh"

namespace dspark {
namespace {

using namespace tc;

constexpr int LBM = 128;                 // requests per M tile (TMEM lanes)
constexpr int LBN = 64;                  // vocabulary columns per tile
constexpr int LGroup = 2;                // tiles per MMA: N = 64 x (up to 2)
constexpr int LAccCols = LGroup * LBN;   // 128 TMEM columns per accumulator (and per E buffer)
constexpr int LKR = 256;                 // Markov rank
constexpr int LAtoms = LKR / 64;         // 64-wide K atoms
constexpr int LWStages = 3;              // W2 atom ring
constexpr int LUTStages = 2;             // U + T tile ring
constexpr int LUBox = 32;                // fp32 columns per box (128 bytes, swizzled)
constexpr int LEpiWarps = 16;
constexpr int LThreads = 64 + 32 * LEpiWarps;
constexpr uint32_t LTmemCols = 512;
constexpr uint32_t LTmemE = 2 * LAccCols;          // E of odd positions at LTmemE + 128, of even at LTmemE
constexpr int LWStageBytes = LAccCols * 128;       // 16384
constexpr int LUTStageBytes = 2 * LBN * LBM * 4;   // U then T: 65536
constexpr int LBarBytes = 512;
constexpr int LXBytes = 4 * LBM * 4;               // the parts' sums of a position
constexpr int LSmemBytes = 1024 + LWStages * LWStageBytes + LUTStages * LUTStageBytes + LBarBytes + LXBytes;
static_assert(LSmemBytes <= 232448, "more dynamic shared memory than one CTA may use");

struct __align__(8) LBars {
  uint64_t full_w[LWStages], empty_w[LWStages];
  uint64_t full_ut[LUTStages], empty_ut[LUTStages];
  uint64_t acc_full[2], acc_empty[2];
  uint64_t e_full[2], drain;
  uint32_t tmem_base;
  int abort;
};
static_assert(sizeof(LBars) <= LBarBytes, "barrier block overflows its shared-memory slot");

struct LabelParams {
  const __nv_bfloat16* W1;
  const int32_t* anchor;
  const int32_t* x;          // [B][G] drafted tokens
  const float* lse_d;        // [B][G]
  const int32_t* ell;        // [B]
  const float2* row_part;    // [B*(G+1)][nsegs] target-row partials
  int nsegs;
  int tail_tile;             // tile staged as [R x 32] boxes (V % 32 != 0), else -1
  const int* stats_done;     // row segments a draft took (nullptr: not checked); the word after the
                             // next is 1 when that draft took only the rows the accept chains reach
  const int* full_rows;      // 1 while verification's statistics cover every row j < ell (nullptr: not checked)
  float* label;              // [B][G], zeroed by the caller
  int* status;
  int B, G, V;
  int ctas_per_mtile, ntiles;
};

__device__ __forceinline__ int l_group_tiles(int g) { return g == 0 ? 1 : LGroup; }

__device__ __forceinline__ int l_tile_begin(int slice, int nslices, int ntiles) {
  return (int)(((long long)ntiles * slice) / nslices);
}

// E[m, 64h .. 64h+63] = W1[tok] into this warp's TMEM lanes (zeros for rows
// that take no part).
__device__ __forceinline__ void l_gather_e(const __nv_bfloat16* W1, int tok, bool active, int h, uint32_t taddr) {
  const uint4* wrow = reinterpret_cast<const uint4*>(W1 + (size_t)tok * LKR);
  uint32_t ev[32];
#pragma unroll
  for (int c = 0; c < 8; ++c) {
    const uint4 val = active ? __ldg(wrow + h * 8 + c) : make_uint4(0, 0, 0, 0);
    ev[4 * c] = val.x; ev[4 * c + 1] = val.y; ev[4 * c + 2] = val.z; ev[4 * c + 3] = val.w;
  }
  tmem_store_32cols(taddr, ev);
}

constexpr float kL2e = 1.4426950408889634f;

template <int R>
__global__ void __launch_bounds__(LThreads, 1)
label_tc(const __grid_constant__ CUtensorMap w2_map, const __grid_constant__ CUtensorMap u_map,
         const __grid_constant__ CUtensorMap t_map, const __grid_constant__ CUtensorMap u4_map,
         const __grid_constant__ CUtensorMap t4_map, const LabelParams p) {
  constexpr int kRepl = LBM / R;
  constexpr int kParts = 4 * kRepl;
  constexpr int CPP = LBN / kParts;
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
  unsigned char* W_s = smem;
  unsigned char* UT_s = W_s + LWStages * LWStageBytes;
  LBars* bars = reinterpret_cast<LBars*>(UT_s + LUTStages * LUTStageBytes);
  float* xs = reinterpret_cast<float*>(reinterpret_cast<unsigned char*>(bars) + LBarBytes);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int mtile = blockIdx.x / p.ctas_per_mtile;
  const int slice = blockIdx.x - mtile * p.ctas_per_mtile;
  const int m0 = mtile * R;
  const int rows_valid = min(R, p.B - m0);
  const int t0 = l_tile_begin(slice, p.ctas_per_mtile, p.ntiles);
  const int ntl = l_tile_begin(slice + 1, p.ctas_per_mtile, p.ntiles) - t0;
  volatile int* abort = &bars->abort;

  if (threadIdx.x == 0) {
    for (int s = 0; s < LWStages; ++s) { mbar_init(&bars->full_w[s], 1); mbar_init(&bars->empty_w[s], 1); }
    for (int s = 0; s < LUTStages; ++s) { mbar_init(&bars->full_ut[s], 1); mbar_init(&bars->empty_ut[s], LEpiWarps); }
    for (int s = 0; s < 2; ++s) { mbar_init(&bars->acc_full[s], 1); mbar_init(&bars->acc_empty[s], LEpiWarps); }
    for (int s = 0; s < 2; ++s) mbar_init(&bars->e_full[s], LEpiWarps);
    mbar_init(&bars->drain, 1);
    bars->abort = 0;
    fence_mbar_init();
  }
  if (blockIdx.x == 0 && threadIdx.x == 0 && p.stats_done &&
      (*p.stats_done < p.B * p.G * p.nsegs || p.stats_done[3] != 0))
    record_status(p.status, DSPARK_ERR_INVALID);
  if (blockIdx.x == 0 && threadIdx.x == 0 && p.full_rows && *p.full_rows != 1)
    record_status(p.status, DSPARK_ERR_INVALID);
  if (warp == 0 && lane == 0) {
    prefetch_tensormap(&w2_map);
    prefetch_tensormap(&u_map);
    prefetch_tensormap(&t_map);
    prefetch_tensormap(&u4_map);
    prefetch_tensormap(&t4_map);
  }
  if (warp == 1) tmem_alloc(&bars->tmem_base, LTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem_base;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    const uint64_t pol_w = policy_evict_last(), pol_u = policy_evict_first();
    uint32_t wcount = 0, ucount = 0;
    bool ok = true;
    for (int k = 1; k <= p.G && ok; ++k) {
      for (int g = 0; g < ntl && ok; g += l_group_tiles(g)) {
        const int v0 = (t0 + g) * LBN;
        for (int a = 0; a < LAtoms && ok; ++a, ++wcount) {
          const int s = wcount % LWStages;
          ok = mbar_wait(&bars->empty_w[s], ((wcount / LWStages) & 1) ^ 1, abort, p.status);
          if (ok && lane == 0) {
            mbar_arrive_expect_tx(&bars->full_w[s], LWStageBytes);
            tma_g2s_2d(W_s + s * LWStageBytes, &w2_map, a * 64, v0, &bars->full_w[s], pol_w);
          }
        }
        const int nsub = min(l_group_tiles(g), ntl - g);
        for (int j = 0; j < nsub && ok; ++j, ++ucount) {
          const int su = ucount % LUTStages;
          ok = mbar_wait(&bars->empty_ut[su], ((ucount / LUTStages) & 1) ^ 1, abort, p.status);
          if (ok && lane == 0) {
            // the U and T tiles of position k, R rows x 64 columns each (rows
            // past B and columns past V are zero-filled)
            const int v = v0 + j * LBN;
            unsigned char* dst = UT_s + su * LUTStageBytes;
            mbar_arrive_expect_tx(&bars->full_ut[su], (uint32_t)(4 * LUBox * R * 4));
            if (t0 + g + j != p.tail_tile) {
              tma_g2s_4d(dst, &u4_map, 0, v / LUBox, k - 1, m0, &bars->full_ut[su], pol_u);
              tma_g2s_4d(dst + R * 256, &t4_map, 0, v / LUBox, k - 1, m0, &bars->full_ut[su], pol_u);
            } else {
              tma_g2s_3d(dst, &u_map, v, k - 1, m0, &bars->full_ut[su], pol_u);
              tma_g2s_3d(dst + R * 128, &u_map, v + LUBox, k - 1, m0, &bars->full_ut[su], pol_u);
              tma_g2s_3d(dst + 2 * R * 128, &t_map, v, k - 1, m0, &bars->full_ut[su], pol_u);
              tma_g2s_3d(dst + 3 * R * 128, &t_map, v + LUBox, k - 1, m0, &bars->full_ut[su], pol_u);
            }
          }
        }
      }
    }
    if (lane == 0 && *abort) {
      for (uint32_t c = (wcount > (uint32_t)LWStages ? wcount - LWStages : 0); c < wcount; ++c)
        mbar_drain(&bars->full_w[c % LWStages], (c / LWStages) & 1);
      for (uint32_t c = (ucount > (uint32_t)LUTStages ? ucount - LUTStages : 0); c < ucount; ++c)
        mbar_drain(&bars->full_ut[c % LUTStages], (c / LUTStages) & 1);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      uint32_t wcount = 0, gcount = 0;
      bool ok = true;
      for (int k = 1; k <= p.G && ok; ++k) {
        // E of position k: buffer k & 1, its ((k - 1) / 2)-th gather
        const int eb = k & 1;
        ok = mbar_wait(&bars->e_full[eb], (uint32_t)((k - 1) >> 1) & 1, abort, p.status);
        tc_fence_after();
        for (int g = 0; g < ntl && ok; g += l_group_tiles(g), ++gcount) {
          const int acc = gcount & 1;
          ok = mbar_wait(&bars->acc_empty[acc], ((gcount >> 1) & 1) ^ 1, abort, p.status);
          if (!ok) break;
          tc_fence_after();
          const uint32_t idesc = idesc_bf16_f32(LBM, LBN * min(l_group_tiles(g), ntl - g));
          const uint32_t d_tmem = tmem + acc * LAccCols;
          for (int a = 0; a < LAtoms && ok; ++a, ++wcount) {
            const int s = wcount % LWStages;
            ok = mbar_wait(&bars->full_w[s], (wcount / LWStages) & 1, abort, p.status);
            if (!ok) break;
            tc_fence_after();
            const uint64_t bd0 = sw128_kmajor_desc(smem_u32(W_s + s * LWStageBytes));
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
              umma_bf16_tmem_a(d_tmem, tmem + LTmemE + eb * LAccCols + a * 32 + kk * 8, bd0 + (uint64_t)(kk * 2),
                               idesc, (a | kk) != 0);
            umma_commit(&bars->empty_w[s]);
          }
          if (ok) umma_commit(&bars->acc_full[acc]);
        }
      }
      umma_commit(&bars->drain);
      mbar_drain(&bars->drain, 0);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;
    const int h = (warp - 2) >> 2;
    const int m = q * 32 + lane;
    const int rep = m / R, r = m - rep * R;
    const int part = rep * 4 + h;
    const int b = m0 + r;
    uint32_t it = 0, gcount = 0;
    bool ok = true;
    // positions 1..ellb of this row are labelled
    const int ellb = r < rows_valid ? min(max(p.ell[b], 0), p.G) : 0;
    const uint32_t e_lanes = tmem + ((uint32_t)(q * 32) << 16) + LTmemE + h * 32;
    // E of positions 1 and 2 (buffers 1 and 0)
    for (int k = 1; k <= min(2, p.G); ++k) {
      const bool act = k <= ellb;
      const int prev = act ? checked_token(k == 1 ? p.anchor[b] : p.x[(size_t)b * p.G + k - 2], p.V, p.status) : 0;
      l_gather_e(p.W1, prev, act, h, e_lanes + (uint32_t)((k & 1) * LAccCols));
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars->e_full[k & 1]);
    }
    // lse_d and lse_t of position 1, in base 2
    float ld2 = 0.f, lt2 = 0.f;
    if (1 <= ellb) {
      ld2 = p.lse_d[(size_t)b * p.G] * kL2e;
      float mt = -INFINITY, st = 0.f;
      merge_partials(p.row_part + (size_t)b * (p.G + 1) * p.nsegs, p.nsegs, mt, st);
      lt2 = (mt + logf(st)) * kL2e;
    }
    for (int k = 1; k <= p.G && ok; ++k) {
      const bool active = k <= ellb;
      float lacc = 0.f;
      for (int i = 0; i < ntl; ++i, ++it) {
        const int sub = i == 0 ? 0 : (i - 1) % LGroup;
        const bool last_sub = i == 0 || sub == LGroup - 1 || i == ntl - 1;
        const int acc_i = gcount & 1;
        const int v0 = (t0 + i) * LBN + part * CPP;
        const int nv = min(CPP, p.V - v0);
        // (the warp leaves together: the TMEM loads below are warp-wide)
        if (sub == 0) ok = __all_sync(0xffffffffu, mbar_wait(&bars->acc_full[acc_i], (gcount >> 1) & 1, abort, p.status));
        if (!ok) break;
        tc_fence_after();
        float v[CPP];
        tmem_load_cols<CPP>(tmem + ((uint32_t)(q * 32) << 16) + acc_i * LAccCols + sub * LBN + part * CPP, v);
        if (last_sub) {
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&bars->acc_empty[acc_i]);
          ++gcount;
        }
        const int su = it % LUTStages;
        ok = __all_sync(0xffffffffu, mbar_wait(&bars->full_ut[su], (it / LUTStages) & 1, abort, p.status));
        if (!ok) break;
        if (active && nv > 0) {
          // this thread's columns: half hf = (part * CPP) / 32 of row r, the
          // 128-byte line 2r + hf of a tile box (hf * R + r of the [R x 32]
          // boxes of a tail tile), 16-byte chunks j0.. stored at chunk
          // j ^ (line & 7) (128-byte swizzle); T R * 256 bytes further
          const int hf = (part * CPP) / LUBox;
          const int line = t0 + i == p.tail_tile ? hf * R + r : 2 * r + hf;
          const unsigned char* urow = UT_s + su * LUTStageBytes + line * 128;
          const unsigned char* trow = urow + R * 256;
          const int j0 = ((part * CPP) % LUBox) / 4, sw = line & 7;
          // lanes with bit 2 set take each pair of chunks in swapped order
          // (rows r and r + 4 share a swizzle phase in a tile box: they then
          // hit different banks); the sum does not depend on the order
          constexpr int NB = CPP / 4;
          const int ps = NB >= 2 ? (lane >> 2) & 1 : 0;
#pragma unroll
          for (int c4 = 0; c4 < NB; ++c4) {
            const int cc = c4 ^ ps;
            const int off = ((j0 + cc) ^ sw) << 4;
            const float4 u4 = *reinterpret_cast<const float4*>(urow + off);
            const float4 t4 = *reinterpret_cast<const float4*>(trow + off);
            const float uv[4] = {u4.x, u4.y, u4.z, u4.w}, tv[4] = {t4.x, t4.y, t4.z, t4.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const float ve = (NB >= 2 && ps) ? v[4 * (c4 ^ (NB >= 2 ? 1 : 0)) + e] : v[4 * c4 + e];
              const float pd = ex2_approx(fmaf(ve + uv[e], kL2e, -ld2));
              const float pt = ex2_approx(fmaf(tv[e], kL2e, -lt2));
              if (4 * cc + e < nv) lacc += fminf(pd, pt);
            }
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars->empty_ut[su]);
      }
      // What position k + 1 needs goes out first: its lse_d, the first
      // eight partials of its target row and the token whose W1 row is E of
      // position k + 2; their latency overlaps the row sums below.
      const bool act1 = k + 1 <= ellb, act2 = k + 2 <= ellb;
      float ldn = 0.f;
      float2 pq[8];
      const float2* rpn = p.row_part + ((size_t)b * (p.G + 1) + k) * p.nsegs;
#pragma unroll
      for (int j = 0; j < 8; ++j) pq[j] = make_float2(-INFINITY, 0.f);
      if (act1) {
        ldn = p.lse_d[(size_t)b * p.G + k];
#pragma unroll
        for (int j = 0; j < 8; ++j)
          if (j < p.nsegs) pq[j] = __ldcg(rpn + j);
      }
      const int tok2 = act2 ? p.x[(size_t)b * p.G + k] : 0;
      // the parts of each row, then one atomicAdd per CTA and row
      xs[part * R + r] = lacc;
      named_bar_sync(1, LEpiWarps * 32);
      if (ok && k + 2 <= p.G) {
        // E of position k + 2 into the buffer position k used: every MMA of
        // position k is complete, its last accumulator having been read
        l_gather_e(p.W1, act2 ? checked_token(tok2, p.V, p.status) : 0, act2, h,
                   e_lanes + (uint32_t)((k & 1) * LAccCols));
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars->e_full[k & 1]);
      }
      if (part == 0 && active && ok) {
        float S = 0.f;
#pragma unroll
        for (int j = 0; j < kParts; ++j) S += xs[j * R + r];
        atomicAdd(&p.label[(size_t)b * p.G + k - 1], S);
      }
      named_bar_sync(1, LEpiWarps * 32);
      if (*abort) ok = false;
      // lse_d and lse_t of position k + 1, in base 2
      ld2 = lt2 = 0.f;
      if (act1) {
        ld2 = ldn * kL2e;
        float mt = -INFINITY, st = 0.f;
#pragma unroll
        for (int j = 0; j < 8; ++j) softmax_merge(mt, st, pq[j].x, pq[j].y);
        if (p.nsegs > 8) merge_partials(rpn + 8, p.nsegs - 8, mt, st);
        lt2 = (mt + logf(st)) * kL2e;
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, LTmemCols);
}

}  // namespace

// The acceptance label of every verified position in one persistent launch
// (label zeroed by the caller; row_part holds the target rows' partials, nsegs
// per row; stats_done, when given, is the draft's count of row segments taken,
// and a short count, or the marker three words further of a draft that took
// only the rows the accept chains reach, is reported as DSPARK_ERR_INVALID;
// full_rows, when given, is the marker of verification's pass over every row
// j < ell, and a marker other than 1 is reported the same way).
cudaError_t launch_acceptance_label_tc(const float* T, const float* U, const void* W1, const void* W2,
                                       const int32_t* anchor, const int32_t* x, const float* lse_d,
                                       const int32_t* ell, const float2* row_part, int nsegs,
                                       const int* stats_done, const int* full_rows, float* label, int B, int G,
                                       int V, int* status, cudaStream_t stream) {
  CUtensorMap wmap, umap, tmap, u4map, t4map;
  cudaError_t e = make_w2_tensor_map(W2, V, &wmap, LAccCols);
  if (e != cudaSuccess) return e;
  int dev = 0, sms = 0;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
  if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
  const int R = B <= 32 ? 32 : (B <= 64 ? 64 : LBM);
  if ((e = make_u_tensor_map(U, B, G, V, R, &umap)) != cudaSuccess) return e;
  if ((e = make_u_tensor_map(T, B, G + 1, V, R, &tmap)) != cudaSuccess) return e;
  // whole tiles by the 4-D view (V >= 32); below that every tile is the tail
  u4map = umap;
  t4map = tmap;
  if (V >= 32) {
    if ((e = make_u_tile_map(U, B, G, V, R, &u4map)) != cudaSuccess) return e;
    if ((e = make_u_tile_map(T, B, G + 1, V, R, &t4map)) != cudaSuccess) return e;
  }
  auto kern = R == 32 ? label_tc<32> : (R == 64 ? label_tc<64> : label_tc<LBM>);
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, LSmemBytes);
  if (e != cudaSuccess) return e;
  const int mtiles = div_up(B, R);
  const int ntiles = div_up(V, LBN);
  int per = std::max(1, sms / mtiles);
  per = std::min(per, ntiles);
  LabelParams lp{};
  lp.W1 = static_cast<const __nv_bfloat16*>(W1);
  lp.anchor = anchor;
  lp.x = x;
  lp.lse_d = lse_d;
  lp.ell = ell;
  lp.row_part = row_part;
  lp.nsegs = nsegs;
  lp.tail_tile = V % 32 != 0 ? ntiles - 1 : -1;
  lp.stats_done = stats_done;
  lp.full_rows = full_rows;
  lp.label = label;
  lp.status = status;
  lp.B = B; lp.G = G; lp.V = V;
  lp.ctas_per_mtile = per;
  lp.ntiles = ntiles;
  kern<<<mtiles * per, LThreads, LSmemBytes, stream>>>(wmap, umap, tmap, u4map, t4map, lp);
  return cudaGetLastError();
}

}  // namespace dspark
