// The hardware-aware prefix scheduler of one round ("[DeepSeek-6] DSpark"
// blog, sections 6-7; study report Theta = tau * SPS(B)) as a block-wide
// device function: the schedule kernel runs it with 1024 threads, the
// tensor-core draft's last CTA with its 512 epilogue threads (same results:
// every reduction has the same shape for up to 4096 candidates).
#pragma once

#include "common.cuh"

namespace dspark {

// ---------------------------------------------------------------------------
// Float-float arithmetic: a value is hi + lo with |lo| <= ulp(hi) / 2, about
// 48 significant bits, on the fp32 pipes (GB300's fp64 units are few and
// their dependent chains long).  Error-free product by fma and sums by the
// classic two-sum (Dekker; Knuth TAOCP vol. 2, 4.2.2); the rn intrinsics keep
// the compiler from contracting the error terms.
// ---------------------------------------------------------------------------
struct ff {
  float hi, lo;
};

__device__ __forceinline__ ff ff_norm(float s, float e) {
  const float r = __fadd_rn(s, e);
  return {r, __fsub_rn(e, __fsub_rn(r, s))};
}

// a * b for a float b
__device__ __forceinline__ ff ff_mul(ff a, float b) {
  const float p = __fmul_rn(a.hi, b);
  float e = fmaf(a.hi, b, -p);
  e = fmaf(a.lo, b, e);
  return ff_norm(p, e);
}

__device__ __forceinline__ ff ff_add(ff a, ff b) {
  const float s = __fadd_rn(a.hi, b.hi);
  const float bb = __fsub_rn(s, a.hi);
  float e = __fadd_rn(__fsub_rn(a.hi, __fsub_rn(s, bb)), __fsub_rn(b.hi, bb));
  e = __fadd_rn(e, __fadd_rn(a.lo, b.lo));
  return ff_norm(s, e);
}

__device__ __forceinline__ ff ff_neg(ff a) { return {-a.hi, -a.lo}; }

__device__ __forceinline__ ff ff_shfl_up(ff a, int off) {
  return {__shfl_up_sync(0xffffffffu, a.hi, off), __shfl_up_sync(0xffffffffu, a.lo, off)};
}

// The sort key of a survival product a in [0, 1] (hi, lo) at candidate index
// i: a's float bits, then lo in units of 2^-20 ulp(hi) (20 bits), then
// 8191 - i, so that a descending integer order is a desc, then index asc.
// Values closer than 2^-43 relative compare as ties and fall back to the index.
__device__ __forceinline__ unsigned long long ff_key(ff a, int i) {
  const uint32_t hb = __float_as_uint(a.hi) & 0x7fffffffu;
  const int e = (int)(hb >> 23);
  uint32_t q = 1u << 19;
  if (e >= 43) {
    const float scale = __uint_as_float((uint32_t)(170 - e + 127) << 23);   // 2^(20 - exponent of ulp(hi))
    const int d = (int)floorf(__fmul_rn(a.lo, scale));
    q = (uint32_t)min(max(d + (1 << 19), 0), (1 << 20) - 1);
  }
  return ((unsigned long long)hb << 33) | ((unsigned long long)q << 13) | (unsigned long long)(8191 - i);
}


// Block-wide scratch of schedule_block besides its dynamic region.
struct SchedShared {
  ff warp_tot[32];
  int first_stop;
  int K;
};

// Barriers of schedule_block for a whole CTA.
struct CtaSync {
  __device__ void operator()() const { __syncthreads(); }
  __device__ bool all(bool p) const { return __syncthreads_and(p) != 0; }
};

// Barriers over the first NT threads of warps 2.. of a CTA (named barrier 1).
template <int NT>
struct NamedSync {
  __device__ void operator()() const { asm volatile("bar.sync 1, %0;" ::"n"(NT) : "memory"); }
  __device__ bool all(bool p) const {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred pi, po;\n\tsetp.ne.u32 pi, %1, 0;\n\tbar.red.and.pred po, 1, %2, pi;\n\t"
        "selp.u32 %0, 1, 0, po;\n\t}"
        : "=r"(r)
        : "r"((uint32_t)p), "n"(NT)
        : "memory");
    return r != 0;
  }
};

// Bytes of smem schedule_block takes: keys and float-float values [NP] each,
// counts [R].
__host__ __device__ inline size_t schedule_smem_bytes(int B, int gamma) {
  int NP = 1;
  while (NP < B * gamma) NP <<= 1;
  return (size_t)NP * (sizeof(unsigned long long) + 2 * sizeof(float)) + sizeof(int) * (size_t)B;
}

// NT threads (tid = 0..NT-1; nt <= NT * 8 candidates for the scan below).
// a_{b,j} = prod_{i<=j} c_{b,i} in float-float.  When SPS strictly
// increases over the batch sizes the greedy can reach, it admits everything
// (see the shortcut below) and nothing is sorted.  Otherwise the candidates are
// sorted by 64-bit keys (ff_key: a desc, then b asc, j asc) with a bitonic
// network that starts from the per-request runs, which are already in
// descending order when gamma is a power of two (c <= 1 makes a
// non-increasing in j); each merge level compares every element with its
// mirror in the partner run, then halves.  The sorted a get an inclusive
// float-float scan S_n; Theta_n = (R + S_n) * SPS(R + n) and the greedy
// count n* is one less than the first n whose Theta does not exceed
// Theta_{n-1}.  That comparison is screened in float32 (a difference far from
// zero decides it) and evaluated in float-float where the float32 difference
// lies within 1e-5 of its terms.
template <int NT, typename Sync>
__device__ __forceinline__ void schedule_block(const float* __restrict__ c, int R, int G, const float* __restrict__ sps,
                                               int mode, unsigned long long round, int32_t* __restrict__ khist,
                                               int32_t* __restrict__ ell_out, int32_t* __restrict__ nstar_out,
                                               double* __restrict__ theta_out, int* __restrict__ status,
                                               unsigned char* smem, SchedShared& sh, int tid, Sync sync) {
  const int N = R * G;
  int NP = 1;
  while (NP < N) NP <<= 1;
  unsigned long long* key = reinterpret_cast<unsigned long long*>(smem);       // [NP] sort keys
  ff* av = reinterpret_cast<ff*>(key + NP);                                      // [NP] a by index, then S_n
  int* ell_s = reinterpret_cast<int*>(av + NP);                                  // [R]
  ff* warp_tot = sh.warp_tot;

  if (mode == DSPARK_SCHED_FIXED) {
    for (int b = tid; b < R; b += NT) ell_out[b] = G;
    if (tid == 0) {
      *nstar_out = N;
      *theta_out = 0.0;
    }
    return;
  }
  for (int i = N + tid; i < NP; i += NT) key[i] = 0ull;   // padding sorts last
  if (tid == 0) {
    sh.first_stop = N + 1;
    sh.K = -1;
    if (mode == DSPARK_SCHED_TOPK && round >= 2) sh.K = khist[(uint32_t)round & 1u];
  }
  // Survival products, one request per thread: its gamma confidences are all
  // loaded before the product chain starts.  `tot` is this thread's sum of a.
  ff tot{0.f, 0.f};
  for (int b = tid; b < R; b += NT) {
    float cj[kMaxGamma];
#pragma unroll
    for (int j = 0; j < kMaxGamma; ++j) cj[j] = j < G ? __ldcg(c + (size_t)b * G + j) : 1.f;
    ff a{1.f, 0.f};
    bool bad = false;
#pragma unroll
    for (int j = 0; j < kMaxGamma; ++j) {
      if (j < G) {
        const int i = b * G + j;
        bad |= !(cj[j] >= 0.f && cj[j] <= 1.f);
        a = ff_mul(a, cj[j]);
        av[i] = a;
        key[i] = ff_key(a, i);
        tot = ff_add(tot, a);
      }
    }
    if (bad) record_status(status, DSPARK_ERR_NONFINITE);
    ell_s[b] = 0;
  }
  // Exact shortcut: when SPS strictly increases over batch sizes R .. R + N,
  // every admitted candidate raises Theta (a >= 0 and R + S > 0), so the greedy
  // admits all N candidates whatever their order; top-K admits them all too
  // when K >= N.  Only Theta* = (R + sum a) * SPS(R + N) is left to compute.
  bool inc = true;
  for (int n = tid + 1; n <= N; n += NT) inc = inc && (sps[R + n] > sps[R + n - 1]);
  const bool all_inc = sync.all(inc);   // also publishes av, key and sh.K
  const int lane = tid & 31, wid = tid >> 5;
  if (all_inc && (mode == DSPARK_SCHED_GREEDY || sh.K < 0 || sh.K >= N)) {
    for (int off = 16; off > 0; off >>= 1)
      tot = ff_add(tot, {__shfl_xor_sync(0xffffffffu, tot.hi, off), __shfl_xor_sync(0xffffffffu, tot.lo, off)});
    if (lane == 0) warp_tot[wid] = tot;
    sync();
    for (int b = tid; b < R; b += NT) ell_out[b] = G;
    if (tid == 0) {
      ff S{0.f, 0.f};
      for (int w = 0; w < NT / 32; ++w) S = ff_add(S, warp_tot[w]);
      const ff x = ff_add({(float)R, 0.f}, S);
      *nstar_out = N;
      *theta_out = ((double)x.hi + (double)x.lo) * (double)sps[R + N];
      if (mode == DSPARK_SCHED_TOPK) khist[(uint32_t)round & 1u] = N;
    }
    return;
  }

  // bitonic merges of sorted runs (descending) from the run length up to NP
  int run = 1;
  if ((G & (G - 1)) == 0) run = G;   // the per-request runs are sorted already
  int lk = 1;
  while ((1 << lk) < 2 * run) ++lk;
  for (int k = 2 * run; k <= NP; k <<= 1, ++lk) {
    // mirror step: element i of a block's first half against element k-1-i
    for (int t = tid; t < NP / 2; t += NT) {
      const int blk = t >> (lk - 1), off = t & ((k >> 1) - 1);
      const int i = (blk << lk) + off, m = (blk << lk) + k - 1 - off;
      const unsigned long long x = key[i], y = key[m];
      if (x < y) { key[i] = y; key[m] = x; }
    }
    sync();
    for (int j = k / 4; j > 0; j >>= 1) {
      for (int t = tid; t < NP / 2; t += NT) {
        const int i = 2 * t - (t & (j - 1)), l = i + j;
        const unsigned long long x = key[i], y = key[l];
        if (x < y) { key[i] = y; key[l] = x; }
      }
      sync();
    }
  }

  // Inclusive float-float scan of the sorted a values: each thread gathers a
  // chunk of up to 8 consecutive sorted values (from av, indexed by
  // candidate) into registers, then a scan of the chunk totals; afterwards
  // av[p] = S_{p+1}.
  const int chunk = max(1, min(8, div_up(N, 256)));
  const int nthr = div_up(N, chunk);
  const int nwarps = div_up(nthr, 32);
  ff loc[8];
  ff run_s{0.f, 0.f};
  if (tid < nthr) {
    const int lo = tid * chunk;
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      if (q < chunk && lo + q < N) {
        run_s = ff_add(run_s, av[8191 - (int)(key[lo + q] & 0x1FFFull)]);
        loc[q] = run_s;
      }
    }
  }
  ff incl = run_s;
  if (wid < nwarps) {
    for (int off = 1; off < 32; off <<= 1) {
      const ff o = ff_shfl_up(incl, off);
      if (lane >= off) incl = ff_add(incl, o);
    }
    if (lane == 31) warp_tot[wid] = incl;
  }
  sync();   // every gather from av is done: av now takes S_n
  if (wid == 0) {
    ff wt = lane < nwarps ? warp_tot[lane] : ff{0.f, 0.f};
    for (int off = 1; off < 32; off <<= 1) {
      const ff o = ff_shfl_up(wt, off);
      if (lane >= off) wt = ff_add(wt, o);
    }
    warp_tot[lane] = wt;
  }
  sync();
  if (tid < nthr) {
    ff base = ff_add(incl, ff_neg(run_s));   // exclusive prefix inside the warp
    if (wid > 0) base = ff_add(base, warp_tot[wid - 1]);
    const int lo = tid * chunk;
#pragma unroll
    for (int q = 0; q < 8; ++q)
      if (q < chunk && lo + q < N) av[lo + q] = ff_add(loc[q], base);
  }
  sync();

  // Theta_n for n = 1..N against Theta_{n-1}; the first n whose Theta does not
  // rise stops the greedy
  const ff Rf{(float)R, 0.f};
  for (int n = tid + 1; n <= N; n += NT) {
    const float pn = sps[R + n], pp = sps[R + n - 1];
    const ff xn = ff_add(Rf, av[n - 1]);
    const ff xp = n >= 2 ? ff_add(Rf, av[n - 2]) : Rf;
    const float tn = xn.hi * pn, tp = xp.hi * pp;
    const float d = tn - tp;
    bool stop;
    if (fabsf(d) > 1e-5f * (fabsf(tn) + fabsf(tp))) {
      stop = d < 0.f;
    } else {
      const ff dd = ff_add(ff_mul(xn, pn), ff_neg(ff_mul(xp, pp)));
      stop = dd.hi < 0.f || (dd.hi == 0.f && dd.lo <= 0.f);
    }
    if (stop) atomicMin(&sh.first_stop, n);
  }
  sync();
  const int nstar = (sh.first_stop <= N) ? sh.first_stop - 1 : N;
  int admitted = nstar;
  if (mode == DSPARK_SCHED_TOPK && round >= 2) admitted = min(max(sh.K, 0), N);
  for (int p = tid; p < admitted; p += NT)
    atomicAdd(&ell_s[(8191 - (int)(key[p] & 0x1FFFull)) / G], 1);
  sync();
  for (int b = tid; b < R; b += NT) ell_out[b] = ell_s[b];
  if (tid == 0) {
    *nstar_out = nstar;
    const ff x = admitted > 0 ? ff_add(Rf, av[admitted - 1]) : Rf;
    *theta_out = ((double)x.hi + (double)x.lo) * (double)sps[R + admitted];
    if (mode == DSPARK_SCHED_TOPK) khist[(uint32_t)round & 1u] = nstar;
  }
}

}  // namespace dspark
