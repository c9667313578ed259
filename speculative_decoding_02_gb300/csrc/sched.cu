// Confidence head (study report Eq.7) and the hardware-aware prefix scheduler
// ("[DeepSeek-6] DSpark" blog, sections 6-7; study report Theta = tau * SPS(B)).
#include "kernels.h"

namespace dspark {
namespace {

// c_k = sigmoid((w[:H] . h_k + w[H:] . W1[x_{k-1}]) / T_k), one warp per (b, k).
constexpr int kConfThreads = 256;
constexpr int kConfBatch = 10;   // 16-byte words of h per lane in flight (H = 2560 bf16: one batch)

// 8 elements of bf16 or f32 storage from 16-byte words (one word of bf16, two of f32).
template <int DT>
__device__ __forceinline__ void unpack8(const uint4* q, float (&v)[8]) {
  if constexpr (DT == DSPARK_BF16) {
    const uint32_t u[4] = {q[0].x, q[0].y, q[0].z, q[0].w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      v[2 * e] = __uint_as_float(u[e] << 16);
      v[2 * e + 1] = __uint_as_float(u[e] & 0xFFFF0000u);
    }
  } else {
    v[0] = __uint_as_float(q[0].x); v[1] = __uint_as_float(q[0].y);
    v[2] = __uint_as_float(q[0].z); v[3] = __uint_as_float(q[0].w);
    v[4] = __uint_as_float(q[1].x); v[5] = __uint_as_float(q[1].y);
    v[6] = __uint_as_float(q[1].z); v[7] = __uint_as_float(q[1].w);
  }
}

__device__ __forceinline__ float dot8_smem(const float* ws, const float (&v)[8], float z) {
  const float4 w0 = *reinterpret_cast<const float4*>(ws);
  const float4 w1 = *reinterpret_cast<const float4*>(ws + 4);
  z = fmaf(w0.x, v[0], z); z = fmaf(w0.y, v[1], z); z = fmaf(w0.z, v[2], z); z = fmaf(w0.w, v[3], z);
  z = fmaf(w1.x, v[4], z); z = fmaf(w1.y, v[5], z); z = fmaf(w1.z, v[6], z); z = fmaf(w1.w, v[7], z);
  return z;
}

// vec: 16-byte aligned h, W1 and w with H and r multiples of 8.  Then w is
// staged in shared memory once per CTA and every 16-byte word of a batch of
// the h row (and the W1 row) is loaded before any arithmetic, so that a warp
// waits for one memory round trip per batch instead of one per step.
template <int HDT, int WDT>
__global__ void __launch_bounds__(kConfThreads)
confidence_kernel(const void* __restrict__ h, const void* __restrict__ W1, const float* __restrict__ w,
                  const float* __restrict__ sts_T, const int32_t* __restrict__ anchor,
                  const int32_t* __restrict__ x, int B, int G, int H, int r, int V, bool vec,
                  float* __restrict__ c_out, int* __restrict__ status) {
  extern __shared__ __align__(16) float w_s[];   // vec: w [H + r]
  if (vec) {
    // 16-byte loads, several in flight per thread
    const int n4 = (H + r) / 4;
#pragma unroll 4
    for (int i = threadIdx.x; i < n4; i += kConfThreads)
      reinterpret_cast<float4*>(w_s)[i] = __ldg(reinterpret_cast<const float4*>(w) + i);
    __syncthreads();
  }
  const int item = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (item >= B * G) return;
  const int b = item / G, k = item - (item / G) * G + 1;
  const int prev = (k == 1) ? anchor[b] : x[(size_t)b * G + k - 2];
  if (prev < 0 || prev >= V) {
    if (lane == 0) {
      if (status) record_status(status, DSPARK_ERR_INVALID);
      c_out[item] = 0.f;
    }
    return;
  }
  float z = 0.f;
  if (vec) {
    constexpr int kHW = HDT == DSPARK_BF16 ? 1 : 2;   // 16-byte words per 8 elements of h
    constexpr int kEW = WDT == DSPARK_BF16 ? 1 : 2;   // ... of W1
    const uint4* hrow = reinterpret_cast<const uint4*>(static_cast<const char*>(h) +
                                                       (size_t)item * H * (HDT == DSPARK_BF16 ? 2 : 4));
    const uint4* erow = reinterpret_cast<const uint4*>(static_cast<const char*>(W1) +
                                                       (size_t)prev * r * (WDT == DSPARK_BF16 ? 2 : 4));
    const int nh = H / 8, ne = r / 8;   // 8-element steps of h and of the W1 row
    float z1 = 0.f;
    // the W1 row (one step per lane for r <= 256) is in flight with the first batch of h
    uint4 e[kEW];
    const bool has_e = lane < ne;
#pragma unroll
    for (int t = 0; t < kEW; ++t) e[t] = has_e ? __ldg(erow + (size_t)lane * kEW + t) : make_uint4(0, 0, 0, 0);
    for (int c0 = 0; c0 < nh; c0 += 32 * kConfBatch) {
      uint4 q[kConfBatch * kHW];
#pragma unroll
      for (int u = 0; u < kConfBatch; ++u) {
        const int ch = c0 + 32 * u + lane;
#pragma unroll
        for (int t = 0; t < kHW; ++t) q[u * kHW + t] = ch < nh ? __ldg(hrow + (size_t)ch * kHW + t) : make_uint4(0, 0, 0, 0);
      }
#pragma unroll
      for (int u = 0; u < kConfBatch; ++u) {
        const int ch = c0 + 32 * u + lane;
        if (ch < nh) {
          float v[8];
          unpack8<HDT>(q + u * kHW, v);
          if (u & 1) z1 = dot8_smem(w_s + 8 * ch, v, z1);
          else z = dot8_smem(w_s + 8 * ch, v, z);
        }
      }
    }
    if (has_e) {
      float v[8];
      unpack8<WDT>(e, v);
      z1 = dot8_smem(w_s + H + 8 * lane, v, z1);
    }
    // rank above 256: the remaining W1 steps
    for (int j = 32 + lane; j < ne; j += 32) {
      uint4 e[kEW];
#pragma unroll
      for (int t = 0; t < kEW; ++t) e[t] = __ldg(erow + (size_t)j * kEW + t);
      float v[8];
      unpack8<WDT>(e, v);
      z1 = dot8_smem(w_s + H + 8 * j, v, z1);
    }
    z += z1;
  } else {
    const size_t hrow = (size_t)item * H;
    for (int i = lane; i < H; i += 32) z = fmaf(w[i], load_weight<HDT>(h, hrow + i), z);
    for (int i = lane; i < r; i += 32) z = fmaf(w[H + i], load_weight<WDT>(W1, (size_t)prev * r + i), z);
  }
  for (int off = 16; off > 0; off >>= 1) z += __shfl_xor_sync(0xffffffffu, z, off);
  if (lane == 0) {
    const float T = sts_T ? sts_T[k - 1] : 1.f;
    c_out[item] = 1.f / (1.f + expf(-z / T));
  }
}

constexpr int kSchedThreads = 1024;

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

// One CTA.  a_{b,j} = prod_{i<=j} c_{b,i} in float-float.  When SPS strictly
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
__global__ void __launch_bounds__(kSchedThreads)
schedule_kernel(const float* __restrict__ c, int R, int G, const float* __restrict__ sps, int mode,
                unsigned long long round_host, const unsigned long long* __restrict__ round_dev,
                int32_t* __restrict__ khist, int32_t* __restrict__ ell_out, int32_t* __restrict__ nstar_out,
                double* __restrict__ theta_out, int* __restrict__ status) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  const int N = R * G;
  int NP = 1;
  while (NP < N) NP <<= 1;
  unsigned long long* key = reinterpret_cast<unsigned long long*>(smem_raw);   // [NP] sort keys
  ff* av = reinterpret_cast<ff*>(key + NP);                                      // [NP] a by index, then S_n
  int* ell_s = reinterpret_cast<int*>(av + NP);                                  // [R]
  __shared__ ff warp_tot[32];
  __shared__ int s_first_stop;
  __shared__ int s_K;
  const int tid = threadIdx.x;

  if (mode == DSPARK_SCHED_FIXED) {
    for (int b = tid; b < R; b += kSchedThreads) ell_out[b] = G;
    if (tid == 0) {
      *nstar_out = N;
      *theta_out = 0.0;
    }
    return;
  }
  const unsigned long long round = round_dev ? __ldcg(round_dev) : round_host;

  for (int i = N + tid; i < NP; i += kSchedThreads) key[i] = 0ull;   // padding sorts last
  if (tid == 0) {
    s_first_stop = N + 1;
    s_K = -1;
    if (mode == DSPARK_SCHED_TOPK && round >= 2) s_K = khist[(uint32_t)round & 1u];
  }
  // Survival products, one request per thread: its gamma confidences are all
  // loaded before the product chain starts.  `tot` is this thread's sum of a.
  ff tot{0.f, 0.f};
  for (int b = tid; b < R; b += kSchedThreads) {
    float cj[kMaxGamma];
#pragma unroll
    for (int j = 0; j < kMaxGamma; ++j) cj[j] = j < G ? c[(size_t)b * G + j] : 1.f;
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
  for (int n = tid + 1; n <= N; n += kSchedThreads) inc = inc && (sps[R + n] > sps[R + n - 1]);
  const bool all_inc = __syncthreads_and(inc) != 0;   // also publishes av, key and s_K
  const int lane = tid & 31, wid = tid >> 5;
  if (all_inc && (mode == DSPARK_SCHED_GREEDY || s_K < 0 || s_K >= N)) {
    for (int off = 16; off > 0; off >>= 1)
      tot = ff_add(tot, {__shfl_xor_sync(0xffffffffu, tot.hi, off), __shfl_xor_sync(0xffffffffu, tot.lo, off)});
    if (lane == 0) warp_tot[wid] = tot;
    __syncthreads();
    for (int b = tid; b < R; b += kSchedThreads) ell_out[b] = G;
    if (tid == 0) {
      ff S{0.f, 0.f};
      for (int w = 0; w < kSchedThreads / 32; ++w) S = ff_add(S, warp_tot[w]);
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
    for (int t = tid; t < NP / 2; t += kSchedThreads) {
      const int blk = t >> (lk - 1), off = t & ((k >> 1) - 1);
      const int i = (blk << lk) + off, m = (blk << lk) + k - 1 - off;
      const unsigned long long x = key[i], y = key[m];
      if (x < y) { key[i] = y; key[m] = x; }
    }
    __syncthreads();
    for (int j = k / 4; j > 0; j >>= 1) {
      for (int t = tid; t < NP / 2; t += kSchedThreads) {
        const int i = 2 * t - (t & (j - 1)), l = i + j;
        const unsigned long long x = key[i], y = key[l];
        if (x < y) { key[i] = y; key[l] = x; }
      }
      __syncthreads();
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
  __syncthreads();   // every gather from av is done: av now takes S_n
  if (wid == 0) {
    ff wt = lane < nwarps ? warp_tot[lane] : ff{0.f, 0.f};
    for (int off = 1; off < 32; off <<= 1) {
      const ff o = ff_shfl_up(wt, off);
      if (lane >= off) wt = ff_add(wt, o);
    }
    warp_tot[lane] = wt;
  }
  __syncthreads();
  if (tid < nthr) {
    ff base = ff_add(incl, ff_neg(run_s));   // exclusive prefix inside the warp
    if (wid > 0) base = ff_add(base, warp_tot[wid - 1]);
    const int lo = tid * chunk;
#pragma unroll
    for (int q = 0; q < 8; ++q)
      if (q < chunk && lo + q < N) av[lo + q] = ff_add(loc[q], base);
  }
  __syncthreads();

  // Theta_n for n = 1..N against Theta_{n-1}; the first n whose Theta does not
  // rise stops the greedy
  const ff Rf{(float)R, 0.f};
  for (int n = tid + 1; n <= N; n += kSchedThreads) {
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
    if (stop) atomicMin(&s_first_stop, n);
  }
  __syncthreads();
  const int nstar = (s_first_stop <= N) ? s_first_stop - 1 : N;
  int admitted = nstar;
  if (mode == DSPARK_SCHED_TOPK && round >= 2) admitted = min(max(s_K, 0), N);
  for (int p = tid; p < admitted; p += kSchedThreads)
    atomicAdd(&ell_s[(8191 - (int)(key[p] & 0x1FFFull)) / G], 1);
  __syncthreads();
  for (int b = tid; b < R; b += kSchedThreads) ell_out[b] = ell_s[b];
  if (tid == 0) {
    *nstar_out = nstar;
    const ff x = admitted > 0 ? ff_add(Rf, av[admitted - 1]) : Rf;
    *theta_out = ((double)x.hi + (double)x.lo) * (double)sps[R + admitted];
    if (mode == DSPARK_SCHED_TOPK) khist[(uint32_t)round & 1u] = nstar;
  }
}

}  // namespace

cudaError_t launch_confidence(const void* h, int hdtype, const void* W1, int wdtype, const float* w,
                              const float* sts_T, const int32_t* anchor, const int32_t* x, int B,
                              int gamma, int H, int r, int V, float* c_out, int* status,
                              cudaStream_t stream) {
  const int items = B * gamma;
  const dim3 grid(div_up(items * 32, kConfThreads));
  // the staged weight must fit in shared memory (H + r up to 24576)
  const bool vec = (H % 8 == 0) && (r % 8 == 0) && (((uintptr_t)h | (uintptr_t)W1 | (uintptr_t)w) % 16 == 0) &&
                   (long long)H + r <= 24576;
  const size_t smem = vec ? sizeof(float) * (size_t)(H + r) : 0;
  cudaError_t e = cudaSuccess;
#define DSPARK_CONF(HD, WD)                                                                                   \
  do {                                                                                                        \
    if (smem > 48 * 1024)                                                                                     \
      e = cudaFuncSetAttribute(confidence_kernel<HD, WD>, cudaFuncAttributeMaxDynamicSharedMemorySize,        \
                               (int)smem);                                                                    \
    if (e == cudaSuccess)                                                                                     \
      confidence_kernel<HD, WD><<<grid, kConfThreads, smem, stream>>>(h, W1, w, sts_T, anchor, x, B, gamma, H, \
                                                                      r, V, vec, c_out, status);              \
  } while (0)
  if (hdtype == DSPARK_BF16 && wdtype == DSPARK_BF16) DSPARK_CONF(DSPARK_BF16, DSPARK_BF16);
  else if (hdtype == DSPARK_BF16) DSPARK_CONF(DSPARK_BF16, DSPARK_F32);
  else if (wdtype == DSPARK_BF16) DSPARK_CONF(DSPARK_F32, DSPARK_BF16);
  else DSPARK_CONF(DSPARK_F32, DSPARK_F32);
#undef DSPARK_CONF
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

size_t schedule_smem_bytes(int B, int gamma) {
  int NP = 1;
  while (NP < B * gamma) NP <<= 1;
  // keys and float-float values [NP] each, counts [B]
  return (size_t)NP * (sizeof(unsigned long long) + 2 * sizeof(float)) + sizeof(int) * (size_t)B;
}

cudaError_t launch_schedule(const float* c, int B, int gamma, const float* sps, int mode,
                            unsigned long long round, const unsigned long long* round_dev, int32_t* khist,
                            int32_t* ell_out, int32_t* nstar_out, double* theta_out, int* status,
                            cudaStream_t stream) {
  const size_t smem = mode == DSPARK_SCHED_FIXED ? 0 : schedule_smem_bytes(B, gamma);
  cudaError_t e = cudaFuncSetAttribute(schedule_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  schedule_kernel<<<1, kSchedThreads, smem, stream>>>(c, B, gamma, sps, mode, round, round_dev, khist, ell_out,
                                                       nstar_out, theta_out, status);
  return cudaGetLastError();
}

}  // namespace dspark
