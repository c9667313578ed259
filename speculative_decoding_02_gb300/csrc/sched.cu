// Confidence head (study report Eq.7) and the hardware-aware prefix scheduler
// ("[DeepSeek-6] DSpark" blog, sections 6-7; study report Theta = tau * SPS(B)).
#include "kernels.h"

namespace dspark {
namespace {

// c_k = sigmoid((w[:H] . h_k + w[H:] . W1[x_{k-1}]) / T_k), one warp per (b, k).
// z + sum_{e < 8} wv[e] * x[i + e] for 8 consecutive elements of x (bf16 or f32
// storage, element offset i a multiple of 8 from a 16-byte aligned base).
template <int DT>
__device__ __forceinline__ float dot8(const void* x, size_t i, const float* __restrict__ wv, float z) {
  const float4 w0 = *reinterpret_cast<const float4*>(wv);
  const float4 w1 = *reinterpret_cast<const float4*>(wv + 4);
  float v[8];
  if constexpr (DT == DSPARK_BF16) {
    const uint4 q = *reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(x) + i);
    const uint32_t u[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      v[2 * e] = __uint_as_float(u[e] << 16);
      v[2 * e + 1] = __uint_as_float(u[e] & 0xFFFF0000u);
    }
  } else {
    const float4 a = *reinterpret_cast<const float4*>(static_cast<const float*>(x) + i);
    const float4 c = *reinterpret_cast<const float4*>(static_cast<const float*>(x) + i + 4);
    v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w; v[4] = c.x; v[5] = c.y; v[6] = c.z; v[7] = c.w;
  }
  z = fmaf(w0.x, v[0], z); z = fmaf(w0.y, v[1], z); z = fmaf(w0.z, v[2], z); z = fmaf(w0.w, v[3], z);
  z = fmaf(w1.x, v[4], z); z = fmaf(w1.y, v[5], z); z = fmaf(w1.z, v[6], z); z = fmaf(w1.w, v[7], z);
  return z;
}

template <int HDT, int WDT>
__global__ void confidence_kernel(const void* __restrict__ h, const void* __restrict__ W1,
                                  const float* __restrict__ w, const float* __restrict__ sts_T,
                                  const int32_t* __restrict__ anchor, const int32_t* __restrict__ x,
                                  int B, int G, int H, int r, int V, bool vec, float* __restrict__ c_out,
                                  int* __restrict__ status) {
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
  const size_t hrow = (size_t)item * H;
  float z = 0.f;
  if (vec) {
    // 8 elements per lane per step: 16-byte loads of bf16 (two 16-byte loads
    // of f32), the weight as two float4 (16-byte aligned bases, H and r
    // multiples of 8 keep every row aligned)
    // four independent partial sums, so that four loads per lane are in
    // flight at once
    float z1 = 0.f, z2 = 0.f, z3 = 0.f;
    int i = 8 * lane;
    for (; i + 768 < H; i += 1024) {
      z = dot8<HDT>(h, hrow + i, w + i, z);
      z1 = dot8<HDT>(h, hrow + i + 256, w + i + 256, z1);
      z2 = dot8<HDT>(h, hrow + i + 512, w + i + 512, z2);
      z3 = dot8<HDT>(h, hrow + i + 768, w + i + 768, z3);
    }
    for (; i < H; i += 256) z = dot8<HDT>(h, hrow + i, w + i, z);
    for (int j = 8 * lane; j < r; j += 256) z1 = dot8<WDT>(W1, (size_t)prev * r + j, w + H + j, z1);
    z = (z + z1) + (z2 + z3);
  } else {
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

// One CTA.  a = prefix products in fp64.  The candidates are sorted as 64-bit
// integers: the bits of a (non-negative, so ordered like the values) with the
// low 13 bits replaced by 8191 - index, index = b*gamma + j-1; a descending
// integer sort (merges of the per-request runs) then gives a desc, b asc,
// j asc (values closer than 2^-39 relative count as ties and fall back to the
// index order).  The exact a
// values stay aside for an inclusive fp64 scan of the sorted list;
// Theta_n = (R + S_n) * SPS(R + n), and the greedy count n* is one less than
// the first n whose Theta does not exceed Theta_{n-1}.
__global__ void __launch_bounds__(kSchedThreads)
schedule_kernel(const float* __restrict__ c, int R, int G, const float* __restrict__ sps, int mode,
                uint32_t round_lo, int round_ge2, int32_t* __restrict__ khist,
                int32_t* __restrict__ ell_out, int32_t* __restrict__ nstar_out,
                double* __restrict__ theta_out, int* __restrict__ status) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  const int N = R * G;
  int NP = 1;
  while (NP < N) NP <<= 1;
  unsigned long long* key = reinterpret_cast<unsigned long long*>(smem_raw);   // [NP]: sort buffer A
  unsigned long long* key2 = key + NP;                                           // [NP]: sort buffer B
  double* av = reinterpret_cast<double*>(key2 + NP);                             // [N]
  int* ell_s = reinterpret_cast<int*>(av + N);                                   // [R]
  __shared__ double warp_tot[32];
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

  for (int b = tid; b < R; b += kSchedThreads) {
    double a = 1.0;
    bool bad = false;
    for (int j = 0; j < G; ++j) {
      const float cj = c[(size_t)b * G + j];
      bad |= !(cj >= 0.f && cj <= 1.f);
      a *= (double)cj;
      const int i = b * G + j;
      av[i] = a;
      key[i] = ((unsigned long long)__double_as_longlong(a) & ~0x1FFFull) | (unsigned long long)(8191 - i);
    }
    if (bad) record_status(status, DSPARK_ERR_NONFINITE);
    ell_s[b] = 0;
  }
  if (tid == 0) {
    s_first_stop = N + 1;
    s_K = -1;
    if (mode == DSPARK_SCHED_TOPK && round_ge2) s_K = khist[round_lo & 1u];
  }
  __syncthreads();

  // Sort the keys descending by merging.  Each request's G keys are already in
  // descending order (c <= 1 makes a non-increasing in j, and equal a break
  // by the smaller j), so ceil(log2 R) rounds of pairwise merges of adjacent
  // runs finish the sort.  In a round every key finds its place on its own:
  // its index in its run plus the number of keys of the partner run that are
  // larger (binary search; keys are distinct through their index bits).
  unsigned long long* src = key;
  unsigned long long* dst = key2;
  for (int run = G; run < N; run <<= 1) {
    for (int i = tid; i < N; i += kSchedThreads) {
      const unsigned long long x = src[i];
      const int r0 = (i / run) * run;             // start of this key's run
      const bool left = ((i / run) & 1) == 0;
      const int p0 = left ? r0 + run : r0 - run;  // start of the partner run
      const int p1 = min(p0 + run, N);
      int rank = 0;
      if (p0 < N) {
        // number of partner keys larger than x (partner run is descending)
        int lo = p0, hi = p1;
        while (lo < hi) {
          const int mid = (lo + hi) >> 1;
          if (src[mid] > x) lo = mid + 1; else hi = mid;
        }
        rank = lo - p0;
      }
      const int base = left ? r0 : p0;            // start of the merged run
      dst[base + (i - r0) + rank] = x;
    }
    __syncthreads();
    unsigned long long* t = src; src = dst; dst = t;
  }
  if (src != key) {
    for (int i = tid; i < N; i += kSchedThreads) key[i] = src[i];
    __syncthreads();
  }

  // the exact a of each sorted position, then an inclusive scan in place:
  // av[p] = S_{p+1}
  const int chunk = div_up(N, kSchedThreads);
  const int lo = tid * chunk, hi = min(N, lo + chunk);
  double loc[8];
  for (int p = lo; p < hi; ++p) loc[p - lo] = av[8191 - (int)(key[p] & 0x1FFFull)];
  __syncthreads();
  double run = 0.0;
  for (int p = lo; p < hi; ++p) {
    run += loc[p - lo];
    av[p] = run;
  }
  double incl = run;
  const int lane = tid & 31, wid = tid >> 5;
  for (int off = 1; off < 32; off <<= 1) {
    const double o = __shfl_up_sync(0xffffffffu, incl, off);
    if (lane >= off) incl += o;
  }
  if (lane == 31) warp_tot[wid] = incl;
  __syncthreads();
  if (wid == 0) {
    double wt = warp_tot[lane];
    for (int off = 1; off < 32; off <<= 1) {
      const double o = __shfl_up_sync(0xffffffffu, wt, off);
      if (lane >= off) wt += o;
    }
    warp_tot[lane] = wt;
  }
  __syncthreads();
  const double base = (incl - run) + (wid > 0 ? warp_tot[wid - 1] : 0.0);
  for (int p = lo; p < hi; ++p) av[p] += base;
  __syncthreads();

  // Theta_n for n = 0..N; the first n >= 1 with Theta_n <= Theta_{n-1} stops
  const double Rd = (double)R;
  for (int n = tid + 1; n <= N; n += kSchedThreads) {
    const double s_prev = n >= 2 ? av[n - 2] : 0.0;
    const double th_prev = (Rd + s_prev) * (double)sps[R + n - 1];
    const double th = (Rd + av[n - 1]) * (double)sps[R + n];
    if (th <= th_prev) atomicMin(&s_first_stop, n);
  }
  __syncthreads();
  const int nstar = (s_first_stop <= N) ? s_first_stop - 1 : N;
  int admitted = nstar;
  if (mode == DSPARK_SCHED_TOPK && round_ge2) admitted = min(max(s_K, 0), N);
  for (int p = tid; p < admitted; p += kSchedThreads)
    atomicAdd(&ell_s[(8191 - (int)(key[p] & 0x1FFFull)) / G], 1);
  __syncthreads();
  for (int b = tid; b < R; b += kSchedThreads) ell_out[b] = ell_s[b];
  if (tid == 0) {
    *nstar_out = nstar;
    const double S = admitted > 0 ? av[admitted - 1] : 0.0;
    *theta_out = (Rd + S) * (double)sps[R + admitted];
    if (mode == DSPARK_SCHED_TOPK) khist[round_lo & 1u] = nstar;
  }
}

}  // namespace

cudaError_t launch_confidence(const void* h, int hdtype, const void* W1, int wdtype, const float* w,
                              const float* sts_T, const int32_t* anchor, const int32_t* x, int B,
                              int gamma, int H, int r, int V, float* c_out, int* status,
                              cudaStream_t stream) {
  const int items = B * gamma;
  const dim3 grid(div_up(items * 32, 256));
  const bool vec = (H % 8 == 0) && (r % 8 == 0) && (((uintptr_t)h | (uintptr_t)W1 | (uintptr_t)w) % 16 == 0);
  if (hdtype == DSPARK_BF16 && wdtype == DSPARK_BF16)
    confidence_kernel<DSPARK_BF16, DSPARK_BF16><<<grid, 256, 0, stream>>>(h, W1, w, sts_T, anchor, x, B, gamma, H, r, V, vec, c_out, status);
  else if (hdtype == DSPARK_BF16)
    confidence_kernel<DSPARK_BF16, DSPARK_F32><<<grid, 256, 0, stream>>>(h, W1, w, sts_T, anchor, x, B, gamma, H, r, V, vec, c_out, status);
  else if (wdtype == DSPARK_BF16)
    confidence_kernel<DSPARK_F32, DSPARK_BF16><<<grid, 256, 0, stream>>>(h, W1, w, sts_T, anchor, x, B, gamma, H, r, V, vec, c_out, status);
  else
    confidence_kernel<DSPARK_F32, DSPARK_F32><<<grid, 256, 0, stream>>>(h, W1, w, sts_T, anchor, x, B, gamma, H, r, V, vec, c_out, status);
  return cudaGetLastError();
}

size_t schedule_smem_bytes(int B, int gamma) {
  int NP = 1;
  while (NP < B * gamma) NP <<= 1;
  return 2 * (size_t)NP * sizeof(unsigned long long) + (size_t)B * gamma * sizeof(double) + sizeof(int) * (size_t)B;
}

cudaError_t launch_schedule(const float* c, int B, int gamma, const float* sps, int mode,
                            uint32_t round_lo, int round_ge2, int32_t* khist, int32_t* ell_out,
                            int32_t* nstar_out, double* theta_out, int* status, cudaStream_t stream) {
  const size_t smem = schedule_smem_bytes(B, gamma);
  cudaError_t e = cudaFuncSetAttribute(schedule_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  schedule_kernel<<<1, kSchedThreads, smem, stream>>>(c, B, gamma, sps, mode, round_lo, round_ge2, khist,
                                                       ell_out, nstar_out, theta_out, status);
  return cudaGetLastError();
}

}  // namespace dspark
