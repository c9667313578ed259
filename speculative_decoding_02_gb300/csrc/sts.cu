// Sequential temperature scaling of the confidence head ("[DeepSeek-6] DSpark"
// blog, section 5; the study report's answer on calibration): on held-out
// samples, position by position from left to right, a grid search picks the
// temperature T_k that makes the prefix product prod_{i<=k} sigmoid(z_i / T_i)
// best match the observed prefix survival, by expected calibration error
// (ECE over kStsBins equal-width bins).
//
// Per position k, two kernels:
//   sts_accumulate  blocks of kStsChunk samples: for every observed sample
//                   (k <= ell) and every grid value, the prediction
//                   P = prod_{i<k} sigmoid(z_i / T_i) * sigmoid(z_k / t) and
//                   its bin; each block leaves its per-bin sums of P - y
//                   (y = 1 if acc >= k) in the workspace.
//   sts_select      one block: per grid value, ECE = sum over bins of
//                   |sum of P - y| / (observed samples), summed over blocks
//                   in a fixed order; the smallest (first on ties) sets T_k.
// Everything is fp64, so that the grid decision is the oracle's.
#include "kernels.h"

namespace dspark {
namespace {

constexpr int kStsThreads = 256;

__device__ __forceinline__ double sigmoid_f64(double x) { return 1.0 / (1.0 + exp(-x)); }

__global__ void __launch_bounds__(kStsThreads)
sts_accumulate(const float* __restrict__ z, const int32_t* __restrict__ ell, const int32_t* __restrict__ acc, int N,
               int G, int k, const float* __restrict__ grid, int ng, const float* __restrict__ T_fixed,
               double* __restrict__ part) {
  extern __shared__ double hist[];   // [ng][kStsBins]
  const int tid = threadIdx.x;
  for (int i = tid; i < ng * kStsBins; i += kStsThreads) hist[i] = 0.0;
  __syncthreads();
  const int n0 = blockIdx.x * kStsChunk, n1 = min(N, n0 + kStsChunk);
  for (int n = n0 + tid; n < n1; n += kStsThreads) {
    if (ell[n] < k) continue;
    double prev = 1.0;
    for (int i = 0; i < k - 1; ++i) prev *= sigmoid_f64((double)z[(size_t)n * G + i] / (double)T_fixed[i]);
    const double zk = (double)z[(size_t)n * G + k - 1];
    const double y = acc[n] >= k ? 1.0 : 0.0;
    for (int g = 0; g < ng; ++g) {
      const double P = prev * sigmoid_f64(zk / (double)grid[g]);
      int m = (int)floor(P * (double)kStsBins);
      m = m < 0 ? 0 : (m > kStsBins - 1 ? kStsBins - 1 : m);
      atomicAdd(&hist[g * kStsBins + m], P - y);
    }
  }
  __syncthreads();
  for (int i = tid; i < ng * kStsBins; i += kStsThreads) part[(size_t)blockIdx.x * ng * kStsBins + i] = hist[i];
}

__global__ void __launch_bounds__(kStsThreads)
sts_select(const int32_t* __restrict__ ell, int N, int k, const float* __restrict__ grid, int ng, int nblk,
           const double* __restrict__ part, float* __restrict__ T_out, float* __restrict__ ece_out) {
  __shared__ int warp_cnt[kStsThreads / 32];
  __shared__ double ece[kMaxStsGrid];
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  int cnt = 0;
  for (int n = tid; n < N; n += kStsThreads) cnt += ell[n] >= k ? 1 : 0;
  for (int off = 16; off > 0; off >>= 1) cnt += __shfl_xor_sync(0xffffffffu, cnt, off);
  if (lane == 0) warp_cnt[wid] = cnt;
  __syncthreads();
  int S = 0;
  for (int w = 0; w < kStsThreads / 32; ++w) S += warp_cnt[w];
  for (int g = tid; g < ng; g += kStsThreads) {
    double e = 0.0;
    for (int m = 0; m < kStsBins; ++m) {
      double s = 0.0;
      for (int b = 0; b < nblk; ++b) s += part[((size_t)b * ng + g) * kStsBins + m];
      e += fabs(s);
    }
    ece[g] = S > 0 ? e / (double)S : 0.0;
  }
  __syncthreads();
  if (tid == 0) {
    if (S == 0) {
      T_out[k - 1] = 1.0f;
      ece_out[k - 1] = 0.0f;
    } else {
      int best = 0;
      for (int g = 1; g < ng; ++g)
        if (ece[g] < ece[best]) best = g;
      T_out[k - 1] = grid[best];
      ece_out[k - 1] = (float)ece[best];
    }
  }
}

}  // namespace

size_t sts_workspace_bytes(int N, int ngrid) {
  return sizeof(double) * (size_t)div_up(N, kStsChunk) * ngrid * kStsBins;
}

cudaError_t launch_sts_fit(const float* z, const int32_t* ell, const int32_t* acc, int N, int gamma,
                           const float* grid, int ngrid, float* T_out, float* ece_out, void* ws,
                           cudaStream_t stream) {
  const int nblk = div_up(N, kStsChunk);
  double* part = static_cast<double*>(ws);
  const size_t smem = sizeof(double) * (size_t)ngrid * kStsBins;
  for (int k = 1; k <= gamma; ++k) {
    sts_accumulate<<<nblk, kStsThreads, smem, stream>>>(z, ell, acc, N, gamma, k, grid, ngrid, T_out, part);
    sts_select<<<1, kStsThreads, 0, stream>>>(ell, N, k, grid, ngrid, nblk, part, T_out, ece_out);
  }
  return cudaGetLastError();
}

}  // namespace dspark
