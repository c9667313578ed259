// Confidence head (study report Eq.7) and the hardware-aware prefix scheduler
// ("[DeepSeek-6] DSpark" blog, sections 6-7; study report Theta = tau * SPS(B)).
#include "conf.cuh"
#include "sched.cuh"
#include "kernels.h"

namespace dspark {
namespace {

// c_k = sigmoid((w[:H] . h_k + w[H:] . W1[x_{k-1}]) / T_k), one warp per (b, k)
// (conf_item in conf.cuh; the tensor-core draft's fused finalize runs the same
// code).  vec: w is staged in shared memory once per CTA.
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
  pdl_wait();   // x from the draft
  const int item = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  if (item >= B * G) return;
  const int b = item / G, k = item - (item / G) * G + 1;
  const int prev = (k == 1) ? anchor[b] : x[(size_t)b * G + k - 2];
  conf_item<HDT, WDT>(h, W1, vec ? w_s : w, sts_T, item, k, prev, H, r, V, vec, threadIdx.x & 31, c_out, status);
}

constexpr int kSchedThreads = 1024;

// One CTA of 1024 threads (schedule_block).
__global__ void __launch_bounds__(kSchedThreads)
schedule_kernel(const float* __restrict__ c, int R, int G, const float* __restrict__ sps, int mode,
                unsigned long long round_host, const unsigned long long* __restrict__ round_dev,
                int32_t* __restrict__ khist, int32_t* __restrict__ ell_out, int32_t* __restrict__ nstar_out,
                double* __restrict__ theta_out, int* __restrict__ status) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  __shared__ SchedShared sh;
  // (no early trigger: the next kernel's CTAs, resident and waiting, would
  // share this CTA's SM while it runs)
  pdl_wait();   // c from the confidence head
  const unsigned long long round = round_dev ? __ldcg(round_dev) : round_host;
  schedule_block<kSchedThreads>(c, R, G, sps, mode, round, khist, ell_out, nstar_out, theta_out, status, smem_raw,
                                sh, (int)threadIdx.x, CtaSync{});
}

}  // namespace

cudaError_t launch_confidence(const void* h, int hdtype, const void* W1, int wdtype, const float* w,
                              const float* sts_T, const int32_t* anchor, const int32_t* x, int B,
                              int gamma, int H, int r, int V, float* c_out, int* status,
                              cudaStream_t stream) {
  const int items = B * gamma;
  const dim3 grid(div_up(items * 32, kConfThreads));
  const bool vec = conf_vec(h, W1, w, H, r);
  const size_t smem = vec ? sizeof(float) * (size_t)(H + r) : 0;
  cudaError_t e = cudaSuccess;
#define DSPARK_CONF(HD, WD)                                                                                   \
  do {                                                                                                        \
    if (smem > 48 * 1024)                                                                                     \
      e = cudaFuncSetAttribute(confidence_kernel<HD, WD>, cudaFuncAttributeMaxDynamicSharedMemorySize,        \
                               (int)smem);                                                                    \
    if (e == cudaSuccess)                                                                                     \
      e = launch_pdl(confidence_kernel<HD, WD>, grid, dim3(kConfThreads), smem, stream, h, W1, w, sts_T,        \
                     anchor, x, B, gamma, H, r, V, vec, c_out, status);                                       \
  } while (0)
  if (hdtype == DSPARK_BF16 && wdtype == DSPARK_BF16) DSPARK_CONF(DSPARK_BF16, DSPARK_BF16);
  else if (hdtype == DSPARK_BF16) DSPARK_CONF(DSPARK_BF16, DSPARK_F32);
  else if (wdtype == DSPARK_BF16) DSPARK_CONF(DSPARK_F32, DSPARK_BF16);
  else DSPARK_CONF(DSPARK_F32, DSPARK_F32);
#undef DSPARK_CONF
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}


cudaError_t launch_schedule(const float* c, int B, int gamma, const float* sps, int mode,
                            unsigned long long round, const unsigned long long* round_dev, int32_t* khist,
                            int32_t* ell_out, int32_t* nstar_out, double* theta_out, int* status,
                            cudaStream_t stream) {
  const size_t smem = mode == DSPARK_SCHED_FIXED ? 0 : schedule_smem_bytes(B, gamma);
  cudaError_t e = cudaFuncSetAttribute(schedule_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  e = launch_pdl(schedule_kernel, dim3(1), dim3(kSchedThreads), smem, stream, c, B, gamma, sps, mode, round,
                 round_dev, khist, ell_out, nstar_out, theta_out, status);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace dspark
