// The confidence head of one (request, position): c_k = sigmoid((w[:H] . h_k +
// w[H:] . W1[x_{k-1}]) / T_k) (study report Eq.7; T_k from sequential
// temperature scaling, 1 without it), one warp per item.  Shared by the
// confidence kernel and the tensor-core draft's fused finalize, so that both
// give the same bits.
#pragma once

#include "common.cuh"

namespace dspark {

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

__device__ __forceinline__ float dot8(const float* ws, const float (&v)[8], float z) {
  const float4 w0 = *reinterpret_cast<const float4*>(ws);
  const float4 w1 = *reinterpret_cast<const float4*>(ws + 4);
  z = fmaf(w0.x, v[0], z); z = fmaf(w0.y, v[1], z); z = fmaf(w0.z, v[2], z); z = fmaf(w0.w, v[3], z);
  z = fmaf(w1.x, v[4], z); z = fmaf(w1.y, v[5], z); z = fmaf(w1.z, v[6], z); z = fmaf(w1.w, v[7], z);
  return z;
}

// Writes c_out[item] (lane 0).  prev = x_{k-1} as stored (an out-of-range
// token gives c = 0 and DSPARK_ERR_INVALID).  vec: 16-byte aligned h, W1 and
// w (w in shared or global memory) with H and r multiples of 8; then every
// 16-byte word of a batch of the h row (and the W1 row) is loaded before any
// arithmetic, so that a warp waits for one memory round trip per batch.
template <int HDT, int WDT>
__device__ __forceinline__ void conf_item(const void* __restrict__ h, const void* __restrict__ W1,
                                          const float* __restrict__ w, const float* __restrict__ sts_T, int item,
                                          int k, int prev, int H, int r, int V, bool vec, int lane,
                                          float* __restrict__ c_out, int* __restrict__ status) {
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
          if (u & 1) z1 = dot8(w + 8 * ch, v, z1);
          else z = dot8(w + 8 * ch, v, z);
        }
      }
    }
    if (has_e) {
      float v[8];
      unpack8<WDT>(e, v);
      z1 = dot8(w + H + 8 * lane, v, z1);
    }
    // rank above 256: the remaining W1 steps
    for (int j = 32 + lane; j < ne; j += 32) {
      uint4 e[kEW];
#pragma unroll
      for (int t = 0; t < kEW; ++t) e[t] = __ldg(erow + (size_t)j * kEW + t);
      float v[8];
      unpack8<WDT>(e, v);
      z1 = dot8(w + H + 8 * j, v, z1);
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

// The vectorised path's conditions (the staged weight of the confidence kernel
// must fit in shared memory: H + r up to 24576).
inline bool conf_vec(const void* h, const void* W1, const float* w, int H, int r) {
  return (H % 8 == 0) && (r % 8 == 0) && (((uintptr_t)h | (uintptr_t)W1 | (uintptr_t)w) % 16 == 0) &&
         (long long)H + r <= 24576;
}

}  // namespace dspark
