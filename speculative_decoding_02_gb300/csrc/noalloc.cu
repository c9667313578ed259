// dspark_markov_draft_noalloc: the Markov draft for callers that cannot
// allocate device memory at the time of the call.
//
// Some callers cannot hand the library a workspace: an inference engine that
// gives all of HBM to its own pool allocator at start-up and forbids other
// allocations, a plugin loaded into a host process that passes it no
// allocator, or code that would otherwise have to call cudaMalloc (which may
// synchronise the device) in the middle of a latency-critical decode loop.
// For them this entry point runs the same draft kernels as dspark_markov_draft,
// but its scratch space is a fixed array in the library's own device memory
// instead of a caller buffer.
//
// The array is a file-scope __device__ variable of DSPARK_NOALLOC_SCRATCH_BYTES
// bytes.  Every GPU on which the library is loaded holds it until the process
// exits.  In host code the array's name is only a host-side stand-in, so the
// device address is looked up with cudaGetSymbolAddress once per device, with
// that device current, on the first call made on it; that first call should
// therefore come before any stream capture.  All calls share the one array:
// two calls whose work overlaps on the GPU race on it and give undefined
// results.  The parts that must start at zero (the argmax keys and the status
// word) are cleared by every call.
#include <mutex>

#include "kernels.h"

namespace dspark {
namespace {

constexpr size_t kNoAllocScratchBytes = DSPARK_NOALLOC_SCRATCH_BYTES;
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

std::mutex g_setup_mutex;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of g_noalloc_scratch on the current device (set up once).
cudaError_t scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_setup_mutex);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return cudaSuccess;
}

// Bytes of scratch the draft touches: the status word, the counters, the
// per-position argmax keys and the per-slice softmax partials.
size_t draft_scratch_bytes(int B, int gamma, int V) {
  const WsLayout L = ws_layout(B, gamma, V);
  return L.draft_part + 8ull * gamma * (size_t)draft_part_slices(V) * B;
}

}  // namespace
}  // namespace dspark

using namespace dspark;

extern "C" int dspark_markov_draft_noalloc(const float* U, const void* W1, const void* W2, int wdtype,
                                           const int32_t* anchor, int B, int gamma, int V, int r,
                                           uint64_t seed, uint64_t round, int32_t* x_out, float* p_out,
                                           float* lse_out, void* stream) {
  if (B <= 0 || gamma <= 0 || V <= 0 || r <= 0) return DSPARK_ERR_INVALID;
  if (gamma > kMaxGamma) return DSPARK_ERR_UNSUPPORTED;
  if (V % 8 != 0 || r % 16 != 0 || r > 256 || B > 65535) return DSPARK_ERR_UNSUPPORTED;
  if ((long long)B * (gamma + 1) * (long long)V >= (1ll << 40)) return DSPARK_ERR_UNSUPPORTED;
  if (wdtype != DSPARK_F32 && wdtype != DSPARK_BF16) return DSPARK_ERR_INVALID;
  if (!U || !W1 || !W2 || !anchor || !x_out || !p_out || !lse_out) return DSPARK_ERR_INVALID;
  if (((uintptr_t)U | (uintptr_t)W1 | (uintptr_t)W2) % 16 != 0) return DSPARK_ERR_INVALID;
  if (round >= (1ull << 29)) return DSPARK_ERR_INVALID;
  if (draft_scratch_bytes(B, gamma, V) > kNoAllocScratchBytes) return DSPARK_ERR_WORKSPACE;
  void* ws = nullptr;
  if (scratch_address(&ws) != cudaSuccess) return DSPARK_ERR_CUDA;
  cudaStream_t s = (cudaStream_t)stream;
  if (cudaMemsetAsync(ws, 0, sizeof(int), s) != cudaSuccess) return DSPARK_ERR_CUDA;
  DraftArgs a{U, W1, W2, wdtype, anchor, B, gamma, V, r, make_rng_key(seed, round), x_out, p_out, lse_out, ws};
  return launch_markov_draft(a, s) == cudaSuccess ? DSPARK_OK : DSPARK_ERR_CUDA;
}
