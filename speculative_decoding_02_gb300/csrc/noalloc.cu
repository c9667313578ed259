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
// bytes.  Once the library's code for it is loaded on a GPU, that GPU holds it
// until the process exits.  With CUDA's lazy module loading that happens when
// its device address is first looked up, so dspark_noalloc_init does the
// lookup for the current device and should be called at start-up, before the
// caller's pool takes the rest of HBM and before any stream capture; the
// first draft call on a device does it otherwise.  In host code the array's
// name is only a host-side stand-in, so the device address comes from
// cudaGetSymbolAddress, with that device current.  All calls share the one
// array: two calls whose work overlaps on the GPU race on it and give
// undefined results.  The parts that must start at zero (the argmax keys, the
// counters and the status word) are cleared by every call; the status word
// then holds what the kernels of the latest call recorded, for
// dspark_noalloc_read_status.
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

extern "C" int dspark_noalloc_init(void) {
  void* ws = nullptr;
  return scratch_address(&ws) == cudaSuccess ? DSPARK_OK : DSPARK_ERR_CUDA;
}

extern "C" int dspark_noalloc_read_status(int* host_status, void* stream) {
  if (!host_status) return DSPARK_ERR_INVALID;
  void* ws = nullptr;
  if (scratch_address(&ws) != cudaSuccess) return DSPARK_ERR_CUDA;
  cudaStream_t s = (cudaStream_t)stream;
  int value = 0;
  if (cudaMemcpyAsync(&value, ws, sizeof(int), cudaMemcpyDeviceToHost, s) != cudaSuccess) return DSPARK_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return DSPARK_ERR_CUDA;
  if (cudaMemsetAsync(ws, 0, sizeof(int), s) != cudaSuccess) return DSPARK_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return DSPARK_ERR_CUDA;
  *host_status = value;
  return DSPARK_OK;
}

extern "C" int dspark_markov_draft_noalloc(const float* U, const void* W1, const void* W2, int wdtype,
                                           const int32_t* anchor, int B, int gamma, int V, int r,
                                           uint64_t seed, uint64_t round, int32_t* x_out, float* p_out,
                                           float* lse_out, void* stream) {
  const int st = draft_arg_checks(U, W1, W2, wdtype, anchor, B, gamma, V, r, x_out, p_out, lse_out);
  if (st != DSPARK_OK) return st;
  if (round >= (1ull << 29)) return DSPARK_ERR_INVALID;
  if (draft_scratch_bytes(B, gamma, V) > kNoAllocScratchBytes) return DSPARK_ERR_WORKSPACE;
  void* ws = nullptr;
  if (scratch_address(&ws) != cudaSuccess) return DSPARK_ERR_CUDA;
  cudaStream_t s = (cudaStream_t)stream;
  if (cudaMemsetAsync(ws, 0, sizeof(int), s) != cudaSuccess) return DSPARK_ERR_CUDA;
  DraftArgs a{U, W1, W2, wdtype, anchor, B, gamma, V, r, make_rng_key(seed, round), x_out, p_out, lse_out, ws};
  return launch_markov_draft(a, s) == cudaSuccess ? DSPARK_OK : DSPARK_ERR_CUDA;
}
