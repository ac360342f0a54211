// engram_forward for callers that cannot allocate device memory.
//
// Some callers have no way to hand the library a workspace: code running
// inside a host framework that owns the device allocator and exposes none of
// it, plugin or extension hosts that accept only plain function calls, and
// latency-critical paths (a serving loop, a callback) where a cudaMalloc --
// which may synchronise the device -- is not allowed.  For them this file
// keeps the forward pass's scratch in a file-scope __device__ array that the
// library image carries: it exists on every GPU that loads the library, from
// module load until process exit, and nothing is allocated per call.
#include <cuda_runtime.h>

#include <mutex>

#include "engram_internal.h"

namespace {

// 32 MiB: the scratch of up to about 4300 tokens of a layer with d = 1024 and
// d_mem = 1024 (the prefill batch of 4096 tokens needs 26.6 MB).
constexpr size_t kStaticScratchBytes = size_t(32) << 20;
constexpr int kMaxDevices = 64;

__device__ __align__(256) unsigned char g_static_scratch[kStaticScratchBytes];

std::mutex g_setup_mutex;
void* g_scratch_ptr[kMaxDevices] = {};

// The device address of g_static_scratch on the current device.  In host code
// the array's name is only a host-side stand-in for the symbol, so the
// address comes from cudaGetSymbolAddress, once per device.
engram_status_t scratch_for_device(int dev, void** out) {
  if (dev < 0 || dev >= kMaxDevices) return ENGRAM_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_setup_mutex);
  if (g_scratch_ptr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_static_scratch) != cudaSuccess || p == nullptr) {
      cudaGetLastError();
      return ENGRAM_ERR_CUDA;
    }
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return ENGRAM_OK;
}

}  // namespace

extern "C" engram_status_t engram_forward_static_scratch(const engram_plan_t* plan, const int32_t* ids, int B, int T,
                                                         const int32_t* proj, int V, const engram_weights_t* w,
                                                         void* H, engram_state_t* state, engram_stream_t stream) {
  if (!plan || B < 0 || T < 0) return ENGRAM_ERR_INVALID_ARG;
  size_t need = 0;
  if (engram_status_t s = engram_plan_workspace_bytes(plan, static_cast<int64_t>(B) * T, &need)) return s;
  if (need > kStaticScratchBytes) return ENGRAM_ERR_WORKSPACE;     // B*T too large for the static scratch
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return ENGRAM_ERR_CUDA;
  if (dev != plan->device) return ENGRAM_ERR_INVALID_ARG;          // the plan belongs to another device
  void* scratch = nullptr;
  if (engram_status_t s = scratch_for_device(dev, &scratch)) return s;
  return engram_forward(plan, ids, B, T, proj, V, w, H, state, scratch, kStaticScratchBytes, stream);
}
