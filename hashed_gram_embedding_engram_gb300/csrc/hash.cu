// Steps 1-3 of "DeepSeek Engram 系列导读", section "Engram 工作原理", Stage A, as a
// standalone kernel (engram_hash): one thread per index z_{t,n,k}, the n-gram
// window read straight from the token ids (L1/L2-resident) and never stored;
// the index arithmetic is in hashing.cuh.  Writes are fully coalesced.
#include <cuda_runtime.h>

#include "engram_internal.h"
#include "hashing.cuh"

namespace engram {
namespace {

__global__ void __launch_bounds__(256) hash_kernel(const __grid_constant__ PlanDev pd, uint32_t* __restrict__ err,
                                                   const int32_t* __restrict__ ids, int B, int T,
                                                   const int32_t* __restrict__ proj, int V,
                                                   const int32_t* __restrict__ prev, int32_t* __restrict__ idx) {
  const int R = pd.R;
  const int64_t total = static_cast<int64_t>(B) * T * R;
  bool bad = false;
  for (int64_t f = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; f < total;
       f += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t tok = f / R;
    const int r = static_cast<int>(f - tok * R);
    const int b = static_cast<int>(tok / T);
    const int t = static_cast<int>(tok - static_cast<int64_t>(b) * T);
    idx[f] = static_cast<int32_t>(hash_index(pd, ids, T, b, t, r, proj, V, prev, bad));
  }
  if (bad) atomicOr(err, kErrIndexRange);
}

}  // namespace

cudaError_t launch_hash(const engram_plan* p, const int32_t* ids, int B, int T, const int32_t* proj, int V,
                        const int32_t* prev_ids, int32_t* idx, cudaStream_t s) {
  const int64_t total = static_cast<int64_t>(B) * T * p->R;
  const int threads = 256;
  int64_t blocks = (total + threads - 1) / threads;
  const int64_t cap = static_cast<int64_t>(p->num_sms) * 8;
  if (blocks > cap) blocks = cap;
  hash_kernel<<<static_cast<int>(blocks), threads, 0, s>>>(p->host, &p->dev->err, ids, B, T, proj, V, prev_ids, idx);
  return cudaGetLastError();
}

}  // namespace engram
