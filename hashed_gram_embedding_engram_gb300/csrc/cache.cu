// HBM hot-row cache in front of tables held in host memory.
//
// "Engram 嵌入扩展：面向高效 DRAM/SSD 卸载的协同设计" (section "AgentX Engram
// DRAM卸载提升性能") keeps the table in host DRAM and reads rows over the host
// link; the Ascend RecSDK Engram blog keeps a hot-embedding cache in device
// memory because n-gram accesses are Zipf-skewed.  This file is that cache for
// the UVA path:
//   * counts    uint32 [total rows]: accesses observed so far (LFU);
//   * slot      int32  [total rows]: the row's slot in the HBM copy, or -1;
//   * rows      [capacity, row bytes] in HBM.
// engram_cache_observe counts the rows a batch will read (Steps 1-3 per head,
// hashing.cuh); engram_cache_build admits the most-counted rows: a histogram
// of the counts gives the smallest threshold whose rows fit, those rows are
// compacted into slots (their order is whatever the atomics give: any order
// serves the same bytes) and copied from the host table, and the remaining
// slots go to rows one count below the threshold.  The cached gather itself
// is row_gather_kernel with a slot lookup per row (gather.cu).
//
// Per-batch row dedup ("Engram 嵌入扩展：面向高效 DRAM/SSD 卸载的协同设计": under
// Zipf-skewed n-gram statistics many lookups of a batch hit the same rows) uses
// the same slot map: before the gather, every distinct row of the batch that
// has no slot is claimed by one of its lookups and copied over the host link,
// once, into that lookup's row of a batch region after the cache's own slots;
// the gather then serves all its lookups from HBM, and afterwards the claimed
// slots are released.  Slot values: -1 no copy in HBM, [0, capacity) the
// hot-row cache, capacity + f lookup f's row of the batch region.
#include <cuda_runtime.h>

#include <vector>

#include "engram_internal.h"
#include "hashing.cuh"

namespace engram {
namespace {

constexpr int kHistBins = 65536;            // counts >= kHistBins - 1 share the last bin

__global__ void __launch_bounds__(256) observe_kernel(const __grid_constant__ PlanDev pd, uint32_t* __restrict__ err,
                                                      const int32_t* __restrict__ ids, int B, int T,
                                                      const int32_t* __restrict__ proj, int V,
                                                      const int32_t* __restrict__ prev, uint32_t* __restrict__ counts) {
  const int R = pd.R;
  const int64_t total = static_cast<int64_t>(B) * T * R;
  bool bad = false;
  for (int64_t f = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; f < total;
       f += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t tok = f / R;
    const int r = static_cast<int>(f - tok * R);
    const int b = static_cast<int>(tok / T);
    const int t = static_cast<int>(tok - static_cast<int64_t>(b) * T);
    const uint32_t z = hash_index(pd, ids, T, b, t, r, proj, V, prev, bad);
    const uint32_t c = atomicAdd(counts + pd.offsets[r] + z, 1u);
    if (c == 0xFFFFFFFFu) atomicSub(counts + pd.offsets[r] + z, 1u);   // saturate instead of wrapping
  }
  if (bad) atomicOr(err, kErrIndexRange);
}

__global__ void __launch_bounds__(256) histogram_kernel(const uint32_t* __restrict__ counts, int64_t n,
                                                        uint32_t* __restrict__ hist) {
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const uint32_t c = counts[i];
    if (c) atomicAdd(hist + (c < kHistBins - 1 ? c : kHistBins - 1), 1u);
  }
}

// Rows with count >= thr take a slot; rows with count == thr - 1 (thr > 1)
// take one while slots remain.  Each admitted row is copied from the table.
__global__ void __launch_bounds__(256) admit_kernel(const uint32_t* __restrict__ counts, int64_t n, uint32_t thr,
                                                    int pass, int64_t capacity, int row_bytes,
                                                    const uint8_t* __restrict__ table, uint8_t* __restrict__ rows,
                                                    int32_t* __restrict__ slot, unsigned long long* __restrict__ used) {
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const uint32_t c = counts[i];
    const bool take = pass == 0 ? (c >= thr && c > 0) : (thr > 1 && c == thr - 1);
    if (!take) continue;
    const unsigned long long s = atomicAdd(used, 1ull);
    if (static_cast<int64_t>(s) >= capacity) continue;        // only in pass 1: the slots are full
    slot[i] = static_cast<int32_t>(s);
    const uint4* src = reinterpret_cast<const uint4*>(table + i * row_bytes);
    uint4* dst = reinterpret_cast<uint4*>(rows + static_cast<int64_t>(s) * row_bytes);
    for (int j = 0; j < row_bytes / 16; ++j) dst[j] = src[j];
  }
}

__global__ void __launch_bounds__(256) decay_kernel(uint32_t* __restrict__ counts, int64_t n) {
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x)
    counts[i] >>= 1;
}

// ---- per-batch dedup

// Every lookup f of the batch: a row without a slot is claimed by the first
// lookup that gets to it (compare-and-swap -1 -> first_slot + f), which
// records the row in owner[f] (others record kNoRow).  No counter is shared:
// the batch region has a row per lookup.
constexpr uint32_t kNoRow = 0xFFFFFFFFu;

__global__ void __launch_bounds__(256) dedup_claim_kernel(const __grid_constant__ PlanDev pd, uint32_t* __restrict__ err,
                                                          const int32_t* __restrict__ ids, int B, int T,
                                                          const int32_t* __restrict__ proj, int V,
                                                          const int32_t* __restrict__ prev, int32_t* __restrict__ slot,
                                                          int32_t first_slot, uint32_t* __restrict__ owner) {
  const int R = pd.R;
  const int64_t total = static_cast<int64_t>(B) * T * R;
  bool bad = false;
  for (int64_t f = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; f < total;
       f += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t tok = f / R;
    const int r = static_cast<int>(f - tok * R);
    const int b = static_cast<int>(tok / T);
    const int t = static_cast<int>(tok - static_cast<int64_t>(b) * T);
    const int64_t g = pd.offsets[r] + hash_index(pd, ids, T, b, t, r, proj, V, prev, bad);
    const bool mine = *reinterpret_cast<volatile int32_t*>(slot + g) == -1 &&
                      atomicCAS(slot + g, -1, first_slot + static_cast<int32_t>(f)) == -1;
    owner[f] = mine ? static_cast<uint32_t>(g) : kNoRow;
  }
  if (bad) atomicOr(err, kErrIndexRange);
}

// The claimed rows from the table (host memory over UVA) into their lookups'
// rows of the batch region: consecutive threads take consecutive 16-byte
// chunks of a row, so each row crosses the link as one request.
__global__ void __launch_bounds__(256) dedup_fetch_kernel(int64_t total, const uint32_t* __restrict__ owner,
                                                          int row_bytes, const uint8_t* __restrict__ table,
                                                          uint8_t* __restrict__ region) {
  const int cpr = row_bytes / 16;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < total * cpr;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t f = i / cpr;
    const uint32_t g = owner[f];
    if (g == kNoRow) continue;
    const int ch = static_cast<int>(i - f * cpr);
    *reinterpret_cast<uint4*>(region + f * row_bytes + ch * 16) =
        __ldg(reinterpret_cast<const uint4*>(table + static_cast<int64_t>(g) * row_bytes + ch * 16));
  }
}

// After the gather: the claimed slots return to -1; the block's claims are
// added to the count of rows fetched (one atomic per block and round).
__global__ void __launch_bounds__(256) dedup_release_kernel(int64_t total, const uint32_t* __restrict__ owner,
                                                            int32_t* __restrict__ slot,
                                                            unsigned long long* __restrict__ fetched) {
  // the loop bound is uniform over the block, so every thread reaches the barrier
  for (int64_t base = static_cast<int64_t>(blockIdx.x) * blockDim.x; base < total;
       base += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t f = base + threadIdx.x;
    const uint32_t g = f < total ? owner[f] : kNoRow;
    if (g != kNoRow) slot[g] = -1;
    const int n = __syncthreads_count(g != kNoRow);
    if (threadIdx.x == 0 && n) atomicAdd(fetched, static_cast<unsigned long long>(n));
  }
}

int grid_rows(const engram_plan* p, int64_t n) {
  int64_t blocks = (n + 255) / 256;
  const int64_t cap = static_cast<int64_t>(p->num_sms) * 16;
  return static_cast<int>(blocks < cap ? (blocks < 1 ? 1 : blocks) : cap);
}

}  // namespace

cudaError_t dedup_claim(const engram_plan* p, const int32_t* ids, int B, int T, const int32_t* proj, int V,
                        const int32_t* prev_ids, int32_t* slot, int32_t first_slot, uint32_t* owner, cudaStream_t s) {
  const int64_t total = static_cast<int64_t>(B) * T * p->R;
  dedup_claim_kernel<<<grid_rows(p, total), 256, 0, s>>>(p->host, &p->dev->err, ids, B, T, proj, V, prev_ids, slot,
                                                         first_slot, owner);
  return cudaGetLastError();
}

cudaError_t dedup_fetch(const engram_plan* p, int64_t total, const uint32_t* owner, int row_bytes, const void* table,
                        void* region, cudaStream_t s) {
  dedup_fetch_kernel<<<grid_rows(p, total * (row_bytes / 16)), 256, 0, s>>>(
      total, owner, row_bytes, static_cast<const uint8_t*>(table), static_cast<uint8_t*>(region));
  return cudaGetLastError();
}

cudaError_t dedup_release(const engram_plan* p, int64_t total, const uint32_t* owner, int32_t* slot,
                          unsigned long long* fetched, cudaStream_t s) {
  dedup_release_kernel<<<grid_rows(p, total), 256, 0, s>>>(total, owner, slot, fetched);
  return cudaGetLastError();
}

cudaError_t cache_observe(const engram_plan* p, const int32_t* ids, int B, int T, const int32_t* proj, int V,
                          const int32_t* prev_ids, uint32_t* counts, cudaStream_t s) {
  const int64_t total = static_cast<int64_t>(B) * T * p->R;
  observe_kernel<<<grid_rows(p, total), 256, 0, s>>>(p->host, &p->dev->err, ids, B, T, proj, V, prev_ids, counts);
  return cudaGetLastError();
}

cudaError_t cache_build(const engram_plan* p, int64_t capacity, int row_bytes, const void* table, uint32_t* counts,
                        int32_t* slot, void* rows, unsigned long long* used, int decay, int64_t* cached,
                        cudaStream_t s) {
  const int64_t n = p->total_rows;
  uint32_t* hist = nullptr;
  if (cudaMallocAsync(&hist, kHistBins * sizeof(uint32_t), s) != cudaSuccess) return cudaErrorMemoryAllocation;
  cudaError_t e = cudaMemsetAsync(hist, 0, kHistBins * sizeof(uint32_t), s);
  if (e == cudaSuccess) {
    histogram_kernel<<<grid_rows(p, n), 256, 0, s>>>(counts, n, hist);
    e = cudaGetLastError();
  }
  std::vector<uint32_t> h(kHistBins);
  if (e == cudaSuccess) e = cudaMemcpyAsync(h.data(), hist, kHistBins * sizeof(uint32_t), cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  cudaFreeAsync(hist, s);
  if (e != cudaSuccess) return e;
  // smallest threshold whose rows (count >= thr) all fit; if not even the
  // most-counted rows all fit, some of them fill the slots (pass 1)
  uint32_t thr = kHistBins;
  int64_t taken = 0;
  int c_max = 0;
  for (int c = kHistBins - 1; c >= 1; --c) {
    if (h[c] && !c_max) c_max = c;
    if (taken + h[c] > capacity) break;
    taken += h[c];
    thr = static_cast<uint32_t>(c);
  }
  if (thr == static_cast<uint32_t>(kHistBins) && c_max > 0) thr = static_cast<uint32_t>(c_max) + 1;
  e = cudaMemsetAsync(slot, 0xFF, static_cast<size_t>(n) * sizeof(int32_t), s);
  if (e == cudaSuccess) e = cudaMemsetAsync(used, 0, sizeof(unsigned long long), s);
  for (int pass = 0; pass < 2 && e == cudaSuccess && thr < static_cast<uint32_t>(kHistBins); ++pass) {
    admit_kernel<<<grid_rows(p, n), 256, 0, s>>>(counts, n, thr, pass, capacity, row_bytes,
                                                 static_cast<const uint8_t*>(table), static_cast<uint8_t*>(rows), slot,
                                                 used);
    e = cudaGetLastError();
  }
  if (e == cudaSuccess && decay) {
    decay_kernel<<<grid_rows(p, n), 256, 0, s>>>(counts, n);
    e = cudaGetLastError();
  }
  unsigned long long u = 0;
  if (e == cudaSuccess) e = cudaMemcpyAsync(&u, used, sizeof(u), cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e == cudaSuccess) *cached = static_cast<int64_t>(u) < capacity ? static_cast<int64_t>(u) : capacity;
  return e;
}

}  // namespace engram
