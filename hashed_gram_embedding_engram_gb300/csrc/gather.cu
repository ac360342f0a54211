// Step 4 of "DeepSeek Engram 系列导读", section "Engram 工作原理", Stage A:
// e_t = concat_{n,k} E_{n,k}[z_{t,n,k}], plus the int8 row dequantisation that
// "Engram 嵌入扩展：面向高效 DRAM/SSD 卸载的协同设计" (section "AgentX Engram
// DRAM卸载提升性能") fuses into the same row-selecting kernel, for tables in HBM
// or in pinned host memory reached over UVA (NVLink-C2C on Grace-Blackwell).
//
// Layout trick: because the R rows of one token are concatenated in (n,k)
// order, the 16-byte chunk number f of the flattened work list
//   f = (token*R + r) * chunks_per_row + c
// is also the 16-byte slot of the output (copy) or 32-byte slot (int8 -> bf16).
// Consecutive threads therefore read consecutive chunks of one row (one
// 64/128-byte transaction per row) and write perfectly contiguous output;
// no shared-memory staging is needed for coalescing.  Each thread keeps
// kItems independent 16-byte loads in flight before it stores anything.
//
// Two entry kernels share this body: gather_kernel reads the indices from
// memory (engram_gather), hash_gather_kernel computes them (Steps 1-3, in
// hashing.cuh) for the row it is about to read (engram_forward), so the
// indices never travel through HBM.  All lanes of a row compute the same index
// in the same instructions, which costs no extra issue slots.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "engram_internal.h"
#include "hashing.cuh"

namespace engram {
namespace {

constexpr int kThreads = 256;
constexpr int kItems = 8;

__device__ __forceinline__ uint4 ld_stream_16(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

// int8 x16 times a scale -> bf16 x16 (one rounding: the binary32 product is exact)
__device__ __forceinline__ void dequant16(uint4 q, float s, uint4& o0, uint4& o1) {
  const uint32_t w[4] = {q.x, q.y, q.z, q.w};
  uint32_t out[8];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int8_t b0 = static_cast<int8_t>(w[j] & 0xFF);
    const int8_t b1 = static_cast<int8_t>((w[j] >> 8) & 0xFF);
    const int8_t b2 = static_cast<int8_t>((w[j] >> 16) & 0xFF);
    const int8_t b3 = static_cast<int8_t>((w[j] >> 24) & 0xFF);
    out[2 * j] = pack_bf16x2(static_cast<float>(b0) * s, static_cast<float>(b1) * s);
    out[2 * j + 1] = pack_bf16x2(static_cast<float>(b2) * s, static_cast<float>(b3) * s);
  }
  o0 = make_uint4(out[0], out[1], out[2], out[3]);
  o1 = make_uint4(out[4], out[5], out[6], out[7]);
}

// Where the indices come from.
struct IdxFromMemory {
  const int32_t* idx;        // [ntok, R]
  __device__ uint32_t operator()(const PlanDev&, int64_t row_item, int, bool&) const {
    return static_cast<uint32_t>(__ldg(idx + row_item));
  }
};
struct IdxFromHash {
  const int32_t* ids;        // [B, T] raw ids
  const int32_t* proj;       // [V]
  const int32_t* prev;       // [B, N-1] or nullptr
  int T;
  int V;
  __device__ uint32_t operator()(const PlanDev& pd, int64_t row_item, int r, bool& bad) const {
    const int64_t tok = row_item / pd.R;
    const int b = static_cast<int>(tok / T);
    const int t = static_cast<int>(tok - static_cast<int64_t>(b) * T);
    return hash_index(pd, ids, T, b, t, r, proj, V, prev, bad);
  }
};

template <int kCpr, bool kInt8, typename Src>
__device__ __forceinline__ void gather_body(const PlanDev& pd, uint32_t* err, const Src& src, int64_t ntok,
                                            const uint8_t* __restrict__ table, const __half* __restrict__ scales,
                                            uint4* __restrict__ out) {
  constexpr int kRowBytes = kCpr * 16;
  const int R = pd.R;
  const int64_t total = ntok * R * kCpr;
  const int64_t span = static_cast<int64_t>(kThreads) * kItems;
  bool bad = false;
  for (int64_t base = static_cast<int64_t>(blockIdx.x) * span; base < total;
       base += static_cast<int64_t>(gridDim.x) * span) {
    uint4 v[kItems];
    float sc[kItems];
    bool ok[kItems];
#pragma unroll
    for (int j = 0; j < kItems; ++j) {
      const int64_t f = base + j * kThreads + threadIdx.x;
      ok[j] = false;
      v[j] = make_uint4(0, 0, 0, 0);
      sc[j] = 0.f;
      if (f < total) {
        const int64_t row_item = f / kCpr;          // token*R + r
        const int c = static_cast<int>(f % kCpr);
        const int r = static_cast<int>(row_item % R);
        const uint32_t z = src(pd, row_item, r, bad);
        if (z < pd.primes[r]) {
          const int64_t row = pd.offsets[r] + z;
          v[j] = ld_stream_16(table + row * kRowBytes + c * 16);
          if constexpr (kInt8) sc[j] = __half2float(scales[row]);
          ok[j] = true;
        } else {
          bad = true;
        }
      }
    }
#pragma unroll
    for (int j = 0; j < kItems; ++j) {
      const int64_t f = base + j * kThreads + threadIdx.x;
      if (f < total) {
        if constexpr (kInt8) {
          uint4 o0 = make_uint4(0, 0, 0, 0), o1 = make_uint4(0, 0, 0, 0);
          if (ok[j]) dequant16(v[j], sc[j], o0, o1);
          out[2 * f] = o0;
          out[2 * f + 1] = o1;
        } else {
          out[f] = v[j];
        }
      }
    }
  }
  if (bad) atomicOr(err, kErrIndexRange);
}

template <int kCpr, bool kInt8>
__global__ void __launch_bounds__(kThreads) gather_kernel(const __grid_constant__ PlanDev pd, uint32_t* __restrict__ err,
                                                          const int32_t* __restrict__ idx, int64_t ntok,
                                                          const uint8_t* __restrict__ table,
                                                          const __half* __restrict__ scales,
                                                          uint4* __restrict__ out) {
  gather_body<kCpr, kInt8>(pd, err, IdxFromMemory{idx}, ntok, table, scales, out);
}

template <int kCpr, bool kInt8>
__global__ void __launch_bounds__(kThreads)
    hash_gather_kernel(const __grid_constant__ PlanDev pd, uint32_t* __restrict__ err,
                       const int32_t* __restrict__ ids, int B, int T, const int32_t* __restrict__ proj, int V,
                       const int32_t* __restrict__ prev, const uint8_t* __restrict__ table,
                       const __half* __restrict__ scales, uint4* __restrict__ out) {
  gather_body<kCpr, kInt8>(pd, err, IdxFromHash{ids, proj, prev, T, V}, static_cast<int64_t>(B) * T, table, scales,
                           out);
}

int grid_blocks(const engram_plan* p, int64_t total) {
  const int64_t span = static_cast<int64_t>(kThreads) * kItems;
  int64_t blocks = (total + span - 1) / span;
  const int64_t cap = static_cast<int64_t>(p->num_sms) * 8;   // 8 x 256 threads resident per SM
  if (blocks > cap) blocks = cap;
  return static_cast<int>(blocks);
}

template <int kCpr, bool kInt8>
cudaError_t launch_idx(const engram_plan* p, const int32_t* idx, int64_t ntok, const void* table,
                       const uint16_t* scales, void* e, cudaStream_t s) {
  gather_kernel<kCpr, kInt8><<<grid_blocks(p, ntok * p->R * kCpr), kThreads, 0, s>>>(
      p->host, &p->dev->err, idx, ntok, static_cast<const uint8_t*>(table), reinterpret_cast<const __half*>(scales),
      static_cast<uint4*>(e));
  return cudaGetLastError();
}

template <int kCpr, bool kInt8>
cudaError_t launch_fused(const engram_plan* p, const int32_t* ids, int B, int T, const int32_t* proj, int V,
                         const int32_t* prev, const void* table, const uint16_t* scales, void* e, cudaStream_t s) {
  const int64_t ntok = static_cast<int64_t>(B) * T;
  hash_gather_kernel<kCpr, kInt8><<<grid_blocks(p, ntok * p->R * kCpr), kThreads, 0, s>>>(
      p->host, &p->dev->err, ids, B, T, proj, V, prev, static_cast<const uint8_t*>(table),
      reinterpret_cast<const __half*>(scales), static_cast<uint4*>(e));
  return cudaGetLastError();
}

int chunks_per_row(const engram_plan* p) {
  const int elem = p->cfg.table_dtype == ENGRAM_F32 ? 4 : (p->cfg.table_dtype == ENGRAM_BF16 ? 2 : 1);
  return p->cfg.row_dim * elem / 16;
}

}  // namespace

#define ENGRAM_DISPATCH_CPR(CALL)                                                  \
  switch (chunks_per_row(p)) {                                                     \
    case 1: return i8 ? CALL(1, true) : CALL(1, false);                            \
    case 2: return i8 ? CALL(2, true) : CALL(2, false);                            \
    case 4: return i8 ? CALL(4, true) : CALL(4, false);                            \
    case 8: return i8 ? CALL(8, true) : CALL(8, false);                            \
    case 16: return i8 ? CALL(16, true) : CALL(16, false);                         \
    default: return cudaErrorInvalidValue;                                         \
  }

cudaError_t launch_gather(const engram_plan* p, const int32_t* idx, int64_t ntok, const void* table,
                          const uint16_t* scales, void* e, cudaStream_t s) {
  const bool i8 = p->cfg.table_dtype == ENGRAM_I8_ROWSCALE_F16;
#define CALL(C, I) launch_idx<C, I>(p, idx, ntok, table, scales, e, s)
  ENGRAM_DISPATCH_CPR(CALL)
#undef CALL
}

cudaError_t launch_hash_gather(const engram_plan* p, const int32_t* ids, int B, int T, const int32_t* proj, int V,
                               const int32_t* prev_ids, const void* table, const uint16_t* scales, void* e,
                               cudaStream_t s) {
  const bool i8 = p->cfg.table_dtype == ENGRAM_I8_ROWSCALE_F16;
#define CALL(C, I) launch_fused<C, I>(p, ids, B, T, proj, V, prev_ids, table, scales, e, s)
  ENGRAM_DISPATCH_CPR(CALL)
#undef CALL
}

#undef ENGRAM_DISPATCH_CPR

}  // namespace engram
