// Step 4 of "DeepSeek Engram 系列导读", section "Engram 工作原理", Stage A:
// e_t = concat_{n,k} E_{n,k}[z_{t,n,k}], plus the int8 row dequantisation that
// "Engram 嵌入扩展：面向高效 DRAM/SSD 卸载的协同设计" (section "AgentX Engram
// DRAM卸载提升性能") fuses into the same row-selecting kernel, for tables in HBM
// or in pinned host memory reached over UVA (NVLink-C2C on Grace-Blackwell).
//
// Layout trick: because the R rows of one token are concatenated in (n,k)
// order, the 16-byte chunk f = r * chunks_per_row + c of a token's rows is
// also the 16-byte slot of its output (copy) or 32-byte slot (int8 -> bf16).
// A warp owns one token: consecutive lanes read consecutive chunks of a row
// (one 64/128-byte transaction per row) and write contiguous output, so no
// shared-memory staging is needed for coalescing; each lane keeps several
// independent 16-byte loads in flight before it stores anything.
//
// The same kernel serves engram_gather (indices read from memory) and
// engram_forward (indices computed from the token ids for the rows about to
// be read, Steps 1-3 -- the arithmetic of hashing.cuh -- so they never
// travel through HBM).  There the warp first loads the token's n-gram window
// (lane i holds x'_{t-i}) and broadcasts it by shuffle; each lane computes the
// index of its chunk's row from the per-row constants of the parameter block
// (the lanes of one row compute the same index in the same instructions).
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "engram_internal.h"
#include "hashing.cuh"
#include "ptx.cuh"

namespace engram {
namespace {

constexpr int kThreads = 128;
constexpr int kWarpItems = 4;    // 16-byte chunks per lane per round

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

// Rows of a table in host memory that have a slot in the HBM hot-row cache
// (cache.cu) are read from there instead; the bytes are the same.
struct RowCache {
  const int32_t* slot;               // [total rows]: slot or -1
  const uint8_t* rows;               // [capacity, row bytes] in HBM
  unsigned long long* stats;         // [2]: rows looked up, rows served from HBM
};

template <int kCpr, bool kInt8, bool kHash, bool kCache = false>
__global__ void __launch_bounds__(kThreads, 8)
    row_gather_kernel(const __grid_constant__ PlanDev pd, uint32_t* __restrict__ err,
                      const int32_t* __restrict__ idx, const int32_t* __restrict__ ids, int T,
                      const int32_t* __restrict__ proj, int V, const int32_t* __restrict__ prev, int64_t ntok,
                      const uint8_t* __restrict__ table, const __half* __restrict__ scales,
                      uint4* __restrict__ out, const RowCache cache) {
  // The per-row constants are read from the parameter block itself (constant
  // bank): no shared memory, so blocks start at once and fit beside the K/V
  // GEMM's blocks on an SM (Stage A of a later layer prefetched on a side stream).
  const int R = pd.R, N = pd.N, K = pd.K;
  ptx::grid_dep_wait();
  ptx::grid_dep_launch();

  constexpr int kRowBytes = kCpr * 16;
  const int lane = threadIdx.x & 31;
  const int per_tok = R * kCpr;
  const int64_t n_warps = static_cast<int64_t>(gridDim.x) * (blockDim.x >> 5);
  bool bad = false;
  uint32_t n_look = 0, n_hit = 0;                       // rows of this lane's chunks 0 (kCache)
  for (int64_t tok = static_cast<int64_t>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5); tok < ntok;
       tok += n_warps) {
    uint64_t xp[kMaxN];
    if constexpr (kHash) {
      const int b = static_cast<int>(tok / T);
      const int t = static_cast<int>(tok - static_cast<int64_t>(b) * T);
      int64_t x = 0;                                   // lane i: x'_{t-i}, pad 0 before the start
      if (lane < N) {
        const int tt = t - lane;
        if (tt >= 0) {
          int raw = __ldg(ids + static_cast<int64_t>(b) * T + tt);
          if (static_cast<unsigned>(raw) >= static_cast<unsigned>(V)) {
            bad = true;
            raw = 0;
          }
          x = __ldg(proj + raw);
        } else if (prev != nullptr) {
          x = __ldg(prev + static_cast<int64_t>(b) * (N - 1) + (N - 1) + tt);
        }
      }
#pragma unroll
      for (int i = 0; i < kMaxN; ++i) xp[i] = static_cast<uint64_t>(__shfl_sync(0xFFFFFFFFu, x, i));
    }
    uint4* dst = out + (kInt8 ? 2 : 1) * tok * per_tok;
    for (int f0 = 0; f0 < per_tok; f0 += 32 * kWarpItems) {
      uint4 v[kWarpItems];
      float sc[kWarpItems];
      bool ok[kWarpItems];
#pragma unroll
      for (int j = 0; j < kWarpItems; ++j) {
        const int f = f0 + j * 32 + lane;
        ok[j] = false;
        v[j] = make_uint4(0, 0, 0, 0);
        sc[j] = 0.f;
        if (f < per_tok) {
          const int r = f / kCpr;
          const int c = f % kCpr;
          uint32_t z;
          const int n = 2 + r / K;
          if constexpr (kHash) {
            const uint64_t* m = pd.mults + pd.mult_base[n] + (r - (n - 2) * K) * n;
            uint64_t h = 0;
#pragma unroll
            for (int i = 0; i < kMaxN; ++i)
              if (i < n) h ^= xp[i] * m[i];
            z = barrett_mod(h, pd.primes[r], pd.mu[r]);
          } else {
            z = static_cast<uint32_t>(__ldg(idx + tok * R + r));
          }
          if (z < pd.primes[r]) {
            const int64_t row = pd.offsets[r] + z;
            const uint8_t* src = table + row * kRowBytes;
            if constexpr (kCache) {
              const int32_t sl = __ldg(cache.slot + row);
              if (sl >= 0) src = cache.rows + static_cast<int64_t>(sl) * kRowBytes;
              if (c == 0) {
                ++n_look;
                n_hit += sl >= 0;
              }
            }
            v[j] = ld_stream_16(src + c * 16);
            if constexpr (kInt8) sc[j] = __half2float(scales[row]);
            ok[j] = true;
          } else {
            bad = true;
          }
        }
      }
#pragma unroll
      for (int j = 0; j < kWarpItems; ++j) {
        const int f = f0 + j * 32 + lane;
        if (f < per_tok) {
          if constexpr (kInt8) {
            uint4 o0 = make_uint4(0, 0, 0, 0), o1 = make_uint4(0, 0, 0, 0);
            if (ok[j]) dequant16(v[j], sc[j], o0, o1);
            dst[2 * f] = o0;
            dst[2 * f + 1] = o1;
          } else {
            dst[f] = v[j];
          }
        }
      }
    }
  }
  if (bad) atomicOr(err, kErrIndexRange);
  if constexpr (kCache) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      n_look += __shfl_xor_sync(0xFFFFFFFFu, n_look, o);
      n_hit += __shfl_xor_sync(0xFFFFFFFFu, n_hit, o);
    }
    if (lane == 0 && n_look) {
      atomicAdd(cache.stats, static_cast<unsigned long long>(n_look));
      atomicAdd(cache.stats + 1, static_cast<unsigned long long>(n_hit));
    }
  }
}

int grid_for_tokens(const engram_plan* p, int64_t ntok) {
  const int64_t warps_per_block = kThreads / 32;
  int64_t blocks = (ntok + warps_per_block - 1) / warps_per_block;
  const int64_t cap = static_cast<int64_t>(p->num_sms) * 8;
  if (blocks > cap) blocks = cap;
  return static_cast<int>(blocks);
}

template <int kCpr, bool kInt8>
cudaError_t launch_idx(const engram_plan* p, const int32_t* idx, int64_t ntok, const void* table,
                       const uint16_t* scales, void* e, cudaStream_t s) {
  return launch_pdl(row_gather_kernel<kCpr, kInt8, false>, dim3(grid_for_tokens(p, ntok)), dim3(kThreads), 0, s,
                    p->host, &p->dev->err, static_cast<const int32_t*>(idx), static_cast<const int32_t*>(nullptr), 1,
                    static_cast<const int32_t*>(nullptr), 0, static_cast<const int32_t*>(nullptr), ntok,
                    static_cast<const uint8_t*>(table), reinterpret_cast<const __half*>(scales),
                    static_cast<uint4*>(e), RowCache{});
}

template <int kCpr, bool kInt8>
cudaError_t launch_fused(const engram_plan* p, const int32_t* ids, int B, int T, const int32_t* proj, int V,
                         const int32_t* prev, const void* table, const uint16_t* scales, void* e, cudaStream_t s) {
  const int64_t ntok = static_cast<int64_t>(B) * T;
  return launch_pdl(row_gather_kernel<kCpr, kInt8, true>, dim3(grid_for_tokens(p, ntok)), dim3(kThreads), 0, s,
                    p->host, &p->dev->err, static_cast<const int32_t*>(nullptr), ids, T, proj, V, prev, ntok,
                    static_cast<const uint8_t*>(table), reinterpret_cast<const __half*>(scales),
                    static_cast<uint4*>(e), RowCache{});
}

template <int kCpr, bool kInt8>
cudaError_t launch_cached(const engram_plan* p, const int32_t* ids, int B, int T, const int32_t* proj, int V,
                          const int32_t* prev, const void* table, const uint16_t* scales, void* e,
                          const RowCache& cache, cudaStream_t s) {
  const int64_t ntok = static_cast<int64_t>(B) * T;
  return launch_pdl(row_gather_kernel<kCpr, kInt8, true, true>, dim3(grid_for_tokens(p, ntok)), dim3(kThreads), 0, s,
                    p->host, &p->dev->err, static_cast<const int32_t*>(nullptr), ids, T, proj, V, prev, ntok,
                    static_cast<const uint8_t*>(table), reinterpret_cast<const __half*>(scales),
                    static_cast<uint4*>(e), cache);
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

cudaError_t launch_hash_gather_cached(const engram_plan* p, const int32_t* ids, int B, int T, const int32_t* proj,
                                      int V, const int32_t* prev_ids, const void* table, const uint16_t* scales,
                                      void* e, const int32_t* slot, const void* rows, unsigned long long* stats,
                                      cudaStream_t s) {
  const bool i8 = p->cfg.table_dtype == ENGRAM_I8_ROWSCALE_F16;
  const RowCache cache{slot, static_cast<const uint8_t*>(rows), stats};
#define CALL(C, I) launch_cached<C, I>(p, ids, B, T, proj, V, prev_ids, table, scales, e, cache, s)
  ENGRAM_DISPATCH_CPR(CALL)
#undef CALL
}

#undef ENGRAM_DISPATCH_CPR

}  // namespace engram
