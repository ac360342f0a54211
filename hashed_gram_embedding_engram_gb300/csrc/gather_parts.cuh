// Building blocks of the row gather (Step 4, with Steps 1-3 computed for the
// rows about to be read): 16-byte streaming loads, the int8 dequantisation,
// the per-row table constants, the two memory hops of a token's n-gram window,
// and one token's row phase (index, source, scale per row) and chunk phase
// (loads and contiguous stores).  gather.cu composes them into the gather
// kernel; decode.cu into the one-launch decode step.  See gather.cu for the
// design.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "engram_internal.h"
#include "hashing.cuh"
#include "ptx.cuh"

namespace engram {
namespace ga {

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

// The per-layer operands of one gather launch; blockIdx.y selects the layer.
// Layers of one launch share the token ids, P and the table shape (N, K, row
// size and type); each has its own parameter block, tables, state and output.
struct GatherLayers {
  const PlanDev* pdg[kMaxGatherLayers];
  uint32_t* err[kMaxGatherLayers];
  const int32_t* prev[kMaxGatherLayers];
  const uint8_t* table[kMaxGatherLayers];
  const __half* scales[kMaxGatherLayers];
  uint4* out[kMaxGatherLayers];
  uint8_t* q8[kMaxGatherLayers];       // e4m3 codes of e [ntok, d_mem] instead of e (the codes kernel)
  float* qscale[kMaxGatherLayers];     // and each token's scale [ntok]
};

// Per-lane table constants of one of the R rows a token reads: the lanes of a
// warp own rows lane and lane + 32 (R <= 64).
struct RowConst {
  uint32_t prime;
  uint64_t mu;
  int64_t offset;
  const uint64_t* mult;                // m_{n,k,0..n-1}
  int n;
};

__device__ __forceinline__ RowConst row_const(const PlanDev* __restrict__ pdg, int K, int r) {
  RowConst c;
  c.prime = __ldg(&pdg->primes[r]);
  c.mu = __ldg(&pdg->mu[r]);
  c.offset = __ldg(&pdg->offsets[r]);
  c.n = 2 + r / K;
  c.mult = pdg->mults + __ldg(&pdg->mult_base[c.n]) + (r - (c.n - 2) * K) * c.n;
  return c;
}

__device__ __forceinline__ uint64_t shfl64(uint64_t v, int src) {
  const uint32_t lo = __shfl_sync(0xFFFFFFFFu, static_cast<uint32_t>(v), src);
  const uint32_t hi = __shfl_sync(0xFFFFFFFFu, static_cast<uint32_t>(v >> 32), src);
  return (static_cast<uint64_t>(hi) << 32) | lo;
}

// 32-bit loads through the non-coherent path, kept in program order with the
// row loads (asm volatile), so the next token's id and projection loads are
// issued exactly where the pipeline below places them.
__device__ __forceinline__ int32_t ld_nc_s32(const int32_t* p) {
  int32_t v;
  asm volatile("ld.global.nc.s32 %0, [%1];" : "=r"(v) : "l"(p));
  return v;
}

// The warp's view of one token's n-gram window, in two memory hops: the raw
// id (or the projected id from `prev`, or the pad), then its projection.
struct WindowHop {
  int32_t v;        // raw id (need_proj) or the projected id itself
  bool need_proj;
};

__device__ __forceinline__ WindowHop window_hop1(const int32_t* __restrict__ ids, const int32_t* __restrict__ prev,
                                                 int64_t tok, int T, int N, int V, int lane, bool& bad) {
  WindowHop h{0, false};
  if (lane < N) {
    const int b = static_cast<int>(tok / T);
    const int t = static_cast<int>(tok - static_cast<int64_t>(b) * T);
    const int tt = t - lane;                           // lane i: x'_{t-i}, pad 0 before the start
    if (tt >= 0) {
      int raw = ld_nc_s32(ids + static_cast<int64_t>(b) * T + tt);
      if (static_cast<unsigned>(raw) >= static_cast<unsigned>(V)) {
        bad = true;
        raw = 0;
      }
      h.v = raw;
      h.need_proj = true;
    } else if (prev != nullptr) {
      h.v = ld_nc_s32(prev + static_cast<int64_t>(b) * (N - 1) + (N - 1) + tt);
    }
  }
  return h;
}

__device__ __forceinline__ int32_t window_hop2(const WindowHop& h, const int32_t* __restrict__ proj) {
  return h.need_proj ? ld_nc_s32(proj + h.v) : h.v;
}

// Row phase of one token: lane r (and r + 32) forms the index of row r (from
// the token's projected window xp, or read: z), its source address (table, or
// the HBM cache) and its int8 scale.  src = 0 marks a row out of range.
template <int kCpr, bool kInt8, bool kHash, bool kCache, bool kWide>
__device__ __forceinline__ void row_phase(const RowConst (&rc)[kWide ? 2 : 1], bool has0, bool has1,
                                          const uint32_t (&xp)[kMaxN], const int32_t (&z_in)[kWide ? 2 : 1],
                                          const uint8_t* __restrict__ table, const __half* __restrict__ scales,
                                          const RowCache& cache, int lane, uint64_t (&src)[kWide ? 2 : 1],
                                          float (&sc)[kWide ? 2 : 1], bool& bad, uint32_t& n_look,
                                          uint32_t& n_hit) {
  constexpr int kRowBytes = kCpr * 16;
  constexpr int kRows = kWide ? 2 : 1;
  (void)lane;
#pragma unroll
  for (int h = 0; h < kRows; ++h) {
    src[h] = 0;
    sc[h] = 0.f;
    const bool has = h == 0 ? has0 : has1;
    if (!has) continue;
    const RowConst& c = rc[h];
    uint32_t z;
    if constexpr (kHash) {
      uint64_t hsh = 0;
#pragma unroll
      for (int i = 0; i < kMaxN; ++i)
        if (i < c.n) hsh ^= static_cast<uint64_t>(xp[i]) * __ldg(c.mult + i);
      z = barrett_mod(hsh, c.prime, c.mu);
    } else {
      z = static_cast<uint32_t>(z_in[h]);
      if (z >= c.prime) {
        bad = true;
        continue;
      }
    }
    const int64_t row = c.offset + z;
    const uint8_t* p = table + row * kRowBytes;
    if constexpr (kCache) {
      const int32_t sl = __ldg(cache.slot + row);
      if (sl >= 0) p = cache.rows + static_cast<int64_t>(sl) * kRowBytes;
      ++n_look;
      n_hit += sl >= 0;
    }
    src[h] = reinterpret_cast<uint64_t>(p);
    if constexpr (kInt8) sc[h] = __half2float(scales[row]);
  }
}

// Chunk phase of one token: lane l takes the token's 16-byte chunks l, l + 32,
// ... (chunk f = r * kCpr + c is also the output's slot f), gets its row's
// address by shuffle, keeps kWarpItems loads in flight, then stores them to
// dst (the token's output row).  after_first() runs once, after the first
// round of loads is issued and before any of them is used.
template <int kCpr, bool kInt8, bool kWide, typename F>
__device__ __forceinline__ void chunk_phase(const uint64_t (&src)[kWide ? 2 : 1], const float (&sc)[kWide ? 2 : 1],
                                            int R, uint4* __restrict__ dst, int lane, F&& after_first) {
  constexpr int kRows = kWide ? 2 : 1;
  const int per_tok = R * kCpr;
  for (int f0 = 0; f0 < per_tok; f0 += 32 * kWarpItems) {
    uint4 v[kWarpItems];
    float s_[kWarpItems];
    bool ok[kWarpItems];
#pragma unroll
    for (int j = 0; j < kWarpItems; ++j) {
      const int f = f0 + j * 32 + lane;
      const int r = f / kCpr;
      const int c = f % kCpr;
      // every lane takes part in the shuffles; lanes past the token's chunks discard theirs
      const int rs = r < R ? r : 0;
      uint64_t sp = shfl64(src[0], rs & 31);
      float sj = kInt8 ? __shfl_sync(0xFFFFFFFFu, sc[0], rs & 31) : 0.f;
      if constexpr (kWide) {
        const uint64_t sp1 = shfl64(src[kRows - 1], rs & 31);
        const float sj1 = kInt8 ? __shfl_sync(0xFFFFFFFFu, sc[kRows - 1], rs & 31) : 0.f;
        if (rs >= 32) {
          sp = sp1;
          sj = sj1;
        }
      }
      ok[j] = f < per_tok && sp != 0;
      v[j] = ok[j] ? ld_stream_16(reinterpret_cast<const uint8_t*>(sp) + c * 16) : make_uint4(0, 0, 0, 0);
      s_[j] = sj;
    }
    if (f0 == 0) after_first();
#pragma unroll
    for (int j = 0; j < kWarpItems; ++j) {
      const int f = f0 + j * 32 + lane;
      if (f < per_tok) {
        if constexpr (kInt8) {
          uint4 o0 = make_uint4(0, 0, 0, 0), o1 = make_uint4(0, 0, 0, 0);
          if (ok[j]) dequant16(v[j], s_[j], o0, o1);
          dst[2 * f] = o0;
          dst[2 * f + 1] = o1;
        } else {
          dst[f] = v[j];
        }
      }
    }
  }
}

// The token's projected window (lane i: x'_{t-i}) from the lanes holding it.
__device__ __forceinline__ void window_broadcast(int32_t x, int N, uint32_t (&xp)[kMaxN]) {
#pragma unroll
  for (int i = 0; i < kMaxN; ++i)
    if (i < N) xp[i] = static_cast<uint32_t>(__shfl_sync(0xFFFFFFFFu, x, i));
}

}  // namespace ga
}  // namespace engram
