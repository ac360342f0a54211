// Steps 6-8 of "DeepSeek Engram 系列导读", section "Engram 工作原理", Stage B,
// and the per-branch gate of its section "多分支 backbone 上的变体":
//   alpha^(m)_t = sigma(RMSNorm(h^(m)_t) . RMSNorm(k^(m)_t) / sqrt(d)),  v~^(m)_t = alpha^(m)_t v_t
//   Y^(m) = SiLU(Conv1D_{w, dilation}(RMSNorm(V~^(m)))) + V~^(m),       H^(m) <- H^(m) + Y^(m)
//
// RMSNorm(v~) = s * v * g_c with the per-(token, branch) scale
//   s = alpha * rinv,  rinv = 1/sqrt(alpha^2 mean(v^2) + eps),
// so after the gate the convolution needs only the v rows and two scalars
// (alpha for the skip term, s for the normalised input).  They are kept as one
// row per token, sa[t] = [s^(1..M), alpha^(1..M), pad] of saw = 4*ceil(2M/4)
// floats: 16-byte rows that a TMA copy can move.
//
//   finalize_kernel   bf16 layers: one warp per token turns the gate partial
//                     sums written by the K/V GEMM's epilogue (gemm.cu) into
//                     the token's sa row.
//   gate_kernel       fp32 layers: one warp per token computes the sa row from
//                     the fp32 [v | k] buffer of the CUDA-core GEMM.
//   conv_kernel       persistent blocks over tiles of (positions, channels):
//                     TMA stages each tile's v rows (with the causal halo), H
//                     rows and sa rows in a two-stage shared-memory ring; a
//                     thread takes chains of 4 outputs a dilation apart, whose
//                     taps cover 7 rows; taps (times g_c) in registers,
//                     compile-time dilation for w = 4 (the pages' conv); SiLU,
//                     the skip and H += Y for every branch.
//   state_kernel      after the chunk: writes RMSNorm(v~) before its weight
//                     (s * v) of the last (w-1)*dilation positions into the
//                     ring, rolls the last N-1 projected ids, advances pos (a
//                     separate launch: the ring slots it writes are slots the
//                     conv still reads).  The ring values are the same float
//                     products the conv forms inside a chunk, so streaming a
//                     sequence reproduces one-shot prefill bit for bit.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>

#include "engram_internal.h"
#include "gate.cuh"
#include "ptx.cuh"

namespace engram {
namespace {

__device__ __forceinline__ void ld4(const float* p, float* out) {
  const float4 u = *reinterpret_cast<const float4*>(p);
  out[0] = u.x;
  out[1] = u.y;
  out[2] = u.z;
  out[3] = u.w;
}

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xFFFFFFFFu, x, o);
  return x;
}

// SiLU(x) = x * sigma(x) = x / (1 + e^-x), with the fast exponential and divide
__device__ __forceinline__ float silu_fast(float x) { return __fdividef(x, 1.f + __expf(-x)); }

// Two fp32 lanes per instruction (sm_100 family): each lane is rounded exactly
// as the scalar instruction would round it.
__device__ __forceinline__ void fma2(float& d0, float& d1, float a0, float a1, float b0, float b1, float c0, float c1) {
  asm("{\n\t.reg .b64 a, b, c, d;\n\tmov.b64 a, {%2, %3};\n\tmov.b64 b, {%4, %5};\n\tmov.b64 c, {%6, %7};\n\t"
      "fma.rn.f32x2 d, a, b, c;\n\tmov.b64 {%0, %1}, d;\n\t}"
      : "=f"(d0), "=f"(d1)
      : "f"(a0), "f"(a1), "f"(b0), "f"(b1), "f"(c0), "f"(c1));
}
__device__ __forceinline__ void mul2(float& d0, float& d1, float a0, float a1, float b0, float b1) {
  asm("{\n\t.reg .b64 a, b, d;\n\tmov.b64 a, {%2, %3};\n\tmov.b64 b, {%4, %5};\n\t"
      "mul.rn.f32x2 d, a, b;\n\tmov.b64 {%0, %1}, d;\n\t}"
      : "=f"(d0), "=f"(d1)
      : "f"(a0), "f"(a1), "f"(b0), "f"(b1));
}
__device__ __forceinline__ void add2(float& d0, float& d1, float a0, float a1, float b0, float b1) {
  asm("{\n\t.reg .b64 a, b, d;\n\tmov.b64 a, {%2, %3};\n\tmov.b64 b, {%4, %5};\n\t"
      "add.rn.f32x2 d, a, b;\n\tmov.b64 {%0, %1}, d;\n\t}"
      : "=f"(d0), "=f"(d1)
      : "f"(a0), "f"(a1), "f"(b0), "f"(b1));
}

// ------------------------------------------------------------------ gate (bf16 layers: from partials)
// Sum over a warp of the n values p[i * stride], i < n, as the adjacent
// pairwise tree: lane l sums its aligned block [l*q, l*q + q) pairwise (zeros
// past n), then the butterfly pairs lanes at distances 1, 2, ..., 16.  With
// q a power of two the result is the tree sum over the values zero-padded to
// a power of two, whatever q is -- so slices that are themselves pairwise
// sums of aligned 32-column chunks (gemm.cu) give the same bits for every
// GEMM tile width.  Every lane returns the same value.
__device__ __forceinline__ float pairwise_warp_sum(const float* p, int stride, int n, int q, int lane) {
  float x;
  if (q == 1) {
    x = lane < n ? __ldg(p + static_cast<int64_t>(lane) * stride) : 0.f;
  } else {
    float stk[12];
    int top = 0;
    for (int i = 0; i < q; ++i) {
      const int j = lane * q + i;
      float y = j < n ? __ldg(p + static_cast<int64_t>(j) * stride) : 0.f;
      for (int k = i; k & 1; k >>= 1) y = stk[--top] + y;
      stk[top++] = y;
    }
    x = stk[0];
  }
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) x += __shfl_xor_sync(0xFFFFFFFFu, x, o);
  return x;
}

// One warp per token: part[0, n_sl) = sum v^2 nodes, part[n_sl + (m*n_sl + j)*3
// + {0,1,2}] = (h.g_h.g_k.k, k^2, h^2) nodes of branch m -> the sa row.  Up to
// 32 nodes (one per lane) the four sums of a branch are loaded together.
// One token's gate scalars from its partials, by one warp (lane 0 writes out[]).
__device__ __forceinline__ void gate_row(const float* p, int n_sl, int q, int M, float inv_d, float inv_sqrt_d,
                                         float eps, int lane, float* out) {
  if (q == 1) {
    const bool has = lane < n_sl;
    float sv = has ? __ldg(p + lane) : 0.f;
    for (int m = 0; m < M; ++m) {
      const float* pm = p + n_sl + (m * n_sl + lane) * 3;
      float dot = has ? __ldg(pm) : 0.f;
      float sk = has ? __ldg(pm + 1) : 0.f;
      float sh = has ? __ldg(pm + 2) : 0.f;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        if (m == 0) sv += __shfl_xor_sync(0xFFFFFFFFu, sv, o);
        dot += __shfl_xor_sync(0xFFFFFFFFu, dot, o);
        sk += __shfl_xor_sync(0xFFFFFFFFu, sk, o);
        sh += __shfl_xor_sync(0xFFFFFFFFu, sh, o);
      }
      if (lane == 0) gate_scalars(sv, dot, sk, sh, inv_d, inv_sqrt_d, eps, out, M, m);
    }
  } else {
    const float sv = pairwise_warp_sum(p, 1, n_sl, q, lane);
    for (int m = 0; m < M; ++m) {
      const float* pm = p + n_sl + m * n_sl * 3;
      const float dot = pairwise_warp_sum(pm, 3, n_sl, q, lane);
      const float sk = pairwise_warp_sum(pm + 1, 3, n_sl, q, lane);
      const float sh = pairwise_warp_sum(pm + 2, 3, n_sl, q, lane);
      if (lane == 0) gate_scalars(sv, dot, sk, sh, inv_d, inv_sqrt_d, eps, out, M, m);
    }
  }
}

__device__ __forceinline__ int nodes_per_lane(int n_sl) {
  int q = 1;
  while (q * 32 < n_sl) q <<= 1;
  return q;
}

__global__ void __launch_bounds__(256) finalize_kernel(const float* __restrict__ part, int n_sl, int pstride,
                                                       int64_t ntok, int M, int d, float eps, float* __restrict__ sa,
                                                       int saw) {
  ptx::grid_dep_wait();
  ptx::grid_dep_launch();
  const int lane = threadIdx.x & 31;
  const float inv_d = 1.f / static_cast<float>(d);
  const float inv_sqrt_d = 1.f / sqrtf(static_cast<float>(d));
  const int q = nodes_per_lane(n_sl);
  const int64_t n_warps = static_cast<int64_t>(gridDim.x) * (blockDim.x >> 5);
  for (int64_t tok = static_cast<int64_t>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5); tok < ntok;
       tok += n_warps)
    gate_row(part + tok * pstride, n_sl, q, M, inv_d, inv_sqrt_d, eps, lane, sa + tok * saw);
}

// ------------------------------------------------------------------ gate (fp32 layers)
__global__ void __launch_bounds__(256) gate_kernel(const float* __restrict__ kv, const float* __restrict__ H,
                                                   int64_t ntok, int M, int d, float eps,
                                                   const float* __restrict__ g_h, const float* __restrict__ g_k,
                                                   float* __restrict__ sa, int saw) {
  const int lane = threadIdx.x & 31;
  const int64_t warps = static_cast<int64_t>(gridDim.x) * (blockDim.x >> 5);
  const float inv_d = 1.f / static_cast<float>(d);
  const float inv_sqrt_d = 1.f / sqrtf(static_cast<float>(d));
  for (int64_t tok = static_cast<int64_t>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5); tok < ntok;
       tok += warps) {
    const float* row = kv + tok * static_cast<int64_t>(M + 1) * d;   // [v | k^(1) | ... | k^(M)]
    float sv = 0.f;
    for (int c = lane * 4; c < d; c += 128) {
      float v[4];
      ld4(row + c, v);
#pragma unroll
      for (int i = 0; i < 4; ++i) sv = fmaf(v[i], v[i], sv);
    }
    sv = warp_sum(sv);
    for (int m = 0; m < M; ++m) {
      const float* k = row + static_cast<int64_t>(1 + m) * d;
      const float* h = H + (tok * M + m) * static_cast<int64_t>(d);
      const float* gh = g_h + static_cast<int64_t>(m) * d;
      const float* gk = g_k + static_cast<int64_t>(m) * d;
      float sh = 0.f, sk = 0.f, dot = 0.f;
      for (int c = lane * 4; c < d; c += 128) {
        float hv[4], kk[4], ga[4], gb[4];
        ld4(h + c, hv);
        ld4(k + c, kk);
        ld4(gh + c, ga);
        ld4(gk + c, gb);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          sh = fmaf(hv[i], hv[i], sh);
          sk = fmaf(kk[i], kk[i], sk);
          dot = fmaf(hv[i] * (ga[i] * gb[i]), kk[i], dot);
        }
      }
      sh = warp_sum(sh);
      sk = warp_sum(sk);
      dot = warp_sum(dot);
      if (lane == 0) gate_scalars(sv, dot, sk, sh, inv_d, inv_sqrt_d, eps, sa + tok * saw, M, m);
    }
  }
}

// ------------------------------------------------------------------ conv + SiLU + skip + residual
constexpr int kConvThreads = 448;                 // compute threads (14 warps); one producer warp more
constexpr int kChain = 4;                          // outputs per thread, a dilation apart
constexpr int kConvStages = 3;
constexpr uint64_t kConvWaitNs = 1000000000ull;   // 1 s: a healthy tile lands in microseconds
constexpr int kConvMaxCS = 256;                    // channels per tile: one TMA box row (<= 256 elements)

// n / d for 0 <= n < 2^31 as one widening multiply and a shift: with
// 2^l >= d and s = 31 + l, m = ceil(2^s / d) fits in 32 bits and
// floor(n * m / 2^s) = floor(n / d), since n * (m - 2^s/d) / 2^s < 2^-l <= 1/d
// (the round-up method of Granlund & Montgomery, "Division by invariant
// integers using multiplication", PLDI 1994).
struct FastDiv {
  uint32_t mul, sh;
  __device__ __forceinline__ uint32_t div(uint32_t n) const {
    return static_cast<uint32_t>((static_cast<uint64_t>(n) * mul) >> sh);
  }
};

FastDiv make_fastdiv(uint32_t d) {
  uint32_t l = 0;
  while ((1ull << l) < d) ++l;
  const uint32_t sh = 31 + l;
  return FastDiv{static_cast<uint32_t>(((1ull << sh) + d - 1) / d), sh};
}

struct ConvArgs {
  FastDiv div_ct, div_tps;   // by n_ct and by tiles_per_seq
  int B, Tn, M, d, dil;
  int S;                 // positions per tile
  int CS;                // channels per tile
  int h0;                // staged rows before a tile's first position: (w-1)*dil, or 0 if a sequence is one tile
  int tiles_per_seq, n_ct, n_tiles;
  int saw;               // floats per sa row
  uint32_t v_off, h_off, sa_off, p_off, stage_bytes, tx_bytes;   // shared-memory layout of one stage
  float* sa_out;         // gate scalars computed in-kernel (KFIN), for the streaming state; or null
  float eps;
  const float* g_c;      // [d]
  const float* conv;     // [d, W]
  const float* ring;     // [B, L, M, d] or null
  const int32_t* pos;    // [B] (with a ring)
  int L;
  uint32_t* err;
};

// 4 channels of H as floats
template <typename T>
struct H4;
template <>
struct H4<__nv_bfloat16> {
  __device__ static void load(const __nv_bfloat16* p, float* out) {
    const uint2 u = *reinterpret_cast<const uint2*>(p);
    out[0] = __uint_as_float(u.x << 16);
    out[1] = __uint_as_float(u.x & 0xFFFF0000u);
    out[2] = __uint_as_float(u.y << 16);
    out[3] = __uint_as_float(u.y & 0xFFFF0000u);
  }
  __device__ static void store(__nv_bfloat16* p, const float* in) {
    __nv_bfloat162 a = __floats2bfloat162_rn(in[0], in[1]);
    __nv_bfloat162 b = __floats2bfloat162_rn(in[2], in[3]);
    *reinterpret_cast<uint2*>(p) = make_uint2(*reinterpret_cast<uint32_t*>(&a), *reinterpret_cast<uint32_t*>(&b));
  }
};
template <>
struct H4<float> {
  __device__ static void load(const float* p, float* out) { ld4(p, out); }
  __device__ static void store(float* p, const float* in) {
    *reinterpret_cast<float4*>(p) = make_float4(in[0], in[1], in[2], in[3]);
  }
};

// Persistent blocks over tiles of (S positions of one sequence, CS channels).
// Each tile's inputs are staged in shared memory by three TMA copies -- the v
// rows of its positions and of the (w-1)*dilation positions before them, the
// H rows of every branch, the sa rows [s^(1..M), alpha^(1..M)] -- in a ring of
// kConvStages stages.  A producer warp refills a stage as soon as all compute
// warps have released it (an "empty" mbarrier), and each compute warp moves
// on to the next tile on its own, so no block-wide barrier separates tiles.
// Rows before a sequence's start (negative coordinates, zero-filled by the
// copy engine, or the previous sequence's rows) are never used: those taps
// come from the caller's ring (RMSNorm(v~) before its weight) or are zero.
// Compute threads map to (4 channels, every npar-th chain of kChain outputs a
// dilation apart, rotated from tile to tile): the kChain + w - 1 rows a
// chain's taps cover are read from shared memory once and scaled once; taps
// (times g_c) in registers; SiLU, the skip and H += Y for every branch,
// stored straight to H.
// DIL > 0: compile-time dilation (the pages' w = 4, dilation = N); DIL = 0: a.dil.
// KFIN: the block also turns the K/V epilogue's gate partial sums into the
// (s, alpha) rows itself (8 slices per quantity, one branch): the producer's
// third copy brings each staged position's 32 partials (128-byte rows,
// 128-byte swizzle) instead of an sa row, and a helper warp -- one row per
// lane, the finalize kernel's tree and arithmetic -- writes the stage's sa
// rows and releases them through sa_ready, one tile ahead of the compute warps.
template <typename TH, int W, int DIL, int MC, int CSC, bool KFIN>
__global__ void __launch_bounds__(kConvThreads + (KFIN ? 64 : 32), 1)
    conv_kernel(const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_h,
                const __grid_constant__ CUtensorMap tm_sa, const ConvArgs a, TH* __restrict__ H) {
  constexpr int kRows = kChain + W - 1;
  constexpr int kWarps = kConvThreads / 32;          // compute warps
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  __shared__ uint64_t full[kConvStages], empty[kConvStages], sa_ready[kConvStages];
  __shared__ int s_abort;
  const int dil = DIL > 0 ? DIL : a.dil;
  const int M = MC > 0 ? MC : a.M;
  const int tid = threadIdx.x;

  auto coords = [&](int tile, int& b, int& t0, int& c0) {
    const int q = static_cast<int>(a.div_ct.div(static_cast<uint32_t>(tile)));
    const int ct = tile - q * a.n_ct;
    b = static_cast<int>(a.div_tps.div(static_cast<uint32_t>(q)));
    t0 = (q - b * a.tiles_per_seq) * a.S;
    c0 = ct * a.CS;
  };

  if (tid == 0) {
    for (int st = 0; st < kConvStages; ++st) {
      ptx::mbar_init(&full[st], 1);
      ptx::mbar_init(&empty[st], kWarps);
      ptx::mbar_init(&sa_ready[st], 1);
    }
    s_abort = 0;
    ptx::fence_mbar_init();
  }
  __syncthreads();
  ptx::grid_dep_wait();
  ptx::grid_dep_launch();

  if constexpr (KFIN) {
    if (tid >= kConvThreads + 32) {
      // ---------------------------------------------------------------- helper warp: gate scalars
      const int lane = tid & 31;
      const float inv_d = 1.f / static_cast<float>(a.d);
      const float inv_sqrt_d = 1.f / sqrtf(static_cast<float>(a.d));
      const int rows = a.S + a.h0;
      int k = 0;
      for (int tile = blockIdx.x; tile < a.n_tiles; tile += gridDim.x, ++k) {
        const int st = k % kConvStages;
        if (!ptx::mbar_wait_bounded(&full[st], static_cast<uint32_t>(k / kConvStages) & 1u, kConvWaitNs)) {
          if (lane == 0) atomicOr(a.err, kErrTimeout);
          break;
        }
        if (*reinterpret_cast<volatile int*>(&s_abort)) break;
        const uint8_t* pp = smem + st * a.stage_bytes + a.p_off;       // [rows][32 floats], 128-byte swizzle
        float* sa_s = reinterpret_cast<float*>(smem + st * a.stage_bytes + a.sa_off);
        int b, t0, c0;
        coords(tile, b, t0, c0);
        for (int r = lane; r < rows; r += 32) {
          float x[32];
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            const float4 q = *reinterpret_cast<const float4*>(pp + r * 128 + ((j ^ (r & 7)) << 4));
            x[4 * j] = q.x;
            x[4 * j + 1] = q.y;
            x[4 * j + 2] = q.z;
            x[4 * j + 3] = q.w;
          }
          float sv[8], dt[8], sk[8], sh[8];
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            sv[i] = x[i];
            dt[i] = x[8 + 3 * i];
            sk[i] = x[9 + 3 * i];
            sh[i] = x[10 + 3 * i];
          }
#pragma unroll
          for (int w = 1; w < 8; w *= 2)
#pragma unroll
            for (int i = 0; i + w < 8; i += 2 * w) {
              sv[i] = sv[i] + sv[i + w];
              dt[i] = dt[i] + dt[i + w];
              sk[i] = sk[i] + sk[i + w];
              sh[i] = sh[i] + sh[i + w];
            }
          float out[2];
          gate_scalars(sv[0], dt[0], sk[0], sh[0], inv_d, inv_sqrt_d, a.eps, out, 1, 0);
          sa_s[r * 4] = out[0];
          sa_s[r * 4 + 1] = out[1];
          const int t = t0 - a.h0 + r;
          if (a.sa_out != nullptr && c0 == 0 && r >= a.h0 && t < a.Tn) {
            float* g = a.sa_out + (static_cast<int64_t>(b) * a.Tn + t) * 4;
            g[0] = out[0];
            g[1] = out[1];
          }
        }
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(&sa_ready[st]);
      }
      return;
    }
  }

  if (tid >= kConvThreads) {
    // ---------------------------------------------------------------- producer warp
    if (tid == kConvThreads) {
      ptx::tma_prefetch_desc(&tm_v);
      ptx::tma_prefetch_desc(&tm_h);
      ptx::tma_prefetch_desc(&tm_sa);
      uint32_t armed = 0;                            // stages with a copy issued and not yet seen complete
      int k = 0;
      for (int tile = blockIdx.x; tile < a.n_tiles; tile += gridDim.x, ++k) {
        const int st = k % kConvStages;
        const uint32_t round = static_cast<uint32_t>(k / kConvStages);
        if (round > 0 && !ptx::mbar_wait_bounded(&empty[st], (round - 1) & 1u, kConvWaitNs)) {
          atomicOr(a.err, kErrTimeout);
          *reinterpret_cast<volatile int*>(&s_abort) = 1;
          break;
        }
        int b, t0, c0;
        coords(tile, b, t0, c0);
        const int32_t row0 = b * a.Tn + t0 - a.h0;   // may be negative: zero fill
        uint8_t* base = smem + st * a.stage_bytes;
        ptx::mbar_arrive_expect_tx(&full[st], a.tx_bytes);
        ptx::tma_load_2d_nohint(base + a.v_off, &tm_v, &full[st], c0, row0);
        ptx::tma_load_2d_nohint(base + a.h_off, &tm_h, &full[st], c0, (b * a.Tn + t0) * M);
        ptx::tma_load_2d_nohint(base + (KFIN ? a.p_off : a.sa_off), &tm_sa, &full[st], 0, row0);
        armed |= 1u << st;
      }
      // copies still in flight land before the block may exit
      const int issued = k;
      for (int j = issued - kConvStages; j < issued; ++j) {
        if (j < 0) continue;
        const int st = j % kConvStages;
        if (armed & (1u << st)) ptx::mbar_wait_bounded(&full[st], static_cast<uint32_t>(j / kConvStages) & 1u,
                                                       kConvWaitNs);
      }
    }
    return;
  }

  // -------------------------------------------------------------------- compute warps
  const int lane = tid & 31;
  const int CS = CSC > 0 ? CSC : a.CS;            // channels per tile (compile-time on the common shape)
  const int saw = MC == 1 ? 4 : a.saw;             // floats per sa row
  const int ng = CS >> 2;                          // channel groups of a tile
  const int npar = kConvThreads / ng;              // chains processed side by side
  const int g = tid % ng, par0 = tid / ng;
  int c_cached = -1;
  float wq[4][W];                                  // taps times g_c for channels c .. c+3
  auto load_taps = [&](int c) {
    float gc[4];
    ld4(a.g_c + c, gc);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
#pragma unroll
      for (int j = 0; j < W; ++j) wq[i][j] = __ldg(a.conv + static_cast<int64_t>(c + i) * W + j) * gc[i];
    }
    c_cached = c;
  };
  if (blockIdx.x < static_cast<unsigned>(a.n_tiles) && par0 < npar) {
    // the first tile's taps, while its copies are in flight
    int b, t0, c0;
    coords(blockIdx.x, b, t0, c0);
    load_taps(c0 + 4 * g);
  }
  int k = 0;
  int rot = par0;                                  // this tile's first chain: rotates by one per tile
  for (int tile = blockIdx.x; tile < a.n_tiles; tile += gridDim.x, ++k) {
    const int st = k % kConvStages;
    if (!ptx::mbar_wait_bounded(&full[st], static_cast<uint32_t>(k / kConvStages) & 1u, kConvWaitNs)) {
      if (lane == 0) atomicOr(a.err, kErrTimeout);
      break;
    }
    if constexpr (KFIN) {
      if (!ptx::mbar_wait_bounded(&sa_ready[st], static_cast<uint32_t>(k / kConvStages) & 1u, kConvWaitNs)) {
        if (lane == 0) atomicOr(a.err, kErrTimeout);
        break;
      }
    }
    if (*reinterpret_cast<volatile int*>(&s_abort)) break;
    int b, t0, c0;
    coords(tile, b, t0, c0);
    const int nt = min(a.S, a.Tn - t0);
    const uint8_t* base = smem + st * a.stage_bytes;
    const float* vs = reinterpret_cast<const float*>(base + a.v_off);    // [S + h0][CS], row r: position t0 - h0 + r
    const TH* hs = reinterpret_cast<const TH*>(base + a.h_off);          // [S * M][CS]
    const float* ss = reinterpret_cast<const float*>(base + a.sa_off);   // [S + h0][saw]
    if (par0 < npar) {
      const int c = c0 + 4 * g;
      if (c != c_cached) load_taps(c);
      const int p0 = a.ring != nullptr ? a.pos[b] : 0;
      const int rstride = dil * CS;                    // floats between tap rows in the staged v
      const int64_t hrow = static_cast<int64_t>(M) * a.d;                 // elements per position of H
      TH* const hbase = H + (static_cast<int64_t>(b) * a.Tn + t0) * hrow + c;   // position t0, branch 0
      // chains of kChain outputs a dilation apart: first output tb = q*kChain*dil + rr
      const int n_chains = (nt + kChain * dil - 1) / (kChain * dil) * dil;
      for (int ch = rot; ch < n_chains; ch += npar) {
        const int tb = (ch / dil) * (kChain * dil) + ch % dil;
        if (tb >= nt) continue;
        if (t0 + tb - (W - 1) * dil >= 0 && tb + (kChain - 1) * dil < nt) {
          // interior chain: every row staged, every output in the tile -- no branches, all loads first
          const int r0 = a.h0 + tb - (W - 1) * dil;
          const float* vp = vs + r0 * CS + 4 * g;
          const float* sp = ss + r0 * saw;
          float vr[kRows][4];
#pragma unroll
          for (int j = 0; j < kRows; ++j) ld4(vp + j * rstride, vr[j]);
          for (int m = 0; m < M; ++m) {
            float u[kRows][4], h[kChain][4], at[kChain];
#pragma unroll
            for (int o = 0; o < kChain; ++o) {
              H4<TH>::load(hs + ((tb + o * dil) * M + m) * CS + 4 * g, h[o]);
              at[o] = sp[(o + W - 1) * dil * saw + M + m];
            }
#pragma unroll
            for (int j = 0; j < kRows; ++j) {
              const float sj = sp[j * dil * saw + m];
              mul2(u[j][0], u[j][1], sj, sj, vr[j][0], vr[j][1]);
              mul2(u[j][2], u[j][3], sj, sj, vr[j][2], vr[j][3]);
            }
#pragma unroll
            for (int o = 0; o < kChain; ++o) {
              float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
              for (int j = 0; j < W; ++j) {
                fma2(acc[0], acc[1], wq[0][j], wq[1][j], u[o + j][0], u[o + j][1], acc[0], acc[1]);
                fma2(acc[2], acc[3], wq[2][j], wq[3][j], u[o + j][2], u[o + j][3], acc[2], acc[3]);
              }
              float y[4];
#pragma unroll
              for (int i = 0; i < 4; ++i) y[i] = silu_fast(acc[i]);
              fma2(y[0], y[1], at[o], at[o], vr[o + W - 1][0], vr[o + W - 1][1], y[0], y[1]);
              fma2(y[2], y[3], at[o], at[o], vr[o + W - 1][2], vr[o + W - 1][3], y[2], y[3]);
              add2(h[o][0], h[o][1], h[o][0], h[o][1], y[0], y[1]);
              add2(h[o][2], h[o][3], h[o][2], h[o][3], y[2], y[3]);
            }
            TH* hp = hbase + static_cast<int64_t>(tb) * hrow + static_cast<int64_t>(m) * a.d;
#pragma unroll
            for (int o = 0; o < kChain; ++o) H4<TH>::store(hp + static_cast<int64_t>(o * dil) * hrow, h[o]);
          }
          continue;
        }
        float vr[kRows][4];                           // v of rows tb + (j - (W-1))*dil, tile-relative
#pragma unroll
        for (int j = 0; j < kRows; ++j) {
          const int tr = tb + (j - (W - 1)) * dil;
          if (t0 + tr >= 0 && tr < nt) {
            ld4(vs + (a.h0 + tr) * CS + 4 * g, vr[j]);
          } else {
#pragma unroll
            for (int i = 0; i < 4; ++i) vr[j][i] = 0.f;
          }
        }
        for (int m = 0; m < M; ++m) {
          float u[kRows][4];                          // conv input RMSNorm(v~) before g_c: s * v, or the ring
#pragma unroll
          for (int j = 0; j < kRows; ++j) {
            const int tr = tb + (j - (W - 1)) * dil;
            if (tr >= nt) {
#pragma unroll
              for (int i = 0; i < 4; ++i) u[j][i] = 0.f;
            } else if (t0 + tr >= 0) {
              const float sj = ss[(a.h0 + tr) * saw + m];
#pragma unroll
              for (int i = 0; i < 4; ++i) u[j][i] = sj * vr[j][i];
            } else if (a.ring != nullptr && p0 + t0 + tr >= 0) {
              ld4(a.ring + ((static_cast<int64_t>(b) * a.L + (p0 + t0 + tr) % a.L) * M + m) * a.d + c, u[j]);
            } else {
#pragma unroll
              for (int i = 0; i < 4; ++i) u[j][i] = 0.f;
            }
          }
#pragma unroll
          for (int o = 0; o < kChain; ++o) {
            const int tt = tb + o * dil;
            if (tt >= nt) break;
            float h[4];
            H4<TH>::load(hs + (tt * M + m) * CS + 4 * g, h);
            const float at = ss[(a.h0 + tt) * saw + M + m];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              float acc = 0.f;
#pragma unroll
              for (int j = 0; j < W; ++j) acc = fmaf(wq[i][j], u[o + j][i], acc);
              h[i] = h[i] + fmaf(at, vr[o + W - 1][i], silu_fast(acc));
            }
            H4<TH>::store(H + ((static_cast<int64_t>(b) * a.Tn + t0 + tt) * M + m) * a.d + c, h);
          }
        }
      }
    }
    __syncwarp();
    if (lane == 0) ptx::mbar_arrive(&empty[st]);    // this warp is done with the stage
    if (++rot == npar) rot = 0;
  }
}

// ------------------------------------------------------------------ one-position decode step
// Steps 6-8 and the streaming state for chunks of one position (decode), in
// one launch: block b is sequence b.  Warp 0 turns the token's gate partials
// into (s, alpha) (gate_row, the finalize kernel's arithmetic; fp32 layers
// read the gate kernel's sa row); every thread forms its 4 channels' conv
// from the caller's ring (the taps at lag > 0) and s * v (lag 0) with the
// conv kernel's operation order, updates H, then writes s * v into the slot
// of the new position -- the slot its own tap at lag (w-1)*dilation just read,
// so no other thread touches it.  Thread 0 then rolls the projected ids and
// advances pos.  The result equals finalize + conv + state bit for bit.
template <typename TH, int W, bool kPart>
__global__ void __launch_bounds__(256) decode_tail_kernel(
    const float* __restrict__ gate_in, int n_sl, int pstride, int saw, float eps, const float* __restrict__ v,
    int64_t sv, int M, int d, int dil, const float* __restrict__ g_c, const float* __restrict__ conv,
    float* __restrict__ ring, int32_t* __restrict__ pos, int L, const int32_t* __restrict__ ids,
    const int32_t* __restrict__ proj, int V, int32_t* __restrict__ prev, int N, float* __restrict__ sa_out,
    uint32_t* __restrict__ err, TH* __restrict__ H) {
  __shared__ float s_sa[2 * kMaxM];
  __shared__ int s_p0;
  ptx::grid_dep_wait();
  ptx::grid_dep_launch();
  const int b = blockIdx.x;
  const int lane = threadIdx.x & 31;
  if (threadIdx.x < 32) {
    if constexpr (kPart) {
      gate_row(gate_in + static_cast<int64_t>(b) * pstride, n_sl, nodes_per_lane(n_sl), M,
               1.f / static_cast<float>(d), 1.f / sqrtf(static_cast<float>(d)), eps, lane, s_sa);
    } else if (lane < 2 * M) {
      s_sa[lane] = gate_in[static_cast<int64_t>(b) * saw + lane];
    }
    if (lane == 0) s_p0 = ring != nullptr ? pos[b] : 0;
  }
  __syncthreads();
  if (sa_out != nullptr && threadIdx.x < 2 * M) sa_out[static_cast<int64_t>(b) * saw + threadIdx.x] = s_sa[threadIdx.x];
  const int p0 = s_p0;
  for (int g = threadIdx.x; g < d / 4; g += blockDim.x) {
    const int c = 4 * g;
    float wq[4][W];
    {
      float gc[4];
      ld4(g_c + c, gc);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
#pragma unroll
        for (int j = 0; j < W; ++j) wq[i][j] = __ldg(conv + static_cast<int64_t>(c + i) * W + j) * gc[i];
      }
    }
    float vt[4];
    ld4(v + static_cast<int64_t>(b) * sv + c, vt);
    for (int m = 0; m < M; ++m) {
      const float sm = s_sa[m];
      float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int j = 0; j < W; ++j) {
        const int lag = (W - 1 - j) * dil;
        if (lag == 0) {
#pragma unroll
          for (int i = 0; i < 4; ++i) acc[i] = fmaf(wq[i][j], sm * vt[i], acc[i]);
        } else if (ring != nullptr && p0 - lag >= 0) {
          float u[4];                                 // the ring holds RMSNorm(v~) before its weight
          ld4(ring + ((static_cast<int64_t>(b) * L + (p0 - lag) % L) * M + m) * d + c, u);
#pragma unroll
          for (int i = 0; i < 4; ++i) acc[i] = fmaf(wq[i][j], u[i], acc[i]);
        }
      }
      TH* hp = H + (static_cast<int64_t>(b) * M + m) * d + c;
      float h[4];
      H4<TH>::load(hp, h);
      const float at = s_sa[M + m];
#pragma unroll
      for (int i = 0; i < 4; ++i) h[i] = h[i] + fmaf(at, vt[i], silu_fast(acc[i]));
      H4<TH>::store(hp, h);
      if (ring != nullptr && L > 0) {
        float* dst = ring + ((static_cast<int64_t>(b) * L + p0 % L) * M + m) * d + c;
        *reinterpret_cast<float4*>(dst) = make_float4(sm * vt[0], sm * vt[1], sm * vt[2], sm * vt[3]);
      }
    }
  }
  if (ring == nullptr) return;
  __syncthreads();                                    // every thread has read pos[b]
  if (threadIdx.x == 0) {
    int32_t old[kMaxN];
    for (int j = 0; j < N - 1; ++j) old[j] = prev[static_cast<int64_t>(b) * (N - 1) + j];
    int raw = ids[b];
    bool bad = false;
    if (static_cast<unsigned>(raw) >= static_cast<unsigned>(V)) {
      bad = true;
      raw = 0;
    }
    for (int j = 0; j + 1 < N - 1; ++j) prev[static_cast<int64_t>(b) * (N - 1) + j] = old[j + 1];
    if (N > 1) prev[static_cast<int64_t>(b) * (N - 1) + N - 2] = proj[raw];
    pos[b] = p0 + 1;
    if (bad) atomicOr(err, kErrIndexRange);
  }
}

template <typename TH, bool kPart>
cudaError_t decode_tail_dispatch(int W, dim3 grid, cudaStream_t s, const float* gate_in, int n_sl, int pstride, int saw,
                                 float eps, const float* v, int64_t sv, int M, int d, int dil, const float* g_c,
                                 const float* conv, float* ring, int32_t* pos, int L, const int32_t* ids,
                                 const int32_t* proj, int V, int32_t* prev, int N, float* sa_out, uint32_t* err,
                                 void* H) {
#define ENGRAM_TAIL(Wv)                                                                                               \
  launch_pdl(decode_tail_kernel<TH, Wv, kPart>, grid, dim3(256), 0, s, gate_in, n_sl, pstride, saw, eps, v, sv, M, d, \
             dil, g_c, conv, ring, pos, L, ids, proj, V, prev, N, sa_out, err, static_cast<TH*>(H))
  switch (W) {
    case 1: return ENGRAM_TAIL(1);
    case 2: return ENGRAM_TAIL(2);
    case 3: return ENGRAM_TAIL(3);
    case 4: return ENGRAM_TAIL(4);
    case 5: return ENGRAM_TAIL(5);
    case 6: return ENGRAM_TAIL(6);
    case 7: return ENGRAM_TAIL(7);
    case 8: return ENGRAM_TAIL(8);
    default: return cudaErrorInvalidValue;
  }
#undef ENGRAM_TAIL
}

// ------------------------------------------------------------------ streaming state
__global__ void __launch_bounds__(256) state_kernel(const float* __restrict__ v_base, int64_t sv,
                                                    const float* __restrict__ sa, int saw, int Tn, int M, int d,
                                                    float* __restrict__ ring, int32_t* __restrict__ pos, int L,
                                                    const int32_t* __restrict__ ids,
                                                    const int32_t* __restrict__ proj, int V,
                                                    int32_t* __restrict__ prev, int N, uint32_t* __restrict__ err) {
  const int b = blockIdx.x;
  const int keep = Tn < L ? Tn : L;            // chunk positions that stay in the ring
  const int p0 = pos[b];
  const int groups = d / 4;
  const int items = keep * M * groups;
  for (int it = threadIdx.x; it < items; it += blockDim.x) {
    const int g = it % groups;
    const int m = (it / groups) % M;
    const int t = Tn - keep + it / (groups * M);
    const int64_t tok = static_cast<int64_t>(b) * Tn + t;
    const int c = g * 4;
    float v[4];
    ld4(v_base + tok * sv + c, v);
    const float sc = sa[tok * saw + m];
    float* dst = ring + ((static_cast<int64_t>(b) * L + (p0 + t) % L) * M + m) * d + c;
#pragma unroll
    for (int i = 0; i < 4; ++i) dst[i] = sc * v[i];
  }
  __syncthreads();                              // every thread has read pos[b]
  if (threadIdx.x == 0) {
    int32_t old[kMaxN];
    for (int j = 0; j < N - 1; ++j) old[j] = prev[static_cast<int64_t>(b) * (N - 1) + j];
    bool bad = false;
    for (int j = 0; j < N - 1; ++j) {
      const int i = Tn + j;                     // index in (old ++ chunk)
      int32_t x;
      if (i < N - 1) {
        x = old[i];
      } else {
        int raw = ids[static_cast<int64_t>(b) * Tn + (i - (N - 1))];
        if (static_cast<unsigned>(raw) >= static_cast<unsigned>(V)) {
          bad = true;
          raw = 0;
        }
        x = proj[raw];
      }
      prev[static_cast<int64_t>(b) * (N - 1) + j] = x;
    }
    pos[b] = p0 + Tn;
    if (bad) atomicOr(err, kErrIndexRange);
  }
}

int grid_for(int64_t items, int threads, int num_sms) {
  int64_t blocks = (items + threads - 1) / threads;
  const int64_t cap = static_cast<int64_t>(num_sms) * 16;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  return static_cast<int>(blocks);
}

template <typename TH, int W, int DIL, int MC, int CSC, bool KFIN>
cudaError_t conv_launch_m(const CUtensorMap& tv, const CUtensorMap& th, const CUtensorMap& ts, const ConvArgs& a,
                          int grid, size_t smem, void* H, cudaStream_t s) {
  static size_t attr_bytes = 0;    // per template instance: the dynamic shared memory opted into so far
  if (smem > attr_bytes) {
    const cudaError_t e = cudaFuncSetAttribute(conv_kernel<TH, W, DIL, MC, CSC, KFIN>,
                                               cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    attr_bytes = smem;
  }
  return launch_pdl(conv_kernel<TH, W, DIL, MC, CSC, KFIN>, dim3(grid), dim3(kConvThreads + (KFIN ? 64 : 32)), smem,
                    s, tv, th, ts, a, static_cast<TH*>(H));
}

// single-branch layers with a compile-time dilation get a compile-time M = 1,
// and a compile-time tile width when it is the widest one; the gate scalars
// are computed in the conv (fin) only on that shape
template <typename TH, int W, int DIL>
cudaError_t conv_launch(const CUtensorMap& tv, const CUtensorMap& th, const CUtensorMap& ts, const ConvArgs& a,
                        int grid, size_t smem, void* H, bool fin, cudaStream_t s) {
  if (DIL > 0 && a.M == 1) {
    if (a.CS == kConvMaxCS) {
      if (fin) return conv_launch_m<TH, W, DIL, 1, kConvMaxCS, true>(tv, th, ts, a, grid, smem, H, s);
      return conv_launch_m<TH, W, DIL, 1, kConvMaxCS, false>(tv, th, ts, a, grid, smem, H, s);
    }
    return conv_launch_m<TH, W, DIL, 1, 0, false>(tv, th, ts, a, grid, smem, H, s);
  }
  return conv_launch_m<TH, W, DIL, 0, 0, false>(tv, th, ts, a, grid, smem, H, s);
}

template <typename TH>
cudaError_t conv_dispatch(int conv_w, const CUtensorMap& tv, const CUtensorMap& th, const CUtensorMap& ts,
                          const ConvArgs& a, int grid, size_t smem, void* H, bool fin, cudaStream_t s) {
#define ENGRAM_CONV(Wv, Dv) conv_launch<TH, Wv, Dv>(tv, th, ts, a, grid, smem, H, fin && (Dv) > 0 && (Wv) == 4, s)
  if (conv_w == 4) {
    switch (a.dil) {   // the pages' short conv: w = 4, dilation = max n-gram order
      case 1: return ENGRAM_CONV(4, 1);
      case 2: return ENGRAM_CONV(4, 2);
      case 3: return ENGRAM_CONV(4, 3);
      case 4: return ENGRAM_CONV(4, 4);
      case 5: return ENGRAM_CONV(4, 5);
      case 6: return ENGRAM_CONV(4, 6);
      case 7: return ENGRAM_CONV(4, 7);
      case 8: return ENGRAM_CONV(4, 8);
      default: break;
    }
  }
  switch (conv_w) {
    case 1: return ENGRAM_CONV(1, 0);
    case 2: return ENGRAM_CONV(2, 0);
    case 3: return ENGRAM_CONV(3, 0);
    case 4: return ENGRAM_CONV(4, 0);
    case 5: return ENGRAM_CONV(5, 0);
    case 6: return ENGRAM_CONV(6, 0);
    case 7: return ENGRAM_CONV(7, 0);
    case 8: return ENGRAM_CONV(8, 0);
    default: return cudaErrorInvalidValue;
  }
#undef ENGRAM_CONV
}

uint32_t round128(uint32_t x) { return (x + 127u) & ~127u; }

// Shared-memory layout of one stage for a tile of S positions and CS channels.
// With fin, a 1024-byte aligned region of 128-byte partial rows follows (the
// 128-byte swizzle pattern repeats every 1024 bytes) and sa is not copied.
void conv_layout(ConvArgs& a, size_t act_bytes, bool fin) {
  const uint32_t rows = static_cast<uint32_t>(a.S + a.h0);
  const uint32_t vb = rows * a.CS * 4u;
  const uint32_t hb = static_cast<uint32_t>(a.S * a.M * a.CS) * static_cast<uint32_t>(act_bytes);
  const uint32_t sb = rows * static_cast<uint32_t>(a.saw) * 4u;
  a.v_off = 0;
  a.h_off = round128(vb);
  a.sa_off = round128(a.h_off + hb);
  if (fin) {
    a.p_off = (a.sa_off + sb + 1023u) & ~1023u;
    a.stage_bytes = (a.p_off + rows * 128u + 1023u) & ~1023u;
    a.tx_bytes = vb + hb + rows * 128u;
  } else {
    a.p_off = 0;
    a.stage_bytes = round128(a.sa_off + sb);
    a.tx_bytes = vb + hb + sb;
  }
}

}  // namespace

int sa_row_floats(int M) { return (2 * M + 3) / 4 * 4; }

cudaError_t launch_finalize(const engram_plan* p, const float* part, int n_sl, int pstride, int64_t ntok, float* sa,
                            cudaStream_t s) {
  return launch_pdl(finalize_kernel, dim3(grid_for(ntok * 32, 256, p->num_sms)), dim3(256), 0, s, part, n_sl, pstride,
                    ntok, p->cfg.M, p->cfg.d, p->cfg.eps, sa, sa_row_floats(p->cfg.M));
}

cudaError_t launch_gate_f32(const engram_plan* p, const float* kv, const float* H, int64_t ntok, const float* g_h,
                            const float* g_k, float* sa, cudaStream_t s) {
  gate_kernel<<<grid_for(ntok * 32, 256, p->num_sms), 256, 0, s>>>(kv, H, ntok, p->cfg.M, p->cfg.d, p->cfg.eps, g_h,
                                                                   g_k, sa, sa_row_floats(p->cfg.M));
  return cudaGetLastError();
}

bool conv_fuses_gate(const engram_plan* p, int n_sl, int pstride) {
  return p->cfg.act_dtype == ENGRAM_BF16 && p->cfg.M == 1 && p->cfg.conv_w == 4 && p->cfg.conv_dilation >= 1 &&
         p->cfg.conv_dilation <= 8 && n_sl == 8 && pstride == 32 && p->cfg.d % kConvMaxCS == 0;
}

cudaError_t launch_conv_residual(const engram_plan* p, const float* v, int64_t sv, const float* sa, int B, int T,
                                 const float* g_c, const float* conv, void* H, const engram_state_t* state,
                                 cudaStream_t s, const float* part, float* sa_out) {
  ConvArgs a{};
  a.B = B;
  a.Tn = T;
  a.M = p->cfg.M;
  a.d = p->cfg.d;
  a.dil = p->cfg.conv_dilation;
  a.saw = sa_row_floats(p->cfg.M);
  a.g_c = g_c;
  a.conv = conv;
  a.ring = state ? state->u_ring : nullptr;
  a.pos = state ? state->pos : nullptr;
  a.L = p->L_ring;
  a.err = &p->dev->err;
  const bool f32 = p->cfg.act_dtype == ENGRAM_F32;
  const size_t act = f32 ? 4 : 2;
  const int halo = (p->cfg.conv_w - 1) * a.dil;
  const int64_t ntok = static_cast<int64_t>(B) * T;
  if (ntok * a.M > INT32_MAX) return cudaErrorInvalidValue;
  // Tile shape.  Channels per tile CS: the widest (<= 256, dividing d) whose
  // tile keeps at least 2/3 of its staged v rows useful (S / (S + halo)),
  // else the one with the best share; S: at most what kConvStages stages hold
  // (S * M <= 256 and S + halo <= 256: one TMA box each), the whole sequence
  // if it fits.  Among multiples of 4 * dilation (whole chains) up to that
  // bound, S then minimises waves-of-tiles x (S + halo + 8): the staged rows
  // of the slowest block plus a per-tile overhead.
  const bool fin = part != nullptr;
  const int64_t budget = (227 * 1024 - 1024) / kConvStages - 3 * 128 - (fin ? 2048 : 0);
  int S = 0, smax_halo = 0;
  double best = -1.0;
  for (int cs = kConvMaxCS; cs >= (fin ? kConvMaxCS : 4); cs >>= 1) {   // fin: the compile-time 256 only
    if (a.d % cs || (static_cast<size_t>(cs) * act) % 16) continue;
    const int64_t per_row = static_cast<int64_t>(cs) * 4 + a.saw * 4 + (fin ? 128 : 0);   // v, sa (partials)
    const int64_t per_pos = per_row + static_cast<int64_t>(a.M) * cs * static_cast<int64_t>(act);
    const int64_t box_cap = std::min<int64_t>(256 / a.M, 256);
    const int64_t s_no_halo = std::min<int64_t>(budget / per_pos, box_cap);
    const int64_t s_halo = std::min<int64_t>(std::max<int64_t>((budget - halo * per_row) / per_pos, 0),
                                             std::min<int64_t>(box_cap, 256 - halo));
    int sc;
    double score;
    if (T <= s_no_halo) {
      sc = T;
      score = 1.0;
    } else if (s_halo >= 1) {
      sc = static_cast<int>(s_halo);
      score = static_cast<double>(sc) / (sc + halo);
    } else {
      continue;
    }
    if (score > best + 1e-9) {
      best = score;
      a.CS = cs;
      S = sc;
      smax_halo = static_cast<int>(s_halo);
    }
    if (best >= 2.0 / 3.0) break;
  }
  if (S == 0) return cudaErrorInvalidValue;
  a.n_ct = a.d / a.CS;
  {
    const int64_t lanes = static_cast<int64_t>(B) * a.n_ct;
    auto cost = [&](int sc) {
      const int64_t tiles = lanes * ((T + sc - 1) / sc);
      const int64_t waves = (tiles + p->num_sms - 1) / p->num_sms;
      return waves * (sc + (sc < T ? halo : 0) + 8);
    };
    int best_s = S;
    int64_t best_cost = cost(S);
    const int step = 4 * a.dil;
    for (int sc = std::min(smax_halo, T - 1) / step * step; sc >= step; sc -= step) {
      const int64_t c = cost(sc);
      if (c < best_cost) {
        best_cost = c;
        best_s = sc;
      }
    }
    S = best_s;
  }
  a.S = S;
  a.tiles_per_seq = (T + S - 1) / S;
  a.h0 = a.tiles_per_seq > 1 ? halo : 0;
  a.div_ct = make_fastdiv(static_cast<uint32_t>(a.n_ct));
  a.div_tps = make_fastdiv(static_cast<uint32_t>(a.tiles_per_seq));
  const int64_t n_tiles = static_cast<int64_t>(B) * a.tiles_per_seq * a.n_ct;
  if (n_tiles > INT32_MAX) return cudaErrorInvalidValue;
  a.n_tiles = static_cast<int>(n_tiles);
  if (fin && a.CS != kConvMaxCS) return cudaErrorInvalidValue;   // the caller falls back to the finalize kernel
  conv_layout(a, act, fin);
  a.sa_out = sa_out;
  a.eps = p->cfg.eps;
  const size_t smem = static_cast<size_t>(kConvStages) * a.stage_bytes + 1024;
  if (smem > 227 * 1024) return cudaErrorInvalidValue;

  CUtensorMap tv, th, ts;
  if (!make_tensor_map_2d(&tv, v, true, static_cast<uint64_t>(a.d), static_cast<uint64_t>(ntok),
                          static_cast<uint64_t>(sv) * 4, static_cast<uint32_t>(a.CS),
                          static_cast<uint32_t>(a.S + a.h0), false) ||
      !make_tensor_map_2d(&th, H, f32, static_cast<uint64_t>(a.d), static_cast<uint64_t>(ntok * a.M),
                          static_cast<uint64_t>(a.d) * act, static_cast<uint32_t>(a.CS),
                          static_cast<uint32_t>(a.S * a.M), false) ||
      !(fin ? make_tensor_map_2d(&ts, part, true, 32, static_cast<uint64_t>(ntok), 32 * 4, 32,
                                 static_cast<uint32_t>(a.S + a.h0), true)
            : make_tensor_map_2d(&ts, sa, true, static_cast<uint64_t>(a.saw), static_cast<uint64_t>(ntok),
                                 static_cast<uint64_t>(a.saw) * 4, static_cast<uint32_t>(a.saw),
                                 static_cast<uint32_t>(a.S + a.h0), false)))
    return cudaErrorInvalidValue;
  const int grid = static_cast<int>(std::min<int64_t>(a.n_tiles, p->num_sms));
  if (f32) return conv_dispatch<float>(p->cfg.conv_w, tv, th, ts, a, grid, smem, H, false, s);
  return conv_dispatch<__nv_bfloat16>(p->cfg.conv_w, tv, th, ts, a, grid, smem, H, fin, s);
}

cudaError_t launch_decode_tail(const engram_plan* p, const float* v, int64_t sv, const float* sa_in, const float* part,
                               int n_sl, int pstride, float* sa_out, int B, const float* g_c, const float* conv,
                               void* H, const int32_t* ids, const int32_t* proj, int V, const engram_state_t* st,
                               cudaStream_t s) {
  const bool f32 = p->cfg.act_dtype == ENGRAM_F32;
  float* ring = st ? st->u_ring : nullptr;
  int32_t* pos = st ? st->pos : nullptr;
  int32_t* prev = st ? st->prev_ids : nullptr;
  const int saw = sa_row_floats(p->cfg.M);
  const dim3 grid(static_cast<unsigned>(B));
  if (f32)
    return decode_tail_dispatch<float, false>(p->cfg.conv_w, grid, s, sa_in, 0, 0, saw, p->cfg.eps, v, sv, p->cfg.M,
                                              p->cfg.d, p->cfg.conv_dilation, g_c, conv, ring, pos, p->L_ring, ids,
                                              proj, V, prev, p->cfg.N, nullptr, &p->dev->err, H);
  return decode_tail_dispatch<__nv_bfloat16, true>(p->cfg.conv_w, grid, s, part, n_sl, pstride, saw, p->cfg.eps, v,
                                                   sv, p->cfg.M, p->cfg.d, p->cfg.conv_dilation, g_c, conv, ring, pos,
                                                   p->L_ring, ids, proj, V, prev, p->cfg.N, sa_out, &p->dev->err, H);
}

cudaError_t launch_state_update(const engram_plan* p, const int32_t* ids, const int32_t* proj, int V, const float* v,
                                int64_t sv, const float* sa, int B, int T, const engram_state_t* st,
                                cudaStream_t s) {
  state_kernel<<<B, 256, 0, s>>>(v, sv, sa, sa_row_floats(p->cfg.M), T, p->cfg.M, p->cfg.d, st->u_ring, st->pos,
                                 p->L_ring, ids, proj, V, st->prev_ids, p->cfg.N, &p->dev->err);
  return cudaGetLastError();
}

}  // namespace engram
