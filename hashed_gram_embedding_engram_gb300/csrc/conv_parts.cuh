// Building blocks of the conv + SiLU + skip + residual (Steps 7-8) over tiles
// staged in shared memory: the per-tile TMA issue, the in-kernel gate
// finalisation of a tile's rows, and the chain computation of one tile by one
// thread.  fusion.cu composes them into the persistent conv kernel; stage_b.cu
// into the kernel that runs the K/V projection and the conv together.  See
// fusion.cu for the design.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "engram_internal.h"
#include "gate.cuh"
#include "ptx.cuh"

namespace engram {
namespace cv {

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
  __host__ __device__ __forceinline__ uint32_t div(uint32_t n) const {
    return static_cast<uint32_t>((static_cast<uint64_t>(n) * mul) >> sh);
  }
};

inline FastDiv make_fastdiv(uint32_t d) {
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


__device__ __forceinline__ void conv_coords(const ConvArgs& a, int tile, int& b, int& t0, int& c0) {
  const int q = static_cast<int>(a.div_ct.div(static_cast<uint32_t>(tile)));
  const int ct = tile - q * a.n_ct;
  b = static_cast<int>(a.div_tps.div(static_cast<uint32_t>(q)));
  t0 = (q - b * a.tiles_per_seq) * a.S;
  c0 = ct * a.CS;
}

// One thread: the first of a tile's three TMA copies into the stage at
// `base` -- its H rows -- after arming the stage's barrier for all three.  H
// is written by no kernel between the previous Stage B and this conv (the
// K/V projection and the gate only read it), so this copy may be issued
// before the dependency wait.
__device__ __forceinline__ void conv_issue_h(const ConvArgs& a, const CUtensorMap* tm_h, uint8_t* base,
                                             uint64_t* full, int tile, int M) {
  int b, t0, c0;
  conv_coords(a, tile, b, t0, c0);
  ptx::mbar_arrive_expect_tx(full, a.tx_bytes);
  ptx::tma_load_2d_nohint(base + a.h_off, tm_h, full, c0, (b * a.Tn + t0) * M);
}

// The other two: v rows with the causal halo and the gate partials (KFIN) or
// sa rows, both written by the kernels just before the conv.
template <bool KFIN>
__device__ __forceinline__ void conv_issue_rest(const ConvArgs& a, const CUtensorMap* tm_v, const CUtensorMap* tm_sa,
                                                uint8_t* base, uint64_t* full, int tile) {
  int b, t0, c0;
  conv_coords(a, tile, b, t0, c0);
  const int32_t row0 = b * a.Tn + t0 - a.h0;       // may be negative: zero fill
  ptx::tma_load_2d_nohint(base + a.v_off, tm_v, full, c0, row0);
  ptx::tma_load_2d_nohint(base + (KFIN ? a.p_off : a.sa_off), tm_sa, full, 0, row0);
}

// One thread: the three TMA copies of a tile into the stage at `base`.
template <bool KFIN>
__device__ __forceinline__ void conv_issue(const ConvArgs& a, const CUtensorMap* tm_v, const CUtensorMap* tm_h,
                                           const CUtensorMap* tm_sa, uint8_t* base, uint64_t* full, int tile, int M) {
  conv_issue_h(a, tm_h, base, full, tile, M);
  conv_issue_rest<KFIN>(a, tm_v, tm_sa, base, full, tile);
}

// One warp: the (s, alpha) rows of a staged tile from its partials (8 slices
// per quantity, one branch), one row per lane, into the stage's sa region.
__device__ __forceinline__ void conv_fin_rows(const ConvArgs& a, const uint8_t* base, int tile, int lane) {
  const float inv_d = 1.f / static_cast<float>(a.d);
  const float inv_sqrt_d = 1.f / sqrtf(static_cast<float>(a.d));
  const int rows = a.S + a.h0;
  const uint8_t* pp = base + a.p_off;             // [rows][32 floats], 128-byte swizzle
  float* sa_s = reinterpret_cast<float*>(const_cast<uint8_t*>(base) + a.sa_off);
  int b, t0, c0;
  conv_coords(a, tile, b, t0, c0);
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
}

// Taps times g_c for channels c .. c+3.
template <int W>
__device__ __forceinline__ void conv_load_taps(const ConvArgs& a, int c, float (&wq)[4][W]) {
  float gc[4];
  ld4(a.g_c + c, gc);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
#pragma unroll
    for (int j = 0; j < W; ++j) wq[i][j] = __ldg(a.conv + static_cast<int64_t>(c + i) * W + j) * gc[i];
  }
}

// One chain of kChain outputs a dilation apart, every row a position of the
// sequence: v rows vp + j * rstride (j = 0 .. kChain + W - 2, lag (W-1-j) * dil
// before the first output), their gate scalars sp + j * sstride (s at m, alpha
// at M + m), H rows hp_s + o * hstride_s in shared memory and hp + o * hstride
// in global memory.  kFull: all kChain outputs; else the first n_out, and the
// rows only the others read are neither loaded nor used.  All loads first.
template <typename TH, int W, bool kFull>
__device__ __forceinline__ void conv_chain(const float* vp, int rstride, const float* sp, int sstride, int saw, int M,
                                           int m, const TH* hp_s, int hstride_s, const float (&wq)[4][W], TH* hp,
                                           int64_t hstride, int n_out) {
  constexpr int kRows = kChain + W - 1;
  (void)saw;
  float vr[kRows][4];
#pragma unroll
  for (int j = 0; j < kRows; ++j) {
    if (kFull || j < n_out + W - 1) {
      ld4(vp + j * rstride, vr[j]);
    } else {
#pragma unroll
      for (int i = 0; i < 4; ++i) vr[j][i] = 0.f;
    }
  }
  float u[kRows][4], h[kChain][4], at[kChain];
#pragma unroll
  for (int o = 0; o < kChain; ++o) {
    if (kFull || o < n_out) {
      H4<TH>::load(hp_s + o * hstride_s, h[o]);
      at[o] = sp[(o + W - 1) * sstride + M + m];
    } else {
#pragma unroll
      for (int i = 0; i < 4; ++i) h[o][i] = 0.f;
      at[o] = 0.f;
    }
  }
#pragma unroll
  for (int j = 0; j < kRows; ++j) {
    const float sj = (kFull || j < n_out + W - 1) ? sp[j * sstride + m] : 0.f;
    mul2(u[j][0], u[j][1], sj, sj, vr[j][0], vr[j][1]);
    mul2(u[j][2], u[j][3], sj, sj, vr[j][2], vr[j][3]);
  }
#pragma unroll
  for (int o = 0; o < kChain; ++o) {
    if (!kFull && o >= n_out) break;
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
#pragma unroll
  for (int o = 0; o < kChain; ++o)
    if (kFull || o < n_out) H4<TH>::store(hp + o * hstride, h[o]);
}

// One thread: the work items rot, rot + npar, ... of the staged tile at
// `base`, channels c = c0 + 4g .. c+3 (taps in wq).  An item is one chain of
// one branch (item = chain * M + branch), so with several branches the chains
// of a tile spread over more threads; a thread reads its chain's v rows from
// shared memory for each item it takes.
template <typename TH, int W, int DIL, int MC, int CSC>
__device__ __forceinline__ void conv_tile(const ConvArgs& a, const uint8_t* base, int tile, int g, int rot, int npar,
                                          const float (&wq)[4][W], TH* __restrict__ H) {
  constexpr int kRows = kChain + W - 1;
  const int dil = DIL > 0 ? DIL : a.dil;
  const int M = MC > 0 ? MC : a.M;
  const int CS = CSC > 0 ? CSC : a.CS;            // channels per tile (compile-time on the common shape)
  const int saw = MC == 1 ? 4 : a.saw;             // floats per sa row
  int b, t0, c0;
  conv_coords(a, tile, b, t0, c0);
  const int nt = min(a.S, a.Tn - t0);
  const float* vs = reinterpret_cast<const float*>(base + a.v_off);    // [S + h0][CS], row r: position t0 - h0 + r
  const TH* hs = reinterpret_cast<const TH*>(base + a.h_off);          // [S * M][CS]
  const float* ss = reinterpret_cast<const float*>(base + a.sa_off);   // [S + h0][saw]
  const int c = c0 + 4 * g;
  const int p0 = a.ring != nullptr ? a.pos[b] : 0;
  const int rstride = dil * CS;                    // floats between tap rows in the staged v
  const int64_t hrow = static_cast<int64_t>(M) * a.d;                 // elements per position of H
  TH* const hbase = H + (static_cast<int64_t>(b) * a.Tn + t0) * hrow + c;   // position t0, branch 0
  // chains of kChain outputs a dilation apart: first output tb = q*kChain*dil + rr
  const int n_chains = (nt + kChain * dil - 1) / (kChain * dil) * dil;
  for (int it = rot; it < n_chains * M; it += npar) {
    const int ch = MC == 1 ? it : it / M;
    const int m = MC == 1 ? 0 : it - ch * M;
    const int tb = (ch / dil) * (kChain * dil) + ch % dil;
    if (tb >= nt) continue;
    // every row the chain reads is a position of the sequence (no ring, no zero rows).  With several
    // branches, whose tiles end inside a chain, a chain that runs past the tile's end also takes
    // this path and computes only its first n_out outputs (same arithmetic); single-branch tiles
    // hold whole chains but for a sequence's last tile, and keep the full-chain form alone.
    const int n_out = min(kChain, (nt - 1 - tb) / dil + 1);
    if (t0 + tb - (W - 1) * dil >= 0 && (MC != 1 || n_out == kChain)) {
      const int r0 = a.h0 + tb - (W - 1) * dil;
      TH* hp = hbase + static_cast<int64_t>(tb) * hrow + static_cast<int64_t>(m) * a.d;
      if (MC == 1 || n_out == kChain)
        conv_chain<TH, W, true>(vs + r0 * CS + 4 * g, rstride, ss + r0 * saw, dil * saw, saw, M, m,
                                hs + (tb * M + m) * CS + 4 * g, dil * M * CS, wq, hp, dil * hrow, kChain);
      else if constexpr (MC != 1)
        conv_chain<TH, W, false>(vs + r0 * CS + 4 * g, rstride, ss + r0 * saw, dil * saw, saw, M, m,
                                 hs + (tb * M + m) * CS + 4 * g, dil * M * CS, wq, hp, dil * hrow, n_out);
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
    {
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

}  // namespace cv
}  // namespace engram
