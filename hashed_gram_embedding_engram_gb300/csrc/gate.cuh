// Gate scalars of Step 6 of "DeepSeek Engram 系列导读" (section "Engram 工作原理"):
//   alpha = sigma(RMSNorm(h) . RMSNorm(k) / sqrt(d)),   v~ = alpha v,
// and the RMSNorm scale of the conv input, RMSNorm(v~) = s * v * g_c with
//   s = alpha / sqrt(alpha^2 mean(v^2) + eps).
// Both follow from four sums over the row: sum v^2, sum h.g_h.g_k.k, sum k^2,
// sum h^2 (the RMSNorm weights g_h, g_k fold into the dot product).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace engram {

// logistic function; __frcp_rn is the correctly rounded reciprocal (same value as 1.f / x)
__device__ __forceinline__ float sigmoidf(float x) { return __frcp_rn(1.f + expf(-x)); }

// s and alpha of branch m from the four sums, into the token's row [s^(1..M), alpha^(1..M)]
__device__ __forceinline__ void gate_scalars(float sv, float dot, float sk, float sh, float inv_d, float inv_sqrt_d,
                                             float eps, float* sa_row, int M, int m) {
  const float rh = 1.f / sqrtf(sh * inv_d + eps);
  const float rk = 1.f / sqrtf(sk * inv_d + eps);
  const float alpha = sigmoidf(dot * rh * rk * inv_sqrt_d);
  sa_row[m] = alpha * (1.f / sqrtf(alpha * alpha * (sv * inv_d) + eps));
  sa_row[M + m] = alpha;
}

// ---- gate scalars of bf16 layers from the K/V epilogue's partial sums
// kNC: the partials were written by an earlier kernel (read through the
// non-coherent path); false: by other blocks of the same launch (read at L2).
template <bool kNC>
__device__ __forceinline__ float ld_part(const float* p) {
  if constexpr (kNC) {
    return __ldg(p);
  } else {
    float v;
    asm volatile("ld.global.cg.f32 %0, [%1];" : "=f"(v) : "l"(p));
    return v;
  }
}

// Sum over a warp of the n values p[i * stride], i < n, as the adjacent
// pairwise tree: lane l sums its aligned block [l*q, l*q + q) pairwise (zeros
// past n), then the butterfly pairs lanes at distances 1, 2, ..., 16.  With
// q a power of two the result is the tree sum over the values zero-padded to
// a power of two, whatever q is -- so slices that are themselves pairwise
// sums of aligned 32-column chunks (gemm.cu) give the same bits for every
// GEMM tile width.  Every lane returns the same value.
template <bool kNC = true>
__device__ __forceinline__ float pairwise_warp_sum(const float* p, int stride, int n, int q, int lane) {
  float x;
  if (q == 1) {
    x = lane < n ? ld_part<kNC>(p + static_cast<int64_t>(lane) * stride) : 0.f;
  } else {
    float stk[12];
    int top = 0;
    for (int i = 0; i < q; ++i) {
      const int j = lane * q + i;
      float y = j < n ? ld_part<kNC>(p + static_cast<int64_t>(j) * stride) : 0.f;
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
template <bool kNC = true>
__device__ __forceinline__ void gate_row(const float* p, int n_sl, int q, int M, float inv_d, float inv_sqrt_d,
                                         float eps, int lane, float* out) {
  if (q == 1) {
    const bool has = lane < n_sl;
    float sv = has ? ld_part<kNC>(p + lane) : 0.f;
    for (int m = 0; m < M; ++m) {
      const float* pm = p + n_sl + (m * n_sl + lane) * 3;
      float dot = has ? ld_part<kNC>(pm) : 0.f;
      float sk = has ? ld_part<kNC>(pm + 1) : 0.f;
      float sh = has ? ld_part<kNC>(pm + 2) : 0.f;
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
    const float sv = pairwise_warp_sum<kNC>(p, 1, n_sl, q, lane);
    for (int m = 0; m < M; ++m) {
      const float* pm = p + n_sl + m * n_sl * 3;
      const float dot = pairwise_warp_sum<kNC>(pm, 3, n_sl, q, lane);
      const float sk = pairwise_warp_sum<kNC>(pm + 1, 3, n_sl, q, lane);
      const float sh = pairwise_warp_sum<kNC>(pm + 2, 3, n_sl, q, lane);
      if (lane == 0) gate_scalars(sv, dot, sk, sh, inv_d, inv_sqrt_d, eps, out, M, m);
    }
  }
}

__device__ __forceinline__ int nodes_per_lane(int n_sl) {
  int q = 1;
  while (q * 32 < n_sl) q <<= 1;
  return q;
}

}  // namespace engram
