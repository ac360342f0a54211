// Gate scalars of Step 6 of "DeepSeek Engram 系列导读" (section "Engram 工作原理"):
//   alpha = sigma(RMSNorm(h) . RMSNorm(k) / sqrt(d)),   v~ = alpha v,
// and the RMSNorm scale of the conv input, RMSNorm(v~) = s * v * g_c with
//   s = alpha / sqrt(alpha^2 mean(v^2) + eps).
// Both follow from four sums over the row: sum v^2, sum h.g_h.g_k.k, sum k^2,
// sum h^2 (the RMSNorm weights g_h, g_k fold into the dot product).
#pragma once

#include <cuda_runtime.h>

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

}  // namespace engram
