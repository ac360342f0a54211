// Steps 1-3 for one index, shared by the standalone hash kernel and the fused
// hash + gather kernel (one definition, so both produce the same indices).
//
//   x'_{t-i} = P[x_{t-i}]  (pad 0 before the sequence start, or the caller's
//                           rolling ids when continuing a sequence)
//   h = XOR_{i<n} (x'_{t-i} * m_{n,k,i})  mod 2^64;   z = h mod p_{n,k}
//
// "DeepSeek Engram 系列导读", section "Engram 工作原理", Stage A, Steps 1-3.
//
// The 64-by-32-bit remainder uses Barrett reduction (P. Barrett, "Implementing
// the RSA public key encryption algorithm on a standard digital signal
// processor", CRYPTO 1986) with mu = floor((2^64-1)/p):
//   q = floor(h * mu / 2^64) is floor(h/p) or one less,
// so r = h - q*p lies in [0, 2p) and one conditional subtraction finishes.
// Proof: mu >= 2^64/p - 1 gives h*mu/2^64 > h/p - 1 (as h < 2^64), and
// mu <= 2^64/p gives h*mu/2^64 <= h/p.
#pragma once

#include "engram_internal.h"

namespace engram {

__device__ __forceinline__ uint32_t barrett_mod(uint64_t h, uint32_t p, uint64_t mu) {
  const uint64_t q = __umul64hi(h, mu);
  uint64_t r = h - q * static_cast<uint64_t>(p);
  if (r >= p) r -= p;
  return static_cast<uint32_t>(r);
}

// Index of head r (order n = 2 + r/K, head k = r%K) at position t of sequence b.
// Raw ids outside [0, V) are read as 0 and reported through `bad`.
__device__ __forceinline__ uint32_t hash_index(const PlanDev& pd, const int32_t* __restrict__ ids, int T, int b,
                                               int t, int r, const int32_t* __restrict__ proj, int V,
                                               const int32_t* __restrict__ prev, bool& bad) {
  const int N = pd.N, K = pd.K;
  const int n = 2 + r / K;
  const int k = r - (n - 2) * K;
  const uint64_t* m = pd.mults + pd.mult_base[n] + k * n;
  uint64_t h = 0;
  for (int i = 0; i < n; ++i) {
    const int tt = t - i;
    int64_t x = 0;                                   // pad id before the sequence start
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
    h ^= static_cast<uint64_t>(x) * m[i];
  }
  return barrett_mod(h, pd.primes[r], pd.mu[r]);
}

}  // namespace engram
