// Steps 1-3 of "DeepSeek Engram 系列导读", section "Engram 工作原理", Stage A:
// vocabulary projection, suffix n-grams and K multiplicative-XOR hash heads per
// order, fused: one thread produces one index z_{t,n,k}, with the n-gram
// window read straight from the token ids (L1/L2-resident) and never stored.
//
//   h = XOR_{i<n} (x'_{t-i} * m_{n,k,i})  mod 2^64;   z = h mod p_{n,k}
//
// The 64-by-32-bit remainder uses Barrett reduction (P. Barrett, "Implementing
// the RSA public key encryption algorithm on a standard digital signal
// processor", CRYPTO 1986) with mu = floor((2^64-1)/p):
//   q = floor(h * mu / 2^64) satisfies q in {floor(h/p) - 1, floor(h/p)},
// so r = h - q*p lies in [0, 2p) and one conditional subtraction finishes.
// Proof sketch: mu >= 2^64/p - 1, hence h*mu/2^64 > h/p - 1 (h < 2^64), and
// mu <= 2^64/p gives h*mu/2^64 <= h/p.
#include <cuda_runtime.h>

#include "engram_internal.h"

namespace engram {
namespace {

__device__ __forceinline__ uint32_t barrett_mod(uint64_t h, uint32_t p, uint64_t mu) {
  const uint64_t q = __umul64hi(h, mu);
  uint64_t r = h - q * static_cast<uint64_t>(p);
  if (r >= p) r -= p;
  return static_cast<uint32_t>(r);
}

__global__ void __launch_bounds__(256) hash_kernel(const PlanDev* __restrict__ pd, uint32_t* __restrict__ err,
                                                   const int32_t* __restrict__ ids, int B, int T,
                                                   const int32_t* __restrict__ proj, int V,
                                                   const int32_t* __restrict__ prev, int32_t* __restrict__ idx) {
  __shared__ uint64_t s_mult[kMaxMults];
  __shared__ uint64_t s_mu[kMaxR];
  __shared__ uint32_t s_p[kMaxR];
  __shared__ int32_t s_base[kMaxN + 1];
  const int R = pd->R, N = pd->N, K = pd->K;
  const int n_mult = pd->mult_base[N] + K * N;
  for (int i = threadIdx.x; i < n_mult; i += blockDim.x) s_mult[i] = pd->mults[i];
  for (int i = threadIdx.x; i < R; i += blockDim.x) {
    s_mu[i] = pd->mu[i];
    s_p[i] = pd->primes[i];
  }
  if (threadIdx.x <= kMaxN) s_base[threadIdx.x] = pd->mult_base[threadIdx.x];
  __syncthreads();

  const int64_t total = static_cast<int64_t>(B) * T * R;
  bool bad = false;
  for (int64_t f = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; f < total;
       f += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t tok = f / R;
    const int r = static_cast<int>(f - tok * R);
    const int b = static_cast<int>(tok / T);
    const int t = static_cast<int>(tok - static_cast<int64_t>(b) * T);
    const int n = 2 + r / K;
    const int k = r - (n - 2) * K;
    const uint64_t* m = s_mult + s_base[n] + k * n;
    uint64_t h = 0;
    for (int i = 0; i < n; ++i) {
      const int tt = t - i;
      int64_t x = 0;                                   // pad id before the sequence start
      if (tt >= 0) {
        int raw = ids[static_cast<int64_t>(b) * T + tt];
        if (static_cast<unsigned>(raw) >= static_cast<unsigned>(V)) {
          bad = true;
          raw = 0;
        }
        x = proj[raw];
      } else if (prev != nullptr) {
        x = prev[static_cast<int64_t>(b) * (N - 1) + (N - 1) + tt];
      }
      h ^= static_cast<uint64_t>(x) * m[i];
    }
    idx[f] = static_cast<int32_t>(barrett_mod(h, s_p[r], s_mu[r]));
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
  hash_kernel<<<static_cast<int>(blocks), threads, 0, s>>>(p->dev, &p->dev->err, ids, B, T, proj, V, prev_ids, idx);
  return cudaGetLastError();
}

}  // namespace engram
