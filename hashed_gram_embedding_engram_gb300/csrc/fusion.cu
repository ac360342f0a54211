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
//   conv_kernel       one thread per (token, 8 channels): the v rows of the W
//                     taps (rows a token shares with its neighbours' taps come
//                     from L1/L2), the ring history before a chunk, the scalar
//                     rows and H are all loaded together; taps (times g_c) in
//                     registers, compile-time dilation for w = 4 (the pages'
//                     conv); SiLU, the skip and H += Y for every branch.
//   state_kernel      after the chunk: writes RMSNorm(v~) before its weight
//                     (s * v) of the last (w-1)*dilation positions into the
//                     ring, rolls the last N-1 projected ids, advances pos (a
//                     separate launch: the ring slots it writes are slots the
//                     conv still reads).  The ring values are the same float
//                     products the conv forms inside a chunk, so streaming a
//                     sequence reproduces one-shot prefill bit for bit.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "engram_internal.h"

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

// logistic function; __frcp_rn is the correctly rounded reciprocal (same value as 1.f / x)
__device__ __forceinline__ float sigmoidf(float x) { return __frcp_rn(1.f + expf(-x)); }

// SiLU(x) = x * sigma(x) = x / (1 + e^-x), with the fast exponential and divide
__device__ __forceinline__ float silu_fast(float x) { return __fdividef(x, 1.f + __expf(-x)); }

// s and alpha from the four sums of one (token, branch), into the token's sa row
__device__ __forceinline__ void gate_scalars(float sv, float dot, float sk, float sh, float inv_d, float inv_sqrt_d,
                                             float eps, float* sa_row, int M, int m) {
  const float rh = 1.f / sqrtf(sh * inv_d + eps);
  const float rk = 1.f / sqrtf(sk * inv_d + eps);
  const float alpha = sigmoidf(dot * rh * rk * inv_sqrt_d);
  sa_row[m] = alpha * (1.f / sqrtf(alpha * alpha * (sv * inv_d) + eps));
  sa_row[M + m] = alpha;
}

// ------------------------------------------------------------------ gate (bf16 layers: from partials)
__global__ void __launch_bounds__(256) finalize_kernel(const float* __restrict__ part, int n_sl, int64_t ntok, int M,
                                                       int d, float eps, float* __restrict__ sa, int saw) {
  const int lane = threadIdx.x & 31;
  const int P = n_sl * (1 + 3 * M);
  const float inv_d = 1.f / static_cast<float>(d);
  const float inv_sqrt_d = 1.f / sqrtf(static_cast<float>(d));
  const int64_t n_warps = static_cast<int64_t>(gridDim.x) * (blockDim.x >> 5);
  for (int64_t tok = static_cast<int64_t>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5); tok < ntok;
       tok += n_warps) {
    const float* p = part + tok * P;
    float sv = 0.f;
    for (int j = lane; j < n_sl; j += 32) sv += p[j];
    sv = warp_sum(sv);
    for (int m = 0; m < M; ++m) {
      float dot = 0.f, sk = 0.f, sh = 0.f;
      for (int j = lane; j < n_sl; j += 32) {
        const float* q = p + n_sl + (m * n_sl + j) * 3;
        dot += q[0];
        sk += q[1];
        sh += q[2];
      }
      dot = warp_sum(dot);
      sk = warp_sum(sk);
      sh = warp_sum(sh);
      if (lane == 0) gate_scalars(sv, dot, sk, sh, inv_d, inv_sqrt_d, eps, sa + tok * saw, M, m);
    }
  }
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
struct ConvArgs {
  int64_t sv;            // row stride of v (elements)
  int B, Tn, M, d, dil;
  int saw;               // floats per sa row
  const float* g_c;      // [d]
  const float* conv;     // [d, W]
  const int32_t* pos;    // [B] (with a ring)
  int L;
};

// 8 channels of H as floats (16-byte bf16 / 2 x 16-byte fp32 accesses)
template <typename T>
struct H8;
template <>
struct H8<__nv_bfloat16> {
  __device__ static void load(const __nv_bfloat16* p, float* out) {
    const uint4 u = *reinterpret_cast<const uint4*>(p);
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      out[2 * i] = __uint_as_float(w[i] << 16);
      out[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
    }
  }
  __device__ static void store(__nv_bfloat16* p, const float* in) {
    uint32_t w[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      __nv_bfloat162 v = __floats2bfloat162_rn(in[2 * i], in[2 * i + 1]);
      w[i] = *reinterpret_cast<uint32_t*>(&v);
    }
    *reinterpret_cast<uint4*>(p) = make_uint4(w[0], w[1], w[2], w[3]);
  }
};
template <>
struct H8<float> {
  __device__ static void load(const float* p, float* out) {
    ld4(p, out);
    ld4(p + 4, out + 4);
  }
  __device__ static void store(float* p, const float* in) {
    *reinterpret_cast<float4*>(p) = make_float4(in[0], in[1], in[2], in[3]);
    *reinterpret_cast<float4*>(p + 4) = make_float4(in[4], in[5], in[6], in[7]);
  }
};

// One thread per (token, 8 channels): grid x = token, grid y = block of 256
// channel groups.  Every load a thread needs -- the v rows of its W taps (the
// rows a token shares with its neighbours' taps come from L1/L2), the ring
// history before a chunk, the scalars of the tap positions, H -- is
// independent of the others and issued together.  DIL > 0: compile-time
// dilation (the pages' w = 4, dilation = N); DIL = 0: a.dil.
template <typename TH, int W, int DIL>
__global__ void __launch_bounds__(256, 3) conv_kernel(const ConvArgs a, const float* __restrict__ v,
                                                   const float* __restrict__ sa, const float* __restrict__ ring,
                                                   TH* __restrict__ H) {
  const int g = blockIdx.y * blockDim.x + threadIdx.x;
  if (g >= a.d / 8) return;
  const int dil = DIL > 0 ? DIL : a.dil;
  const int64_t tok = blockIdx.x;
  const int b = static_cast<int>(static_cast<uint32_t>(blockIdx.x) / static_cast<uint32_t>(a.Tn));
  const int t = static_cast<int>(blockIdx.x) - b * a.Tn;
  const int M = a.M, d = a.d, c = 8 * g, saw = a.saw;
  float vt[W][8];                                   // v rows of the tap positions inside the chunk
#pragma unroll
  for (int j = 0; j < W; ++j) {
    const int lag = (W - 1 - j) * dil;
    if (t - lag >= 0) {
      const float* vp = v + (tok - lag) * a.sv + c;
      ld4(vp, vt[j]);
      ld4(vp + 4, vt[j] + 4);
    } else {
#pragma unroll
      for (int i = 0; i < 8; ++i) vt[j][i] = 0.f;
    }
  }
  float wq[8][W];                                   // taps times the RMSNorm weight g_c
  {
    float gc[8];
    ld4(a.g_c + c, gc);
    ld4(a.g_c + c + 4, gc + 4);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      if constexpr (W == 4) {
        ld4(a.conv + static_cast<int64_t>(c + i) * W, wq[i]);
      } else {
#pragma unroll
        for (int j = 0; j < W; ++j) wq[i][j] = __ldg(a.conv + static_cast<int64_t>(c + i) * W + j);
      }
#pragma unroll
      for (int j = 0; j < W; ++j) wq[i][j] *= gc[i];
    }
  }
  const int p0 = ring != nullptr ? a.pos[b] : 0;
  TH* hp = H + tok * M * static_cast<int64_t>(d) + c;
  for (int m = 0; m < M; ++m) {
    float h[8];
    H8<TH>::load(hp + static_cast<int64_t>(m) * d, h);
    float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int j = 0; j < W; ++j) {
      const int lag = (W - 1 - j) * dil;
      if (t - lag >= 0) {
        const float sj = __ldg(sa + (tok - lag) * saw + m);
#pragma unroll
        for (int i = 0; i < 8; ++i) acc[i] = fmaf(wq[i][j], sj * vt[j][i], acc[i]);
      } else if (ring != nullptr && p0 + t - lag >= 0) {
        float u[8];                                 // the ring holds RMSNorm(v~) before its weight
        const float* rp = ring + ((static_cast<int64_t>(b) * a.L + (p0 + t - lag) % a.L) * M + m) * d + c;
        ld4(rp, u);
        ld4(rp + 4, u + 4);
#pragma unroll
        for (int i = 0; i < 8; ++i) acc[i] = fmaf(wq[i][j], u[i], acc[i]);
      }
    }
    const float at = __ldg(sa + tok * saw + M + m);
#pragma unroll
    for (int i = 0; i < 8; ++i) h[i] += silu_fast(acc[i]) + at * vt[W - 1][i];
    H8<TH>::store(hp + static_cast<int64_t>(m) * d, h);
  }
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

template <typename TH, int W, int DIL>
cudaError_t conv_launch(const engram_plan* p, ConvArgs a, const float* v, int64_t sv, const float* sa,
                        const float* ring, void* H, cudaStream_t s) {
  (void)p;
  a.sv = sv;
  const int groups = a.d / 8;
  const dim3 grid(static_cast<unsigned>(a.B) * static_cast<unsigned>(a.Tn), (groups + 255) / 256);
  conv_kernel<TH, W, DIL><<<grid, 256, 0, s>>>(a, v, sa, ring, static_cast<TH*>(H));
  return cudaGetLastError();
}

template <typename TH>
cudaError_t conv_dispatch(const engram_plan* p, const ConvArgs& a, const float* v, int64_t sv, const float* sa,
                          const float* ring, void* H, cudaStream_t s) {
  if (p->cfg.conv_w == 4) {
    switch (a.dil) {   // the pages' short conv: w = 4, dilation = max n-gram order
      case 1: return conv_launch<TH, 4, 1>(p, a, v, sv, sa, ring, H, s);
      case 2: return conv_launch<TH, 4, 2>(p, a, v, sv, sa, ring, H, s);
      case 3: return conv_launch<TH, 4, 3>(p, a, v, sv, sa, ring, H, s);
      case 4: return conv_launch<TH, 4, 4>(p, a, v, sv, sa, ring, H, s);
      case 5: return conv_launch<TH, 4, 5>(p, a, v, sv, sa, ring, H, s);
      case 6: return conv_launch<TH, 4, 6>(p, a, v, sv, sa, ring, H, s);
      case 7: return conv_launch<TH, 4, 7>(p, a, v, sv, sa, ring, H, s);
      case 8: return conv_launch<TH, 4, 8>(p, a, v, sv, sa, ring, H, s);
      default: break;
    }
  }
  switch (p->cfg.conv_w) {
    case 1: return conv_launch<TH, 1, 0>(p, a, v, sv, sa, ring, H, s);
    case 2: return conv_launch<TH, 2, 0>(p, a, v, sv, sa, ring, H, s);
    case 3: return conv_launch<TH, 3, 0>(p, a, v, sv, sa, ring, H, s);
    case 4: return conv_launch<TH, 4, 0>(p, a, v, sv, sa, ring, H, s);
    case 5: return conv_launch<TH, 5, 0>(p, a, v, sv, sa, ring, H, s);
    case 6: return conv_launch<TH, 6, 0>(p, a, v, sv, sa, ring, H, s);
    case 7: return conv_launch<TH, 7, 0>(p, a, v, sv, sa, ring, H, s);
    case 8: return conv_launch<TH, 8, 0>(p, a, v, sv, sa, ring, H, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

int sa_row_floats(int M) { return (2 * M + 3) / 4 * 4; }

cudaError_t launch_finalize(const engram_plan* p, const float* part, int n_sl, int64_t ntok, float* sa,
                            cudaStream_t s) {
  finalize_kernel<<<grid_for(ntok * 32, 256, p->num_sms), 256, 0, s>>>(part, n_sl, ntok, p->cfg.M, p->cfg.d,
                                                                       p->cfg.eps, sa, sa_row_floats(p->cfg.M));
  return cudaGetLastError();
}

cudaError_t launch_gate_f32(const engram_plan* p, const float* kv, const float* H, int64_t ntok, const float* g_h,
                            const float* g_k, float* sa, cudaStream_t s) {
  gate_kernel<<<grid_for(ntok * 32, 256, p->num_sms), 256, 0, s>>>(kv, H, ntok, p->cfg.M, p->cfg.d, p->cfg.eps, g_h,
                                                                   g_k, sa, sa_row_floats(p->cfg.M));
  return cudaGetLastError();
}

cudaError_t launch_conv_residual(const engram_plan* p, const float* v, int64_t sv, const float* sa, int B, int T,
                                 const float* g_c, const float* conv, void* H, const engram_state_t* state,
                                 cudaStream_t s) {
  ConvArgs a{};
  a.B = B;
  a.Tn = T;
  a.M = p->cfg.M;
  a.d = p->cfg.d;
  a.dil = p->cfg.conv_dilation;
  a.saw = sa_row_floats(p->cfg.M);
  a.g_c = g_c;
  a.conv = conv;
  a.pos = state ? state->pos : nullptr;
  a.L = p->L_ring;
  const float* ring = state ? state->u_ring : nullptr;
  if (p->cfg.act_dtype == ENGRAM_F32) return conv_dispatch<float>(p, a, v, sv, sa, ring, H, s);
  return conv_dispatch<__nv_bfloat16>(p, a, v, sv, sa, ring, H, s);
}

cudaError_t launch_state_update(const engram_plan* p, const int32_t* ids, const int32_t* proj, int V, const float* v,
                                int64_t sv, const float* sa, int B, int T, const engram_state_t* st,
                                cudaStream_t s) {
  state_kernel<<<B, 256, 0, s>>>(v, sv, sa, sa_row_floats(p->cfg.M), T, p->cfg.M, p->cfg.d, st->u_ring, st->pos,
                                 p->L_ring, ids, proj, V, st->prev_ids, p->cfg.N, &p->dev->err);
  return cudaGetLastError();
}

}  // namespace engram
