// Steps 6-8 of "DeepSeek Engram 系列导读", section "Engram 工作原理", Stage B,
// and the per-branch gate of its section "多分支 backbone 上的变体":
//   alpha^(m)_t = sigma(RMSNorm(h^(m)_t) . RMSNorm(k^(m)_t) / sqrt(d)),  v~^(m)_t = alpha^(m)_t v_t
//   Y^(m) = SiLU(Conv1D_{w, dilation}(RMSNorm(V~^(m)))) + V~^(m),       H^(m) <- H^(m) + Y^(m)
//
// Kernel split (all HBM-bound, fp32 arithmetic):
//   bf16 layers: the K/V GEMM's epilogue (gemm.cu) already reduced every k tile
//   to partial sums and wrote v in fp32.
//     finalize_kernel  one thread per (token, branch): partials -> alpha and
//                      rinv = 1/sqrt(mean((alpha v)^2) + eps).  Since
//                      RMSNorm(v~) = (alpha v) * rinv * g_c, the convolution
//                      needs only v and these two scalars.
//   fp32 layers (CUDA-core GEMM, [v | k] buffer in fp32):
//     gate_kernel      one warp per token: the same scalars from h, k and v.
//   conv_kernel   one thread per (token, 4 channels of H): the
//                 causal dilated taps read v rows at t - j*dilation (rows of
//                 neighbouring tokens, served by L1/L2), the history before a
//                 chunk from the caller's ring, then SiLU, skip and the
//                 residual update of all M branches in place.
//   state_kernel  after the chunk: writes the last (w-1)*dilation conv inputs
//                 into the ring, rolls the last N-1 projected ids, advances pos.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "engram_internal.h"

namespace engram {
namespace {

template <typename T>
struct Vec;   // 16-byte vectors of T widened to float
template <>
struct Vec<__nv_bfloat16> {
  static constexpr int kN = 8;
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
struct Vec<float> {
  static constexpr int kN = 4;
  __device__ static void load(const float* p, float* out) {
    const float4 u = *reinterpret_cast<const float4*>(p);
    out[0] = u.x;
    out[1] = u.y;
    out[2] = u.z;
    out[3] = u.w;
  }
  __device__ static void store(float* p, const float* in) {
    *reinterpret_cast<float4*>(p) = make_float4(in[0], in[1], in[2], in[3]);
  }
};

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xFFFFFFFFu, x, o);
  return x;
}

__device__ __forceinline__ float sigmoidf(float x) { return 1.f / (1.f + expf(-x)); }

// ------------------------------------------------------------------ gate
template <typename T>
__global__ void __launch_bounds__(256) gate_kernel(const T* __restrict__ kv, const T* __restrict__ H, int64_t ntok,
                                                   int M, int d, float eps, const float* __restrict__ g_h,
                                                   const float* __restrict__ g_k, float* __restrict__ alpha,
                                                   float* __restrict__ rinv) {
  constexpr int V = Vec<T>::kN;
  const int lane = threadIdx.x & 31;
  const int64_t warps = static_cast<int64_t>(gridDim.x) * (blockDim.x >> 5);
  const float inv_d = 1.f / static_cast<float>(d);
  const float inv_sqrt_d = 1.f / sqrtf(static_cast<float>(d));
  for (int64_t tok = static_cast<int64_t>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5); tok < ntok;
       tok += warps) {
    const T* row = kv + tok * static_cast<int64_t>(M + 1) * d;   // [v | k^(1) | ... | k^(M)]
    float sv = 0.f;
    for (int c = lane * V; c < d; c += 32 * V) {
      float v[V];
      Vec<T>::load(row + c, v);
#pragma unroll
      for (int i = 0; i < V; ++i) sv = fmaf(v[i], v[i], sv);
    }
    sv = warp_sum(sv);
    const float ms_v = sv * inv_d;
    for (int m = 0; m < M; ++m) {
      const T* k = row + static_cast<int64_t>(1 + m) * d;
      const T* h = H + (tok * M + m) * static_cast<int64_t>(d);
      const float* gh = g_h + static_cast<int64_t>(m) * d;
      const float* gk = g_k + static_cast<int64_t>(m) * d;
      float sh = 0.f, sk = 0.f, dot = 0.f;
      for (int c = lane * V; c < d; c += 32 * V) {
        float hv[V], kv_[V];
        Vec<T>::load(h + c, hv);
        Vec<T>::load(k + c, kv_);
#pragma unroll
        for (int i = 0; i < V; ++i) {
          sh = fmaf(hv[i], hv[i], sh);
          sk = fmaf(kv_[i], kv_[i], sk);
          dot = fmaf(hv[i] * gh[c + i], kv_[i] * gk[c + i], dot);
        }
      }
      sh = warp_sum(sh);
      sk = warp_sum(sk);
      dot = warp_sum(dot);
      const float rh = 1.f / sqrtf(sh * inv_d + eps);
      const float rk = 1.f / sqrtf(sk * inv_d + eps);
      const float a = sigmoidf(dot * rh * rk * inv_sqrt_d);
      if (lane == 0) {
        alpha[tok * M + m] = a;
        rinv[tok * M + m] = 1.f / sqrtf(a * a * ms_v + eps);
      }
    }
  }
}

// ------------------------------------------------------------------ finalize the gate
// partials from the fused GEMM epilogue -> alpha and rinv per (token, branch)
__global__ void __launch_bounds__(256) finalize_kernel(const float* __restrict__ part, int64_t ntok, int M, int d,
                                                       int n_vt, float eps, float* __restrict__ alpha,
                                                       float* __restrict__ rinv) {
  const int P = n_vt * (1 + 3 * M);
  const float inv_d = 1.f / static_cast<float>(d);
  const float inv_sqrt_d = 1.f / sqrtf(static_cast<float>(d));
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < ntok * M;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t tok = i / M;
    const int m = static_cast<int>(i - tok * M);
    const float* p = part + tok * P;
    float sv = 0.f, dot = 0.f, sk = 0.f, sh = 0.f;
    for (int j = 0; j < n_vt; ++j) {
      sv += p[j];
      const float* q = p + n_vt + (m * n_vt + j) * 3;
      dot += q[0];
      sk += q[1];
      sh += q[2];
    }
    const float rh = 1.f / sqrtf(sh * inv_d + eps);
    const float rk = 1.f / sqrtf(sk * inv_d + eps);
    const float a = sigmoidf(dot * rh * rk * inv_sqrt_d);
    alpha[i] = a;
    rinv[i] = 1.f / sqrtf(a * a * (sv * inv_d) + eps);
  }
}

template <int VN>
__device__ __forceinline__ void load_v(const float* p, float* out) {
#pragma unroll
  for (int i = 0; i < VN; i += 4) {
    const float4 q = *reinterpret_cast<const float4*>(p + i);
    out[i] = q.x;
    out[i + 1] = q.y;
    out[i + 2] = q.z;
    out[i + 3] = q.w;
  }
}

// ------------------------------------------------------------------ conv + SiLU + skip + residual
// 4 channels per thread (8-byte bf16 / 16-byte fp32 H accesses), register use
// capped so that 3 blocks of 256 threads stay resident per SM: the kernel is
// latency-bound unless many tokens are in flight.
template <typename T>
struct Vec4;
template <>
struct Vec4<__nv_bfloat16> {
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
struct Vec4<float> {
  __device__ static void load(const float* p, float* out) { Vec<float>::load(p, out); }
  __device__ static void store(float* p, const float* in) { Vec<float>::store(p, in); }
};

// v rows are fp32 with row stride sv (the fused path's v buffer, or the fp32 kv buffer).
template <typename TH, int W>
__global__ void __launch_bounds__(256, 3) conv_kernel(const float* __restrict__ v_base, int64_t sv,
                                                      const float* __restrict__ alpha,
                                                      const float* __restrict__ rinv, int B, int Tn, int M, int d,
                                                      int dil, const float* __restrict__ g_c,
                                                      const float* __restrict__ conv, TH* __restrict__ H,
                                                      const float* __restrict__ ring,
                                                      const int32_t* __restrict__ pos, int L) {
  constexpr int V = 4;
  const int groups = d / V;
  const int64_t total = static_cast<int64_t>(B) * Tn * groups;
  for (int64_t item = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; item < total;
       item += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t tok = item / groups;
    const int c = static_cast<int>(item - tok * groups) * V;
    const int b = static_cast<int>(tok / Tn);
    const int t = static_cast<int>(tok - static_cast<int64_t>(b) * Tn);

    // taps of the 4 channels: conv[c+i][j]
    float w[V][W];
    if constexpr (W == 4) {
#pragma unroll
      for (int i = 0; i < V; ++i) Vec<float>::load(conv + static_cast<int64_t>(c + i) * W, w[i]);
    } else {
#pragma unroll
      for (int i = 0; i < V; ++i)
#pragma unroll
        for (int j = 0; j < W; ++j) w[i][j] = __ldg(conv + static_cast<int64_t>(c + i) * W + j);
    }
    float gc[V];
    Vec<float>::load(g_c + c, gc);
    // v rows at the taps' positions inside this chunk
    float v[W][V];
#pragma unroll
    for (int j = 0; j < W; ++j) {
      const int lag = (W - 1 - j) * dil;
      if (t - lag >= 0) {
        Vec<float>::load(v_base + (tok - lag) * sv + c, v[j]);
      } else {
#pragma unroll
        for (int i = 0; i < V; ++i) v[j][i] = 0.f;
      }
    }
    const int p0 = ring ? pos[b] : 0;
    for (int m = 0; m < M; ++m) {
      float acc[V];
#pragma unroll
      for (int i = 0; i < V; ++i) acc[i] = 0.f;
#pragma unroll
      for (int j = 0; j < W; ++j) {
        const int lag = (W - 1 - j) * dil;
        float u[V];
        if (t - lag >= 0) {
          const int64_t tj = tok - lag;
          const float a = alpha[tj * M + m], ri = rinv[tj * M + m];
#pragma unroll
          for (int i = 0; i < V; ++i) u[i] = ((a * v[j][i]) * ri) * gc[i];
        } else {
          const int abs_pos = p0 + t - lag;
          if (ring != nullptr && abs_pos >= 0) {
            Vec<float>::load(ring + ((static_cast<int64_t>(b) * L + abs_pos % L) * M + m) * d + c, u);
          } else {
#pragma unroll
            for (int i = 0; i < V; ++i) u[i] = 0.f;
          }
        }
#pragma unroll
        for (int i = 0; i < V; ++i) acc[i] = fmaf(w[i][j], u[i], acc[i]);
      }
      const float a_t = alpha[tok * M + m];
      TH* hp = H + (tok * M + m) * static_cast<int64_t>(d) + c;
      float h[V];
      Vec4<TH>::load(hp, h);
#pragma unroll
      for (int i = 0; i < V; ++i) h[i] += acc[i] * sigmoidf(acc[i]) + a_t * v[W - 1][i];
      Vec4<TH>::store(hp, h);
    }
  }
}

// ------------------------------------------------------------------ streaming state
__global__ void __launch_bounds__(256) state_kernel(const float* __restrict__ v_base, int64_t sv,
                                                    const float* __restrict__ alpha, const float* __restrict__ rinv,
                                                    int Tn, int M, int d, const float* __restrict__ g_c,
                                                    float* __restrict__ ring, int32_t* __restrict__ pos, int L,
                                                    const int32_t* __restrict__ ids,
                                                    const int32_t* __restrict__ proj, int V,
                                                    int32_t* __restrict__ prev, int N, uint32_t* __restrict__ err) {
  constexpr int VN = 4;
  const int b = blockIdx.x;
  const int keep = Tn < L ? Tn : L;            // chunk positions that stay in the ring
  const int p0 = pos[b];
  const int groups = d / VN;
  const int items = keep * M * groups;
  for (int it = threadIdx.x; it < items; it += blockDim.x) {
    const int g = it % groups;
    const int m = (it / groups) % M;
    const int t = Tn - keep + it / (groups * M);
    const int64_t tok = static_cast<int64_t>(b) * Tn + t;
    const int c = g * VN;
    float v[VN];
    load_v<VN>(v_base + tok * sv + c, v);
    const float a = alpha[tok * M + m], ri = rinv[tok * M + m];
    float* dst = ring + ((static_cast<int64_t>(b) * L + (p0 + t) % L) * M + m) * d + c;
#pragma unroll
    for (int i = 0; i < VN; ++i) dst[i] = ((a * v[i]) * ri) * g_c[c + i];
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

template <typename TH, int W>
void conv_launch(const engram_plan* p, const float* v, int64_t sv, const float* alpha, const float* rinv, int B,
                 int Tn, const float* g_c, const float* conv, void* H, const engram_state_t* st, cudaStream_t s) {
  const int d = p->cfg.d;
  const int64_t items = static_cast<int64_t>(B) * Tn * (d / 4);
  conv_kernel<TH, W><<<grid_for(items, 256, p->num_sms), 256, 0, s>>>(
      v, sv, alpha, rinv, B, Tn, p->cfg.M, d, p->cfg.conv_dilation, g_c, conv, static_cast<TH*>(H),
      st ? st->u_ring : nullptr, st ? st->pos : nullptr, p->L_ring);
}

template <typename TH>
cudaError_t conv_dispatch(const engram_plan* p, const float* v, int64_t sv, const float* alpha, const float* rinv,
                          int B, int Tn, const float* g_c, const float* conv, void* H, const engram_state_t* st,
                          cudaStream_t s) {
  switch (p->cfg.conv_w) {
    case 1: conv_launch<TH, 1>(p, v, sv, alpha, rinv, B, Tn, g_c, conv, H, st, s); break;
    case 2: conv_launch<TH, 2>(p, v, sv, alpha, rinv, B, Tn, g_c, conv, H, st, s); break;
    case 3: conv_launch<TH, 3>(p, v, sv, alpha, rinv, B, Tn, g_c, conv, H, st, s); break;
    case 4: conv_launch<TH, 4>(p, v, sv, alpha, rinv, B, Tn, g_c, conv, H, st, s); break;
    case 5: conv_launch<TH, 5>(p, v, sv, alpha, rinv, B, Tn, g_c, conv, H, st, s); break;
    case 6: conv_launch<TH, 6>(p, v, sv, alpha, rinv, B, Tn, g_c, conv, H, st, s); break;
    case 7: conv_launch<TH, 7>(p, v, sv, alpha, rinv, B, Tn, g_c, conv, H, st, s); break;
    case 8: conv_launch<TH, 8>(p, v, sv, alpha, rinv, B, Tn, g_c, conv, H, st, s); break;
    default: return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_gate_f32(const engram_plan* p, const float* kv, const float* H, int64_t ntok, const float* g_h,
                            const float* g_k, float* alpha, float* rinv, cudaStream_t s) {
  const int grid = grid_for(ntok * 32, 256, p->num_sms);
  gate_kernel<float><<<grid, 256, 0, s>>>(kv, H, ntok, p->cfg.M, p->cfg.d, p->cfg.eps, g_h, g_k, alpha, rinv);
  return cudaGetLastError();
}

cudaError_t launch_finalize(const engram_plan* p, const float* part, int n_vt, int64_t ntok, float* alpha,
                            float* rinv, cudaStream_t s) {
  finalize_kernel<<<grid_for(ntok * p->cfg.M, 256, p->num_sms), 256, 0, s>>>(part, ntok, p->cfg.M, p->cfg.d, n_vt,
                                                                            p->cfg.eps, alpha, rinv);
  return cudaGetLastError();
}

cudaError_t launch_conv_residual(const engram_plan* p, const float* v, int64_t sv, const float* alpha,
                                 const float* rinv, int B, int T, const float* g_c, const float* conv, void* H,
                                 const engram_state_t* state, cudaStream_t s) {
  if (p->cfg.act_dtype == ENGRAM_F32)
    return conv_dispatch<float>(p, v, sv, alpha, rinv, B, T, g_c, conv, H, state, s);
  return conv_dispatch<__nv_bfloat16>(p, v, sv, alpha, rinv, B, T, g_c, conv, H, state, s);
}

cudaError_t launch_state_update(const engram_plan* p, const int32_t* ids, const int32_t* proj, int V, const float* v,
                                int64_t sv, const float* alpha, const float* rinv, int B, int T, const float* g_c,
                                const engram_state_t* st, cudaStream_t s) {
  state_kernel<<<B, 256, 0, s>>>(v, sv, alpha, rinv, T, p->cfg.M, p->cfg.d, g_c, st->u_ring, st->pos, p->L_ring, ids,
                                 proj, V, st->prev_ids, p->cfg.N, &p->dev->err);
  return cudaGetLastError();
}

}  // namespace engram
