// Steps 6-8 and the streaming state of one sequence at one new position
// (decode), by one block: the body of the decode tail kernel (fusion.cu) and
// of the one-launch decode step (decode.cu), so both give the same bits.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "conv_parts.cuh"
#include "engram_internal.h"
#include "gate.cuh"

namespace engram {
namespace cv {

// Four floats of v: through the non-coherent path when an earlier kernel wrote
// them (kNC), else at L2 (written by other blocks of the same launch).
template <bool kNC>
__device__ __forceinline__ void ld4_v(const float* p, float* out) {
  if constexpr (kNC) {
    ld4(p, out);
  } else {
    asm volatile("ld.global.cg.v4.f32 {%0, %1, %2, %3}, [%4];"
                 : "=f"(out[0]), "=f"(out[1]), "=f"(out[2]), "=f"(out[3])
                 : "l"(p));
  }
}

// What one thread of sequence b's tail loads that no kernel of the step
// writes: the state (pos, the ring rows at lag > 0, the projected ids to roll)
// written by the previous step, the conv taps times g_c and H of its first
// channel group (branch 0).  Only v and the gate partials come from the K/V
// projection, so a tail launched right after it can load all this before its
// dependency wait (a kernel's predecessors other than the immediately
// preceding one have completed before it starts).
// (The projected ids to roll live in a separate array: they are indexed by a
// run-time count, which would move the whole struct to local memory.)
template <int W>
struct TailPre {
  int p0;                  // pos[b] (0 without a ring)
  bool bad_id;             // thread 0: the new raw id is outside [0, V)
  bool pre;                // this thread has a first channel group
  float wq0[4][W], u0[W][4], h0[4];
};

template <typename TH, int W>
__device__ __forceinline__ void decode_tail_pre(TailPre<W>& t, int32_t (&roll)[kMaxN], int b, int tid, int M, int d,
                                                int dil,
                                                const float* __restrict__ g_c, const float* __restrict__ conv,
                                                const float* __restrict__ ring, const int32_t* __restrict__ pos, int L,
                                                const int32_t* __restrict__ ids, const int32_t* __restrict__ proj,
                                                int V, const int32_t* __restrict__ prev, int N,
                                                const TH* __restrict__ H) {
  t.p0 = ring != nullptr ? pos[b] : 0;             // written by thread 0 at the end, after the last barrier
  t.bad_id = false;
  if (tid == 0 && ring != nullptr) {
    for (int j = 0; j + 1 < N - 1; ++j) roll[j] = prev[static_cast<int64_t>(b) * (N - 1) + j + 1];
    int raw = ids[b];
    if (static_cast<unsigned>(raw) >= static_cast<unsigned>(V)) {
      t.bad_id = true;
      raw = 0;
    }
    if (N > 1) roll[N - 2] = proj[raw];
  }
  const int g0 = tid;
  t.pre = g0 < d / 4;
  if (t.pre) {
    const int c = 4 * g0;
    float gc[4];
    ld4(g_c + c, gc);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
#pragma unroll
      for (int j = 0; j < W; ++j) t.wq0[i][j] = __ldg(conv + static_cast<int64_t>(c + i) * W + j) * gc[i];
    }
#pragma unroll
    for (int j = 0; j < W; ++j) {
      const int lag = (W - 1 - j) * dil;
      if (lag > 0 && ring != nullptr && t.p0 - lag >= 0)
        ld4(ring + ((static_cast<int64_t>(b) * L + (t.p0 - lag) % L) * M) * d + c, t.u0[j]);
    }
    H4<TH>::load(H + static_cast<int64_t>(b) * M * d + c, t.h0);
  }
}

// Sequence b, by the block's threads tid < nthr (every thread of the block
// calls it: it synchronises the block), from what decode_tail_pre loaded.
// Warp 0 turns the token's gate partials into (s, alpha) (kPart, gate_row) or
// reads them (fp32 layers: the gate kernel's sa row) into s_sa[2M]; every
// thread forms its 4 channels' conv from the caller's ring (the taps at
// lag > 0) and s * v (lag 0) with the conv kernel's operation order, updates
// H, then writes s * v into the slot of the new position -- the slot its own
// tap at lag (w-1)*dilation just read, so no other thread touches it.
// Thread 0 then rolls the projected ids and advances pos.  Each thread loads
// its first channel group's v before the barrier that publishes the gate, so
// that load overlaps warp 0's gate.  v and gate_in: see ld4_v / ld_part for kNC.
// sync(): a barrier over the nthr threads that run this sequence (the block,
// or a named barrier over part of it when a block runs two sequences at once).
template <typename TH, int W, bool kPart, bool kNC, typename Sync>
__device__ __forceinline__ void decode_tail_main(
    const TailPre<W>& t, const int32_t (&roll)[kMaxN], int b, int tid, int nthr, float* s_sa, const float* gate_in, int n_sl, int pstride,
    int saw, float eps, const float* v, int64_t sv, int M, int d, int dil, const float* __restrict__ g_c,
    const float* __restrict__ conv, float* __restrict__ ring, int32_t* __restrict__ pos, int L,
    int32_t* __restrict__ prev, int N, float* __restrict__ sa_out, uint32_t* __restrict__ err,
    TH* __restrict__ H, Sync&& sync) {
  const int lane = tid & 31;
  const int p0 = t.p0;
  const int g0 = tid;
  float vt0[4];
  if (t.pre) ld4_v<kNC>(v + static_cast<int64_t>(b) * sv + 4 * g0, vt0);
  if (tid < 32) {
    if constexpr (kPart) {
      gate_row<kNC>(gate_in + static_cast<int64_t>(b) * pstride, n_sl, nodes_per_lane(n_sl), M,
               1.f / static_cast<float>(d), 1.f / sqrtf(static_cast<float>(d)), eps, lane, s_sa);
    } else if (lane < 2 * M) {
      s_sa[lane] = gate_in[static_cast<int64_t>(b) * saw + lane];
    }
  }
  sync();
  if (sa_out != nullptr && tid < 2 * M) sa_out[static_cast<int64_t>(b) * saw + tid] = s_sa[tid];
  for (int g = tid; g < d / 4; g += nthr) {
    const int c = 4 * g;
    const bool first = g == g0;                    // its inputs of branch 0 are already in registers
    float wq[4][W];
    float vt[4];
    if (first) {
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        vt[i] = vt0[i];
#pragma unroll
        for (int j = 0; j < W; ++j) wq[i][j] = t.wq0[i][j];
      }
    } else {
      float gc[4];
      ld4(g_c + c, gc);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
#pragma unroll
        for (int j = 0; j < W; ++j) wq[i][j] = __ldg(conv + static_cast<int64_t>(c + i) * W + j) * gc[i];
      }
      ld4_v<kNC>(v + static_cast<int64_t>(b) * sv + c, vt);
    }
    for (int m = 0; m < M; ++m) {
      const float sm = s_sa[m];
      const bool have = first && m == 0;
      float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int j = 0; j < W; ++j) {
        const int lag = (W - 1 - j) * dil;
        if (lag == 0) {
#pragma unroll
          for (int i = 0; i < 4; ++i) acc[i] = fmaf(wq[i][j], sm * vt[i], acc[i]);
        } else if (ring != nullptr && p0 - lag >= 0) {
          float u[4];                                 // the ring holds RMSNorm(v~) before its weight
          if (have) {
#pragma unroll
            for (int i = 0; i < 4; ++i) u[i] = t.u0[j][i];
          } else {
            ld4(ring + ((static_cast<int64_t>(b) * L + (p0 - lag) % L) * M + m) * d + c, u);
          }
#pragma unroll
          for (int i = 0; i < 4; ++i) acc[i] = fmaf(wq[i][j], u[i], acc[i]);
        }
      }
      TH* hp = H + (static_cast<int64_t>(b) * M + m) * d + c;
      float h[4];
      if (have) {
#pragma unroll
        for (int i = 0; i < 4; ++i) h[i] = t.h0[i];
      } else {
        H4<TH>::load(hp, h);
      }
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
  if (ring == nullptr) return;                        // the same for every thread of the sequence
  sync();                                             // every thread has read pos[b]
  if (tid == 0) {
    for (int j = 0; j < N - 1; ++j) prev[static_cast<int64_t>(b) * (N - 1) + j] = roll[j];
    pos[b] = p0 + 1;
    if (t.bad_id) atomicOr(err, kErrIndexRange);
  }
}


// Both parts back to back (the one-launch decode, whose phases are ordered by
// its own counters).
template <typename TH, int W, bool kPart, bool kNC, typename Sync>
__device__ __forceinline__ void decode_tail_seq(
    int b, int tid, int nthr, float* s_sa, const float* gate_in, int n_sl, int pstride, int saw, float eps,
    const float* v, int64_t sv, int M, int d, int dil, const float* __restrict__ g_c,
    const float* __restrict__ conv, float* __restrict__ ring, int32_t* __restrict__ pos, int L,
    const int32_t* __restrict__ ids, const int32_t* __restrict__ proj, int V, int32_t* __restrict__ prev, int N,
    float* __restrict__ sa_out, uint32_t* __restrict__ err, TH* __restrict__ H, Sync&& sync) {
  TailPre<W> t;
  int32_t roll[kMaxN];
  decode_tail_pre<TH, W>(t, roll, b, tid, M, d, dil, g_c, conv, ring, pos, L, ids, proj, V, prev, N, H);
  decode_tail_main<TH, W, kPart, kNC>(t, roll, b, tid, nthr, s_sa, gate_in, n_sl, pstride, saw, eps, v, sv, M, d, dil, g_c,
                                      conv, ring, pos, L, prev, N, sa_out, err, H, static_cast<Sync&&>(sync));
}

}  // namespace cv
}  // namespace engram
