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

#include "conv_host.h"
#include "conv_parts.cuh"
#include "engram_internal.h"
#include "gate.cuh"
#include "ptx.cuh"
#include "tail_parts.cuh"

namespace engram {
namespace {

using namespace cv;

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
// KFIN: the block also turns the K/V epilogue's gate partial sums into the
// (s, alpha) rows itself (8 slices per quantity, one branch): the producer's
// third copy brings each staged position's 32 partials (128-byte rows,
// 128-byte swizzle) instead of an sa row, and a helper warp -- one row per
// lane, the finalize kernel's tree and arithmetic -- writes the stage's sa
// rows and releases them through sa_ready, one tile ahead of the compute warps.
// DIL > 0: compile-time dilation (the pages' w = 4, dilation = N); DIL = 0: a.dil.
template <typename TH, int W, int DIL, int MC, int CSC, bool KFIN>
__global__ void __launch_bounds__(kConvThreads + (KFIN ? 64 : 32), 1)
    conv_kernel(const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_h,
                const __grid_constant__ CUtensorMap tm_sa, const ConvArgs a, TH* __restrict__ H) {
  constexpr int kWarps = kConvThreads / 32;          // compute warps
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  __shared__ uint64_t full[kConvStages], empty[kConvStages], sa_ready[kConvStages];
  __shared__ int s_abort;
  const int M = MC > 0 ? MC : a.M;
  const int tid = threadIdx.x;

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
  // Only the producer waits for the kernels before this one: every copy of
  // their results (v, the gate partials or sa rows) is issued after its wait,
  // and the other warps read those results, and write H, only after a stage
  // they wait for has landed.  H itself, the state and the weights are
  // written by no kernel of this Stage B.
  ptx::grid_dep_launch();

  if constexpr (KFIN) {
    if (tid >= kConvThreads + 32) {
      // ---------------------------------------------------------------- helper warp: gate scalars
      const int lane = tid & 31;
      int k = 0;
      for (int tile = blockIdx.x; tile < a.n_tiles; tile += gridDim.x, ++k) {
        const int st = k % kConvStages;
        if (!ptx::mbar_wait_bounded(&full[st], static_cast<uint32_t>(k / kConvStages) & 1u, kConvWaitNs)) {
          if (lane == 0) atomicOr(a.err, kErrTimeout);
          break;
        }
        if (*reinterpret_cast<volatile int*>(&s_abort)) break;
        conv_fin_rows(a, smem + st * a.stage_bytes, tile, lane);
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
      // the H rows of the first tiles (one per stage) while the previous kernel finishes
      int n_pre = 0;
      for (int tile = blockIdx.x; tile < a.n_tiles && n_pre < kConvStages; tile += gridDim.x, ++n_pre) {
        conv_issue_h(a, &tm_h, smem + n_pre * a.stage_bytes, &full[n_pre], tile, M);
        armed |= 1u << n_pre;
      }
      ptx::grid_dep_wait();
      int k = 0;
      for (int tile = blockIdx.x; tile < a.n_tiles; tile += gridDim.x, ++k) {
        const int st = k % kConvStages;
        const uint32_t round = static_cast<uint32_t>(k / kConvStages);
        if (k < n_pre) {
          conv_issue_rest<KFIN>(a, &tm_v, &tm_sa, smem + st * a.stage_bytes, &full[st], tile);
          continue;
        }
        if (round > 0 && !ptx::mbar_wait_bounded(&empty[st], (round - 1) & 1u, kConvWaitNs)) {
          atomicOr(a.err, kErrTimeout);
          *reinterpret_cast<volatile int*>(&s_abort) = 1;
          break;
        }
        conv_issue<KFIN>(a, &tm_v, &tm_h, &tm_sa, smem + st * a.stage_bytes, &full[st], tile, M);
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
  const int CS = CSC > 0 ? CSC : a.CS;
  const int ng = CS >> 2;                          // channel groups of a tile
  const int npar = kConvThreads / ng;              // chains processed side by side
  const int g = tid % ng, par0 = tid / ng;
  int c_cached = -1;
  float wq[4][W];                                  // taps times g_c for channels c .. c+3
  if (blockIdx.x < static_cast<unsigned>(a.n_tiles) && par0 < npar) {
    // the first tile's taps, while its copies are in flight
    int b, t0, c0;
    conv_coords(a, blockIdx.x, b, t0, c0);
    c_cached = c0 + 4 * g;
    conv_load_taps<W>(a, c_cached, wq);
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
    if (par0 < npar) {
      int b, t0, c0;
      conv_coords(a, tile, b, t0, c0);
      if (c0 + 4 * g != c_cached) {
        c_cached = c0 + 4 * g;
        conv_load_taps<W>(a, c_cached, wq);
      }
      conv_tile<TH, W, DIL, MC, CSC>(a, smem + st * a.stage_bytes, tile, g, rot, npar, wq, H);
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
// advances pos.  The result equals finalize + conv + state bit for bit.  Each
// thread loads its first channel group's taps, ring rows and H before the
// dependency wait (none of them comes from the K/V projection) and its v
// before the barrier that publishes the gate, so those loads overlap the
// projection's tail and warp 0's gate.  Three blocks fit an SM (80 registers
// a thread): 256 sequences' blocks are all resident beside the projection's
// blocks (64 SMs at decode sizes), so all of them load ahead of the wait.
template <typename TH, int W, bool kPart>
__global__ void __launch_bounds__(256, 3) decode_tail_kernel(
    const float* __restrict__ gate_in, int n_sl, int pstride, int saw, float eps, const float* __restrict__ v,
    int64_t sv, int M, int d, int dil, const float* __restrict__ g_c, const float* __restrict__ conv,
    float* __restrict__ ring, int32_t* __restrict__ pos, int L, const int32_t* __restrict__ ids,
    const int32_t* __restrict__ proj, int V, int32_t* __restrict__ prev, int N, float* __restrict__ sa_out,
    uint32_t* __restrict__ err, TH* __restrict__ H) {
  __shared__ float s_sa[2 * kMaxM];
  // the state, taps and H: written by no kernel of this call (the previous
  // kernel, the K/V projection, writes only v and the partials), so they load
  // while the projection finishes
  TailPre<W> t;
  int32_t roll[kMaxN];
  decode_tail_pre<TH, W>(t, roll, blockIdx.x, threadIdx.x, M, d, dil, g_c, conv, ring, pos, L, ids, proj, V, prev, N,
                         H);
  ptx::grid_dep_wait();
  ptx::grid_dep_launch();
  decode_tail_main<TH, W, kPart, true>(t, roll, blockIdx.x, threadIdx.x, blockDim.x, s_sa, gate_in, n_sl, pstride, saw, eps,
                                       v, sv, M, d, dil, g_c, conv, ring, pos, L, prev, N, sa_out, err, H,
                                       [] { __syncthreads(); });
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
  // four hyper-connection branches (the pages' multi-branch variant) at the pages' w = 4
  if (DIL > 0 && W == 4 && a.M == 4) return conv_launch_m<TH, W, DIL, 4, 0, false>(tv, th, ts, a, grid, smem, H, s);
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
  return launch_pdl(finalize_kernel, dim3(grid_for(ntok * 32, 256, stage_b_sms(p))), dim3(256), 0, s, part, n_sl, pstride,
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

cudaError_t conv_prepare(const engram_plan* p, const float* v, int64_t sv, const float* sa, int B, int T,
                         const float* g_c, const float* conv, void* H, const engram_state_t* state, const float* part,
                         float* sa_out, ConvArgs* out, CUtensorMap* tv_out, CUtensorMap* th_out, CUtensorMap* ts_out,
                         size_t* smem_out, size_t smem_cap) {
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
  const int64_t budget = (static_cast<int64_t>(smem_cap) - 1024) / kConvStages - 3 * 128 - (fin ? 2048 : 0);
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
      const int64_t waves = (tiles + stage_b_sms(p) - 1) / stage_b_sms(p);
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
  if (smem > smem_cap) return cudaErrorInvalidValue;

  CUtensorMap& tv = *tv_out;
  CUtensorMap& th = *th_out;
  CUtensorMap& ts = *ts_out;
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
  *out = a;
  *smem_out = smem;
  return cudaSuccess;
}

cudaError_t launch_conv_residual(const engram_plan* p, const float* v, int64_t sv, const float* sa, int B, int T,
                                 const float* g_c, const float* conv, void* H, const engram_state_t* state,
                                 cudaStream_t s, const float* part, float* sa_out) {
  ConvArgs a;
  CUtensorMap tv, th, ts;
  size_t smem = 0;
  const cudaError_t e =
      conv_prepare(p, v, sv, sa, B, T, g_c, conv, H, state, part, sa_out, &a, &tv, &th, &ts, &smem, 227 * 1024);
  if (e != cudaSuccess) return e;
  const int grid = static_cast<int>(std::min<int64_t>(a.n_tiles, stage_b_sms(p)));
  if (p->cfg.act_dtype == ENGRAM_F32) return conv_dispatch<float>(p->cfg.conv_w, tv, th, ts, a, grid, smem, H, false, s);
  return conv_dispatch<__nv_bfloat16>(p->cfg.conv_w, tv, th, ts, a, grid, smem, H, part != nullptr, s);
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
