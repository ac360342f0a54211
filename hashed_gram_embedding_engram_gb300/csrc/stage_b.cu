// Steps 5-8 of "DeepSeek Engram 系列导读", section "Engram 工作原理", Stage B,
// in ONE cooperative launch for the common bf16 shape (one branch, w = 4,
// 128-column v/k slices): the K/V projection with its fused gate epilogue
// (gemm_parts.cuh) and the conv + SiLU + skip + residual with the in-kernel
// gate finalisation (conv_parts.cuh), linked by a dataflow of row blocks
// instead of a kernel boundary.
//
// Why: the projection has 8 column tiles per 128-row block, 256 tiles in all
// for 4096 tokens -- 1.7 waves over 152 SMs, so in the second wave a third of
// the SMs idle; and a separate conv launch cannot start before the last tile
// is stored.  Here a block that runs out of projection tiles goes straight on
// to conv tiles whose rows are complete.
// Measured on GB300 (4096 tokens, warm, per call): 31.8 us against 26.5 us
// for the two launches.  The cooperative launch starts 3.3 us after the
// counter reset (no overlap with the previous kernel), the projection's tiles
// end 1.6 us later than alone (per-tile store completion and fences before
// each signal), and with 10 compute warps instead of 14 the conv after the
// last projection tile takes as long as the standalone conv; the ~48 blocks
// freed early get through 3-4 conv tiles each, less than those losses.  The
// two-launch form is therefore the default.
//
// One block per SM (all co-resident: a cooperative launch), 12 warps.
//   projection phase: warp 0 TMA producer, warp 1 MMA issuer, warps 2-9 the
//     fused epilogue; after each tile every epilogue warp makes its global
//     writes visible (TMA stores complete, proxy + memory fences) and adds 1
//     to row_done[row block] with release semantics; warps 10-11 idle.
//   block barrier; warp 1 frees TMEM; the operand ring is reused for conv
//     stages.
//   conv phase: warp 10 takes conv tiles from a global queue in row order
//     (atomicAdd), waits (acquire, bounded) until every row block the tile's
//     copies touch has all 8 x 8 epilogue arrivals, then issues the tile's TMA
//     copies into a 3-stage ring; warp 11 turns each staged tile's gate
//     partials into (s, alpha) rows; warps 0-9 compute the chains (5 chains
//     side by side over 64 four-channel groups).  A tile index of -1 in a
//     stage ends the phase.
// A block enters the conv phase only after its own projection tiles, and
// those never wait on conv work, so every wait is on work that resident
// blocks finish by themselves.  The conv writes H rows only of row blocks
// whose projection -- the only reader of H here -- has finished.
//
// The counters (row_done, then the queue head) live in the caller's
// workspace and are zeroed by a one-block kernel launched just before, on
// the same stream.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>

#include "conv_host.h"
#include "conv_parts.cuh"
#include "engram_internal.h"
#include "gemm_parts.cuh"
#include "ptx.cuh"

namespace engram {
namespace {

constexpr int kSbThreads = 384;
constexpr int kSbBN = 256;
constexpr int kSbCompute = 320;                  // conv compute threads: warps 0-9
constexpr int kSbCS = 256;                       // conv channels per tile (compile time)
using G = gk::Cfg<kSbBN, true>;
constexpr size_t kSbGemmBytes = static_cast<size_t>(G::kStages) * G::kStageBytes + G::kEpiBytes;
constexpr size_t kSbStatic = 1024;               // upper bound of the kernel's static shared memory
constexpr size_t kSbSmemCap = 227 * 1024 - kSbStatic;

struct SbSync {
  uint32_t* row_done;    // [m_tiles]
  uint32_t* queue;       // conv tile queue head
  uint32_t target;       // arrivals that complete a row block: 8 x column tiles
  int rows;              // tokens
};

__global__ void sync_zero_kernel(uint32_t* p, int n) {
  ptx::grid_dep_wait();          // the previous user of these counters has finished
  for (int i = threadIdx.x; i < n; i += blockDim.x) p[i] = 0u;
  ptx::grid_dep_launch();
}

// Wait until every row block that tile `tile`'s copies read is complete.
__device__ __forceinline__ bool wait_rows(const cv::ConvArgs& a, const SbSync& sy, int tile) {
  int b, t0, c0;
  cv::conv_coords(a, tile, b, t0, c0);
  const int first = b * a.Tn + t0 - a.h0;
  const int r_lo = max(first, 0);
  const int r_hi = min(first + a.S + a.h0, sy.rows) - 1;
  const uint64_t start = ptx::globaltimer_ns();
  for (int m = r_lo / gk::kBM; m <= r_hi / gk::kBM; ++m) {
    while (ptx::ld_acquire_gpu(sy.row_done + m) < sy.target) {
      if (ptx::globaltimer_ns() - start > cv::kConvWaitNs) return false;
      ptx::nanosleep(64);
    }
  }
  ptx::fence_proxy_async_global();   // the copies below see what the generic proxy released
  return true;
}

template <int DIL>
__global__ void __launch_bounds__(kSbThreads, 1)
    stage_b_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmH,
                   const __grid_constant__ CUtensorMap cv_v, const __grid_constant__ CUtensorMap cv_h,
                   const __grid_constant__ CUtensorMap cv_p, int Mr, int Nc, int Kd, const gk::EngramEpilogue epi,
                   const cv::ConvArgs a, __nv_bfloat16* __restrict__ H, const SbSync sy) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  __shared__ gk::Bars gbars;
  __shared__ uint64_t full[cv::kConvStages], empty[cv::kConvStages], sa_ready[cv::kConvStages];
  __shared__ int s_tile[cv::kConvStages];
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  uint32_t* err = a.err;

  gk::GemmCtx c = gk::gemm_ctx<kSbBN, true>(smem, Mr, Nc, Kd, err, &gbars);
  gk::gemm_setup<kSbBN, true>(c, warp, lane);
  if (threadIdx.x == 0) {
    for (int st = 0; st < cv::kConvStages; ++st) {
      ptx::mbar_init(&full[st], 1);
      ptx::mbar_init(&empty[st], kSbCompute / 32);
      ptx::mbar_init(&sa_ready[st], 1);
    }
    ptx::fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    ptx::tma_prefetch_desc(&tmA);
    ptx::tma_prefetch_desc(&tmB);
    ptx::tma_prefetch_desc(&tmV);
    ptx::tma_prefetch_desc(&tmH);
    gk::gemm_prefetch_b<kSbBN, true>(c, &tmB);
  }
  if (warp == 10 && lane == 0) {
    ptx::tma_prefetch_desc(&cv_v);
    ptx::tma_prefetch_desc(&cv_h);
    ptx::tma_prefetch_desc(&cv_p);
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  c.tmem = gbars.tmem_base;
  ptx::grid_dep_wait();
  ptx::grid_dep_launch();

  // ------------------------------------------------------------ projection phase
  if (warp == 0) {
    if (lane == 0) gk::gemm_producer<kSbBN, true>(c, &tmA, &tmB);
  } else if (warp == 1) {
    if (lane == 0) gk::gemm_mma<kSbBN, true>(c);
  } else if (warp < 10) {
    gk::gemm_epilogue<kSbBN, true, true>(c, epi, &tmV, &tmH, nullptr, warp, lane, sy.row_done);
  }
  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    ptx::tc_fence_after();
    ptx::tmem_dealloc(c.tmem, G::kTmemCols);
  }
  // a projection timeout ends this block's conv phase too (other blocks time out on its row blocks)
  const bool gemm_ok = *reinterpret_cast<volatile int*>(&gbars.abort) == 0;

  // ------------------------------------------------------------ conv phase
  if (warp == 10) {
    if (lane == 0) {
      uint32_t armed = 0;
      int k = 0;
      bool ok = gemm_ok, post_end = true;
      for (;; ++k) {
        const int st = k % cv::kConvStages;
        const uint32_t round = static_cast<uint32_t>(k / cv::kConvStages);
        if (round > 0 && !ptx::mbar_wait_bounded(&empty[st], (round - 1) & 1u, cv::kConvWaitNs)) {
          // compute warps stopped releasing stages: they have given up already
          atomicOr(err, kErrTimeout);
          post_end = false;
          break;
        }
        int tile = ok ? static_cast<int>(atomicAdd(sy.queue, 1u)) : a.n_tiles;
        if (tile < a.n_tiles && !wait_rows(a, sy, tile)) {
          atomicOr(err, kErrTimeout);
          tile = a.n_tiles;
        }
        if (tile >= a.n_tiles) break;
        *reinterpret_cast<volatile int*>(&s_tile[st]) = tile;
        cv::conv_issue<true>(a, &cv_v, &cv_h, &cv_p, smem + st * a.stage_bytes, &full[st], tile, 1);
        armed |= 1u << st;
      }
      // copies issued in the last kConvStages iterations land before the ring is left (or
      // handed to the end marker); older ones were consumed before their stage came back
      for (int j = k - cv::kConvStages; j < k; ++j) {
        if (j < 0) continue;
        const int sj = j % cv::kConvStages;
        if (armed & (1u << sj))
          ptx::mbar_wait_bounded(&full[sj], static_cast<uint32_t>(j / cv::kConvStages) & 1u, cv::kConvWaitNs);
      }
      if (post_end) {
        const int st = k % cv::kConvStages;
        *reinterpret_cast<volatile int*>(&s_tile[st]) = -1;
        ptx::mbar_arrive(&full[st]);
      }
    }
  } else if (warp == 11) {
    // gate scalars of each staged tile, one tile ahead of the compute warps
    for (int k = 0;; ++k) {
      const int st = k % cv::kConvStages;
      if (!ptx::mbar_wait_bounded(&full[st], static_cast<uint32_t>(k / cv::kConvStages) & 1u, cv::kConvWaitNs)) {
        if (lane == 0) atomicOr(err, kErrTimeout);
        break;
      }
      const int tile = *reinterpret_cast<volatile int*>(&s_tile[st]);
      if (tile < 0) break;
      cv::conv_fin_rows(a, smem + st * a.stage_bytes, tile, lane);
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(&sa_ready[st]);
    }
  } else {
    constexpr int ng = kSbCS / 4;                   // four-channel groups of a tile
    constexpr int npar = kSbCompute / ng;           // chains side by side
    const int g = threadIdx.x % ng, par0 = threadIdx.x / ng;
    int c_cached = -1;
    float wq[4][4];
    int rot = par0;
    for (int k = 0;; ++k) {
      const int st = k % cv::kConvStages;
      const uint32_t par = static_cast<uint32_t>(k / cv::kConvStages) & 1u;
      if (!ptx::mbar_wait_bounded(&full[st], par, cv::kConvWaitNs)) {
        if (lane == 0) atomicOr(err, kErrTimeout);
        break;
      }
      const int tile = *reinterpret_cast<volatile int*>(&s_tile[st]);
      if (tile < 0) break;
      if (!ptx::mbar_wait_bounded(&sa_ready[st], par, cv::kConvWaitNs)) {
        if (lane == 0) atomicOr(err, kErrTimeout);
        break;
      }
      int b, t0, c0;
      cv::conv_coords(a, tile, b, t0, c0);
      if (c0 + 4 * g != c_cached) {
        c_cached = c0 + 4 * g;
        cv::conv_load_taps<4>(a, c_cached, wq);
      }
      cv::conv_tile<__nv_bfloat16, 4, DIL, 1, kSbCS>(a, smem + st * a.stage_bytes, tile, g, rot, npar, wq, H);
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(&empty[st]);
      if (++rot == npar) rot = 0;
    }
  }
  __syncthreads();
}

template <int DIL>
cudaError_t sb_launch(const CUtensorMap& ta, const CUtensorMap& tb, const CUtensorMap& tv, const CUtensorMap& th,
                      const CUtensorMap& cvv, const CUtensorMap& cvh, const CUtensorMap& cvp, int Mr, int Nc, int Kd,
                      const gk::EngramEpilogue& epi, const cv::ConvArgs& a, __nv_bfloat16* H, const SbSync& sy,
                      int grid, size_t smem, cudaStream_t s) {
  static size_t attr_bytes = 0;    // per template instance: the dynamic shared memory opted into so far
  if (smem > attr_bytes) {
    const cudaError_t e = cudaFuncSetAttribute(stage_b_kernel<DIL>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                               static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    attr_bytes = smem;
  }
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kSbThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  cudaError_t e = cudaLaunchKernelEx(&cfg, stage_b_kernel<DIL>, ta, tb, tv, th, cvv, cvh, cvp, Mr, Nc, Kd, epi, a, H,
                                     sy);
  if (e != cudaSuccess) {
    // without overlap of the previous kernel's tail, if the two attributes do not combine here
    (void)cudaGetLastError();
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, stage_b_kernel<DIL>, ta, tb, tv, th, cvv, cvh, cvp, Mr, Nc, Kd, epi, a, H, sy);
  }
  return e;
}

}  // namespace

cudaError_t launch_zero_words(uint32_t* p, int n, cudaStream_t s) {
  return launch_pdl(sync_zero_kernel, dim3(1), dim3(256), 0, s, p, n);
}

size_t stage_b_sync_words(int64_t ntok) { return static_cast<size_t>((ntok + gk::kBM - 1) / gk::kBM) + 1; }

bool stage_b_fused_applies(const engram_plan* p, int64_t ntok, int T) {
  if (T < 2 || p->cfg.act_dtype != ENGRAM_BF16 || p->cfg.M != 1 || p->cfg.conv_w != 4 || p->cfg.conv_dilation < 1 ||
      p->cfg.conv_dilation > 8 || p->cfg.d % kSbCS != 0 || p->d_mem % gk::kBK != 0 || ntok > INT32_MAX / 2)
    return false;
  // 256-column projection tiles give the conv's gate finalisation its 8 slices per quantity
  return p->cfg.d / (kSbBN / 2) == 8;
}

cudaError_t launch_stage_b_fused(const engram_plan* p, const void* e, const void* w_kv, int B, int T, void* H,
                                 const float* g_h, const float* g_k, const float* g_c, const float* conv, float* v32,
                                 float* part, float* sa_out, const engram_state_t* state, uint32_t* sync,
                                 cudaStream_t s) {
  const int64_t ntok = static_cast<int64_t>(B) * T;
  const int d = p->cfg.d, Kd = p->d_mem, Nc = 2 * d;
  const int Mr = static_cast<int>(ntok);
  gk::EngramEpilogue epi{v32, part, static_cast<const __nv_bfloat16*>(H), g_h, g_k, d, 1, d / (kSbBN / 2), 0,
                         nullptr, nullptr};
  epi.pstride = (epi.n_sl * 4 + 3) / 4 * 4;
  if (epi.n_sl != 8 || epi.pstride != 32) return cudaErrorInvalidValue;
  CUtensorMap ta, tb, tv, th;
  if (!make_tensor_map_2d(&ta, e, false, static_cast<uint64_t>(Kd), static_cast<uint64_t>(Mr),
                          static_cast<uint64_t>(Kd) * 2, gk::kBK, gk::kBM, true) ||
      !make_tensor_map_2d(&tb, w_kv, false, static_cast<uint64_t>(Kd), static_cast<uint64_t>(Nc),
                          static_cast<uint64_t>(Kd) * 2, gk::kBK, kSbBN, true) ||
      !make_tensor_map_2d(&tv, v32, true, static_cast<uint64_t>(d), static_cast<uint64_t>(Mr),
                          static_cast<uint64_t>(d) * 4, 32, 32, true) ||
      !make_tensor_map_3d_bf16(&th, H, static_cast<uint64_t>(d), 1, static_cast<uint64_t>(Mr),
                               static_cast<uint64_t>(d) * 2, static_cast<uint64_t>(d) * 2, 64, 1, 32, true))
    return cudaErrorInvalidValue;
  cv::ConvArgs a;
  CUtensorMap cvv, cvh, cvp;
  size_t conv_smem = 0;
  cudaError_t err = conv_prepare(p, v32, d, nullptr, B, T, g_c, conv, H, state, part, sa_out, &a, &cvv, &cvh, &cvp,
                                 &conv_smem, kSbSmemCap);
  if (err != cudaSuccess) return err;
  if (a.CS != kSbCS || a.M != 1) return cudaErrorInvalidValue;
  const size_t smem = std::max(kSbGemmBytes + 1024, conv_smem);
  if (smem > kSbSmemCap) return cudaErrorInvalidValue;
  const int words = static_cast<int>(stage_b_sync_words(ntok));
  SbSync sy{sync, sync + (words - 1), 8u * static_cast<uint32_t>(Nc / kSbBN), Mr};
  err = launch_pdl(sync_zero_kernel, dim3(1), dim3(256), 0, s, sync, words);
  if (err != cudaSuccess) return err;
  const int grid = p->num_sms;
  switch (p->cfg.conv_dilation) {
#define ENGRAM_SB(D) \
  case D: return sb_launch<D>(ta, tb, tv, th, cvv, cvh, cvp, Mr, Nc, Kd, epi, a, static_cast<__nv_bfloat16*>(H), sy, grid, smem, s)
    ENGRAM_SB(1);
    ENGRAM_SB(2);
    ENGRAM_SB(3);
    ENGRAM_SB(4);
    ENGRAM_SB(5);
    ENGRAM_SB(6);
    ENGRAM_SB(7);
    ENGRAM_SB(8);
#undef ENGRAM_SB
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace engram
