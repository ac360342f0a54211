// Step 5 of "DeepSeek Engram 系列导读", section "Engram 工作原理", Stage B:
// k_t = W_K e_t, v_t = W_V e_t, computed for all branches as ONE GEMM
//   kv[Mr, Nc] = e[Mr, Kd] . W_kv[Nc, Kd]^T,  Nc = (M+1)*d,  W_kv = [W_V; W_K^(1..M)],
// the fusion that the page's section "多分支 backbone 上的变体" suggests for the
// hyper-connection variant (it names FP8; this kernel runs bf16 -> fp32).
//
// sm_103a design (one CTA per SM, persistent over output tiles):
//   warp 0      TMA producer: 128x64 A and BNx64 B tiles, 128-byte swizzle,
//               into a kStages-deep shared-memory ring (mbarrier full/empty).
//   warp 1      allocates TMEM (2 x BN fp32 columns: two accumulators) and one
//               elected lane issues tcgen05.mma (M=128, N=BN, K=16) per 16-wide
//               K slice; tcgen05.commit frees ring stages and publishes tiles.
//   warps 2-9   epilogue: two warps per TMEM lane quadrant, each taking half
//               of the tile's columns; tcgen05.ld 32 lanes x 32 columns at a
//               time, round to bf16 and store (or the Engram epilogue below);
//               overlaps the MMA of the next tile (the accumulators ping-pong).
// Every mbarrier wait is bounded in time: on expiry the kernel records
// kErrTimeout, drains its own TMA loads and MMAs (again bounded), frees TMEM
// and returns.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "engram_internal.h"
#include "gemm_parts.cuh"
#include "ptx.cuh"

namespace engram {
namespace {

using namespace gk;

template <int BN, bool kFused>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_bf16_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                     const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmH,
                     __nv_bfloat16* __restrict__ C, int Mr, int Nc, int Kd, uint32_t* __restrict__ err,
                     const EngramEpilogue epi) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  GemmCtx c = gemm_ctx<BN, kFused>(smem, Mr, Nc, Kd, err);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  gemm_setup<BN, kFused>(c, warp, lane);
  if (warp == 0 && lane == 0) {
    ptx::tma_prefetch_desc(&tmA);
    ptx::tma_prefetch_desc(&tmB);
    if constexpr (kFused) {
      ptx::tma_prefetch_desc(&tmV);
      ptx::tma_prefetch_desc(&tmH);
    }
    gemm_prefetch_b<BN, kFused>(c, &tmB);
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  c.tmem = c.bars->tmem_base;
  // the set-up above overlaps the previous kernel's tail; e, W_kv and H are read only after this
  ptx::grid_dep_wait();
  ptx::grid_dep_launch();

  if (warp == 0) {
    if (lane == 0) gemm_producer<BN, kFused>(c, &tmA, &tmB);
  } else if (warp == 1) {
    if (lane == 0) gemm_mma<BN, kFused>(c);
  } else {
    gemm_epilogue<BN, kFused, false>(c, epi, &tmV, &tmH, C, warp, lane, nullptr);
  }

  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    ptx::tc_fence_after();
    ptx::tmem_dealloc(c.tmem, Cfg<BN, kFused>::kTmemCols);
  }
}

// The same persistent kernel on e4m3 operands: e and W_kv quantised per row
// (one scale per token, one per output row of W_kv), kind::f8f6f4 MMAs with
// K = 32 per instruction at twice the bf16 rate, and the Engram epilogue on
// the rescaled accumulators.  The fused-projection suggestion of the page's
// section "多分支 backbone 上的变体" names FP8 for this GEMM.
template <int BN>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_e4m3_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                     const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmH, int Mr, int Nc,
                     int Kd, uint32_t* __restrict__ err, const EngramEpilogue epi) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  GemmCtx c = gemm_ctx<BN, true, true>(smem, Mr, Nc, Kd, err);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  gemm_setup<BN, true, true>(c, warp, lane);
  if (warp == 0 && lane == 0) {
    ptx::tma_prefetch_desc(&tmA);
    ptx::tma_prefetch_desc(&tmB);
    ptx::tma_prefetch_desc(&tmV);
    ptx::tma_prefetch_desc(&tmH);
    gemm_prefetch_b<BN, true, true>(c, &tmB);
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  c.tmem = c.bars->tmem_base;
  ptx::grid_dep_wait();
  ptx::grid_dep_launch();

  if (warp == 0) {
    if (lane == 0) gemm_producer<BN, true, true>(c, &tmA, &tmB);
  } else if (warp == 1) {
    if (lane == 0) gemm_mma<BN, true, true>(c);
  } else {
    gemm_epilogue<BN, true, false, true>(c, epi, &tmV, &tmH, nullptr, warp, lane, nullptr);
  }

  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    ptx::tc_fence_after();
    ptx::tmem_dealloc(c.tmem, Cfg<BN, true, true>::kTmemCols);
  }
}

// ---------------------------------------------------------------- host side
// Row-major bf16 [rows, cols] -> 2D map with a box of box_rows x 64 elements, 128-byte swizzle.
bool make_map(CUtensorMap* map, const void* base, int64_t rows, int cols, int box_rows) {
  return make_tensor_map_2d(map, base, false, static_cast<uint64_t>(cols), static_cast<uint64_t>(rows),
                            static_cast<uint64_t>(cols) * 2, kBK, static_cast<uint32_t>(box_rows), true);
}

template <int BN, bool kFused>
cudaError_t run(const void* A, const void* B, void* C, int64_t Mr, int Nc, int Kd, int num_sms, uint32_t* err,
                EngramEpilogue epi, cudaStream_t s) {
  using G = Cfg<BN, kFused>;
  CUtensorMap ta, tb, tv, th;
  if (!make_map(&ta, A, Mr, Kd, kBM) || !make_map(&tb, B, Nc, Kd, BN)) return cudaErrorInvalidValue;
  if constexpr (kFused) {
    // v32 [Mr, d] fp32 in 32 x 32 boxes; H [Mr, M, d] bf16 in (64 columns, 1 branch, 32 rows) boxes
    if (!make_tensor_map_2d(&tv, epi.v32, true, static_cast<uint64_t>(epi.d), static_cast<uint64_t>(Mr),
                            static_cast<uint64_t>(epi.d) * 4, 32, 32, true) ||
        !make_tensor_map_3d_bf16(&th, epi.H, static_cast<uint64_t>(epi.d), static_cast<uint64_t>(epi.M),
                                 static_cast<uint64_t>(Mr), static_cast<uint64_t>(epi.d) * 2,
                                 static_cast<uint64_t>(epi.d) * epi.M * 2, 64, 1, 32, true))
      return cudaErrorInvalidValue;
  } else {
    tv = ta;
    th = ta;
  }
  static bool attr_set = false;   // per template instance; idempotent if raced
  if (!attr_set) {
    cudaError_t e =
        cudaFuncSetAttribute(gemm_bf16_kernel<BN, kFused>, cudaFuncAttributeMaxDynamicSharedMemorySize, G::kSmem);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  const int64_t tiles = ((Mr + kBM - 1) / kBM) * ((Nc + BN - 1) / BN);
  const int grid = static_cast<int>(tiles < num_sms ? tiles : num_sms);
  if constexpr (kFused) {
    epi.n_sl = epi.d / (BN / 2);
    epi.pstride = (epi.n_sl * (1 + 3 * epi.M) + 3) / 4 * 4;
  }
  return launch_pdl(gemm_bf16_kernel<BN, kFused>, dim3(grid), dim3(kThreads), G::kSmem, s, ta, tb, tv, th,
                    static_cast<__nv_bfloat16*>(C), static_cast<int>(Mr), Nc, Kd, err, epi);
}

template <int BN>
cudaError_t run_e4m3(const uint8_t* A, const uint8_t* B, int64_t Mr, int Nc, int Kd, int num_sms, uint32_t* err,
                     EngramEpilogue epi, cudaStream_t s) {
  using G = Cfg<BN, true, true>;
  CUtensorMap ta, tb, tv, th;
  if (!make_tensor_map_2d_u8(&ta, A, static_cast<uint64_t>(Kd), static_cast<uint64_t>(Mr), static_cast<uint64_t>(Kd),
                             128, kBM, true) ||
      !make_tensor_map_2d_u8(&tb, B, static_cast<uint64_t>(Kd), static_cast<uint64_t>(Nc), static_cast<uint64_t>(Kd),
                             128, BN, true) ||
      !make_tensor_map_2d(&tv, epi.v32, true, static_cast<uint64_t>(epi.d), static_cast<uint64_t>(Mr),
                          static_cast<uint64_t>(epi.d) * 4, 32, 32, true) ||
      !make_tensor_map_3d_bf16(&th, epi.H, static_cast<uint64_t>(epi.d), static_cast<uint64_t>(epi.M),
                               static_cast<uint64_t>(Mr), static_cast<uint64_t>(epi.d) * 2,
                               static_cast<uint64_t>(epi.d) * epi.M * 2, 64, 1, 32, true))
    return cudaErrorInvalidValue;
  static bool attr_set = false;   // per template instance; idempotent if raced
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(gemm_e4m3_kernel<BN>, cudaFuncAttributeMaxDynamicSharedMemorySize, G::kSmem);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  const int64_t tiles = ((Mr + kBM - 1) / kBM) * ((Nc + BN - 1) / BN);
  const int grid = static_cast<int>(tiles < num_sms ? tiles : num_sms);
  epi.n_sl = epi.d / (BN / 2);
  epi.pstride = (epi.n_sl * (1 + 3 * epi.M) + 3) / 4 * 4;
  return launch_pdl(gemm_e4m3_kernel<BN>, dim3(grid), dim3(kThreads), G::kSmem, s, ta, tb, tv, th,
                    static_cast<int>(Mr), Nc, Kd, err, epi);
}

// Widest N tile (256, 128, 64) that divides `div` and still gives every SM a tile.
int pick_bn(int64_t Mr, int Nc, int div, int num_sms) {
  const int64_t m_tiles = (Mr + kBM - 1) / kBM;
  for (int bn : {256, 128}) {
    if (div % bn == 0 && m_tiles * (Nc / bn) >= num_sms) return bn;
  }
  if (div % 64 == 0) return 64;
  return div % 128 == 0 ? 128 : 0;
}

// ---------------------------------------------------------------- fp32 (CUDA cores)
constexpr int kFT = 64;   // output tile
constexpr int kFK = 16;   // K step

__global__ void __launch_bounds__(256) gemm_f32_kernel(const float* __restrict__ A, const float* __restrict__ B,
                                                       float* __restrict__ C, int Mr, int Nc, int Kd) {
  __shared__ float sA[kFK][kFT + 1];
  __shared__ float sB[kFK][kFT + 1];
  const int tx = threadIdx.x % 16, ty = threadIdx.x / 16;
  const int m0 = blockIdx.y * kFT, n0 = blockIdx.x * kFT;
  float acc[4][4] = {};
  for (int k0 = 0; k0 < Kd; k0 += kFK) {
    for (int i = threadIdx.x; i < kFT * kFK; i += 256) {
      const int rr = i / kFK, kk = i % kFK;
      const int am = m0 + rr, bn = n0 + rr, k = k0 + kk;
      sA[kk][rr] = (am < Mr && k < Kd) ? A[static_cast<int64_t>(am) * Kd + k] : 0.f;
      sB[kk][rr] = (bn < Nc && k < Kd) ? B[static_cast<int64_t>(bn) * Kd + k] : 0.f;
    }
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < kFK; ++kk) {
      float a[4], b[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        a[i] = sA[kk][ty * 4 + i];
        b[i] = sB[kk][tx * 4 + i];
      }
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int m = m0 + ty * 4 + i, n = n0 + tx * 4 + j;
      if (m < Mr && n < Nc) C[static_cast<int64_t>(m) * Nc + n] = acc[i][j];
    }
}

}  // namespace

cudaError_t gemm_bf16_tcgen05(const void* A, const void* B, void* C, int64_t Mr, int Nc, int Kd, int num_sms,
                              uint32_t* err, cudaStream_t s) {
  if (Nc % 32 || Kd % 64 || Mr <= 0) return cudaErrorInvalidValue;
  EngramEpilogue none{};
  switch (pick_bn(Mr, Nc, Nc % 64 == 0 ? Nc : 32, num_sms)) {
    case 256: return run<256, false>(A, B, C, Mr, Nc, Kd, num_sms, err, none, s);
    case 64: return run<64, false>(A, B, C, Mr, Nc, Kd, num_sms, err, none, s);
    default: return run<128, false>(A, B, C, Mr, Nc, Kd, num_sms, err, none, s);
  }
}

cudaError_t gemm_bf16_engram(const void* e, const void* w_kv, int64_t Mr, int d, int M, int Kd, const void* H,
                             const float* g_h, const float* g_k, float* v32, float* part, int* n_sl, int* pstride,
                             int num_sms, uint32_t* err, cudaStream_t s, bool cta_pairs) {
  const int Nc = (M + 1) * d;
  if (d % 64 || Kd % 64 || Mr <= 0) return cudaErrorInvalidValue;
  EngramEpilogue epi{v32, part, static_cast<const __nv_bfloat16*>(H), g_h, g_k, d, M, 0, 0, nullptr, nullptr};
  const int bn = pick_bn(Mr, Nc, d, num_sms);
  // on request, the widest tiles run on CTA pairs: half of B per SM, same bits
  if (cta_pairs && bn == 256 && gemm_pair_applies(Mr, d, Kd))
    return gemm_bf16_engram_pair(e, w_kv, Mr, d, M, Kd, H, g_h, g_k, v32, part, n_sl, pstride, num_sms, err, s);
  *n_sl = d / (bn / 2);
  *pstride = (*n_sl * (1 + 3 * M) + 3) / 4 * 4;
  switch (bn) {
    case 256: return run<256, true>(e, w_kv, nullptr, Mr, Nc, Kd, num_sms, err, epi, s);
    case 128: return run<128, true>(e, w_kv, nullptr, Mr, Nc, Kd, num_sms, err, epi, s);
    default: return run<64, true>(e, w_kv, nullptr, Mr, Nc, Kd, num_sms, err, epi, s);
  }
}

cudaError_t gemm_e4m3_engram(const uint8_t* e8, const float* s_e, const uint8_t* w8, const float* s_w, int64_t Mr,
                             int d, int M, int Kd, const void* H, const float* g_h, const float* g_k, float* v32,
                             float* part, int* n_sl, int* pstride, int num_sms, uint32_t* err, cudaStream_t s) {
  const int Nc = (M + 1) * d;
  if (d % 64 || Kd % 128 || Mr <= 0) return cudaErrorInvalidValue;
  EngramEpilogue epi{v32, part, static_cast<const __nv_bfloat16*>(H), g_h, g_k, d, M, 0, 0, s_e, s_w};
  const int bn = pick_bn(Mr, Nc, d, num_sms);
  *n_sl = d / (bn / 2);
  *pstride = (*n_sl * (1 + 3 * M) + 3) / 4 * 4;
  switch (bn) {
    case 256: return run_e4m3<256>(e8, w8, Mr, Nc, Kd, num_sms, err, epi, s);
    case 128: return run_e4m3<128>(e8, w8, Mr, Nc, Kd, num_sms, err, epi, s);
    default: return run_e4m3<64>(e8, w8, Mr, Nc, Kd, num_sms, err, epi, s);
  }
}

cudaError_t gemm_f32_simt(const float* A, const float* B, float* C, int64_t Mr, int Nc, int Kd, cudaStream_t s) {
  dim3 grid((Nc + kFT - 1) / kFT, static_cast<unsigned>((Mr + kFT - 1) / kFT));
  gemm_f32_kernel<<<grid, 256, 0, s>>>(A, B, C, static_cast<int>(Mr), Nc, Kd);
  return cudaGetLastError();
}

cudaError_t launch_kv_projection(const engram_plan* p, const void* e, int64_t ntok, const void* w_kv, void* kv,
                                 cudaStream_t s) {
  const int Nc = (p->cfg.M + 1) * p->cfg.d;
  if (p->cfg.act_dtype == ENGRAM_F32)
    return gemm_f32_simt(static_cast<const float*>(e), static_cast<const float*>(w_kv), static_cast<float*>(kv), ntok,
                         Nc, p->d_mem, s);
  return gemm_bf16_tcgen05(e, w_kv, kv, ntok, Nc, p->d_mem, p->num_sms, &p->dev->err, s);
}

}  // namespace engram
