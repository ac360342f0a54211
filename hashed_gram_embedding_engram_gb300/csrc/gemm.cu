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
#include "ptx.cuh"

namespace engram {
namespace {

constexpr int kBM = 128;
constexpr int kBK = 64;                        // one 128-byte swizzle atom of bf16
constexpr int kThreads = 320;                 // producer, MMA, 8 epilogue warps
constexpr uint64_t kWaitLimitNs = 1000000000ull;   // 1 s: a healthy stage turns over in < 1 us

constexpr int kEpiWarpBytes = 8192;            // fused epilogue: per-warp staging of v chunks / the H slice

template <int BN, bool kFused>
struct Cfg {
  static constexpr int kStages = kFused ? (BN == 256 ? 3 : (BN == 128 ? 4 : 6)) : (BN == 256 ? 4 : (BN == 128 ? 6 : 8));
  static constexpr int kABytes = kBM * kBK * 2;
  static constexpr int kBBytes = BN * kBK * 2;
  static constexpr int kStageBytes = kABytes + kBBytes;
  static constexpr int kEpiBytes = kFused ? 8 * kEpiWarpBytes : 0;
  static constexpr int kTmemCols = 2 * BN < 32 ? 32 : 2 * BN;
  static constexpr int kBarBytes = 256;
  static constexpr int kSmem = 1024 + kStages * kStageBytes + kEpiBytes + kBarBytes;
  static constexpr uint32_t kIdesc = ptx::idesc_bf16_f32(kBM, BN);
  static constexpr int kHBoxes = BN / 2 > 64 ? BN / 128 : 1;   // 64-column H boxes per warp slice
};

struct EngramEpilogue {
  float* v32;                     // [Mr, d]
  float* part;                    // [Mr, n_sl * (1 + 3M)]
  const __nv_bfloat16* H;         // [Mr, M, d]
  const float* g_h;               // [M, d]
  const float* g_k;               // [M, d]
  int d;
  int M;
  int n_sl;                       // d / (BN / 2): column slices per row of v
  int pstride;                    // floats per row of part: n_sl * (1 + 3M) rounded up to 4
};

struct Bars {
  uint64_t full[8];
  uint64_t empty[8];
  uint64_t tfull[2];
  uint64_t tempty[2];
  uint64_t hbar[8];               // fused epilogue: H slice of each epilogue warp landed
  uint64_t drain;
  uint32_t tmem_base;
  int abort;
};

__device__ __forceinline__ bool wait_or_abort(uint64_t* bar, uint32_t parity, Bars* b, uint32_t* err) {
  if (ptx::mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = ptx::globaltimer_ns();
  while (true) {
    for (int i = 0; i < 32; ++i)
      if (ptx::mbar_try_wait(bar, parity)) return true;
    if (*reinterpret_cast<volatile int*>(&b->abort)) return false;
    if (ptx::globaltimer_ns() - t0 > kWaitLimitNs) {
      atomicOr(err, kErrTimeout);
      *reinterpret_cast<volatile int*>(&b->abort) = 1;
      return false;
    }
  }
}

// Engram epilogue of the K/V projection (Steps 5-6 fused).  Output columns
// [0, d) are v: stored in fp32 with a per-slice partial of sum(v^2).  Columns
// [(1+m)d, (2+m)d) are k^(m): never stored; each slice contributes the partial
// sums the gate needs, taken from the fp32 accumulators and H^(m):
//   dot = sum h*g_h*g_k*k,  sk = sum k^2,  sh = sum h^2   (over the slice's columns).
// A slice is the half tile (BN/2 columns) one epilogue warp handles; with
// n_sl = d / (BN/2) slices per row of v (and of each k^(m)), token t has
// part[t*P + j] = sum v^2 of v slice j, and
// part[t*P + n_sl + (m*n_sl + j)*3 + {0,1,2}] = (dot, sk, sh) of k^(m) slice j.
// Rows of part are pstride floats apart (padded to 16 bytes).  Each sum is a
// sequential fmaf chain over the 32 columns of one tcgen05.ld chunk; a
// slice's chunks are combined as an adjacent pairwise tree, which the gate
// finalisation continues over the slices (fusion.cu), so the gate's sums have
// the same bits for every tile width BN.
//
// TMEM gives each lane one row, so global accesses lane by lane would touch 32
// cache lines per instruction.  Both directions go through the warp's 8 KB of
// shared memory in the 128-byte swizzled layout instead (16-byte chunk j of
// row r at r*128 + 16*(j ^ (r % 8)), conflict-free for row-per-lane access):
// v chunks of 32 x 32 fp32 leave by TMA tensor stores, and the warp's H slice
// (32 rows x BN/2 columns) arrives by TMA while the tile's MMAs run.
template <int BN>
__device__ __forceinline__ void fused_epilogue(const EngramEpilogue& epi, const CUtensorMap* tmV, uint8_t* eb,
                                               uint32_t t_row, int row, int row0, int Mr, int n0, int c_lo, int lane) {
  constexpr int SW = BN / 2;
  constexpr int kChunks = SW / 32;          // 1, 2 or 4
  const int d = epi.d;
  const int P = epi.pstride;
  const int swz = lane & 7;
  if (n0 < d) {
    float stk[3];
    int top = 0;
#pragma unroll
    for (int ci = 0; ci < kChunks; ++ci) {
      const int c = c_lo + ci * 32;
      uint32_t r[32];
      ptx::tmem_ld_32x32b_x32(t_row + c, r);
      ptx::tmem_ld_wait();
      float sv = 0.f;
#pragma unroll
      for (int j = 0; j < 32; ++j) sv = fmaf(__uint_as_float(r[j]), __uint_as_float(r[j]), sv);
#pragma unroll
      for (int k = ci; k & 1; k >>= 1) sv = stk[--top] + sv;
      stk[top++] = sv;
      uint8_t* sb = eb + (ci & 1) * 4096;
      if (lane == 0) {
        if (ci == 0) ptx::bulk_wait_read<0>();     // earlier tiles' stores have left both buffers
        else if (ci >= 2) ptx::bulk_wait_read<1>();  // the store from this buffer two chunks ago
      }
      __syncwarp();
#pragma unroll
      for (int j = 0; j < 8; ++j)
        *reinterpret_cast<uint4*>(sb + lane * 128 + ((j ^ swz) << 4)) =
            make_uint4(r[4 * j], r[4 * j + 1], r[4 * j + 2], r[4 * j + 3]);
      ptx::fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        ptx::tma_store_2d(tmV, sb, n0 + c, row0);
        ptx::bulk_commit();
      }
    }
    if (row < Mr) epi.part[static_cast<int64_t>(row) * P + (n0 + c_lo) / SW] = stk[0];
  } else {
    const int m = (n0 - d) / d;
    const int col = n0 - d - m * d;
    const int j = (col + c_lo) / SW;
    const float* gh = epi.g_h + static_cast<int64_t>(m) * d + col;
    const float* gk = epi.g_k + static_cast<int64_t>(m) * d + col;
    float s_dot[3], s_sk[3], s_sh[3];
    int top = 0;
#pragma unroll
    for (int ci = 0; ci < kChunks; ++ci) {
      const int c = c_lo + ci * 32;
      uint32_t r[32];
      ptx::tmem_ld_32x32b_x32(t_row + c, r);
      ptx::tmem_ld_wait();
      float dot = 0.f, sk = 0.f, sh = 0.f;
      const uint8_t* hb = eb + (ci >> 1) * 4096 + lane * 128;     // this row of the chunk's 64-column box
      const float4* gh4 = reinterpret_cast<const float4*>(gh + c);
      const float4* gk4 = reinterpret_cast<const float4*>(gk + c);
#pragma unroll
      for (int q4 = 0; q4 < 4; ++q4) {
        const uint4 hv = *reinterpret_cast<const uint4*>(hb + ((((ci & 1) * 4 + q4) ^ swz) << 4));
        const uint32_t hw[4] = {hv.x, hv.y, hv.z, hv.w};
        const float4 ga = __ldg(gh4 + 2 * q4), gb = __ldg(gh4 + 2 * q4 + 1);
        const float4 ka = __ldg(gk4 + 2 * q4), kb = __ldg(gk4 + 2 * q4 + 1);
        const float g[8] = {ga.x * ka.x, ga.y * ka.y, ga.z * ka.z, ga.w * ka.w,
                            gb.x * kb.x, gb.y * kb.y, gb.z * kb.z, gb.w * kb.w};
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const float h = __uint_as_float(i & 1 ? (hw[i >> 1] & 0xFFFF0000u) : (hw[i >> 1] << 16));
          const float k = __uint_as_float(r[q4 * 8 + i]);
          dot = fmaf(h * g[i], k, dot);
          sk = fmaf(k, k, sk);
          sh = fmaf(h, h, sh);
        }
      }
#pragma unroll
      for (int k = ci; k & 1; k >>= 1) {
        --top;
        dot = s_dot[top] + dot;
        sk = s_sk[top] + sk;
        sh = s_sh[top] + sh;
      }
      s_dot[top] = dot;
      s_sk[top] = sk;
      s_sh[top] = sh;
      ++top;
    }
    if (row < Mr) {
      float* dst = epi.part + static_cast<int64_t>(row) * P + epi.n_sl + (m * epi.n_sl + j) * 3;
      dst[0] = s_dot[0];
      dst[1] = s_sk[0];
      dst[2] = s_sh[0];
    }
  }
}

template <int BN, bool kFused>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_bf16_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                     const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmH,
                     __nv_bfloat16* __restrict__ C, int Mr, int Nc, int Kd, uint32_t* __restrict__ err,
                     const EngramEpilogue epi) {
  using G = Cfg<BN, kFused>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* epi_smem = smem + G::kStages * G::kStageBytes;          // 1024-byte aligned
  Bars* bars = reinterpret_cast<Bars*>(epi_smem + G::kEpiBytes);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int m_tiles = (Mr + kBM - 1) / kBM;
  const int n_tiles = (Nc + BN - 1) / BN;
  const int num_tiles = m_tiles * n_tiles;
  const int k_blocks = (Kd + kBK - 1) / kBK;

  if (threadIdx.x == 0) {
    for (int s = 0; s < G::kStages; ++s) {
      ptx::mbar_init(&bars->full[s], 1);
      ptx::mbar_init(&bars->empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      ptx::mbar_init(&bars->tfull[a], 1);
      ptx::mbar_init(&bars->tempty[a], 8);     // one arrive per epilogue warp
    }
    for (int w = 0; w < 8; ++w) ptx::mbar_init(&bars->hbar[w], 1);
    ptx::mbar_init(&bars->drain, 1);
    bars->abort = 0;
    ptx::fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    ptx::tma_prefetch_desc(&tmA);
    ptx::tma_prefetch_desc(&tmB);
    if constexpr (kFused) {
      ptx::tma_prefetch_desc(&tmV);
      ptx::tma_prefetch_desc(&tmH);
    }
  }
  if (warp == 1) {
    ptx::tmem_alloc(&bars->tmem_base, G::kTmemCols);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = bars->tmem_base;
  // the set-up above overlaps the previous kernel's tail; e, W_kv and H are read only after this
  ptx::grid_dep_wait();
  ptx::grid_dep_launch();

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------ TMA producer
      const uint64_t keep = ptx::policy_evict_last();    // W_kv is re-read by every row tile
      int stage = 0;
      uint32_t phase = 0;
      uint32_t armed = 0, armed_parity = 0;               // per stage: armed at least once / parity
      bool ok = true;
      for (int tile = blockIdx.x; ok && tile < num_tiles; tile += gridDim.x) {
        const int m0 = (tile / n_tiles) * kBM;
        const int n0 = (tile % n_tiles) * BN;
        for (int kb = 0; kb < k_blocks; ++kb) {
          if (!wait_or_abort(&bars->empty[stage], phase ^ 1, bars, err)) {
            ok = false;
            break;
          }
          uint8_t* sa = smem + stage * G::kStageBytes;
          ptx::mbar_arrive_expect_tx(&bars->full[stage], G::kStageBytes);
          ptx::tma_load_2d_nohint(sa, &tmA, &bars->full[stage], kb * kBK, m0);
          ptx::tma_load_2d(sa + G::kABytes, &tmB, &bars->full[stage], kb * kBK, n0, keep);
          armed |= 1u << stage;
          armed_parity = (armed_parity & ~(1u << stage)) | (phase << stage);
          if (++stage == G::kStages) {
            stage = 0;
            phase ^= 1;
          }
        }
      }
      // our own copies in flight must land before the CTA can exit
      for (int s = 0; s < G::kStages; ++s)
        if (armed & (1u << s)) ptx::mbar_wait_bounded(&bars->full[s], (armed_parity >> s) & 1u, kWaitLimitNs);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ------------------------------------------------ MMA issuer
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      bool ok = true;
      for (int tile = blockIdx.x; ok && tile < num_tiles; tile += gridDim.x) {
        if (!wait_or_abort(&bars->tempty[acc], acc_phase ^ 1, bars, err)) break;
        ptx::tc_fence_after();
        const uint32_t d_tmem = tmem + static_cast<uint32_t>(acc * BN);
        for (int kb = 0; kb < k_blocks; ++kb) {
          if (!wait_or_abort(&bars->full[stage], phase, bars, err)) {
            ok = false;
            break;
          }
          ptx::tc_fence_after();
          const uint32_t a_addr = ptx::smem_u32(smem + stage * G::kStageBytes);
          const uint32_t b_addr = a_addr + G::kABytes;
#pragma unroll
          for (int k = 0; k < kBK / 16; ++k) {
            ptx::mma_bf16(d_tmem, ptx::sdesc_kmajor_sw128(a_addr + k * 32), ptx::sdesc_kmajor_sw128(b_addr + k * 32),
                          G::kIdesc, (kb | k) != 0);
          }
          ptx::mma_commit(&bars->empty[stage]);
          if (++stage == G::kStages) {
            stage = 0;
            phase ^= 1;
          }
        }
        if (!ok) break;
        ptx::mma_commit(&bars->tfull[acc]);
        acc ^= 1;
        if (acc == 0) acc_phase ^= 1;
      }
      // every MMA this thread issued has finished before TMEM is freed
      ptx::mma_commit(&bars->drain);
      ptx::mbar_wait_bounded(&bars->drain, 0, kWaitLimitNs);
    }
  } else {
    // -------------------------------------------------- epilogue (warps 2..9)
    const int q = warp & 3;                 // TMEM lane quadrant this warp may access
    const int ew = warp - 2;
    const int c_lo = (ew >> 2) * (BN / 2);  // half of the tile's columns
    uint8_t* eb = epi_smem + ew * kEpiWarpBytes;
    int acc = 0;
    uint32_t acc_phase = 0;
    uint32_t h_phase = 0;
    bool h_pending = false;
    for (int tile = blockIdx.x; tile < num_tiles; tile += gridDim.x) {
      const int m0 = (tile / n_tiles) * kBM;
      const int n0 = (tile % n_tiles) * BN;
      const int row = m0 + q * 32 + lane;
      const bool ktile = kFused && n0 >= epi.d;
      if (ktile) {
        // this warp's H slice (32 rows x BN/2 columns) lands while the tile's MMAs run
        if (lane == 0) {
          ptx::bulk_wait_read<0>();            // staged v of an earlier tile has left this buffer
          ptx::fence_proxy_async_smem();
          const int m = (n0 - epi.d) / epi.d;
          const int col = n0 - epi.d - m * epi.d + c_lo;
          ptx::mbar_arrive_expect_tx(&bars->hbar[ew], G::kHBoxes * 4096);
#pragma unroll
          for (int bx = 0; bx < G::kHBoxes; ++bx)
            ptx::tma_load_3d(eb + bx * 4096, &tmH, &bars->hbar[ew], col + bx * 64, m, m0 + q * 32);
        }
        h_pending = true;
      }
      if (!wait_or_abort(&bars->tfull[acc], acc_phase, bars, err)) break;
      ptx::tc_fence_after();
      if (ktile) {
        if (!wait_or_abort(&bars->hbar[ew], h_phase, bars, err)) break;
        h_phase ^= 1;
        h_pending = false;
      }
      const uint32_t t_row = tmem + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(acc * BN);
      if constexpr (!kFused) {
#pragma unroll 1
        for (int c = c_lo; c < c_lo + BN / 2; c += 32) {
          uint32_t r[32];
          ptx::tmem_ld_32x32b_x32(t_row + c, r);
          ptx::tmem_ld_wait();
          if (row < Mr && n0 + c < Nc) {
            uint32_t packed[16];
#pragma unroll
            for (int j = 0; j < 16; ++j) {
              __nv_bfloat162 v = __floats2bfloat162_rn(__uint_as_float(r[2 * j]), __uint_as_float(r[2 * j + 1]));
              packed[j] = *reinterpret_cast<uint32_t*>(&v);
            }
            uint4* dst = reinterpret_cast<uint4*>(C + static_cast<int64_t>(row) * Nc + n0 + c);
#pragma unroll
            for (int j = 0; j < 4; ++j)
              dst[j] = make_uint4(packed[4 * j], packed[4 * j + 1], packed[4 * j + 2], packed[4 * j + 3]);
          }
        }
      } else {
        fused_epilogue<BN>(epi, &tmV, eb, t_row, row, m0 + q * 32, Mr, n0, c_lo, lane);
      }
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(&bars->tempty[acc]);
      acc ^= 1;
      if (acc == 0) acc_phase ^= 1;
    }
    if constexpr (kFused) {
      if (lane == 0) {
        // an H load that a timeout left in flight lands before the block exits; v stores complete
        if (h_pending) ptx::mbar_wait_bounded(&bars->hbar[ew], h_phase, kWaitLimitNs);
        ptx::bulk_wait_all();
      }
    }
  }

  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, G::kTmemCols);
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
                             int num_sms, uint32_t* err, cudaStream_t s) {
  const int Nc = (M + 1) * d;
  if (d % 64 || Kd % 64 || Mr <= 0) return cudaErrorInvalidValue;
  EngramEpilogue epi{v32, part, static_cast<const __nv_bfloat16*>(H), g_h, g_k, d, M, 0, 0};
  const int bn = pick_bn(Mr, Nc, d, num_sms);
  *n_sl = d / (bn / 2);
  *pstride = (*n_sl * (1 + 3 * M) + 3) / 4 * 4;
  switch (bn) {
    case 256: return run<256, true>(e, w_kv, nullptr, Mr, Nc, Kd, num_sms, err, epi, s);
    case 128: return run<128, true>(e, w_kv, nullptr, Mr, Nc, Kd, num_sms, err, epi, s);
    default: return run<64, true>(e, w_kv, nullptr, Mr, Nc, Kd, num_sms, err, epi, s);
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
