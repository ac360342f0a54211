// Step 5 of "DeepSeek Engram 系列导读", section "Engram 工作原理", Stage B, on
// CTA pairs: the fused K/V projection
//   kv[Mr, Nc] = e[Mr, Kd] . W_kv[Nc, Kd]^T,  Nc = (M+1)*d,  W_kv = [W_V; W_K^(1..M)],
// with the same Engram epilogue as gemm.cu (v stored in fp32, k turned into
// the gate's partial sums), in 256 x 256 output tiles per pair of SMs.
//
// Why pairs: a one-SM 128 x 256 tile consumes 48 KB of operands per 64-deep
// k-block.  With tcgen05.mma.cta_group::2 two SMs of a cluster compute a
// 256 x 256 tile together: each SM stages its own 128 rows of e and HALF of
// the tile's 256 rows of W_kv (16 KB + 16 KB per k-block), and one MMA
// instruction reads A from each SM's shared memory and B from both; each SM's
// TMEM receives its 128 rows x 256 columns.  Operand traffic per FLOP, into
// and out of each SM's shared memory, drops by a third.
// Measured on GB300 (4096 x 2048 x 1024, event-timed): 24.2 us against
// 22.2 us for the one-SM form.  A globaltimer timeline of both (L2 flushed, e
// just written) shows why: the pair's first tile runs its mainloop at 94 % of
// the MMA rate (5.6 us against 6.1 us on one SM: the 4-stage ring covers the
// refill latency), but the cluster barrier and the paired TMEM allocation
// start it 1.3 us later, and its second tile's mainloop takes 6.9-7.2 us while
// the first wave's epilogues -- all v tiles, 128 KB of stores per SM -- go out
// through the same TMA unit.  It is selectable (engram_plan_set_cta_pairs)
// and gives the same bits.
//
// Roles (320 threads per CTA, one CTA per SM, persistent over pair tiles):
//   warp 0      both CTAs: TMA producer of the CTA's own A rows and B half into
//               a 4-stage ring; every copy completes on the LEADER's (rank 0)
//               full barrier, for which the leader expects both CTAs' bytes.
//   warp 1      both CTAs allocate the same 512 TMEM columns (two 256-column
//               accumulators); one thread of the leader issues the M = 256
//               MMAs and commits each stage's release to both CTAs' empty
//               barriers and each finished tile to both CTAs' tfull barriers.
//   warps 2-9   both CTAs: the Engram epilogue of the CTA's 128 rows (gemm.cu),
//               then one arrive on the leader's tempty barrier (16 per tile).
// Every wait is bounded (1 s; on expiry: error word, unwind).  Both CTAs meet
// at a cluster barrier before the collective TMEM free; a CTA that gave up
// first lets any copy it had issued land (a short grace period), so no copy
// or remote arrive can target a CTA that has exited.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "engram_internal.h"
#include "gemm_parts.cuh"
#include "ptx.cuh"

namespace engram {
namespace {

using namespace gk;

constexpr int kPairBM = 256;                       // output rows per pair tile (128 per CTA)
constexpr int kPairBN = 256;                       // output columns per pair tile
constexpr int kPairStages = 4;
constexpr int kPairABytes = 128 * 128;             // this CTA's 128 rows x 64 bf16
constexpr int kPairBBytes = 128 * 128;             // this CTA's half of B: 128 rows x 64 bf16
constexpr int kPairStageBytes = kPairABytes + kPairBBytes;
using EpiCfg = Cfg<kPairBN, true>;                 // per-CTA epilogue of a 128 x 256 accumulator
constexpr int kPairSmem = 1024 + kPairStages * kPairStageBytes + EpiCfg::kEpiBytes + EpiCfg::kBarBytes;
constexpr int kPairTmemCols = 2 * kPairBN;
constexpr uint32_t kPairIdesc = ptx::idesc_bf16_f32(kPairBM, kPairBN);
constexpr uint64_t kGraceNs = 200000;             // after an abort: copies already issued land

__device__ __forceinline__ bool wait_cluster_or_abort(uint64_t* bar, uint32_t parity, Bars* b, uint32_t* err) {
  if (ptx::mbar_try_wait_cluster(bar, parity)) return true;
  const uint64_t t0 = ptx::globaltimer_ns();
  while (true) {
    for (int i = 0; i < 32; ++i)
      if (ptx::mbar_try_wait_cluster(bar, parity)) return true;
    if (*reinterpret_cast<volatile int*>(&b->abort)) return false;
    if (ptx::globaltimer_ns() - t0 > kWaitLimitNs) {
      atomicOr(err, kErrTimeout);
      *reinterpret_cast<volatile int*>(&b->abort) = 1;
      return false;
    }
  }
}

// Pair tiles in launch order: every v tile (output columns [0, d)) before any
// k tile, so the pairs' first wave does the v tiles, whose epilogue (v stored)
// is the longer one and then overlaps the next tile's MMAs, and the last tile
// of a pair is a k tile.  Tile t -> (row of pairs, 256-column block).
struct TileMap {
  int m_tiles, nv, nk;           // rows of pairs; column blocks of v; of k
  __device__ __forceinline__ void at(int t, int& mt, int& nt) const {
    const int tv = m_tiles * nv;
    if (t < tv) {
      mt = t / nv;
      nt = t - mt * nv;
    } else {
      const int u = t - tv;
      mt = u / nk;
      nt = nv + (u - mt * nk);
    }
  }
};

struct PairCtx {
  uint8_t* smem;
  uint8_t* epi_smem;
  Bars* bars;
  uint32_t rank;       // 0: leader (issues the MMAs), 1: peer
  int pair, n_pairs;
  int n_tiles, num_tiles, k_blocks, Mr;
  TileMap map;
  uint32_t* err;
};

// Warp 0, lane 0 of both CTAs.
__device__ __forceinline__ void pair_producer(const PairCtx& c, const CUtensorMap* tmA, const CUtensorMap* tmB) {
  Bars* bars = c.bars;
  const uint64_t keep = ptx::policy_evict_last();   // W_kv is re-read by every row of pairs
  const uint32_t full0 = ptx::mapa_shared(ptx::smem_u32(&bars->full[0]), 0);
  int stage = 0;
  uint32_t phase = 0;
  uint32_t armed = 0, armed_parity = 0;
  bool ok = true;
  for (int tile = c.pair; ok && tile < c.num_tiles; tile += c.n_pairs) {
    int mt, nt;
    c.map.at(tile, mt, nt);
    const int m0 = mt * kPairBM + static_cast<int>(c.rank) * 128;
    const int nb = nt * kPairBN + static_cast<int>(c.rank) * 128;
    for (int kb = 0; kb < c.k_blocks; ++kb) {
      if (!wait_or_abort(&bars->empty[stage], phase ^ 1, bars, c.err)) {
        ok = false;
        break;
      }
      if (c.rank == 0) {
        ptx::mbar_arrive_expect_tx(&bars->full[stage], 2 * kPairStageBytes);
        armed |= 1u << stage;
        armed_parity = (armed_parity & ~(1u << stage)) | (phase << stage);
      }
      uint8_t* sa = c.smem + stage * kPairStageBytes;
      const uint32_t fb = full0 + static_cast<uint32_t>(stage * sizeof(uint64_t));
      ptx::tma_load_2d_pair(sa, tmA, fb, kb * kBK, m0, 0ull);
      ptx::tma_load_2d_pair(sa + kPairABytes, tmB, fb, kb * kBK, nb, keep);
      if (++stage == kPairStages) {
        stage = 0;
        phase ^= 1;
      }
    }
  }
  // the leader's full barriers count both CTAs' copies: once a phase it armed
  // completes, every copy of that phase has landed
  if (c.rank == 0)
    for (int s = 0; s < kPairStages; ++s)
      if (armed & (1u << s)) ptx::mbar_wait_bounded(&bars->full[s], (armed_parity >> s) & 1u, kWaitLimitNs);
}

// Warp 1, lane 0 of the leader.
__device__ __forceinline__ void pair_mma(const PairCtx& c, uint32_t tmem) {
  Bars* bars = c.bars;
  int stage = 0;
  uint32_t phase = 0;
  int acc = 0;
  uint32_t acc_phase = 0;
  bool ok = true;
  for (int tile = c.pair; ok && tile < c.num_tiles; tile += c.n_pairs) {
    // both CTAs' epilogues have read this accumulator
    if (!wait_cluster_or_abort(&bars->tempty[acc], acc_phase ^ 1, bars, c.err)) break;
    ptx::tc_fence_after();
    const uint32_t d_tmem = tmem + static_cast<uint32_t>(acc * kPairBN);
    for (int kb = 0; kb < c.k_blocks; ++kb) {
      if (!wait_or_abort(&bars->full[stage], phase, bars, c.err)) {
        ok = false;
        break;
      }
      ptx::tc_fence_after();
      const uint32_t a_addr = ptx::smem_u32(c.smem + stage * kPairStageBytes);
      const uint32_t b_addr = a_addr + kPairABytes;
#pragma unroll
      for (int k = 0; k < 4; ++k)            // 16 bf16 of K per instruction
        ptx::mma_bf16_pair(d_tmem, ptx::sdesc_kmajor_sw128(a_addr + k * 32), ptx::sdesc_kmajor_sw128(b_addr + k * 32),
                           kPairIdesc, (kb | k) != 0);
      const uint32_t eb = ptx::smem_u32(&bars->empty[stage]);
      ptx::mma_commit_pair(eb);
      ptx::mma_commit_pair(ptx::mapa_shared(eb, 1));
      if (++stage == kPairStages) {
        stage = 0;
        phase ^= 1;
      }
    }
    if (!ok) break;
    const uint32_t tb = ptx::smem_u32(&bars->tfull[acc]);
    ptx::mma_commit_pair(tb);
    ptx::mma_commit_pair(ptx::mapa_shared(tb, 1));
    acc ^= 1;
    if (acc == 0) acc_phase ^= 1;
  }
  // every MMA issued has finished (in both CTAs' TMEM) before TMEM is freed
  ptx::mma_commit_pair(ptx::smem_u32(&bars->drain));
  ptx::mbar_wait_bounded(&bars->drain, 0, kWaitLimitNs);
}

// Warps 2..9 of both CTAs: the CTA's 128 rows of each pair tile.
__device__ __forceinline__ void pair_epilogue(const PairCtx& c, uint32_t tmem, const EngramEpilogue& epi,
                                              const CUtensorMap* tmV, const CUtensorMap* tmH, int warp, int lane) {
  Bars* bars = c.bars;
  const int q = warp & 3;                   // TMEM lane quadrant this warp may access
  const int ew = warp - 2;
  const int c_lo = (ew >> 2) * (kPairBN / 2);
  uint8_t* eb = c.epi_smem + ew * kEpiWarpBytes;
  float* gs = reinterpret_cast<float*>(c.epi_smem + 8 * kEpiWarpBytes + ew * EpiCfg::kGWarpBytes);
  const uint32_t tempty0 = ptx::mapa_shared(ptx::smem_u32(&bars->tempty[0]), 0);
  int acc = 0;
  uint32_t acc_phase = 0;
  uint32_t h_phase = 0;
  bool h_pending = false;
  for (int tile = c.pair; tile < c.num_tiles; tile += c.n_pairs) {
    int mt, nt;
    c.map.at(tile, mt, nt);
    const int m0 = mt * kPairBM + static_cast<int>(c.rank) * 128;
    const int n0 = nt * kPairBN;
    const int row = m0 + q * 32 + lane;
    const bool ktile = n0 >= epi.d;
    if (ktile) {
      if (lane == 0) {
        ptx::bulk_wait_read<0>();            // staged v of an earlier tile has left this buffer
        ptx::fence_proxy_async_smem();
        const int m = (n0 - epi.d) / epi.d;
        const int col = n0 - epi.d - m * epi.d + c_lo;
        ptx::mbar_arrive_expect_tx(&bars->hbar[ew], EpiCfg::kHBoxes * 4096 + EpiCfg::kGWarpBytes);
        const int64_t go = static_cast<int64_t>(m) * epi.d + col;
        ptx::bulk_load(gs, epi.g_h + go, EpiCfg::kGWarpBytes / 2, &bars->hbar[ew]);
        ptx::bulk_load(gs + kPairBN / 2, epi.g_k + go, EpiCfg::kGWarpBytes / 2, &bars->hbar[ew]);
#pragma unroll
        for (int bx = 0; bx < EpiCfg::kHBoxes; ++bx)
          ptx::tma_load_3d(eb + bx * 4096, tmH, &bars->hbar[ew], col + bx * 64, m, m0 + q * 32);
      }
      h_pending = true;
    }
    if (!wait_or_abort(&bars->tfull[acc], acc_phase, bars, c.err)) break;
    ptx::tc_fence_after();
    if (ktile) {
      if (!wait_or_abort(&bars->hbar[ew], h_phase, bars, c.err)) break;
      h_phase ^= 1;
      h_pending = false;
    }
    const uint32_t t_row = tmem + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(acc * kPairBN);
    fused_epilogue<kPairBN, false>(epi, tmV, eb, gs, t_row, row, m0 + q * 32, c.Mr, n0, c_lo, lane);
    ptx::tc_fence_before();
    __syncwarp();
    if (lane == 0) ptx::mbar_arrive_cluster(tempty0 + static_cast<uint32_t>(acc * sizeof(uint64_t)));
    acc ^= 1;
    if (acc == 0) acc_phase ^= 1;
  }
  if (lane == 0) {
    if (h_pending) ptx::mbar_wait_bounded(&bars->hbar[ew], h_phase, kWaitLimitNs);
    ptx::bulk_wait_all();
  }
}

__global__ void __launch_bounds__(kThreads, 1)
    gemm_pair_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                     const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmH, int Mr, int Nc,
                     int Kd, uint32_t* __restrict__ err, const EngramEpilogue epi) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  PairCtx c;
  c.smem = smem;
  c.epi_smem = smem + kPairStages * kPairStageBytes;
  c.bars = reinterpret_cast<Bars*>(c.epi_smem + EpiCfg::kEpiBytes);
  c.rank = ptx::cluster_ctarank();
  c.pair = static_cast<int>(blockIdx.x >> 1);
  c.n_pairs = static_cast<int>(gridDim.x >> 1);
  c.n_tiles = Nc / kPairBN;
  c.num_tiles = ((Mr + kPairBM - 1) / kPairBM) * c.n_tiles;
  c.k_blocks = Kd / kBK;
  c.map.m_tiles = (Mr + kPairBM - 1) / kPairBM;
  c.map.nv = epi.d / kPairBN;
  c.map.nk = c.n_tiles - c.map.nv;
  c.Mr = Mr;
  c.err = err;
  Bars* bars = c.bars;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kPairStages; ++s) {
      ptx::mbar_init(&bars->full[s], 1);
      ptx::mbar_init(&bars->empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      ptx::mbar_init(&bars->tfull[a], 1);
      ptx::mbar_init(&bars->tempty[a], 16);   // 8 epilogue warps in each CTA of the pair
    }
    for (int w = 0; w < 8; ++w) ptx::mbar_init(&bars->hbar[w], 1);
    ptx::mbar_init(&bars->drain, 1);
    bars->abort = 0;
    ptx::fence_mbar_init();
  }
  if (warp == 1) {
    ptx::tmem_alloc_pair(&bars->tmem_base, kPairTmemCols);
    ptx::tmem_relinquish_pair();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  // this CTA's barriers are initialised: tell the peer now, wait for its
  // signal only before the first access to the peer's barriers
  ptx::cluster_arrive();
  if (warp == 0 && lane == 0) {
    ptx::tma_prefetch_desc(&tmA);
    ptx::tma_prefetch_desc(&tmB);
    ptx::tma_prefetch_desc(&tmV);
    ptx::tma_prefetch_desc(&tmH);
    // W_kv is written by no kernel before this one: the B halves of the first
    // tiles go to L2 while the previous kernel drains
    if (c.pair < c.num_tiles) {
      int mt, nt;
      c.map.at(c.pair, mt, nt);
      const int nb = nt * kPairBN + static_cast<int>(c.rank) * 128;
      for (int kb = 0; kb < c.k_blocks; ++kb) ptx::tma_prefetch_l2_2d(&tmB, kb * kBK, nb);
    }
  }
  const uint32_t tmem = bars->tmem_base;
  ptx::cluster_wait();
  ptx::grid_dep_wait();
  ptx::grid_dep_launch();

  if (warp == 0) {
    if (lane == 0) pair_producer(c, &tmA, &tmB);
  } else if (warp == 1) {
    if (lane == 0 && c.rank == 0) pair_mma(c, tmem);
  } else {
    pair_epilogue(c, tmem, epi, &tmV, &tmH, warp, lane);
  }

  __syncthreads();
  if (threadIdx.x == 0 && *reinterpret_cast<volatile int*>(&bars->abort)) {
    const uint64_t t0 = ptx::globaltimer_ns();
    while (ptx::globaltimer_ns() - t0 < kGraceNs) {
    }
  }
  ptx::cluster_sync();                        // both CTAs done with each other's barriers and TMEM
  if (warp == 1) {
    __syncwarp();
    ptx::tc_fence_after();
    ptx::tmem_dealloc_pair(tmem, kPairTmemCols);
  }
}

// Pairs that can be resident at once (clusters of two SMs with this kernel's
// shared memory), per device.
int max_pairs(int num_sms) {
  static int cached[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  if (cached[dev] > 0) return cached[dev];
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(static_cast<unsigned>(num_sms & ~1));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kPairSmem;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, gemm_pair_kernel, &cfg) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  cached[dev] = n;
  return n;
}

}  // namespace

bool gemm_pair_applies(int64_t Mr, int d, int Kd) {
  return Mr >= kPairBM && d % kPairBN == 0 && Kd % kBK == 0;
}

cudaError_t gemm_bf16_engram_pair(const void* e, const void* w_kv, int64_t Mr, int d, int M, int Kd, const void* H,
                                  const float* g_h, const float* g_k, float* v32, float* part, int* n_sl,
                                  int* pstride, int num_sms, uint32_t* err, cudaStream_t s) {
  if (!gemm_pair_applies(Mr, d, Kd) || Mr > INT32_MAX) return cudaErrorInvalidValue;
  const int Nc = (M + 1) * d;
  EngramEpilogue epi{v32, part, static_cast<const __nv_bfloat16*>(H), g_h, g_k, d, M, 0, 0, nullptr, nullptr};
  epi.n_sl = d / (kPairBN / 2);
  epi.pstride = (epi.n_sl * (1 + 3 * M) + 3) / 4 * 4;
  *n_sl = epi.n_sl;
  *pstride = epi.pstride;
  CUtensorMap ta, tb, tv, th;
  if (!make_tensor_map_2d(&ta, e, false, static_cast<uint64_t>(Kd), static_cast<uint64_t>(Mr),
                          static_cast<uint64_t>(Kd) * 2, kBK, 128, true) ||
      !make_tensor_map_2d(&tb, w_kv, false, static_cast<uint64_t>(Kd), static_cast<uint64_t>(Nc),
                          static_cast<uint64_t>(Kd) * 2, kBK, 128, true) ||
      !make_tensor_map_2d(&tv, v32, true, static_cast<uint64_t>(d), static_cast<uint64_t>(Mr),
                          static_cast<uint64_t>(d) * 4, 32, 32, true) ||
      !make_tensor_map_3d_bf16(&th, H, static_cast<uint64_t>(d), static_cast<uint64_t>(M), static_cast<uint64_t>(Mr),
                               static_cast<uint64_t>(d) * 2, static_cast<uint64_t>(d) * M * 2, 64, 1, 32, true))
    return cudaErrorInvalidValue;
  static bool attr_set = false;   // idempotent if raced
  if (!attr_set) {
    cudaError_t r = cudaFuncSetAttribute(gemm_pair_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kPairSmem);
    if (r != cudaSuccess) return r;
    attr_set = true;
  }
  const int64_t tiles = ((Mr + kPairBM - 1) / kPairBM) * (Nc / kPairBN);
  int pairs = max_pairs(num_sms);
  if (pairs <= 0) return cudaErrorInvalidConfiguration;
  if (pairs > num_sms / 2) pairs = num_sms / 2 > 0 ? num_sms / 2 : 1;   // the SMs granted to this launch
  if (tiles < pairs) pairs = static_cast<int>(tiles);
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(static_cast<unsigned>(2 * pairs));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kPairSmem;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, gemm_pair_kernel, ta, tb, tv, th, static_cast<int>(Mr), Nc, Kd, err, epi);
}

}  // namespace engram
