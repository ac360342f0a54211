// Building blocks of the tcgen05 K/V projection: configuration, shared-memory
// barriers, the fused Engram epilogue and the three warp roles of the
// persistent kernel (TMA producer, MMA issuer, epilogue).  gemm.cu composes
// them into the standalone GEMM; stage_b.cu into the kernel that also runs
// the conv.  See gemm.cu for the design.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "engram_internal.h"
#include "ptx.cuh"

namespace engram {
namespace gk {

constexpr int kBM = 128;
constexpr int kBK = 64;                        // bf16 elements per k-block: one 128-byte swizzle atom
constexpr int kThreads = 320;                 // producer, MMA, 8 epilogue warps
constexpr uint64_t kWaitLimitNs = 1000000000ull;   // 1 s: a healthy stage turns over in < 1 us

constexpr int kEpiWarpBytes = 8192;            // fused epilogue: per-warp staging of v chunks / the H slice

// kF8: e4m3 operands (128 elements per 128-byte k-block, kind::f8f6f4) with
// per-row scales applied in the epilogue; else bf16 (64 per k-block, kind::f16).
template <int BN, bool kFused, bool kF8 = false>
struct Cfg {
  static constexpr int kStages = kFused ? (BN == 256 ? 3 : (BN == 128 ? 4 : 6)) : (BN == 256 ? 4 : (BN == 128 ? 6 : 8));
  static constexpr int kBKe = kF8 ? 128 : kBK;  // elements per k-block
  static constexpr int kABytes = kBM * 128;
  static constexpr int kBBytes = BN * 128;
  static constexpr int kStageBytes = kABytes + kBBytes;
  // fused: 8 warps x (the warp's staging, then its columns' g_h and g_k: BN/2 floats each)
  static constexpr int kGWarpBytes = kFused ? BN * 4 : 0;
  static constexpr int kEpiBytes = kFused ? 8 * (kEpiWarpBytes + kGWarpBytes) : 0;
  static constexpr int kTmemCols = 2 * BN < 32 ? 32 : 2 * BN;
  static constexpr int kBarBytes = 256;
  static constexpr int kSmem = 1024 + kStages * kStageBytes + kEpiBytes + kBarBytes;
  static constexpr uint32_t kIdesc = kF8 ? ptx::idesc_e4m3_f32(kBM, BN) : ptx::idesc_bf16_f32(kBM, BN);
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
  const float* s_row;             // e4m3 operands: [Mr] scale of each row of e
  const float* s_col;             // e4m3 operands: [(M+1)d] scale of each row of W_kv
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
// Rows of part are pstride floats apart (padded to 16 bytes).  Within one
// 32-column tcgen05.ld chunk each sum is four interleaved fmaf chains (column
// j of the chunk in chain j % 4, so the dependent chains are 8 deep, not 32),
// combined as (c0 + c1) + (c2 + c3); a
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
// e4m3 operands (kF8): the accumulator of row t, column n is the dot product
// of the quantised codes; each is first multiplied by s_row[t] * s_col[n].
template <bool kF8>
__device__ __forceinline__ void dequant_chunk(const EngramEpilogue& epi, float srow, int n, uint32_t (&r)[32]) {
  if constexpr (kF8) {
    const float4* sc = reinterpret_cast<const float4*>(epi.s_col + n);
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      const float4 c4 = __ldg(sc + q);
      r[4 * q] = __float_as_uint(__uint_as_float(r[4 * q]) * (srow * c4.x));
      r[4 * q + 1] = __float_as_uint(__uint_as_float(r[4 * q + 1]) * (srow * c4.y));
      r[4 * q + 2] = __float_as_uint(__uint_as_float(r[4 * q + 2]) * (srow * c4.z));
      r[4 * q + 3] = __float_as_uint(__uint_as_float(r[4 * q + 3]) * (srow * c4.w));
    }
  }
}

// gs: the warp's copy of g_h (then g_k) over its BN/2 columns of a k tile.
template <int BN, bool kF8 = false>
__device__ __forceinline__ void fused_epilogue(const EngramEpilogue& epi, const CUtensorMap* tmV, uint8_t* eb,
                                               const float* gs, uint32_t t_row, int row, int row0, int Mr, int n0,
                                               int c_lo, int lane) {
  constexpr int SW = BN / 2;
  const float srow = kF8 && row < Mr ? __ldg(epi.s_row + row) : 0.f;
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
      dequant_chunk<kF8>(epi, srow, n0 + c, r);
      float a[4] = {0.f, 0.f, 0.f, 0.f};       // column j of the chunk goes to chain j % 4
#pragma unroll
      for (int j = 0; j < 32; ++j) a[j & 3] = fmaf(__uint_as_float(r[j]), __uint_as_float(r[j]), a[j & 3]);
      float sv = (a[0] + a[1]) + (a[2] + a[3]);
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
    (void)col;
    float s_dot[3], s_sk[3], s_sh[3];
    int top = 0;
#pragma unroll
    for (int ci = 0; ci < kChunks; ++ci) {
      const int c = c_lo + ci * 32;
      uint32_t r[32];
      ptx::tmem_ld_32x32b_x32(t_row + c, r);
      ptx::tmem_ld_wait();
      dequant_chunk<kF8>(epi, srow, n0 + c, r);
      float d4[4] = {0.f, 0.f, 0.f, 0.f}, k4[4] = {0.f, 0.f, 0.f, 0.f}, h4[4] = {0.f, 0.f, 0.f, 0.f};
      const uint8_t* hb = eb + (ci >> 1) * 4096 + lane * 128;     // this row of the chunk's 64-column box
      const float4* gh4 = reinterpret_cast<const float4*>(gs + ci * 32);        // shared: broadcast reads
      const float4* gk4 = reinterpret_cast<const float4*>(gs + SW + ci * 32);
#pragma unroll
      for (int q4 = 0; q4 < 4; ++q4) {
        const uint4 hv = *reinterpret_cast<const uint4*>(hb + ((((ci & 1) * 4 + q4) ^ swz) << 4));
        const uint32_t hw[4] = {hv.x, hv.y, hv.z, hv.w};
        const float4 ga = gh4[2 * q4], gb = gh4[2 * q4 + 1];
        const float4 ka = gk4[2 * q4], kb = gk4[2 * q4 + 1];
        const float g[8] = {ga.x * ka.x, ga.y * ka.y, ga.z * ka.z, ga.w * ka.w,
                            gb.x * kb.x, gb.y * kb.y, gb.z * kb.z, gb.w * kb.w};
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const float h = __uint_as_float(i & 1 ? (hw[i >> 1] & 0xFFFF0000u) : (hw[i >> 1] << 16));
          const float k = __uint_as_float(r[q4 * 8 + i]);
          d4[i & 3] = fmaf(h * g[i], k, d4[i & 3]);
          k4[i & 3] = fmaf(k, k, k4[i & 3]);
          h4[i & 3] = fmaf(h, h, h4[i & 3]);
        }
      }
      float dot = (d4[0] + d4[1]) + (d4[2] + d4[3]);
      float sk = (k4[0] + k4[1]) + (k4[2] + k4[3]);
      float sh = (h4[0] + h4[1]) + (h4[2] + h4[3]);
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

// Per-CTA view of one launch.
struct GemmCtx {
  uint8_t* smem;        // 1024-byte aligned: kStages operand stages
  uint8_t* epi_smem;    // fused: 8 x kEpiWarpBytes epilogue staging
  Bars* bars;
  uint32_t tmem;
  int m_tiles, n_tiles, num_tiles, k_blocks;
  int Mr, Nc, Kd;
  uint32_t* err;
};

// `bars`: where the barrier block lives; null = right after the epilogue staging.
template <int BN, bool kFused, bool kF8 = false>
__device__ __forceinline__ GemmCtx gemm_ctx(uint8_t* smem, int Mr, int Nc, int Kd, uint32_t* err,
                                            Bars* bars = nullptr) {
  using G = Cfg<BN, kFused, kF8>;
  GemmCtx c;
  c.smem = smem;
  c.epi_smem = smem + G::kStages * G::kStageBytes;
  c.bars = bars != nullptr ? bars : reinterpret_cast<Bars*>(c.epi_smem + G::kEpiBytes);
  c.tmem = 0;
  c.m_tiles = (Mr + kBM - 1) / kBM;
  c.n_tiles = (Nc + BN - 1) / BN;
  c.num_tiles = c.m_tiles * c.n_tiles;
  c.k_blocks = (Kd + G::kBKe - 1) / G::kBKe;
  c.Mr = Mr;
  c.Nc = Nc;
  c.Kd = Kd;
  c.err = err;
  return c;
}

// Barrier initialisation (thread 0) and TMEM allocation (warp 1); the caller
// then synchronises the block with tcgen05 fences around the barrier and
// reads the TMEM base from bars->tmem_base.
template <int BN, bool kFused, bool kF8 = false>
__device__ __forceinline__ void gemm_setup(const GemmCtx& c, int warp, int lane) {
  using G = Cfg<BN, kFused, kF8>;
  Bars* bars = c.bars;
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
  (void)lane;
  if (warp == 1) {
    ptx::tmem_alloc(&bars->tmem_base, G::kTmemCols);
    ptx::tmem_relinquish();
  }
}

// Warp 0, lane 0, before the dependency wait: W_kv into L2, each column
// panel by one block (the blocks of the first row block).  W_kv is not
// written by the kernel before, and a prefetch changes no data, so it may
// overlap that kernel.
template <int BN, bool kFused, bool kF8 = false>
__device__ __forceinline__ void gemm_prefetch_b(const GemmCtx& c, const CUtensorMap* tmB) {
  using G = Cfg<BN, kFused, kF8>;
  if (static_cast<int>(blockIdx.x) >= c.n_tiles || static_cast<int>(blockIdx.x) >= c.num_tiles) return;
  const int n0 = (static_cast<int>(blockIdx.x) % c.n_tiles) * BN;
  for (int kb = 0; kb < c.k_blocks; ++kb) ptx::tma_prefetch_l2_2d(tmB, kb * G::kBKe, n0);
}

// Warp 0, lane 0.
template <int BN, bool kFused, bool kF8 = false>
__device__ __forceinline__ void gemm_producer(const GemmCtx& c, const CUtensorMap* tmA, const CUtensorMap* tmB) {
  using G = Cfg<BN, kFused, kF8>;
  Bars* bars = c.bars;
  uint8_t* smem = c.smem;
  uint32_t* err = c.err;
  const int n_tiles = c.n_tiles, num_tiles = c.num_tiles, k_blocks = c.k_blocks;
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
      ptx::tma_load_2d_nohint(sa, tmA, &bars->full[stage], kb * G::kBKe, m0);
      ptx::tma_load_2d(sa + G::kABytes, tmB, &bars->full[stage], kb * G::kBKe, n0, keep);
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

// Warp 1, lane 0.
template <int BN, bool kFused, bool kF8 = false>
__device__ __forceinline__ void gemm_mma(const GemmCtx& c) {
  using G = Cfg<BN, kFused, kF8>;
  Bars* bars = c.bars;
  uint8_t* smem = c.smem;
  uint32_t* err = c.err;
  const uint32_t tmem = c.tmem;
  const int num_tiles = c.num_tiles, k_blocks = c.k_blocks;
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
      for (int k = 0; k < 4; ++k) {            // 32 bytes of K per instruction: 16 bf16 or 32 e4m3
        if constexpr (kF8)
          ptx::mma_e4m3(d_tmem, ptx::sdesc_kmajor_sw128(a_addr + k * 32), ptx::sdesc_kmajor_sw128(b_addr + k * 32),
                        G::kIdesc, (kb | k) != 0);
        else
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

// Warps 2..9.  kSignal: after each tile, the warp's global writes are made
// visible device-wide (its TMA stores completed, proxy and memory fences) and
// the warp adds one to row_done[tile's row block] with release semantics, so
// a row block is complete once its counter reaches 8 x (column tiles).
template <int BN, bool kFused, bool kSignal, bool kF8 = false>
__device__ __forceinline__ void gemm_epilogue(const GemmCtx& c, const EngramEpilogue& epi, const CUtensorMap* tmV_,
                                              const CUtensorMap* tmH_, __nv_bfloat16* C, int warp, int lane,
                                              uint32_t* row_done) {
  static_assert(kFused || !kF8, "e4m3 operands only with the Engram epilogue");
  using G = Cfg<BN, kFused, kF8>;
  Bars* bars = c.bars;
  uint8_t* epi_smem = c.epi_smem;
  uint32_t* err = c.err;
  const uint32_t tmem = c.tmem;
  const int n_tiles = c.n_tiles, num_tiles = c.num_tiles, Mr = c.Mr, Nc = c.Nc;
  const CUtensorMap& tmV = *tmV_;
  const CUtensorMap& tmH = *tmH_;
  const int q = warp & 3;                 // TMEM lane quadrant this warp may access
  const int ew = warp - 2;
  const int c_lo = (ew >> 2) * (BN / 2);  // half of the tile's columns
  uint8_t* eb = epi_smem + ew * kEpiWarpBytes;
  float* gs = reinterpret_cast<float*>(epi_smem + 8 * kEpiWarpBytes + ew * G::kGWarpBytes);
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
        ptx::mbar_arrive_expect_tx(&bars->hbar[ew], G::kHBoxes * 4096 + G::kGWarpBytes);
        // the slice's RMSNorm weights, read by every lane of every row: one copy into shared memory
        const int64_t go = static_cast<int64_t>(m) * epi.d + col;
        ptx::bulk_load(gs, epi.g_h + go, G::kGWarpBytes / 2, &bars->hbar[ew]);
        ptx::bulk_load(gs + BN / 2, epi.g_k + go, G::kGWarpBytes / 2, &bars->hbar[ew]);
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
      fused_epilogue<BN, kF8>(epi, &tmV, eb, gs, t_row, row, m0 + q * 32, Mr, n0, c_lo, lane);
    }
    ptx::tc_fence_before();
    __syncwarp();
    if (lane == 0) ptx::mbar_arrive(&bars->tempty[acc]);
    if constexpr (kSignal) {
      if (lane == 0) {
        ptx::bulk_wait_all();                 // this tile's v stores are in global memory
        ptx::fence_proxy_async_global();
      }
      __threadfence();                        // and every lane's partial sums
      __syncwarp();
      if (lane == 0) ptx::red_release_gpu_add(row_done + tile / n_tiles, 1u);
    }
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

}  // namespace gk
}  // namespace engram
