// Step 4 of "DeepSeek Engram 系列导读", section "Engram 工作原理", Stage A:
// e_t = concat_{n,k} E_{n,k}[z_{t,n,k}], plus the int8 row dequantisation that
// "Engram 嵌入扩展：面向高效 DRAM/SSD 卸载的协同设计" (section "AgentX Engram
// DRAM卸载提升性能") fuses into the same row-selecting kernel, for tables in HBM
// or in pinned host memory reached over UVA (NVLink-C2C on Grace-Blackwell).
//
// Layout trick: because the R rows of one token are concatenated in (n,k)
// order, the 16-byte chunk f = r * chunks_per_row + c of a token's rows is
// also the 16-byte slot of its output (copy) or 32-byte slot (int8 -> bf16).
// A warp owns one token: consecutive lanes read consecutive chunks of a row
// (one 64/128-byte transaction per row) and write contiguous output, so no
// shared-memory staging is needed for coalescing; each lane keeps several
// independent 16-byte loads in flight before it stores anything.
//
// The same kernel serves engram_gather (indices read from memory) and
// engram_forward (indices computed from the token ids for the rows about to
// be read, Steps 1-3 -- the arithmetic of hashing.cuh -- so they never
// travel through HBM).  There the warp first loads the token's n-gram window
// (lane i holds x'_{t-i}) and broadcasts it by shuffle; lane r computes the
// index of row r once, and the lanes reading that row's chunks get its
// address by shuffle.
//
// Variants: tokens of at most 16 rows and 64 chunks (int8 rows of 64 bytes)
// take half a warp each (row_gather_half_kernel), so a warp carries two
// tokens' rows at once; for the FP8 projection the row kernel can write the
// token's e4m3 codes and scale instead of e (kQ8, the rule of e4m3.cuh).
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "e4m3.cuh"
#include "engram_internal.h"
#include "gather_parts.cuh"
#include "ptx.cuh"

namespace engram {
namespace {

using namespace ga;

constexpr int kThreads = 128;

// Each warp walks its tokens tok, tok + n_warps, ... as a two-stage software
// pipeline: while one token's table rows are in flight, the next token's
// n-gram window is fetched (its raw ids before the row loads are issued, their
// projections right after), so a warp's consecutive tokens overlap their
// dependent memory round trips instead of paying them one after another.
//
// Per token (one warp).  Row phase: lane r (and r + 32) owns row r of the
// token -- its index (computed from the n-gram window, or read), its source
// address (table, or the HBM cache) and its int8 scale -- so each row's index
// is computed once.  Chunk phase: lane l takes the token's 16-byte chunks
// l, l + 32, ... (chunk f = r * kCpr + c is also the output's slot f), gets
// its row's address by shuffle and keeps kWarpItems independent loads in
// flight before storing; consecutive lanes read consecutive chunks of a row
// and write contiguous output.  The per-row constants come from the device
// copy of the parameter block, read before the dependency wait (they are
// written at plan creation only).
// kWide: R > 32, two rows per lane.
// kBlk: threads per block -- 128 (eight blocks per SM), or 1024 for tables in
// host memory, so that a grid of hostgrid_sms blocks holds that many whole SMs
// and leaves the others to the work running beside the lookup.
// (The row and chunk phases are written out here, not through ga::row_phase
// and ga::chunk_phase as in decode.cu: this form measured 7 % faster.)
// kQ8 (bf16 rows, a token's chunks within one round of loads): instead of
// e, the token's e4m3 codes and scale for the FP8 projection, from the row
// the warp holds in registers (the arithmetic of e4m3.cuh, so the bytes of
// the quantisation kernel run on e).
template <int kCpr, bool kInt8, bool kHash, bool kCache = false, bool kWide = false, int kBlk = kThreads,
          bool kQ8 = false>
__global__ void __launch_bounds__(kBlk, kThreads * 8 / kBlk)
    row_gather_kernel(const GatherLayers ls, int R, int N, int K, const int32_t* __restrict__ idx,
                      const int32_t* __restrict__ ids, int T, const int32_t* __restrict__ proj, int V, int64_t ntok,
                      const RowCache cache) {
  constexpr int kRowBytes = kCpr * 16;
  const int lane = threadIdx.x & 31;
  // this block's layer: blockIdx.y (the layers share ids, proj and the table shape)
  const int ly = static_cast<int>(blockIdx.y);
  const PlanDev* __restrict__ pdg = ls.pdg[ly];
  uint32_t* __restrict__ err = ls.err[ly];
  const int32_t* __restrict__ prev = ls.prev[ly];
  const uint8_t* __restrict__ table = ls.table[ly];
  const __half* __restrict__ scales = ls.scales[ly];
  uint4* __restrict__ out = ls.out[ly];
  uint8_t* __restrict__ q8 = ls.q8[ly];
  float* __restrict__ qscale = ls.qscale[ly];
  constexpr int kRows = kWide ? 2 : 1;
  const bool has0 = lane < R, has1 = kWide && lane + 32 < R;
  RowConst rc[kRows];
  if (has0) rc[0] = row_const(pdg, K, lane);
  if (kWide && has1) rc[kRows - 1] = row_const(pdg, K, lane + 32);
  if constexpr (kHash) {
    // P (read at random, written by no kernel) into L2 while the ids load: one 128-byte line per thread
    const int64_t line = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (ly == 0 && line * 32 < V) ptx::prefetch_l2(proj + line * 32);
  }
  ptx::grid_dep_wait();
  ptx::grid_dep_launch();

  const int per_tok = R * kCpr;
  const int64_t n_warps = static_cast<int64_t>(gridDim.x) * (blockDim.x >> 5);
  bool bad = false;
  uint32_t n_look = 0, n_hit = 0;                       // this lane's rows (kCache)
  int64_t tok = static_cast<int64_t>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5);
  // pipeline state: the current token's projected window id (kHash) or row index (read)
  int32_t x_cur = 0;
  int32_t z_cur[kRows] = {};
  if (tok < ntok) {
    if constexpr (kHash) {
      x_cur = window_hop2(window_hop1(ids, prev, tok, T, N, V, lane, bad), proj);
    } else {
      if (has0) z_cur[0] = ld_nc_s32(idx + tok * R + lane);
      if (kWide && has1) z_cur[kRows - 1] = ld_nc_s32(idx + tok * R + lane + 32);
    }
  }
  for (; tok < ntok; tok += n_warps) {
    const int64_t tn = tok + n_warps;
    const bool more = tn < ntok;
    // next token, first hop (raw ids, or its row indices)
    WindowHop hop{0, false};
    int32_t z_next[kRows] = {};
    if (more) {
      if constexpr (kHash) {
        hop = window_hop1(ids, prev, tn, T, N, V, lane, bad);
      } else {
        if (has0) z_next[0] = ld_nc_s32(idx + tn * R + lane);
        if (kWide && has1) z_next[kRows - 1] = ld_nc_s32(idx + tn * R + lane + 32);
      }
    }
    uint32_t xp[kMaxN];                                // projected ids: non-negative int32
    if constexpr (kHash) {
#pragma unroll
      for (int i = 0; i < kMaxN; ++i)
        if (i < N) xp[i] = static_cast<uint32_t>(__shfl_sync(0xFFFFFFFFu, x_cur, i));
    }
    // ---- row phase: index, source and scale of rows lane and lane + 32
    uint64_t src[kRows] = {};                          // 0: the row is out of range (zero output)
    float sc[kRows] = {};
#pragma unroll
    for (int h = 0; h < kRows; ++h) {
      const bool has = h == 0 ? has0 : has1;
      if (!has) continue;
      const RowConst& c = rc[h];
      uint32_t z;
      if constexpr (kHash) {
        uint64_t hsh = 0;
#pragma unroll
        for (int i = 0; i < kMaxN; ++i)
          if (i < c.n) hsh ^= static_cast<uint64_t>(xp[i]) * __ldg(c.mult + i);
        z = barrett_mod(hsh, c.prime, c.mu);
      } else {
        z = static_cast<uint32_t>(z_cur[h]);
        if (z >= c.prime) {
          bad = true;
          continue;
        }
      }
      const int64_t row = c.offset + z;
      const uint8_t* p = table + row * kRowBytes;
      if constexpr (kCache) {
        const int32_t sl = __ldg(cache.slot + row);
        if (sl >= 0) p = cache.rows + static_cast<int64_t>(sl) * kRowBytes;
        ++n_look;
        n_hit += sl >= 0;
      }
      src[h] = reinterpret_cast<uint64_t>(p);
      if constexpr (kInt8) sc[h] = __half2float(scales[row]);
    }
    // ---- chunk phase
    uint4* dst = out + (kInt8 ? 2 : 1) * tok * per_tok;
    for (int f0 = 0; f0 < per_tok; f0 += 32 * kWarpItems) {
      uint4 v[kWarpItems];
      float s_[kWarpItems];
      bool ok[kWarpItems];
#pragma unroll
      for (int j = 0; j < kWarpItems; ++j) {
        const int f = f0 + j * 32 + lane;
        const int r = f / kCpr;
        const int c = f % kCpr;
        // every lane takes part in the shuffles; lanes past the token's chunks discard theirs
        const int rs = r < R ? r : 0;
        uint64_t sp = shfl64(src[0], rs & 31);
        float sj = kInt8 ? __shfl_sync(0xFFFFFFFFu, sc[0], rs & 31) : 0.f;
        if constexpr (kWide) {
          const uint64_t sp1 = shfl64(src[kRows - 1], rs & 31);
          const float sj1 = kInt8 ? __shfl_sync(0xFFFFFFFFu, sc[kRows - 1], rs & 31) : 0.f;
          if (rs >= 32) {
            sp = sp1;
            sj = sj1;
          }
        }
        ok[j] = f < per_tok && sp != 0;
        v[j] = ok[j] ? ld_stream_16(reinterpret_cast<const uint8_t*>(sp) + c * 16) : make_uint4(0, 0, 0, 0);
        s_[j] = sj;
      }
      if (f0 == 0) {
        // next token, second hop, while this token's rows are in flight
        if constexpr (kHash) {
          if (more) x_cur = window_hop2(hop, proj);
        }
      }
      if constexpr (kQ8) {
        // the token's whole row is in this round's registers: its amax, scale and codes
        float amax = 0.f;
#pragma unroll
        for (int j = 0; j < kWarpItems; ++j)
          if (f0 + j * 32 + lane < per_tok) amax = e4m3::amax8(v[j], amax);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, o));
        const float inv = e4m3::inv_of(amax);
        if (lane == 0) qscale[tok] = e4m3::scale_of(amax);
        uint2* qd = reinterpret_cast<uint2*>(q8 + tok * per_tok * 8);
#pragma unroll
        for (int j = 0; j < kWarpItems; ++j) {
          const int f = f0 + j * 32 + lane;
          if (f < per_tok) qd[f] = e4m3::quant8(v[j], inv);
        }
      } else {
#pragma unroll
        for (int j = 0; j < kWarpItems; ++j) {
          const int f = f0 + j * 32 + lane;
          if (f < per_tok) {
            if constexpr (kInt8) {
              uint4 o0 = make_uint4(0, 0, 0, 0), o1 = make_uint4(0, 0, 0, 0);
              if (ok[j]) dequant16(v[j], s_[j], o0, o1);
              dst[2 * f] = o0;
              dst[2 * f + 1] = o1;
            } else {
              dst[f] = v[j];
            }
          }
        }
      }
    }
    if constexpr (!kHash) {
#pragma unroll
      for (int h = 0; h < kRows; ++h) z_cur[h] = z_next[h];
    }
  }
  if (bad) atomicOr(err, kErrIndexRange);
  if constexpr (kCache) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      n_look += __shfl_xor_sync(0xFFFFFFFFu, n_look, o);
      n_hit += __shfl_xor_sync(0xFFFFFFFFu, n_hit, o);
    }
    if (lane == 0 && n_look) {
      atomicAdd(cache.stats, static_cast<unsigned long long>(n_look));
      atomicAdd(cache.stats + 1, static_cast<unsigned long long>(n_hit));
    }
  }
}

// Steps 1-4 for tokens of at most 16 rows and 64 chunks (int8 rows of 64
// bytes at R = 16): one token's chunk phase would fill only half of a warp's
// load slots, so each half-warp owns a token -- two tokens per warp pass,
// twice a warp's rows in flight with the same registers.  Lane h*16 + i holds
// row i, and window entry i, of half h's token; otherwise the row kernel's
// pipeline, phases and arithmetic, per half.
template <int kCpr, bool kInt8, bool kCache, int kBlk>
__global__ void __launch_bounds__(kBlk, kThreads * 8 / kBlk)
    row_gather_half_kernel(const GatherLayers ls, int R, int N, int K, const int32_t* __restrict__ ids, int T,
                           const int32_t* __restrict__ proj, int V, int64_t ntok, const RowCache cache) {
  constexpr int kRowBytes = kCpr * 16;
  const int lane = threadIdx.x & 31;
  const int hl = lane & 15, hb = lane & 16;            // lane within the half; the half's first lane
  const int ly = static_cast<int>(blockIdx.y);
  const PlanDev* __restrict__ pdg = ls.pdg[ly];
  uint32_t* __restrict__ err = ls.err[ly];
  const int32_t* __restrict__ prev = ls.prev[ly];
  const uint8_t* __restrict__ table = ls.table[ly];
  const __half* __restrict__ scales = ls.scales[ly];
  uint4* __restrict__ out = ls.out[ly];
  const bool has = hl < R;
  RowConst rc{};
  if (has) rc = row_const(pdg, K, hl);
  {
    const int64_t line = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (ly == 0 && line * 32 < V) ptx::prefetch_l2(proj + line * 32);
  }
  ptx::grid_dep_wait();
  ptx::grid_dep_launch();

  const int per_tok = R * kCpr;                          // <= 64: four chunks per lane of a half
  const int64_t stride = 2 * static_cast<int64_t>(gridDim.x) * (blockDim.x >> 5);
  bool bad = false;
  uint32_t n_look = 0, n_hit = 0;
  // a warp's pair of tokens: base (lanes 0-15) and base + 1 (lanes 16-31); base is warp-uniform
  int64_t base = 2 * (static_cast<int64_t>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5));
  int32_t x_cur = 0;
  if (base + (hb >> 4) < ntok) x_cur = window_hop2(window_hop1(ids, prev, base + (hb >> 4), T, N, V, hl, bad), proj);
  for (; base < ntok; base += stride) {
    const int64_t tok = base + (hb >> 4);
    const bool live = tok < ntok;
    const int64_t tn = tok + stride;
    const bool more = tn < ntok;
    WindowHop hop{0, false};
    if (more) hop = window_hop1(ids, prev, tn, T, N, V, hl, bad);
    uint32_t xp[kMaxN];
#pragma unroll
    for (int i = 0; i < kMaxN; ++i)
      if (i < N) xp[i] = static_cast<uint32_t>(__shfl_sync(0xFFFFFFFFu, x_cur, hb + i));
    // ---- row phase: lane hl < R of each half, row hl of the half's token
    uint64_t src = 0;
    float sc = 0.f;
    if (has && live) {
      uint64_t hsh = 0;
#pragma unroll
      for (int i = 0; i < kMaxN; ++i)
        if (i < rc.n) hsh ^= static_cast<uint64_t>(xp[i]) * __ldg(rc.mult + i);
      const int64_t row = rc.offset + barrett_mod(hsh, rc.prime, rc.mu);
      const uint8_t* p = table + row * kRowBytes;
      if constexpr (kCache) {
        const int32_t sl = __ldg(cache.slot + row);
        if (sl >= 0) p = cache.rows + static_cast<int64_t>(sl) * kRowBytes;
        ++n_look;
        n_hit += sl >= 0;
      }
      src = reinterpret_cast<uint64_t>(p);
      if constexpr (kInt8) sc = __half2float(scales[row]);
    }
    // ---- chunk phase: chunk f = j * 16 + hl of the half's token
    uint4* dst = out + (kInt8 ? 2 : 1) * tok * per_tok;
    uint4 v[kWarpItems];
    float s_[kWarpItems];
    bool ok[kWarpItems];
#pragma unroll
    for (int j = 0; j < kWarpItems; ++j) {
      const int f = j * 16 + hl;
      const int r = f / kCpr;
      const int c = f % kCpr;
      const int rs = r < R ? r : 0;
      const uint64_t sp = shfl64(src, hb + rs);
      s_[j] = kInt8 ? __shfl_sync(0xFFFFFFFFu, sc, hb + rs) : 0.f;
      ok[j] = live && f < per_tok && sp != 0;
      v[j] = ok[j] ? ld_stream_16(reinterpret_cast<const uint8_t*>(sp) + c * 16) : make_uint4(0, 0, 0, 0);
    }
    // next pair's second hop while these rows are in flight
    if (more) x_cur = window_hop2(hop, proj);
#pragma unroll
    for (int j = 0; j < kWarpItems; ++j) {
      const int f = j * 16 + hl;
      if (live && f < per_tok) {
        if constexpr (kInt8) {
          uint4 o0 = make_uint4(0, 0, 0, 0), o1 = make_uint4(0, 0, 0, 0);
          if (ok[j]) dequant16(v[j], s_[j], o0, o1);
          dst[2 * f] = o0;
          dst[2 * f + 1] = o1;
        } else {
          dst[f] = v[j];
        }
      }
    }
  }
  if (bad) atomicOr(err, kErrIndexRange);
  if constexpr (kCache) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      n_look += __shfl_xor_sync(0xFFFFFFFFu, n_look, o);
      n_hit += __shfl_xor_sync(0xFFFFFFFFu, n_hit, o);
    }
    if (lane == 0 && n_look) {
      atomicAdd(cache.stats, static_cast<unsigned long long>(n_look));
      atomicAdd(cache.stats + 1, static_cast<unsigned long long>(n_hit));
    }
  }
}

// SMs a gather over the host link occupies: one 1024-thread block each.  An
// SM keeps 32 warps' row loads in flight (a token's rows each, the next
// token's window behind them), so a quarter of the SMs already carries the
// ~200 GB/s the link delivers (NVLink-C2C, as measured with pinned copies);
// the rest stay free for work that runs beside the lookup.
constexpr int kHostBlk = 1024;

int grid_for_tokens(const engram_plan* p, int64_t ntok, bool host_table = false) {
  const int64_t warps_per_block = (host_table ? kHostBlk : kThreads) / 32;
  int64_t blocks = (ntok + warps_per_block - 1) / warps_per_block;
  const int64_t cap = host_table ? hostgrid_sms(p) : static_cast<int64_t>(p->num_sms) * 8;
  if (blocks > cap) blocks = cap;
  return static_cast<int>(blocks);
}

GatherLayers one_layer(const engram_plan* p, const int32_t* prev, const void* table, const uint16_t* scales,
                       void* e) {
  GatherLayers ls{};
  ls.pdg[0] = p->dev;
  ls.err[0] = &p->dev->err;
  ls.prev[0] = prev;
  ls.table[0] = static_cast<const uint8_t*>(table);
  ls.scales[0] = reinterpret_cast<const __half*>(scales);
  ls.out[0] = static_cast<uint4*>(e);
  return ls;
}

template <int kCpr, bool kInt8>
cudaError_t launch_idx(const engram_plan* p, const int32_t* idx, int64_t ntok, const void* table,
                       const uint16_t* scales, void* e, cudaStream_t s) {
  auto k = p->R > 32 ? row_gather_kernel<kCpr, kInt8, false, false, true> : row_gather_kernel<kCpr, kInt8, false>;
  return launch_pdl(k, dim3(grid_for_tokens(p, ntok)), dim3(kThreads), 0, s, one_layer(p, nullptr, table, scales, e),
                    p->R, p->cfg.N, p->cfg.K, idx, static_cast<const int32_t*>(nullptr), 1,
                    static_cast<const int32_t*>(nullptr), 0, ntok, RowCache{});
}

// Steps 1-4 for n_layers layers of one shape in one launch (grid.y = layer);
// with tables in host memory, the grid's share of the SMs is split among them.
template <int kCpr, bool kInt8>
cudaError_t launch_fused(const engram_plan* p, int n_layers, const GatherLayers& ls, const int32_t* ids, int B, int T,
                         const int32_t* proj, int V, cudaStream_t s, bool host_table, const RowCache* cache,
                         bool q8 = false) {
  const int64_t ntok = static_cast<int64_t>(B) * T;
  int gx = grid_for_tokens(p, ntok, host_table);
  const int cap = host_table ? hostgrid_sms(p) : p->num_sms * 8;   // one wave over all layers
  if (static_cast<int64_t>(gx) * n_layers > cap) gx = cap / n_layers > 0 ? cap / n_layers : 1;
  const dim3 grid(gx, n_layers);
  const dim3 block(host_table ? kHostBlk : kThreads);
  const bool wide = p->R > 32;
  if (q8) {
    if constexpr (!kInt8) {
      // e4m3 codes of bf16 rows: the token's chunks within one round of loads
      if (cache != nullptr || wide || p->R * kCpr > 32 * kWarpItems || p->cfg.table_dtype != ENGRAM_BF16)
        return cudaErrorInvalidValue;
      auto k = host_table ? row_gather_kernel<kCpr, false, true, false, false, kHostBlk, true>
                          : row_gather_kernel<kCpr, false, true, false, false, kThreads, true>;
      return launch_pdl(k, grid, block, 0, s, ls, p->R, p->cfg.N, p->cfg.K, static_cast<const int32_t*>(nullptr), ids,
                        T, proj, V, ntok, RowCache{});
    }
    return cudaErrorInvalidValue;
  }
  if constexpr (kCpr <= 4) {
    if (p->R <= 16 && kCpr * p->R <= 64) {
      // half a warp per token
      const RowCache rcache = cache != nullptr ? *cache : RowCache{};
      auto k = cache != nullptr ? row_gather_half_kernel<kCpr, kInt8, true, kThreads>
                                : row_gather_half_kernel<kCpr, kInt8, false, kThreads>;
      if (host_table)
        k = cache != nullptr ? row_gather_half_kernel<kCpr, kInt8, true, kHostBlk>
                             : row_gather_half_kernel<kCpr, kInt8, false, kHostBlk>;
      return launch_pdl(k, grid, block, 0, s, ls, p->R, p->cfg.N, p->cfg.K, ids, T, proj, V, ntok, rcache);
    }
  }
  if (cache != nullptr) {
    auto k = wide ? row_gather_kernel<kCpr, kInt8, true, true, true> : row_gather_kernel<kCpr, kInt8, true, true>;
    if (host_table)
      k = wide ? row_gather_kernel<kCpr, kInt8, true, true, true, kHostBlk>
               : row_gather_kernel<kCpr, kInt8, true, true, false, kHostBlk>;
    return launch_pdl(k, grid, block, 0, s, ls, p->R, p->cfg.N, p->cfg.K, static_cast<const int32_t*>(nullptr), ids,
                      T, proj, V, ntok, *cache);
  }
  auto k = wide ? row_gather_kernel<kCpr, kInt8, true, false, true> : row_gather_kernel<kCpr, kInt8, true>;
  if (host_table)
    k = wide ? row_gather_kernel<kCpr, kInt8, true, false, true, kHostBlk>
             : row_gather_kernel<kCpr, kInt8, true, false, false, kHostBlk>;
  return launch_pdl(k, grid, block, 0, s, ls, p->R, p->cfg.N, p->cfg.K, static_cast<const int32_t*>(nullptr), ids, T,
                    proj, V, ntok, RowCache{});
}

int chunks_per_row(const engram_plan* p) {
  const int elem = p->cfg.table_dtype == ENGRAM_F32 ? 4 : (p->cfg.table_dtype == ENGRAM_BF16 ? 2 : 1);
  return p->cfg.row_dim * elem / 16;
}

}  // namespace

#define ENGRAM_DISPATCH_CPR(CALL)                                                  \
  switch (chunks_per_row(p)) {                                                     \
    case 1: return i8 ? CALL(1, true) : CALL(1, false);                            \
    case 2: return i8 ? CALL(2, true) : CALL(2, false);                            \
    case 4: return i8 ? CALL(4, true) : CALL(4, false);                            \
    case 8: return i8 ? CALL(8, true) : CALL(8, false);                            \
    case 16: return i8 ? CALL(16, true) : CALL(16, false);                         \
    default: return cudaErrorInvalidValue;                                         \
  }

cudaError_t launch_gather(const engram_plan* p, const int32_t* idx, int64_t ntok, const void* table,
                          const uint16_t* scales, void* e, cudaStream_t s) {
  const bool i8 = p->cfg.table_dtype == ENGRAM_I8_ROWSCALE_F16;
#define CALL(C, I) launch_idx<C, I>(p, idx, ntok, table, scales, e, s)
  ENGRAM_DISPATCH_CPR(CALL)
#undef CALL
}

cudaError_t launch_hash_gather(const engram_plan* p, const int32_t* ids, int B, int T, const int32_t* proj, int V,
                               const int32_t* prev_ids, const void* table, const uint16_t* scales, void* e,
                               cudaStream_t s, bool host_table) {
  const bool i8 = p->cfg.table_dtype == ENGRAM_I8_ROWSCALE_F16;
  const GatherLayers ls = one_layer(p, prev_ids, table, scales, e);
#define CALL(C, I) launch_fused<C, I>(p, 1, ls, ids, B, T, proj, V, s, host_table, nullptr)
  ENGRAM_DISPATCH_CPR(CALL)
#undef CALL
}

cudaError_t launch_hash_gather_cached(const engram_plan* p, const int32_t* ids, int B, int T, const int32_t* proj,
                                      int V, const int32_t* prev_ids, const void* table, const uint16_t* scales,
                                      void* e, const int32_t* slot, const void* rows, unsigned long long* stats,
                                      cudaStream_t s, bool host_table) {
  const bool i8 = p->cfg.table_dtype == ENGRAM_I8_ROWSCALE_F16;
  const RowCache cache{slot, static_cast<const uint8_t*>(rows), stats};
  const GatherLayers ls = one_layer(p, prev_ids, table, scales, e);
#define CALL(C, I) launch_fused<C, I>(p, 1, ls, ids, B, T, proj, V, s, host_table, &cache)
  ENGRAM_DISPATCH_CPR(CALL)
#undef CALL
}

cudaError_t launch_hash_gather_layers(const engram_plan* const* plans, int n_layers, const int32_t* ids, int B, int T,
                                      const int32_t* proj, int V, const int32_t* const* prev_ids,
                                      const void* const* tables, const uint16_t* const* scales, void* const* e,
                                      cudaStream_t s, bool host_table) {
  if (n_layers < 1 || n_layers > kMaxGatherLayers) return cudaErrorInvalidValue;
  const engram_plan* p = plans[0];
  GatherLayers ls{};
  for (int l = 0; l < n_layers; ++l) {
    ls.pdg[l] = plans[l]->dev;
    ls.err[l] = &plans[l]->dev->err;
    ls.prev[l] = prev_ids != nullptr ? prev_ids[l] : nullptr;
    ls.table[l] = static_cast<const uint8_t*>(tables[l]);
    ls.scales[l] = scales != nullptr ? reinterpret_cast<const __half*>(scales[l]) : nullptr;
    ls.out[l] = static_cast<uint4*>(e[l]);
  }
  const bool i8 = p->cfg.table_dtype == ENGRAM_I8_ROWSCALE_F16;
#define CALL(C, I) launch_fused<C, I>(p, n_layers, ls, ids, B, T, proj, V, s, host_table, nullptr)
  ENGRAM_DISPATCH_CPR(CALL)
#undef CALL
}

bool gather_e4m3_applies(const engram_plan* p) {
  return p->cfg.table_dtype == ENGRAM_BF16 && p->cfg.act_dtype == ENGRAM_BF16 && p->R <= 32 &&
         p->R * chunks_per_row(p) <= 32 * kWarpItems;
}

cudaError_t launch_hash_gather_layers_e4m3(const engram_plan* const* plans, int n_layers, const int32_t* ids, int B,
                                           int T, const int32_t* proj, int V, const int32_t* const* prev_ids,
                                           const void* const* tables, uint8_t* const* e8, float* const* e_scale,
                                           cudaStream_t s, bool host_table) {
  if (n_layers < 1 || n_layers > kMaxGatherLayers || !gather_e4m3_applies(plans[0])) return cudaErrorInvalidValue;
  const engram_plan* p = plans[0];
  GatherLayers ls{};
  for (int l = 0; l < n_layers; ++l) {
    ls.pdg[l] = plans[l]->dev;
    ls.err[l] = &plans[l]->dev->err;
    ls.prev[l] = prev_ids != nullptr ? prev_ids[l] : nullptr;
    ls.table[l] = static_cast<const uint8_t*>(tables[l]);
    ls.q8[l] = e8[l];
    ls.qscale[l] = e_scale[l];
  }
  const bool i8 = false;
#define CALL(C, I) launch_fused<C, I>(p, n_layers, ls, ids, B, T, proj, V, s, host_table, nullptr, true)
  ENGRAM_DISPATCH_CPR(CALL)
#undef CALL
}

cudaError_t launch_hash_gather_e4m3(const engram_plan* p, const int32_t* ids, int B, int T, const int32_t* proj, int V,
                                    const int32_t* prev_ids, const void* table, uint8_t* e8, float* e_scale,
                                    cudaStream_t s, bool host_table) {
  return launch_hash_gather_layers_e4m3(&p, 1, ids, B, T, proj, V, prev_ids ? &prev_ids : nullptr, &table, &e8,
                                        &e_scale, s, host_table);
}

#undef ENGRAM_DISPATCH_CPR

}  // namespace engram
