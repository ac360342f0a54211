// A decode step -- one new token for each of B sequences -- of the whole
// Engram layer of "DeepSeek Engram 系列导读" (section "Engram 工作原理"), Steps
// 1-8, in ONE cooperative launch.
//
// Why: at one position per sequence the layer moves a few MB (W_kv once, 16
// table rows and the conv ring per sequence) and is bound by latency, not
// bandwidth: as three kernels (gather, K/V projection, tail) every kernel
// boundary costs a launch and a pipeline drain.  The indices of Stage A depend
// on the tokens only, so one launch can walk ids -> rows -> projection ->
// gate, conv, residual and state.
//
// One block per SM (all co-resident: a cooperative launch), 320 threads, in
// three phases linked by counters in the caller's workspace:
//   1. gather: every warp of the grid takes tokens (warp w of block c: token
//      w * grid + c, ...) and writes its e row (the gather kernel's row and
//      chunk phases); the block then adds 1 to `gathered` with release
//      semantics (its rows made visible to the copy engine first).
//   2. K/V projection: the blocks with a 128 x 64 output tile run the roles of
//      the tcgen05 GEMM (gemm_parts.cuh: TMA producer, MMA issuer, the fused
//      epilogue that stores v and the gate's partial sums); the producer first
//      waits (acquire, bounded) until every block has gathered; after each
//      tile every epilogue warp publishes its stores and adds 1 to the tile's
//      row-block counter (release).
//   3. tail: block c takes sequences c, c + grid, ..., two at a time on the
//      two halves of the block; thread 0 waits (acquire, bounded) until their
//      row blocks have all their epilogue arrivals, then each half runs the
//      decode tail of its sequence (tail_parts.cuh: gate, conv from the ring,
//      H += Y, ring slot, projected ids, position).
// A phase waits only on earlier phases of resident blocks, which never wait
// on later ones, so every wait ends; each is bounded in time anyway (an
// expired wait records ENGRAM_ERR_TIMEOUT and the block skips the rest).  The
// results are the three-launch path's bits: the same per-token arithmetic,
// GEMM tiles and tail.  The counters are zeroed by a one-block kernel
// launched just before on the same stream.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "engram_internal.h"
#include "gather_parts.cuh"
#include "gemm_parts.cuh"
#include "ptx.cuh"
#include "tail_parts.cuh"

namespace engram {
namespace {

constexpr int kDecBN = 64;                         // K/V tile: 128 tokens x 64 output columns
using DG = gk::Cfg<kDecBN, true>;
constexpr int kDecW = 4;                           // conv taps (the pages' short conv)
constexpr uint64_t kDecWaitNs = 1000000000ull;     // 1 s: a healthy phase ends in microseconds

struct DecodeArgs {
  const PlanDev* pdg;        // per-row table constants
  int R, N, K, V, B;
  uint32_t* err;
  const int32_t* ids;        // [B] raw ids of the new position
  const int32_t* proj;       // [V]
  int32_t* prev;             // [B, N-1] projected ids before it (read in phase 1, rolled in phase 3)
  const uint8_t* table;
  const __half* scales;
  uint4* e;                  // [B, d_mem] gathered rows
  int do_gather;             // 0: e is given (Stage A ran earlier)
  const float* v;            // [B, d] fp32, from the epilogue
  const float* part;         // gate partials, pstride floats per token
  int n_sl, pstride, saw;
  float eps;
  int M, d, dil, L;
  const float* g_c;
  const float* conv;
  float* ring;
  int32_t* pos;
  float* sa_out;
  __nv_bfloat16* H;
  uint32_t* gathered;        // blocks done with phase 1
  uint32_t* done;            // [m_tiles] epilogue arrivals per 128-token row block
  uint32_t done_target;      // 8 warps x column tiles
};

// Wait (acquire at GPU scope, bounded) until *p >= target.
__device__ __forceinline__ bool wait_at_least(const uint32_t* p, uint32_t target) {
  const uint64_t t0 = ptx::globaltimer_ns();
  while (ptx::ld_acquire_gpu(p) < target) {
    if (ptx::globaltimer_ns() - t0 > kDecWaitNs) return false;
    ptx::nanosleep(64);
  }
  return true;
}

template <int kCpr, bool kInt8>
__global__ void __launch_bounds__(gk::kThreads, 1)
    decode_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                  const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmH, int Nc, int Kd,
                  const gk::EngramEpilogue epi, const DecodeArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  __shared__ float s_sa[2][2 * kMaxM];
  __shared__ int s_ok;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  gk::GemmCtx c = gk::gemm_ctx<kDecBN, true>(smem, a.B, Nc, Kd, a.err);
  gk::gemm_setup<kDecBN, true>(c, warp, lane);
  if (warp == 0 && lane == 0) {
    ptx::tma_prefetch_desc(&tmA);
    ptx::tma_prefetch_desc(&tmB);
    ptx::tma_prefetch_desc(&tmV);
    ptx::tma_prefetch_desc(&tmH);
    gk::gemm_prefetch_b<kDecBN, true>(c, &tmB);     // W_kv is written by no kernel: into L2 now
  }
  const bool has0 = lane < a.R;
  ga::RowConst rc[1];
  if (has0) rc[0] = ga::row_const(a.pdg, a.K, lane);
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  c.tmem = c.bars->tmem_base;
  ptx::grid_dep_wait();
  ptx::grid_dep_launch();

  // ---------------------------------------------------------------- 1. gather
  if (a.do_gather) {
    bool bad = false;
    uint32_t n_look = 0, n_hit = 0;
    const int per_tok = a.R * kCpr;
    const int n_w = static_cast<int>(gridDim.x) * (gk::kThreads / 32);
    for (int tok = warp * static_cast<int>(gridDim.x) + static_cast<int>(blockIdx.x); tok < a.B; tok += n_w) {
      const int32_t x = ga::window_hop2(ga::window_hop1(a.ids, a.prev, tok, 1, a.N, a.V, lane, bad), a.proj);
      uint32_t xp[kMaxN] = {};
      ga::window_broadcast(x, a.N, xp);
      const int32_t z_none[1] = {0};
      uint64_t src[1];
      float sc[1];
      ga::row_phase<kCpr, kInt8, true, false, false>(rc, has0, false, xp, z_none, a.table, a.scales, ga::RowCache{},
                                                     lane, src, sc, bad, n_look, n_hit);
      ga::chunk_phase<kCpr, kInt8, false>(src, sc, a.R, a.e + static_cast<int64_t>(kInt8 ? 2 : 1) * tok * per_tok,
                                          lane, [] {});
    }
    if (bad) atomicOr(a.err, kErrIndexRange);
    ptx::fence_proxy_async_global();             // the rows, for other blocks' TMA loads
    __syncthreads();
    if (threadIdx.x == 0) {
      __threadfence();
      ptx::red_release_gpu_add(a.gathered, 1u);
    }
  }

  // ---------------------------------------------------------------- 2. K/V projection
  if (static_cast<int>(blockIdx.x) < c.num_tiles) {
    if (warp == 0) {
      if (lane == 0) {
        bool ok = true;
        if (a.do_gather) {
          ok = wait_at_least(a.gathered, gridDim.x);
          ptx::fence_proxy_async_global();       // the copies below see what the generic proxy released
        }
        if (ok) {
          gk::gemm_producer<kDecBN, true>(c, &tmA, &tmB);
        } else {
          atomicOr(a.err, kErrTimeout);
          *reinterpret_cast<volatile int*>(&c.bars->abort) = 1;
        }
      }
    } else if (warp == 1) {
      if (lane == 0) gk::gemm_mma<kDecBN, true>(c);
    } else {
      gk::gemm_epilogue<kDecBN, true, true>(c, epi, &tmV, &tmH, nullptr, warp, lane, a.done);
    }
  }
  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    ptx::tc_fence_after();
    ptx::tmem_dealloc(c.tmem, DG::kTmemCols);
  }

  // ---------------------------------------------------------------- 3. tail
  // sequences b0 = c, c + 2 grid, ... with b1 = b0 + grid beside them: two at
  // a time on the two halves of the block (named barriers), else one on all of it
  const int G = static_cast<int>(gridDim.x);
  for (int b0 = blockIdx.x; b0 < a.B; b0 += 2 * G) {
    const int b1 = b0 + G;
    const bool two = b1 < a.B;
    if (threadIdx.x == 0) {
      bool ok = wait_at_least(a.done + b0 / gk::kBM, a.done_target);
      if (ok && two) ok = wait_at_least(a.done + b1 / gk::kBM, a.done_target);
      s_ok = ok ? 1 : 0;
    }
    __syncthreads();
    if (!s_ok) {
      if (threadIdx.x == 0) atomicOr(a.err, kErrTimeout);
      break;
    }
    if (two) {
      constexpr int kHalf = gk::kThreads / 2;      // five warps each
      const int grp = static_cast<int>(threadIdx.x) >= kHalf ? 1 : 0;
      cv::decode_tail_seq<__nv_bfloat16, kDecW, true, false>(
          grp ? b1 : b0, threadIdx.x - grp * kHalf, kHalf, s_sa[grp], a.part, a.n_sl, a.pstride, a.saw, a.eps, a.v,
          a.d, a.M, a.d, a.dil, a.g_c, a.conv, a.ring, a.pos, a.L, a.ids, a.proj, a.V, a.prev, a.N, a.sa_out, a.err,
          a.H, [grp] { ptx::named_barrier(1 + grp, kHalf); });
    } else {
      cv::decode_tail_seq<__nv_bfloat16, kDecW, true, false>(
          b0, threadIdx.x, blockDim.x, s_sa[0], a.part, a.n_sl, a.pstride, a.saw, a.eps, a.v, a.d, a.M, a.d, a.dil,
          a.g_c, a.conv, a.ring, a.pos, a.L, a.ids, a.proj, a.V, a.prev, a.N, a.sa_out, a.err, a.H,
          [] { __syncthreads(); });
    }
    __syncthreads();                             // s_sa and s_ok are the next pair's
  }
}

// Blocks of the one-launch decode that can be resident at once on this device
// (one per SM at this shared memory); 0 if the kernel cannot be configured.
template <int kCpr, bool kInt8>
int resident_blocks(int num_sms) {
  static int cached[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  if (cached[dev] > 0) return cached[dev];
  if (cudaFuncSetAttribute(decode_kernel<kCpr, kInt8>, cudaFuncAttributeMaxDynamicSharedMemorySize, DG::kSmem) !=
      cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, decode_kernel<kCpr, kInt8>, gk::kThreads, DG::kSmem) !=
      cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  cached[dev] = per_sm * num_sms;
  return cached[dev];
}

template <int kCpr, bool kInt8>
cudaError_t decode_launch(const CUtensorMap& ta, const CUtensorMap& tb, const CUtensorMap& tv, const CUtensorMap& th,
                          int Nc, int Kd, const gk::EngramEpilogue& epi, const DecodeArgs& a, int num_sms,
                          cudaStream_t s) {
  const int blocks = resident_blocks<kCpr, kInt8>(num_sms);
  if (blocks <= 0) return cudaErrorCooperativeLaunchTooLarge;
  const int grid = blocks < num_sms ? blocks : num_sms;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(static_cast<unsigned>(grid));
  cfg.blockDim = dim3(gk::kThreads);
  cfg.dynamicSmemBytes = DG::kSmem;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  cudaError_t e = cudaLaunchKernelEx(&cfg, decode_kernel<kCpr, kInt8>, ta, tb, tv, th, Nc, Kd, epi, a);
  if (e != cudaSuccess && e != cudaErrorCooperativeLaunchTooLarge) {
    // without overlap of the previous kernel's tail, if the two attributes do not combine here
    (void)cudaGetLastError();
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, decode_kernel<kCpr, kInt8>, ta, tb, tv, th, Nc, Kd, epi, a);
  }
  return e;
}

}  // namespace

bool decode_fused_applies(const engram_plan* p, int T) {
  return T == 1 && p->cfg.act_dtype == ENGRAM_BF16 && p->R <= 32 && p->cfg.conv_w == kDecW &&
         p->cfg.d % kDecBN == 0 && p->d_mem % gk::kBK == 0 && p->cfg.table_dtype != ENGRAM_F32;
}

cudaError_t launch_decode_fused(const engram_plan* p, const int32_t* ids, int B, const int32_t* proj, int V,
                                const void* table, const uint16_t* scales, const void* e, bool do_gather,
                                const engram_weights_t* w, void* H, const engram_state_t* state,
                                const Workspace& ws, cudaStream_t s) {
  const int d = p->cfg.d, M = p->cfg.M, Kd = p->d_mem, Nc = (M + 1) * d;
  const int64_t Mr = B;
  gk::EngramEpilogue epi{ws.v32, ws.part, static_cast<const __nv_bfloat16*>(H), w->g_h, w->g_k, d, M, 0, 0,
                         nullptr, nullptr};
  epi.n_sl = d / (kDecBN / 2);
  epi.pstride = (epi.n_sl * (1 + 3 * M) + 3) / 4 * 4;
  CUtensorMap ta, tb, tv, th;
  if (!make_tensor_map_2d(&ta, e, false, static_cast<uint64_t>(Kd), static_cast<uint64_t>(Mr),
                          static_cast<uint64_t>(Kd) * 2, gk::kBK, gk::kBM, true) ||
      !make_tensor_map_2d(&tb, w->w_kv, false, static_cast<uint64_t>(Kd), static_cast<uint64_t>(Nc),
                          static_cast<uint64_t>(Kd) * 2, gk::kBK, kDecBN, true) ||
      !make_tensor_map_2d(&tv, ws.v32, true, static_cast<uint64_t>(d), static_cast<uint64_t>(Mr),
                          static_cast<uint64_t>(d) * 4, 32, 32, true) ||
      !make_tensor_map_3d_bf16(&th, H, static_cast<uint64_t>(d), static_cast<uint64_t>(M),
                               static_cast<uint64_t>(Mr), static_cast<uint64_t>(d) * 2,
                               static_cast<uint64_t>(d) * M * 2, 64, 1, 32, true))
    return cudaErrorInvalidValue;
  const int m_tiles = static_cast<int>((Mr + gk::kBM - 1) / gk::kBM);
  DecodeArgs a{};
  a.pdg = p->dev;
  a.R = p->R;
  a.N = p->cfg.N;
  a.K = p->cfg.K;
  a.V = V;
  a.B = B;
  a.err = &p->dev->err;
  a.ids = ids;
  a.proj = proj;
  a.prev = state ? state->prev_ids : nullptr;
  a.table = static_cast<const uint8_t*>(table);
  a.scales = reinterpret_cast<const __half*>(scales);
  a.e = static_cast<uint4*>(const_cast<void*>(e));
  a.do_gather = do_gather ? 1 : 0;
  a.v = ws.v32;
  a.part = ws.part;
  a.n_sl = epi.n_sl;
  a.pstride = epi.pstride;
  a.saw = sa_row_floats(M);
  a.eps = p->cfg.eps;
  a.M = M;
  a.d = d;
  a.dil = p->cfg.conv_dilation;
  a.L = p->L_ring;
  a.g_c = w->g_c;
  a.conv = w->conv;
  a.ring = state ? state->u_ring : nullptr;
  a.pos = state ? state->pos : nullptr;
  a.sa_out = ws.sa;
  a.H = static_cast<__nv_bfloat16*>(H);
  a.gathered = ws.sync;
  a.done = ws.sync + 1;
  a.done_target = 8u * static_cast<uint32_t>(Nc / kDecBN);
  cudaError_t err = launch_zero_words(ws.sync, m_tiles + 1, s);
  if (err != cudaSuccess) return err;
  const bool i8 = p->cfg.table_dtype == ENGRAM_I8_ROWSCALE_F16;
  const int cpr = p->cfg.row_dim * (i8 ? 1 : 2) / 16;
#define ENGRAM_DEC(C, I) decode_launch<C, I>(ta, tb, tv, th, Nc, Kd, epi, a, p->num_sms, s)
  switch (cpr) {
    case 1: return i8 ? ENGRAM_DEC(1, true) : ENGRAM_DEC(1, false);
    case 2: return i8 ? ENGRAM_DEC(2, true) : ENGRAM_DEC(2, false);
    case 4: return i8 ? ENGRAM_DEC(4, true) : ENGRAM_DEC(4, false);
    case 8: return i8 ? ENGRAM_DEC(8, true) : ENGRAM_DEC(8, false);
    case 16: return i8 ? ENGRAM_DEC(16, true) : ENGRAM_DEC(16, false);
    default: return cudaErrorInvalidValue;
  }
#undef ENGRAM_DEC
}

}  // namespace engram
