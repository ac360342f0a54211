// Internal declarations shared by the host API and the kernel files.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <utility>
#include <vector>

#include "../../include/engram.h"

namespace engram {

constexpr int kMaxR = 64;          // (N-1)*K
constexpr int kMaxMults = 320;     // sum_{n=2..N} K*n with (N-1)*K <= 64, N <= 8
constexpr int kMaxN = 8;
constexpr int kMaxConvW = 8;
constexpr int kMaxM = 8;
constexpr int kMaxGatherLayers = 8;   // layers one engram_stage_a_layers launch gathers for

// bits of the device error word
constexpr uint32_t kErrIndexRange = 1u;
constexpr uint32_t kErrTimeout = 2u;

// Parameter block of a plan.  A device copy holds the error word; kernels get
// the parameters by value (a __grid_constant__ argument, read from the
// constant bank), so no block starts with a dependent global load.
struct PlanDev {
  uint32_t err;                    // error word (atomicOr from kernels)
  int32_t R;
  int32_t N;
  int32_t K;
  uint32_t primes[kMaxR];          // rows of table r = (n-2)*K + k
  uint64_t mu[kMaxR];              // floor(2^64 / p_r) for the Barrett remainder
  int64_t offsets[kMaxR];          // first row of table r in the concatenated table
  int32_t mult_base[kMaxN + 1];    // index of m_{n,0,0} in mults, per order n
  uint64_t mults[kMaxMults];
};

}  // namespace engram

struct engram_plan {
  engram_config_t cfg;             // host copy; the two array pointers are cleared
  int R;
  int d_mem;
  int L_ring;                      // (conv_w - 1) * conv_dilation
  int64_t max_tokens;
  int64_t total_rows;
  int device;
  int num_sms;
  std::vector<uint32_t> primes;
  std::vector<uint64_t> mults;
  std::vector<int64_t> offsets;
  engram::PlanDev* dev;            // device copy of the parameter block (its err word is live)
  engram::PlanDev host;            // host copy, passed to kernels by value
  // tracing: events recorded around each kernel of the last engram_forward
  static constexpr int kMaxMarks = 8;
  cudaEvent_t marks[kMaxMarks];
  bool timing;
  mutable int n_marks;
  bool fused_stage_b;              // Stage B as one cooperative launch where launch_stage_b_fused applies
  bool cta_pairs;                  // the K/V projection's 256-column tiles on CTA pairs (gemm_pair.cu)
  bool fused_decode;               // chunks of one position as one cooperative launch (decode.cu)
  int sm_limit;                    // SMs Stage B's persistent kernels may use (0: all)
  int host_sms;                    // blocks of a Stage A over host-memory tables (0: a quarter of the SMs)
};

namespace engram {

// An SM split (smsplit.cu): each group's stream and SM count, and events for
// ordering the two streams (kSplitEvents of them, created with the split).
constexpr int kMaxPieces = 64;
constexpr int kSplitEvents = kMaxPieces + 3;
cudaStream_t split_stream(const engram_sm_split* sp, int group);
int split_sms(const engram_sm_split* sp, int group);
cudaEvent_t split_event(const engram_sm_split* sp, int i);

// SMs a Stage A over tables in host memory occupies (gather.cu): one 1024-thread block each.
inline int hostgrid_sms(const engram_plan* p) {
  if (p->host_sms > 0) return p->host_sms < p->num_sms ? p->host_sms : p->num_sms;
  return p->num_sms / 4 > 0 ? p->num_sms / 4 : 1;
}

// SMs the persistent Stage B kernels (K/V projection, conv) size their grids and tiles for.
inline int stage_b_sms(const engram_plan* p) {
  return p->sm_limit > 0 && p->sm_limit < p->num_sms ? p->sm_limit : p->num_sms;
}

// Launch `k` with programmatic stream serialisation: its blocks may be
// scheduled while the previous kernel on `s` drains; the kernel itself waits
// (grid_dep_wait in ptx.cuh) before it reads or writes anything shared.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*k)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s, Args&&... args) {
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, k, std::forward<Args>(args)...);
}

// Workspace carve-up for engram_forward / engram_stage_b, 256-byte aligned parts.
struct Workspace {
  int32_t* idx;      // [ntok, R]
  void* e;           // [ntok, d_mem] act dtype
  float* kv;         // f32 layers: [ntok, (M+1)d] = [v | k^(1..M)]
  float* v32;        // bf16 layers: [ntok, d] v in fp32 (fused K/V epilogue)
  float* part;       // bf16 layers: gate partial sums, at most (d/32)(1+3M) per token (rows padded to 4)
  float* sa;         // [ntok, sa_row_floats(M)]: s^(1..M) = alpha/sqrt(mean(v~^2)+eps), then alpha^(1..M)
  uint32_t* sync;    // bf16 layers: stage_b_sync_words(ntok) counters of the fused Stage-B kernel
  uint8_t* e8;       // bf16 layers: [ntok, d_mem] e4m3 codes of e (FP8 projection)
  float* e_scale;    // bf16 layers: [ntok] their per-token scales
  size_t bytes;
};
Workspace carve_workspace(const engram_plan* p, int64_t ntok, void* base);

// ---- launchers (each returns cudaGetLastError() after the launch) ----
cudaError_t launch_hash(const engram_plan* p, const int32_t* ids, int B, int T, const int32_t* proj, int V,
                        const int32_t* prev_ids, int32_t* idx, cudaStream_t s);
cudaError_t launch_gather(const engram_plan* p, const int32_t* idx, int64_t ntok, const void* table,
                          const uint16_t* scales, void* e, cudaStream_t s);
// Steps 1-4 fused: indices computed per row inside the gather, never stored.
// host_table: the rows are read from pinned host memory over the host link;
// the grid then holds a share of the SMs sized for the link (one 1024-thread
// block on each of hostgrid_sms SMs), leaving the rest to concurrent work (the
// Stage-A prefetch beside earlier layers).
cudaError_t launch_hash_gather(const engram_plan* p, const int32_t* ids, int B, int T, const int32_t* proj, int V,
                               const int32_t* prev_ids, const void* table, const uint16_t* scales, void* e,
                               cudaStream_t s, bool host_table = false);
// Steps 1-4 of n_layers layers in one launch (the layers share ids, P and the
// table shape; each has its own plan, tables, state ids and output).
cudaError_t launch_hash_gather_layers(const engram_plan* const* plans, int n_layers, const int32_t* ids, int B, int T,
                                      const int32_t* proj, int V, const int32_t* const* prev_ids,
                                      const void* const* tables, const uint16_t* const* scales, void* const* e,
                                      cudaStream_t s, bool host_table = false);
// Steps 1-4 writing e's e4m3 codes and per-token scales instead of e (the FP8
// projection's input), for bf16 tables of at most 32 rows and 128 chunks per
// token (gather_e4m3_applies); else cudaErrorInvalidValue.
bool gather_e4m3_applies(const engram_plan* p);
cudaError_t launch_hash_gather_e4m3(const engram_plan* p, const int32_t* ids, int B, int T, const int32_t* proj, int V,
                                    const int32_t* prev_ids, const void* table, uint8_t* e8, float* e_scale,
                                    cudaStream_t s, bool host_table);
cudaError_t launch_hash_gather_layers_e4m3(const engram_plan* const* plans, int n_layers, const int32_t* ids, int B,
                                           int T, const int32_t* proj, int V, const int32_t* const* prev_ids,
                                           const void* const* tables, uint8_t* const* e8, float* const* e_scale,
                                           cudaStream_t s, bool host_table);
// The same through the HBM hot-row cache (slot map, cached rows, [lookups, hits] counters).
cudaError_t launch_hash_gather_cached(const engram_plan* p, const int32_t* ids, int B, int T, const int32_t* proj,
                                      int V, const int32_t* prev_ids, const void* table, const uint16_t* scales,
                                      void* e, const int32_t* slot, const void* rows, unsigned long long* stats,
                                      cudaStream_t s, bool host_table = false);
// Hot-row cache maintenance (cache.cu).
cudaError_t cache_observe(const engram_plan* p, const int32_t* ids, int B, int T, const int32_t* proj, int V,
                          const int32_t* prev_ids, uint32_t* counts, cudaStream_t s);
cudaError_t cache_build(const engram_plan* p, int64_t capacity, int row_bytes, const void* table, uint32_t* counts,
                        int32_t* slot, void* rows, unsigned long long* used, int decay, int64_t* cached,
                        cudaStream_t s);
// Per-batch row dedup through the cache's slot map (cache.cu): each distinct
// row without a slot is claimed by one lookup f (slot first_slot + f; owner[f]
// = its table row, else 0xFFFFFFFF) and copied into row f of the batch region;
// after the gather the release returns the slots to -1 and adds the claims to
// *fetched.
cudaError_t dedup_claim(const engram_plan* p, const int32_t* ids, int B, int T, const int32_t* proj, int V,
                        const int32_t* prev_ids, int32_t* slot, int32_t first_slot, uint32_t* owner, cudaStream_t s);
cudaError_t dedup_fetch(const engram_plan* p, int64_t total, const uint32_t* owner, int row_bytes, const void* table,
                        void* region, cudaStream_t s);
cudaError_t dedup_release(const engram_plan* p, int64_t total, const uint32_t* owner, int32_t* slot,
                          unsigned long long* fetched, cudaStream_t s);
cudaError_t launch_kv_projection(const engram_plan* p, const void* e, int64_t ntok, const void* w_kv, void* kv,
                                 cudaStream_t s);
// Floats per row of the per-token gate scalars: [s^(1..M), alpha^(1..M)] padded to 16 bytes.
int sa_row_floats(int M);
cudaError_t launch_gate_f32(const engram_plan* p, const float* kv, const float* H, int64_t ntok, const float* g_h,
                            const float* g_k, float* sa, cudaStream_t s);
// bf16 layers: the K/V epilogue's partial sums (n_sl nodes per quantity, rows
// pstride floats apart) -> sa rows.
cudaError_t launch_finalize(const engram_plan* p, const float* part, int n_sl, int pstride, int64_t ntok, float* sa,
                            cudaStream_t s);
// Conv + SiLU + skip + residual over B sequences of T positions (v fp32 with
// row stride sv; sa rows [s^(1..M), alpha^(1..M)] per token).
// With `part` (bf16 layers where conv_fuses_gate holds) the conv computes the
// gate scalars from the K/V epilogue's partials itself (sa_out: where to also
// store them for the streaming state, or null) and sa is not read.
cudaError_t launch_conv_residual(const engram_plan* p, const float* v, int64_t sv, const float* sa, int B, int T,
                                 const float* g_c, const float* conv, void* H, const engram_state_t* state,
                                 cudaStream_t s, const float* part = nullptr, float* sa_out = nullptr);
// Whether the conv can compute the gate scalars itself for this layer shape
// (one branch, 8 slices per quantity: 32 partials per row).
bool conv_fuses_gate(const engram_plan* p, int n_sl, int pstride);
// Steps 6-8 and the state update for one position per sequence (decode) in one
// launch: gate scalars from sa_in (fp32 layers) or the partials (bf16 layers,
// also written to sa_out), conv from the ring, H += Y, ring/prev_ids/pos update.
cudaError_t launch_decode_tail(const engram_plan* p, const float* v, int64_t sv, const float* sa_in, const float* part,
                               int n_sl, int pstride, float* sa_out, int B, const float* g_c, const float* conv,
                               void* H, const int32_t* ids, const int32_t* proj, int V, const engram_state_t* st,
                               cudaStream_t s);
cudaError_t launch_state_update(const engram_plan* p, const int32_t* ids, const int32_t* proj, int V, const float* v,
                                int64_t sv, const float* sa, int B, int T, const engram_state_t* state,
                                cudaStream_t s);

// bf16 GEMM on tcgen05: C[Mr, Nc] = A[Mr, Kd] . B[Nc, Kd]^T, all row-major bf16.
cudaError_t gemm_bf16_tcgen05(const void* A, const void* B, void* C, int64_t Mr, int Nc, int Kd, int num_sms,
                              uint32_t* err, cudaStream_t s);
// The same GEMM with the Engram epilogue: v (columns [0,d)) to v32 in fp32,
// gate partial sums of every tile to part (n_sl nodes per quantity, rows
// pstride floats apart; both returned); k is never stored.
// cta_pairs: where the tiles are 256 columns wide, run them on CTA pairs
// (gemm_bf16_engram_pair); the same bits either way.
cudaError_t gemm_bf16_engram(const void* e, const void* w_kv, int64_t Mr, int d, int M, int Kd, const void* H,
                             const float* g_h, const float* g_k, float* v32, float* part, int* n_sl, int* pstride,
                             int num_sms, uint32_t* err, cudaStream_t s, bool cta_pairs = false);
// The same GEMM and epilogue on CTA pairs (tcgen05.mma.cta_group::2, 256 x 256
// tiles per pair of SMs; gemm_pair.cu): bit-identical results, 256-column
// slices (n_sl = d / 128).  Applies when Mr >= 256, d % 256 == 0, Kd % 64 == 0.
bool gemm_pair_applies(int64_t Mr, int d, int Kd);
cudaError_t gemm_bf16_engram_pair(const void* e, const void* w_kv, int64_t Mr, int d, int M, int Kd, const void* H,
                                  const float* g_h, const float* g_k, float* v32, float* part, int* n_sl,
                                  int* pstride, int num_sms, uint32_t* err, cudaStream_t s);
// The same projection on e4m3 operands: e8 [Mr, Kd] and w8 [(M+1)d, Kd]
// quantised per row with scales s_e [Mr] and s_w [(M+1)d] (quant.cu); the
// epilogue multiplies each accumulator by its two scales.  Kd % 128 == 0.
cudaError_t gemm_e4m3_engram(const uint8_t* e8, const float* s_e, const uint8_t* w8, const float* s_w, int64_t Mr,
                             int d, int M, int Kd, const void* H, const float* g_h, const float* g_k, float* v32,
                             float* part, int* n_sl, int* pstride, int num_sms, uint32_t* err, cudaStream_t s);
// Per-row e4m3 quantisation of a bf16 [rows, cols] array (quant.cu):
// scale[i] = amax_i / 448 and q[i, j] = e4m3_satfinite(x[i, j] * (448 / amax_i)),
// both quotients in binary32; an all-zero row gets scale 1 and zero codes.
cudaError_t launch_quantize_rows_e4m3(const void* x, int64_t rows, int cols, uint8_t* q, float* scale, int num_sms,
                                      cudaStream_t s);
// 2-D tiled TMA descriptor of a row-major [rows, inner] array (fp32 or bf16),
// rows row_stride_bytes apart, box of box_rows x box_inner elements.
bool make_tensor_map_2d(CUtensorMap* map, const void* base, bool is_f32, uint64_t inner, uint64_t rows,
                        uint64_t row_stride_bytes, uint32_t box_inner, uint32_t box_rows, bool swizzle128);
// The same for a byte array (fp8 operands).
bool make_tensor_map_2d_u8(CUtensorMap* map, const void* base, uint64_t inner, uint64_t rows,
                           uint64_t row_stride_bytes, uint32_t box_inner, uint32_t box_rows, bool swizzle128);
// 3-D tiled TMA descriptor of a bf16 array with dims d0 (contiguous), d1, d2 and
// byte strides stride1, stride2 between consecutive indices of d1 and d2.
bool make_tensor_map_3d_bf16(CUtensorMap* map, const void* base, uint64_t d0, uint64_t d1, uint64_t d2,
                             uint64_t stride1_bytes, uint64_t stride2_bytes, uint32_t box0, uint32_t box1,
                             uint32_t box2, bool swizzle128);
// Stage B (Steps 5-8) of a bf16, one-branch, w = 4 layer with 128-column
// projection slices (d = 1024) and T > 1, as one cooperative launch (stage_b.cu):
// the K/V projection with its gate epilogue and the conv with the in-kernel
// gate finalisation, the conv tiles starting as soon as their row blocks are
// projected.  Bit-identical to gemm_bf16_engram + launch_conv_residual(part).
// sync: stage_b_sync_words(B*T) words of device memory (any contents).
bool stage_b_fused_applies(const engram_plan* p, int64_t ntok, int T);
size_t stage_b_sync_words(int64_t ntok);
cudaError_t launch_stage_b_fused(const engram_plan* p, const void* e, const void* w_kv, int B, int T, void* H,
                                 const float* g_h, const float* g_k, const float* g_c, const float* conv, float* v32,
                                 float* part, float* sa_out, const engram_state_t* state, uint32_t* sync,
                                 cudaStream_t s);
// Zero n words of device memory (one block, stream-ordered, programmatic
// dependent launch: it waits for the previous kernel before writing).
cudaError_t launch_zero_words(uint32_t* p, int n, cudaStream_t s);
// A whole decode step (chunks of one position, T = 1) of a bf16 layer with
// R <= 32 and conv_w = 4 as one cooperative launch (decode.cu): the gather
// (unless do_gather is false and e already holds the rows), the K/V
// projection in 128 x 64 tiles with its gate epilogue, and the decode tail,
// linked by counters in ws.sync.  Bit-identical to the gather + projection +
// decode tail launches.
bool decode_fused_applies(const engram_plan* p, int T);
cudaError_t launch_decode_fused(const engram_plan* p, const int32_t* ids, int B, const int32_t* proj, int V,
                                const void* table, const uint16_t* scales, const void* e, bool do_gather,
                                const engram_weights_t* w, void* H, const engram_state_t* state,
                                const Workspace& ws, cudaStream_t s);
// fp32 GEMM on the CUDA cores, same shapes.
cudaError_t gemm_f32_simt(const float* A, const float* B, float* C, int64_t Mr, int Nc, int Kd, cudaStream_t s);

}  // namespace engram
