// Host side of the C ABI: argument checks, the plan, workspace layout, dispatch.
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <cstring>
#include <new>

#include <nvtx3/nvToolsExt.h>

#include "engram_internal.h"

using engram::PlanDev;

namespace {

constexpr uint64_t kU64Max = ~0ull;

// Tracing: an NVTX range over each entry point that enqueues work (host side:
// the enqueue itself; a profiler shows the GPU work it launched beneath it).
// NVTX is header-only and inert unless a profiler is attached.
struct NvtxRange {
  explicit NvtxRange(const char* name) { nvtxRangePushA(name); }
  ~NvtxRange() { nvtxRangePop(); }
  NvtxRange(const NvtxRange&) = delete;
  NvtxRange& operator=(const NvtxRange&) = delete;
};

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

bool aligned16(const void* ptr) { return (reinterpret_cast<uintptr_t>(ptr) & 15u) == 0; }

size_t act_bytes(engram_dtype_t t) { return t == ENGRAM_F32 ? 4 : 2; }

size_t table_elem_bytes(engram_dtype_t t) {
  switch (t) {
    case ENGRAM_F32: return 4;
    case ENGRAM_BF16: return 2;
    default: return 1;
  }
}

engram_status_t cuda_status(cudaError_t e) { return e == cudaSuccess ? ENGRAM_OK : ENGRAM_ERR_CUDA; }

// Resolve a pointer the kernels will dereference.  Device and managed memory
// are used as is; pinned or registered host memory through its device alias;
// pageable host memory is refused.
engram_status_t device_view(const void* ptr, const void** out, bool* on_host = nullptr) {
  if (on_host) *on_host = false;
  cudaPointerAttributes a;
  cudaError_t e = cudaPointerGetAttributes(&a, ptr);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return ENGRAM_ERR_NOT_MAPPED;
  }
  switch (a.type) {
    case cudaMemoryTypeDevice:
    case cudaMemoryTypeManaged:
      *out = ptr;
      return ENGRAM_OK;
    case cudaMemoryTypeHost:
      if (a.devicePointer == nullptr) return ENGRAM_ERR_NOT_MAPPED;
      *out = a.devicePointer;
      if (on_host) *on_host = true;
      return ENGRAM_OK;
    default:
      return ENGRAM_ERR_NOT_MAPPED;
  }
}

// Tracing: record the plan's next event on `s` (no-op unless timing is on).
// Under stream capture the event becomes an event-record node of the graph
// (cudaEventRecordExternal), so every replay records it again.
void mark(const engram_plan* p, cudaStream_t s) {
  if (!p->timing || p->n_marks >= engram_plan::kMaxMarks) return;
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(s, &cs) == cudaSuccess && cs == cudaStreamCaptureStatusActive)
    cudaEventRecordWithFlags(p->marks[p->n_marks++], s, cudaEventRecordExternal);
  else
    cudaEventRecord(p->marks[p->n_marks++], s);
}

engram_status_t check_tokens(const engram_plan* p, int B, int T) {
  if (B < 0 || T < 0) return ENGRAM_ERR_INVALID_ARG;
  if (static_cast<int64_t>(B) * T > p->max_tokens) return ENGRAM_ERR_INVALID_ARG;
  return ENGRAM_OK;
}

engram_status_t check_weights(const engram_plan* p, const engram_weights_t* w, bool need_table) {
  if (!w) return ENGRAM_ERR_INVALID_ARG;
  if (!w->g_h || !w->g_k || !w->g_c || !w->conv) return ENGRAM_ERR_INVALID_ARG;
  if (!aligned16(w->g_h) || !aligned16(w->g_k) || !aligned16(w->g_c) || !aligned16(w->conv))
    return ENGRAM_ERR_INVALID_ARG;
  if ((w->w_kv_fp8 != nullptr) != (w->w_kv_scale != nullptr)) return ENGRAM_ERR_INVALID_ARG;
  if (w->w_kv_fp8) {
    if (p->cfg.act_dtype != ENGRAM_BF16 || p->d_mem % 128) return ENGRAM_ERR_UNSUPPORTED;
    if (!aligned16(w->w_kv_fp8) || !aligned16(w->w_kv_scale)) return ENGRAM_ERR_INVALID_ARG;
  } else if (!w->w_kv || !aligned16(w->w_kv)) {
    return ENGRAM_ERR_INVALID_ARG;
  }
  if (need_table) {
    if (!w->table) return ENGRAM_ERR_INVALID_ARG;
    if ((p->cfg.table_dtype == ENGRAM_I8_ROWSCALE_F16) != (w->scales != nullptr)) return ENGRAM_ERR_INVALID_ARG;
  }
  return ENGRAM_OK;
}

engram_status_t check_state(const engram_plan* p, const engram_state_t* st) {
  if (!st) return ENGRAM_OK;
  if (!st->prev_ids || !st->u_ring || !st->pos) return ENGRAM_ERR_INVALID_ARG;
  if (!aligned16(st->u_ring)) return ENGRAM_ERR_INVALID_ARG;
  (void)p;
  return ENGRAM_OK;
}

}  // namespace

namespace engram {

Workspace carve_workspace(const engram_plan* p, int64_t ntok, void* base) {
  Workspace w{};
  const size_t ab = act_bytes(p->cfg.act_dtype);
  const size_t M = p->cfg.M, d = p->cfg.d;
  const size_t n = static_cast<size_t>(ntok);
  size_t off = 0;
  auto take = [&](size_t bytes) {
    size_t at = off;
    off = align_up(off + bytes, 256);
    return base ? static_cast<char*>(base) + at : nullptr;
  };
  w.idx = reinterpret_cast<int32_t*>(take(n * p->R * 4));
  w.e = take(n * p->d_mem * ab);
  if (p->cfg.act_dtype == ENGRAM_F32) {
    w.kv = reinterpret_cast<float*>(take(n * (M + 1) * d * 4));
  } else {
    w.v32 = reinterpret_cast<float*>(take(n * d * 4));
    // widest case: 32-column slices, rows padded to 16 bytes
    w.part = reinterpret_cast<float*>(take(n * (((d / 32) * (1 + 3 * M) + 3) / 4 * 4) * 4));
    w.sync = reinterpret_cast<uint32_t*>(take(engram::stage_b_sync_words(ntok) * 4));
    w.e8 = reinterpret_cast<uint8_t*>(take(n * p->d_mem));
    w.e_scale = reinterpret_cast<float*>(take(n * 4));
  }
  w.sa = reinterpret_cast<float*>(take(n * engram::sa_row_floats(static_cast<int>(M)) * 4));
  w.bytes = off;
  return w;
}

}  // namespace engram

extern "C" {

const char* engram_status_string(engram_status_t s) {
  switch (s) {
    case ENGRAM_OK: return "ok";
    case ENGRAM_ERR_INVALID_ARG: return "invalid argument";
    case ENGRAM_ERR_UNSUPPORTED: return "unsupported configuration or device";
    case ENGRAM_ERR_NOT_MAPPED: return "host pointer not mapped for device access (pin or register it)";
    case ENGRAM_ERR_INDEX_RANGE: return "index out of range (row zero-filled)";
    case ENGRAM_ERR_CUDA: return "CUDA runtime error";
    case ENGRAM_ERR_TIMEOUT: return "in-kernel wait timed out";
    case ENGRAM_ERR_WORKSPACE: return "workspace missing or too small";
  }
  return "unknown status";
}

engram_status_t engram_plan_create(const engram_config_t* cfg, int64_t max_tokens, engram_plan_t** out) {
  if (!cfg || !out) return ENGRAM_ERR_INVALID_ARG;
  *out = nullptr;
  const engram_config_t& c = *cfg;
  if (c.N < 2 || c.N > engram::kMaxN || c.K < 1) return ENGRAM_ERR_INVALID_ARG;
  const int R = (c.N - 1) * c.K;
  if (R > engram::kMaxR) return ENGRAM_ERR_INVALID_ARG;
  if (c.M < 1 || c.M > engram::kMaxM || c.d < 8 || c.d % 8) return ENGRAM_ERR_INVALID_ARG;
  if (c.conv_w < 1 || c.conv_w > engram::kMaxConvW || c.conv_dilation < 1 || (c.conv_w - 1) * c.conv_dilation > 192)
    return ENGRAM_ERR_INVALID_ARG;
  if (!(c.eps > 0.f) || !std::isfinite(c.eps)) return ENGRAM_ERR_INVALID_ARG;
  if (!c.primes || !c.multipliers) return ENGRAM_ERR_INVALID_ARG;
  if (max_tokens <= 0 || max_tokens > INT32_MAX) return ENGRAM_ERR_INVALID_ARG;
  if (c.row_dim < 1 || (static_cast<size_t>(c.row_dim) * table_elem_bytes(c.table_dtype)) % 16)
    return ENGRAM_ERR_INVALID_ARG;
  // table / activation pairs: copy f32->f32, bf16->bf16, dequant int8->bf16
  const bool pair_ok = (c.table_dtype == ENGRAM_F32 && c.act_dtype == ENGRAM_F32) ||
                       (c.table_dtype == ENGRAM_BF16 && c.act_dtype == ENGRAM_BF16) ||
                       (c.table_dtype == ENGRAM_I8_ROWSCALE_F16 && c.act_dtype == ENGRAM_BF16);
  if (!pair_ok) return ENGRAM_ERR_UNSUPPORTED;
  const int d_mem = R * c.row_dim;
  if (c.act_dtype == ENGRAM_BF16 && (d_mem % 64 || c.d % 64)) return ENGRAM_ERR_UNSUPPORTED;
  if (static_cast<int64_t>(c.M + 1) * c.d > INT32_MAX / 2) return ENGRAM_ERR_INVALID_ARG;

  int dev = 0, sms = 0, major = 0, minor = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return ENGRAM_ERR_CUDA;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return ENGRAM_ERR_CUDA;
  if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess) return ENGRAM_ERR_CUDA;
  if (cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess) return ENGRAM_ERR_CUDA;
  if (major != 10 || minor != 3) return ENGRAM_ERR_UNSUPPORTED;   // built for sm_103a only

  engram_plan* p = new (std::nothrow) engram_plan();
  if (!p) return ENGRAM_ERR_CUDA;
  p->cfg = c;
  p->cfg.primes = nullptr;
  p->cfg.multipliers = nullptr;
  p->R = R;
  p->d_mem = d_mem;
  p->L_ring = (c.conv_w - 1) * c.conv_dilation;
  p->max_tokens = max_tokens;
  p->device = dev;
  p->num_sms = sms;
  p->fused_stage_b = false;
  p->cta_pairs = false;
  p->fused_decode = false;
  p->sm_limit = 0;
  p->host_sms = 0;

  PlanDev h{};
  h.R = R;
  h.N = c.N;
  h.K = c.K;
  int64_t rows = 0;
  for (int r = 0; r < R; ++r) {
    const uint32_t prime = c.primes[r];
    if (prime < 2 || prime > static_cast<uint32_t>(INT32_MAX)) {
      delete p;
      return ENGRAM_ERR_INVALID_ARG;
    }
    h.primes[r] = prime;
    h.mu[r] = kU64Max / prime;    // floor((2^64-1)/p): Barrett reciprocal (see hash.cu)
    h.offsets[r] = rows;
    rows += prime;
    p->primes.push_back(prime);
    p->offsets.push_back(h.offsets[r]);
  }
  p->total_rows = rows;
  int base = 0;
  for (int n = 2; n <= c.N; ++n) {
    h.mult_base[n] = base;
    base += c.K * n;
  }
  for (int i = 0; i < base; ++i) {
    h.mults[i] = c.multipliers[i];
    p->mults.push_back(c.multipliers[i]);
  }
  p->host = h;
  if (cudaMalloc(&p->dev, sizeof(PlanDev)) != cudaSuccess) {
    delete p;
    return ENGRAM_ERR_CUDA;
  }
  if (cudaMemcpy(p->dev, &h, sizeof(PlanDev), cudaMemcpyHostToDevice) != cudaSuccess) {
    cudaFree(p->dev);
    delete p;
    return ENGRAM_ERR_CUDA;
  }
  *out = p;
  return ENGRAM_OK;
}

engram_status_t engram_plan_destroy(engram_plan_t* plan) {
  if (!plan) return ENGRAM_OK;
  if (plan->timing)
    for (int i = 0; i < engram_plan::kMaxMarks; ++i) cudaEventDestroy(plan->marks[i]);
  cudaError_t e = cudaFree(plan->dev);
  delete plan;
  return cuda_status(e);
}

engram_status_t engram_plan_workspace_bytes(const engram_plan_t* plan, int64_t ntok, size_t* bytes) {
  if (!plan || !bytes || ntok < 0) return ENGRAM_ERR_INVALID_ARG;
  *bytes = engram::carve_workspace(plan, ntok, nullptr).bytes;
  return ENGRAM_OK;
}

engram_status_t engram_hash(const engram_plan_t* plan, const int32_t* ids, int B, int T, const int32_t* proj,
                            int V, const int32_t* prev_ids, int32_t* idx_out, engram_stream_t stream) {
  NvtxRange nvtx_range("engram_hash");
  if (!plan) return ENGRAM_ERR_INVALID_ARG;
  if (engram_status_t s = check_tokens(plan, B, T)) return s;
  if (static_cast<int64_t>(B) * T == 0) return ENGRAM_OK;
  if (!ids || !proj || !idx_out || V <= 0) return ENGRAM_ERR_INVALID_ARG;
  return cuda_status(engram::launch_hash(plan, ids, B, T, proj, V, prev_ids, idx_out, (cudaStream_t)stream));
}

engram_status_t engram_gather(const engram_plan_t* plan, const int32_t* idx, int64_t ntok, const void* table,
                              const uint16_t* scales, void* e_out, engram_stream_t stream) {
  NvtxRange nvtx_range("engram_gather");
  if (!plan || ntok < 0 || ntok > plan->max_tokens) return ENGRAM_ERR_INVALID_ARG;
  if (ntok == 0) return ENGRAM_OK;
  if (!idx || !table || !e_out || !aligned16(e_out)) return ENGRAM_ERR_INVALID_ARG;
  const bool i8 = plan->cfg.table_dtype == ENGRAM_I8_ROWSCALE_F16;
  if (i8 != (scales != nullptr)) return ENGRAM_ERR_INVALID_ARG;
  const void* tab = nullptr;
  if (engram_status_t s = device_view(table, &tab)) return s;
  if (!aligned16(tab)) return ENGRAM_ERR_INVALID_ARG;
  const void* sc = nullptr;
  if (i8) {
    if (engram_status_t s = device_view(scales, &sc)) return s;
  }
  return cuda_status(engram::launch_gather(plan, idx, ntok, tab, static_cast<const uint16_t*>(sc), e_out,
                                           (cudaStream_t)stream));
}

engram_status_t engram_stage_a(const engram_plan_t* plan, const int32_t* ids, int B, int T, const int32_t* proj,
                               int V, const int32_t* prev_ids, const void* table, const uint16_t* scales,
                               void* e_out, engram_stream_t stream) {
  NvtxRange nvtx_range("engram_stage_a");
  if (!plan) return ENGRAM_ERR_INVALID_ARG;
  if (engram_status_t s = check_tokens(plan, B, T)) return s;
  if (static_cast<int64_t>(B) * T == 0) return ENGRAM_OK;
  if (!ids || !proj || V <= 0 || !table || !e_out || !aligned16(e_out)) return ENGRAM_ERR_INVALID_ARG;
  const bool i8 = plan->cfg.table_dtype == ENGRAM_I8_ROWSCALE_F16;
  if (i8 != (scales != nullptr)) return ENGRAM_ERR_INVALID_ARG;
  const void* tab = nullptr;
  bool host = false;
  if (engram_status_t s = device_view(table, &tab, &host)) return s;
  if (!aligned16(tab)) return ENGRAM_ERR_INVALID_ARG;
  const void* sc = nullptr;
  if (i8) {
    if (engram_status_t s = device_view(scales, &sc)) return s;
  }
  return cuda_status(engram::launch_hash_gather(plan, ids, B, T, proj, V, prev_ids, tab,
                                                static_cast<const uint16_t*>(sc), e_out, (cudaStream_t)stream,
                                                host));
}

engram_status_t engram_stage_a_layers(int n_layers, const engram_plan_t* const* plans, const int32_t* ids, int B,
                                      int T, const int32_t* proj, int V, const int32_t* const* prev_ids,
                                      const void* const* tables, const uint16_t* const* scales, void* const* e_out,
                                      engram_stream_t stream) {
  NvtxRange nvtx_range("engram_stage_a_layers");
  if (n_layers < 1 || n_layers > engram::kMaxGatherLayers || !plans || !tables || !e_out)
    return ENGRAM_ERR_INVALID_ARG;
  const engram_plan_t* p0 = plans[0];
  if (!p0) return ENGRAM_ERR_INVALID_ARG;
  const bool i8 = p0->cfg.table_dtype == ENGRAM_I8_ROWSCALE_F16;
  if (i8 != (scales != nullptr)) return ENGRAM_ERR_INVALID_ARG;
  for (int l = 0; l < n_layers; ++l) {
    const engram_plan_t* p = plans[l];
    if (!p || p->device != p0->device || p->cfg.N != p0->cfg.N || p->cfg.K != p0->cfg.K ||
        p->cfg.row_dim != p0->cfg.row_dim || p->cfg.table_dtype != p0->cfg.table_dtype ||
        p->cfg.act_dtype != p0->cfg.act_dtype)
      return ENGRAM_ERR_INVALID_ARG;
    if (engram_status_t s = check_tokens(p, B, T)) return s;
  }
  if (static_cast<int64_t>(B) * T == 0) return ENGRAM_OK;
  if (!ids || !proj || V <= 0) return ENGRAM_ERR_INVALID_ARG;
  const void* tab[engram::kMaxGatherLayers] = {};
  const uint16_t* sc[engram::kMaxGatherLayers] = {};
  bool host0 = false;
  for (int l = 0; l < n_layers; ++l) {
    if (!tables[l] || !e_out[l] || !aligned16(e_out[l])) return ENGRAM_ERR_INVALID_ARG;
    bool host = false;
    if (engram_status_t s = device_view(tables[l], &tab[l], &host)) return s;
    if (!aligned16(tab[l])) return ENGRAM_ERR_INVALID_ARG;
    if (l == 0) host0 = host;
    if (host != host0) return ENGRAM_ERR_INVALID_ARG;
    if (i8) {
      const void* v = nullptr;
      if (!scales[l]) return ENGRAM_ERR_INVALID_ARG;
      if (engram_status_t s = device_view(scales[l], &v)) return s;
      sc[l] = static_cast<const uint16_t*>(v);
    }
  }
  return cuda_status(engram::launch_hash_gather_layers(plans, n_layers, ids, B, T, proj, V, prev_ids, tab,
                                                       i8 ? sc : nullptr, e_out, (cudaStream_t)stream, host0));
}

engram_status_t engram_stage_a_layers_e4m3(int n_layers, const engram_plan_t* const* plans, const int32_t* ids,
                                           int B, int T, const int32_t* proj, int V, const int32_t* const* prev_ids,
                                           const void* const* tables, uint8_t* const* e8_out,
                                           float* const* e_scale_out, engram_stream_t stream) {
  NvtxRange nvtx_range("engram_stage_a_layers_e4m3");
  if (n_layers < 1 || n_layers > engram::kMaxGatherLayers || !plans || !tables || !e8_out || !e_scale_out)
    return ENGRAM_ERR_INVALID_ARG;
  const engram_plan_t* p0 = plans[0];
  if (!p0) return ENGRAM_ERR_INVALID_ARG;
  for (int l = 0; l < n_layers; ++l) {
    const engram_plan_t* p = plans[l];
    if (!p || p->device != p0->device || p->cfg.N != p0->cfg.N || p->cfg.K != p0->cfg.K ||
        p->cfg.row_dim != p0->cfg.row_dim || p->cfg.table_dtype != p0->cfg.table_dtype ||
        p->cfg.act_dtype != p0->cfg.act_dtype)
      return ENGRAM_ERR_INVALID_ARG;
    if (engram_status_t s = check_tokens(p, B, T)) return s;
  }
  if (!engram::gather_e4m3_applies(p0)) return ENGRAM_ERR_UNSUPPORTED;
  if (static_cast<int64_t>(B) * T == 0) return ENGRAM_OK;
  if (!ids || !proj || V <= 0) return ENGRAM_ERR_INVALID_ARG;
  const void* tab[engram::kMaxGatherLayers] = {};
  bool host0 = false;
  for (int l = 0; l < n_layers; ++l) {
    if (!tables[l] || !e8_out[l] || !e_scale_out[l] || !aligned16(e8_out[l]) || !aligned16(e_scale_out[l]))
      return ENGRAM_ERR_INVALID_ARG;
    bool host = false;
    if (engram_status_t s = device_view(tables[l], &tab[l], &host)) return s;
    if (!aligned16(tab[l])) return ENGRAM_ERR_INVALID_ARG;
    if (l == 0) host0 = host;
    if (host != host0) return ENGRAM_ERR_INVALID_ARG;
  }
  return cuda_status(engram::launch_hash_gather_layers_e4m3(plans, n_layers, ids, B, T, proj, V, prev_ids, tab,
                                                            e8_out, e_scale_out, (cudaStream_t)stream, host0));
}

engram_status_t engram_stage_a_e4m3(const engram_plan_t* plan, const int32_t* ids, int B, int T, const int32_t* proj,
                                    int V, const int32_t* prev_ids, const void* table, uint8_t* e8_out,
                                    float* e_scale_out, engram_stream_t stream) {
  return engram_stage_a_layers_e4m3(1, &plan, ids, B, T, proj, V, prev_ids ? &prev_ids : nullptr, &table, &e8_out,
                                    &e_scale_out, stream);
}

engram_status_t engram_kv_projection(const engram_plan_t* plan, const void* e, int64_t ntok, const void* w_kv,
                                     void* kv_out, engram_stream_t stream) {
  NvtxRange nvtx_range("engram_kv_projection");
  if (!plan || ntok < 0 || ntok > plan->max_tokens) return ENGRAM_ERR_INVALID_ARG;
  if (ntok == 0) return ENGRAM_OK;
  if (!e || !w_kv || !kv_out || !aligned16(e) || !aligned16(w_kv) || !aligned16(kv_out))
    return ENGRAM_ERR_INVALID_ARG;
  return cuda_status(engram::launch_kv_projection(plan, e, ntok, w_kv, kv_out, (cudaStream_t)stream));
}

// Steps 5-8 from e (already gathered into ws.e or the caller's buffer).
// e8 / e_scale: e's e4m3 codes and scales from the codes gather (FP8 weights only), used instead of
// quantising e (which may then be null)
static engram_status_t run_stage_b(const engram_plan_t* plan, const engram::Workspace& ws, const void* e,
                                   const int32_t* ids, const int32_t* proj, int V, int B, int T,
                                   const engram_weights_t* w, void* H, engram_state_t* state, cudaStream_t s,
                                   const uint8_t* e8 = nullptr, const float* e_scale = nullptr) {
  const int64_t ntok = static_cast<int64_t>(B) * T;
  const int d = plan->cfg.d, M = plan->cfg.M;
  const float* v = nullptr;
  int64_t sv = 0;
  mark(plan, s);
  if (plan->cfg.act_dtype == ENGRAM_F32) {
    if (engram::gemm_f32_simt(static_cast<const float*>(e), static_cast<const float*>(w->w_kv), ws.kv, ntok,
                              (M + 1) * d, plan->d_mem, s) != cudaSuccess)
      return ENGRAM_ERR_CUDA;
    mark(plan, s);
    if (engram::launch_gate_f32(plan, ws.kv, static_cast<const float*>(H), ntok, w->g_h, w->g_k, ws.sa, s) !=
        cudaSuccess)
      return ENGRAM_ERR_CUDA;
    v = ws.kv;
    sv = static_cast<int64_t>(M + 1) * d;
  } else {
    const bool f8 = w->w_kv_fp8 != nullptr;
    if (!f8 && plan->fused_decode && engram::decode_fused_applies(plan, T)) {
      // one position per sequence, rows already gathered: projection and tail as one cooperative launch
      const cudaError_t de =
          engram::launch_decode_fused(plan, ids, B, proj, V, nullptr, nullptr, e, false, w, H, state, ws, s);
      if (de == cudaSuccess) {
        mark(plan, s);
        return ENGRAM_OK;
      }
      if (de != cudaErrorCooperativeLaunchTooLarge) return ENGRAM_ERR_CUDA;
      (void)cudaGetLastError();
    }
    cudaError_t fe = cudaErrorNotSupported;
    if (!f8 && plan->fused_stage_b && engram::stage_b_fused_applies(plan, ntok, T)) {
      // projection and conv in one cooperative launch (after a one-block kernel zeroing its counters)
      fe = engram::launch_stage_b_fused(plan, e, w->w_kv, B, T, H, w->g_h, w->g_k, w->g_c, w->conv, ws.v32, ws.part,
                                        state ? ws.sa : nullptr, state, ws.sync, s);
      if (fe == cudaErrorCooperativeLaunchTooLarge) {
        (void)cudaGetLastError();     // fewer SMs than the plan saw (e.g. a partitioned device): two launches
      } else if (fe != cudaSuccess) {
        return ENGRAM_ERR_CUDA;
      }
    }
    if (fe == cudaSuccess) {
      mark(plan, s);
      if (state) {
        if (engram::launch_state_update(plan, ids, proj, V, ws.v32, d, ws.sa, B, T, state, s) != cudaSuccess)
          return ENGRAM_ERR_CUDA;
        mark(plan, s);
      }
      return ENGRAM_OK;
    }
    int n_sl = 0, pstride = 0;
    if (f8) {
      // e4m3 projection: each token's row of e quantised (unless the gather wrote the codes), then the GEMM on them
      if (e8 == nullptr) {
        if (engram::launch_quantize_rows_e4m3(e, ntok, plan->d_mem, ws.e8, ws.e_scale, engram::stage_b_sms(plan),
                                              s) != cudaSuccess)
          return ENGRAM_ERR_CUDA;
        mark(plan, s);
        e8 = ws.e8;
        e_scale = ws.e_scale;
      }
      if (engram::gemm_e4m3_engram(e8, e_scale, w->w_kv_fp8, w->w_kv_scale, ntok, d, M, plan->d_mem, H, w->g_h,
                                   w->g_k, ws.v32, ws.part, &n_sl, &pstride, engram::stage_b_sms(plan),
                                   &plan->dev->err, s) !=
          cudaSuccess)
        return ENGRAM_ERR_CUDA;
    } else if (engram::gemm_bf16_engram(e, w->w_kv, ntok, d, M, plan->d_mem, H, w->g_h, w->g_k, ws.v32, ws.part,
                                        &n_sl, &pstride, engram::stage_b_sms(plan), &plan->dev->err, s,
                                        plan->cta_pairs) !=
               cudaSuccess) {
      return ENGRAM_ERR_CUDA;
    }
    mark(plan, s);
    if (T == 1) {
      // one position per sequence (decode): gate, conv, residual and state in one launch
      if (engram::launch_decode_tail(plan, ws.v32, d, nullptr, ws.part, n_sl, pstride, ws.sa, B, w->g_c, w->conv, H,
                                     ids, proj, V, state, s) != cudaSuccess)
        return ENGRAM_ERR_CUDA;
      mark(plan, s);
      return ENGRAM_OK;
    }
    if (engram::conv_fuses_gate(plan, n_sl, pstride)) {
      // the conv computes the gate scalars from the partials itself
      if (engram::launch_conv_residual(plan, ws.v32, d, nullptr, B, T, w->g_c, w->conv, H, state, s, ws.part,
                                       state ? ws.sa : nullptr) != cudaSuccess)
        return ENGRAM_ERR_CUDA;
      mark(plan, s);
      if (state) {
        if (engram::launch_state_update(plan, ids, proj, V, ws.v32, d, ws.sa, B, T, state, s) != cudaSuccess)
          return ENGRAM_ERR_CUDA;
        mark(plan, s);
      }
      return ENGRAM_OK;
    }
    if (engram::launch_finalize(plan, ws.part, n_sl, pstride, ntok, ws.sa, s) != cudaSuccess) return ENGRAM_ERR_CUDA;
    v = ws.v32;
    sv = d;
  }
  mark(plan, s);
  if (T == 1) {
    if (engram::launch_decode_tail(plan, v, sv, ws.sa, nullptr, 0, 0, nullptr, B, w->g_c, w->conv, H, ids, proj, V,
                                   state, s) != cudaSuccess)
      return ENGRAM_ERR_CUDA;
    mark(plan, s);
    return ENGRAM_OK;
  }
  if (engram::launch_conv_residual(plan, v, sv, ws.sa, B, T, w->g_c, w->conv, H, state, s) != cudaSuccess)
    return ENGRAM_ERR_CUDA;
  mark(plan, s);
  if (state) {
    if (engram::launch_state_update(plan, ids, proj, V, v, sv, ws.sa, B, T, state, s) != cudaSuccess)
      return ENGRAM_ERR_CUDA;
    mark(plan, s);
  }
  return ENGRAM_OK;
}

engram_status_t engram_stage_b(const engram_plan_t* plan, const int32_t* ids, int B, int T, const int32_t* proj,
                               int V, const void* e, const engram_weights_t* w, void* H, engram_state_t* state,
                               void* workspace, size_t workspace_bytes, engram_stream_t stream) {
  NvtxRange nvtx_range("engram_stage_b");
  if (!plan) return ENGRAM_ERR_INVALID_ARG;
  if (engram_status_t s = check_tokens(plan, B, T)) return s;
  const int64_t ntok = static_cast<int64_t>(B) * T;
  if (ntok == 0) return ENGRAM_OK;
  if (!e || !H || !aligned16(e) || !aligned16(H)) return ENGRAM_ERR_INVALID_ARG;
  if (state && (!ids || !proj || V <= 0)) return ENGRAM_ERR_INVALID_ARG;
  if (engram_status_t s = check_weights(plan, w, false)) return s;
  if (engram_status_t s = check_state(plan, state)) return s;
  engram::Workspace ws = engram::carve_workspace(plan, ntok, workspace);
  if (!workspace || workspace_bytes < ws.bytes || (reinterpret_cast<uintptr_t>(workspace) & 255u))
    return ENGRAM_ERR_WORKSPACE;
  plan->n_marks = 0;
  return run_stage_b(plan, ws, e, ids, proj, V, B, T, w, H, state, (cudaStream_t)stream);
}

engram_status_t engram_stage_b_e4m3(const engram_plan_t* plan, const int32_t* ids, int B, int T, const int32_t* proj,
                                    int V, const uint8_t* e8, const float* e_scale, const engram_weights_t* w, void* H,
                                    engram_state_t* state, void* workspace, size_t workspace_bytes,
                                    engram_stream_t stream) {
  NvtxRange nvtx_range("engram_stage_b_e4m3");
  if (!plan) return ENGRAM_ERR_INVALID_ARG;
  if (engram_status_t s = check_tokens(plan, B, T)) return s;
  const int64_t ntok = static_cast<int64_t>(B) * T;
  if (ntok == 0) return ENGRAM_OK;
  if (!e8 || !e_scale || !H || !aligned16(e8) || !aligned16(e_scale) || !aligned16(H)) return ENGRAM_ERR_INVALID_ARG;
  if (!w || !w->w_kv_fp8) return ENGRAM_ERR_INVALID_ARG;
  if (state && (!ids || !proj || V <= 0)) return ENGRAM_ERR_INVALID_ARG;
  if (engram_status_t s = check_weights(plan, w, false)) return s;
  if (engram_status_t s = check_state(plan, state)) return s;
  engram::Workspace ws = engram::carve_workspace(plan, ntok, workspace);
  if (!workspace || workspace_bytes < ws.bytes || (reinterpret_cast<uintptr_t>(workspace) & 255u))
    return ENGRAM_ERR_WORKSPACE;
  plan->n_marks = 0;
  return run_stage_b(plan, ws, nullptr, ids, proj, V, B, T, w, H, state, (cudaStream_t)stream, e8, e_scale);
}

engram_status_t engram_forward(const engram_plan_t* plan, const int32_t* ids, int B, int T, const int32_t* proj,
                               int V, const engram_weights_t* w, void* H, engram_state_t* state, void* workspace,
                               size_t workspace_bytes, engram_stream_t stream) {
  NvtxRange nvtx_range("engram_forward");
  if (!plan) return ENGRAM_ERR_INVALID_ARG;
  if (engram_status_t s = check_tokens(plan, B, T)) return s;
  const int64_t ntok = static_cast<int64_t>(B) * T;
  if (ntok == 0) return ENGRAM_OK;
  if (!ids || !proj || V <= 0 || !H || !aligned16(H)) return ENGRAM_ERR_INVALID_ARG;
  if (engram_status_t s = check_weights(plan, w, true)) return s;
  if (engram_status_t s = check_state(plan, state)) return s;
  engram::Workspace ws = engram::carve_workspace(plan, ntok, workspace);
  if (!workspace || workspace_bytes < ws.bytes || (reinterpret_cast<uintptr_t>(workspace) & 255u))
    return ENGRAM_ERR_WORKSPACE;
  const void* tab = nullptr;
  bool host = false;
  if (engram_status_t s = device_view(w->table, &tab, &host)) return s;
  if (!aligned16(tab)) return ENGRAM_ERR_INVALID_ARG;
  const void* sc = nullptr;
  if (w->scales) {
    if (engram_status_t s = device_view(w->scales, &sc)) return s;
  }
  cudaStream_t s = (cudaStream_t)stream;
  const int32_t* prev = state ? state->prev_ids : nullptr;
  plan->n_marks = 0;
  mark(plan, s);
  if (plan->fused_decode && w->w_kv_fp8 == nullptr && engram::decode_fused_applies(plan, T)) {
    // one position per sequence: the whole layer as one cooperative launch
    const cudaError_t de = engram::launch_decode_fused(plan, ids, B, proj, V, tab, static_cast<const uint16_t*>(sc),
                                                       ws.e, true, w, H, state, ws, s);
    if (de == cudaSuccess) {
      mark(plan, s);
      return ENGRAM_OK;
    }
    if (de != cudaErrorCooperativeLaunchTooLarge) return ENGRAM_ERR_CUDA;
    (void)cudaGetLastError();     // fewer co-resident blocks than SMs (e.g. a partitioned device): three launches
  }
  if (w->w_kv_fp8 != nullptr && engram::gather_e4m3_applies(plan)) {
    // FP8 projection: the gather writes e's codes and scales itself (no e, no quantisation launch)
    if (engram::launch_hash_gather_e4m3(plan, ids, B, T, proj, V, prev, tab, ws.e8, ws.e_scale, s, host) !=
        cudaSuccess)
      return ENGRAM_ERR_CUDA;
    return run_stage_b(plan, ws, nullptr, ids, proj, V, B, T, w, H, state, s, ws.e8, ws.e_scale);
  }
  if (engram::launch_hash_gather(plan, ids, B, T, proj, V, prev, tab, static_cast<const uint16_t*>(sc), ws.e, s,
                                 host) != cudaSuccess)
    return ENGRAM_ERR_CUDA;
  return run_stage_b(plan, ws, ws.e, ids, proj, V, B, T, w, H, state, s);
}

}  // extern "C"

struct engram_cache {
  const engram_plan* plan;
  int64_t capacity;
  int row_bytes;
  const void* table;                 // device view of the table
  bool table_on_host = false;        // pinned or registered host memory (rows cross the host link)
  uint32_t* counts;                  // [total rows]
  int32_t* slot;                     // [total rows]
  void* rows;                        // [capacity + batch_cap, row_bytes]: cached rows, then the dedup region
  unsigned long long* stats;         // [0] lookups, [1] served from HBM, [2] slots used by the last build,
                                     // [3] rows fetched by the dedup
  int64_t cached;
  int64_t batch_cap;                 // lookups the dedup region has a row for (0: no dedup)
  uint32_t* batch_rows;              // [batch_cap] the table row each lookup claimed, or 0xFFFFFFFF
  // dedup pipeline over pieces of the batch: claims on the caller's stream, fetches over the
  // host link on `fetch`, gathers from HBM on `gather`
  static constexpr int kChunks = 4;
  cudaStream_t fetch = nullptr, gather = nullptr;
  cudaEvent_t claimed[kChunks] = {}, fetched[kChunks] = {}, fork = nullptr, join = nullptr;
};

extern "C" {

engram_status_t engram_cache_create(const engram_plan_t* plan, int64_t capacity, const void* table,
                                    engram_cache_t** out) {
  if (!plan || !table || !out) return ENGRAM_ERR_INVALID_ARG;
  *out = nullptr;
  if (capacity < 0 || capacity > plan->total_rows || capacity > INT32_MAX) return ENGRAM_ERR_INVALID_ARG;
  const void* tab = nullptr;
  bool host = false;
  if (engram_status_t s = device_view(table, &tab, &host)) return s;
  if (!aligned16(tab)) return ENGRAM_ERR_INVALID_ARG;
  engram_cache* c = new (std::nothrow) engram_cache();
  if (!c) return ENGRAM_ERR_CUDA;
  c->plan = plan;
  c->table_on_host = host;
  c->capacity = capacity;
  c->row_bytes = static_cast<int>(plan->cfg.row_dim * table_elem_bytes(plan->cfg.table_dtype));
  c->table = tab;
  const size_t n = static_cast<size_t>(plan->total_rows);
  bool ok = cudaMalloc(&c->counts, n * sizeof(uint32_t)) == cudaSuccess &&
            cudaMalloc(&c->slot, n * sizeof(int32_t)) == cudaSuccess &&
            cudaMalloc(&c->rows, static_cast<size_t>(capacity > 0 ? capacity : 1) * c->row_bytes) == cudaSuccess &&
            cudaMalloc(&c->stats, 8 * sizeof(unsigned long long)) == cudaSuccess;
  ok = ok && cudaMemset(c->counts, 0, n * sizeof(uint32_t)) == cudaSuccess &&
       cudaMemset(c->slot, 0xFF, n * sizeof(int32_t)) == cudaSuccess &&
       cudaMemset(c->stats, 0, 8 * sizeof(unsigned long long)) == cudaSuccess;
  if (!ok) {
    cudaGetLastError();
    engram_cache_destroy(c);
    return ENGRAM_ERR_CUDA;
  }
  *out = c;
  return ENGRAM_OK;
}

engram_status_t engram_cache_destroy(engram_cache_t* c) {
  if (!c) return ENGRAM_OK;
  cudaError_t e = cudaSuccess;
  for (void* ptr : {static_cast<void*>(c->counts), static_cast<void*>(c->slot), c->rows, static_cast<void*>(c->stats),
                    static_cast<void*>(c->batch_rows)})
    if (ptr && cudaFree(ptr) != cudaSuccess) e = cudaErrorUnknown;
  for (int i = 0; i < engram_cache::kChunks; ++i)
    for (cudaEvent_t ev : {c->claimed[i], c->fetched[i]})
      if (ev && cudaEventDestroy(ev) != cudaSuccess) e = cudaErrorUnknown;
  for (cudaEvent_t ev : {c->fork, c->join})
    if (ev && cudaEventDestroy(ev) != cudaSuccess) e = cudaErrorUnknown;
  for (cudaStream_t st : {c->fetch, c->gather})
    if (st && cudaStreamDestroy(st) != cudaSuccess) e = cudaErrorUnknown;
  delete c;
  return cuda_status(e);
}

engram_status_t engram_cache_observe(engram_cache_t* c, const int32_t* ids, int B, int T, const int32_t* proj, int V,
                                     const int32_t* prev_ids, engram_stream_t stream) {
  NvtxRange nvtx_range("engram_cache_observe");
  if (!c) return ENGRAM_ERR_INVALID_ARG;
  if (engram_status_t s = check_tokens(c->plan, B, T)) return s;
  if (static_cast<int64_t>(B) * T == 0) return ENGRAM_OK;
  if (!ids || !proj || V <= 0) return ENGRAM_ERR_INVALID_ARG;
  return cuda_status(engram::cache_observe(c->plan, ids, B, T, proj, V, prev_ids, c->counts, (cudaStream_t)stream));
}

engram_status_t engram_cache_build(engram_cache_t* c, int decay, engram_stream_t stream, int64_t* cached_rows) {
  NvtxRange nvtx_range("engram_cache_build");
  if (!c) return ENGRAM_ERR_INVALID_ARG;
  int64_t cached = 0;
  if (engram::cache_build(c->plan, c->capacity, c->row_bytes, c->table, c->counts, c->slot, c->rows, c->stats + 2,
                          decay, &cached, (cudaStream_t)stream) != cudaSuccess)
    return ENGRAM_ERR_CUDA;
  c->cached = cached;
  if (cached_rows) *cached_rows = cached;
  return ENGRAM_OK;
}

engram_status_t engram_stage_a_cached(const engram_cache_t* c, const int32_t* ids, int B, int T, const int32_t* proj,
                                      int V, const int32_t* prev_ids, const uint16_t* scales, void* e_out,
                                      engram_stream_t stream) {
  NvtxRange nvtx_range("engram_stage_a_cached");
  if (!c) return ENGRAM_ERR_INVALID_ARG;
  const engram_plan* plan = c->plan;
  if (engram_status_t s = check_tokens(plan, B, T)) return s;
  if (static_cast<int64_t>(B) * T == 0) return ENGRAM_OK;
  if (!ids || !proj || V <= 0 || !e_out || !aligned16(e_out)) return ENGRAM_ERR_INVALID_ARG;
  const bool i8 = plan->cfg.table_dtype == ENGRAM_I8_ROWSCALE_F16;
  if (i8 != (scales != nullptr)) return ENGRAM_ERR_INVALID_ARG;
  const void* sc = nullptr;
  if (i8) {
    if (engram_status_t s = device_view(scales, &sc)) return s;
  }
  cudaStream_t s = (cudaStream_t)stream;
  const int64_t lookups = static_cast<int64_t>(B) * T * plan->R;
  const bool dedup = c->batch_cap > 0 && lookups <= c->batch_cap;
  const int chunks = dedup && c->gather ? (B < engram_cache::kChunks ? B : engram_cache::kChunks) : 1;
  if (chunks > 1) {
    // pieces of whole sequences: piece i+1 is claimed while piece i's claimed rows cross the host
    // link and piece i-1 is gathered from HBM.  A row claimed by an earlier piece is served from its
    // slot and not fetched again; every claim is released after the last gather.
    const int R = plan->R, Nm1 = plan->cfg.N - 1;
    const size_t e_row = static_cast<size_t>(plan->d_mem) * act_bytes(plan->cfg.act_dtype);
    uint8_t* region = static_cast<uint8_t*>(c->rows) + static_cast<size_t>(c->capacity) * c->row_bytes;
    if (cudaEventRecord(c->fork, s) != cudaSuccess || cudaStreamWaitEvent(c->fetch, c->fork, 0) != cudaSuccess ||
        cudaStreamWaitEvent(c->gather, c->fork, 0) != cudaSuccess)
      return ENGRAM_ERR_CUDA;
    for (int k = 0; k < chunks; ++k) {
      const int b0 = static_cast<int>(static_cast<int64_t>(B) * k / chunks);
      const int b1 = static_cast<int>(static_cast<int64_t>(B) * (k + 1) / chunks);
      const int64_t f0 = static_cast<int64_t>(b0) * T * R;
      const int64_t n = static_cast<int64_t>(b1 - b0) * T * R;
      const int32_t* ids_k = ids + static_cast<int64_t>(b0) * T;
      const int32_t* prev_k = prev_ids ? prev_ids + static_cast<int64_t>(b0) * Nm1 : nullptr;
      if (engram::dedup_claim(plan, ids_k, b1 - b0, T, proj, V, prev_k, c->slot,
                              static_cast<int32_t>(c->capacity + f0), c->batch_rows + f0, s) != cudaSuccess ||
          cudaEventRecord(c->claimed[k], s) != cudaSuccess ||
          cudaStreamWaitEvent(c->fetch, c->claimed[k], 0) != cudaSuccess ||
          engram::dedup_fetch(plan, n, c->batch_rows + f0, c->row_bytes, c->table,
                              region + static_cast<size_t>(f0) * c->row_bytes, c->fetch) != cudaSuccess ||
          cudaEventRecord(c->fetched[k], c->fetch) != cudaSuccess ||
          cudaStreamWaitEvent(c->gather, c->fetched[k], 0) != cudaSuccess ||
          engram::launch_hash_gather_cached(plan, ids_k, b1 - b0, T, proj, V, prev_k, c->table,
                                            static_cast<const uint16_t*>(sc),
                                            static_cast<uint8_t*>(e_out) + static_cast<size_t>(b0) * T * e_row,
                                            c->slot, c->rows, c->stats, c->gather) != cudaSuccess)
        return ENGRAM_ERR_CUDA;
    }
    if (cudaEventRecord(c->join, c->gather) != cudaSuccess || cudaStreamWaitEvent(s, c->join, 0) != cudaSuccess ||
        engram::dedup_release(plan, lookups, c->batch_rows, c->slot, c->stats + 3, s) != cudaSuccess)
      return ENGRAM_ERR_CUDA;
    return ENGRAM_OK;
  }
  if (dedup) {
    // distinct uncached rows of the batch: one fetch each over the host link, into the batch region
    uint8_t* region = static_cast<uint8_t*>(c->rows) + static_cast<size_t>(c->capacity) * c->row_bytes;
    if (engram::dedup_claim(plan, ids, B, T, proj, V, prev_ids, c->slot, static_cast<int32_t>(c->capacity),
                            c->batch_rows, s) != cudaSuccess ||
        engram::dedup_fetch(plan, lookups, c->batch_rows, c->row_bytes, c->table, region, s) != cudaSuccess)
      return ENGRAM_ERR_CUDA;
  }
  // with the dedup every lookup is served from HBM; otherwise the misses cross the host link
  if (engram::launch_hash_gather_cached(plan, ids, B, T, proj, V, prev_ids, c->table, static_cast<const uint16_t*>(sc),
                                        e_out, c->slot, c->rows, c->stats, s, c->table_on_host && !dedup) !=
      cudaSuccess)
    return ENGRAM_ERR_CUDA;
  if (dedup && engram::dedup_release(plan, lookups, c->batch_rows, c->slot, c->stats + 3, s) != cudaSuccess)
    return ENGRAM_ERR_CUDA;
  return ENGRAM_OK;
}

engram_status_t engram_cache_set_dedup(engram_cache_t* c, int64_t batch_rows) {
  if (!c || batch_rows < 0 || c->capacity + batch_rows > INT32_MAX) return ENGRAM_ERR_INVALID_ARG;
  if (batch_rows == c->batch_cap) return ENGRAM_OK;
  if (cudaDeviceSynchronize() != cudaSuccess) return ENGRAM_ERR_CUDA;
  const size_t keep = static_cast<size_t>(c->capacity) * c->row_bytes;
  const size_t total = keep + static_cast<size_t>(batch_rows) * c->row_bytes;
  void* rows = nullptr;
  uint32_t* br = nullptr;
  bool ok = cudaMalloc(&rows, total > 0 ? total : c->row_bytes) == cudaSuccess &&
            (batch_rows == 0 || cudaMalloc(&br, static_cast<size_t>(batch_rows) * sizeof(uint32_t)) == cudaSuccess);
  ok = ok && (keep == 0 || cudaMemcpy(rows, c->rows, keep, cudaMemcpyDeviceToDevice) == cudaSuccess);
  if (!ok) {
    cudaGetLastError();
    if (rows) cudaFree(rows);
    if (br) cudaFree(br);
    return ENGRAM_ERR_CUDA;
  }
  cudaFree(c->rows);
  if (c->batch_rows) cudaFree(c->batch_rows);
  c->rows = rows;
  c->batch_rows = br;
  c->batch_cap = batch_rows;
  if (batch_rows > 0 && !c->gather) {
    // the pipeline's streams and events (its fork/join are stream-ordered and capturable)
    auto ev = [](cudaEvent_t* e) { return cudaEventCreateWithFlags(e, cudaEventDisableTiming) == cudaSuccess; };
    bool made = cudaStreamCreateWithFlags(&c->fetch, cudaStreamNonBlocking) == cudaSuccess &&
                cudaStreamCreateWithFlags(&c->gather, cudaStreamNonBlocking) == cudaSuccess && ev(&c->fork) &&
                ev(&c->join);
    for (int i = 0; made && i < engram_cache::kChunks; ++i) made = ev(&c->claimed[i]) && ev(&c->fetched[i]);
    if (!made) {
      cudaGetLastError();
      for (int i = 0; i < engram_cache::kChunks; ++i)
        for (cudaEvent_t* e : {&c->claimed[i], &c->fetched[i]})
          if (*e) {
            cudaEventDestroy(*e);
            *e = nullptr;
          }
      for (cudaEvent_t* e : {&c->fork, &c->join})
        if (*e) {
          cudaEventDestroy(*e);
          *e = nullptr;
        }
      for (cudaStream_t* st : {&c->fetch, &c->gather})
        if (*st) {
          cudaStreamDestroy(*st);
          *st = nullptr;
        }                                 // the dedup then runs unpipelined
    }
  }
  return ENGRAM_OK;
}

engram_status_t engram_forward_split(engram_plan_t* plan, const engram_sm_split_t* split, int n_pieces,
                                     const engram_cache_t* cache, const int32_t* ids, int B, int T,
                                     const int32_t* proj, int V, const engram_weights_t* w, void* H,
                                     engram_state_t* state, void* workspace, size_t workspace_bytes,
                                     engram_stream_t stream) {
  NvtxRange nvtx_range("engram_forward_split");
  if (!plan || !split) return ENGRAM_ERR_INVALID_ARG;
  if (cache && cache->plan != plan) return ENGRAM_ERR_INVALID_ARG;
  if (cache && cache->batch_cap > 0) return ENGRAM_ERR_UNSUPPORTED;      // the dedup runs its own pipeline
  if (engram_status_t s = check_tokens(plan, B, T)) return s;
  const int64_t ntok = static_cast<int64_t>(B) * T;
  if (ntok == 0) return ENGRAM_OK;
  if (n_pieces < 1 || n_pieces > B || n_pieces > engram::kMaxPieces) return ENGRAM_ERR_INVALID_ARG;
  if (!ids || !proj || V <= 0 || !H || !aligned16(H)) return ENGRAM_ERR_INVALID_ARG;
  if (engram_status_t s = check_weights(plan, w, true)) return s;
  if (engram_status_t s = check_state(plan, state)) return s;
  engram::Workspace ws = engram::carve_workspace(plan, ntok, workspace);
  if (!workspace || workspace_bytes < ws.bytes || (reinterpret_cast<uintptr_t>(workspace) & 255u))
    return ENGRAM_ERR_WORKSPACE;
  const void* tab = nullptr;
  bool host = false;
  if (engram_status_t s = device_view(w->table, &tab, &host)) return s;
  if (!aligned16(tab)) return ENGRAM_ERR_INVALID_ARG;
  const void* sc = nullptr;
  if (w->scales) {
    if (engram_status_t s = device_view(w->scales, &sc)) return s;
  }
  const cudaStream_t s = (cudaStream_t)stream;
  const cudaStream_t sa = engram::split_stream(split, 0), sb = engram::split_stream(split, 1);
  const size_t ab = act_bytes(plan->cfg.act_dtype);
  const int64_t e_row = static_cast<int64_t>(plan->d_mem) * ab;                    // bytes of e per token
  const int64_t h_row = static_cast<int64_t>(plan->cfg.M) * plan->cfg.d * ab;      // bytes of H per token
  const int L = plan->L_ring, N = plan->cfg.N, Md = plan->cfg.M * plan->cfg.d;
  const bool codes = w->w_kv_fp8 != nullptr && !cache && engram::gather_e4m3_applies(plan);
  // each group's grids sized for its SMs; the two-launch Stage B on one SM per CTA (its
  // one-launch and CTA-pair forms need every SM or clusters): the same bits in every form
  struct Saved {
    engram_plan* p;
    int sm_limit, host_sms;
    bool timing, fused_stage_b, cta_pairs;
    ~Saved() {
      p->sm_limit = sm_limit;
      p->host_sms = host_sms;
      p->timing = timing;
      p->fused_stage_b = fused_stage_b;
      p->cta_pairs = cta_pairs;
    }
  } saved{plan, plan->sm_limit, plan->host_sms, plan->timing, plan->fused_stage_b, plan->cta_pairs};
  plan->sm_limit = engram::split_sms(split, 1);
  plan->host_sms = engram::split_sms(split, 0);
  plan->timing = false;
  plan->fused_stage_b = false;
  plan->cta_pairs = false;
  plan->n_marks = 0;
  auto order = [](cudaStream_t before, cudaStream_t after, cudaEvent_t ev) {
    return cudaEventRecord(ev, before) == cudaSuccess && cudaStreamWaitEvent(after, ev, 0) == cudaSuccess;
  };
  // both groups' streams start after the work already on `stream`
  if (!order(s, sa, engram::split_event(split, 0)) || cudaStreamWaitEvent(sb, engram::split_event(split, 0), 0))
    return ENGRAM_ERR_CUDA;
  // piece boundaries: with three pieces or more, the first and the last are half the size of the others,
  // so that the pipeline's fill (the first lookup) and drain (the last Stage B) are short
  auto piece_start = [&](int i) -> int {
    if (i <= 0) return 0;
    if (i >= n_pieces) return B;
    if (n_pieces <= 2) return static_cast<int>(static_cast<int64_t>(B) * i / n_pieces);
    return static_cast<int>((static_cast<int64_t>(B) * (2 * i - 1) + (n_pieces - 1)) / (2 * (n_pieces - 1)));
  };
  engram_status_t status = ENGRAM_OK;
  for (int i = 0; i < n_pieces && status == ENGRAM_OK; ++i) {
    const int lo = piece_start(i), hi = piece_start(i + 1);
    const int nb = hi - lo;
    if (nb == 0) continue;
    const int64_t t0 = static_cast<int64_t>(lo) * T;
    void* e_i = static_cast<char*>(ws.e) + t0 * e_row;
    engram_state_t st_i{};
    if (state) {
      st_i.prev_ids = state->prev_ids + static_cast<int64_t>(lo) * (N - 1);
      st_i.u_ring = state->u_ring + static_cast<int64_t>(lo) * L * Md;
      st_i.pos = state->pos + lo;
    }
    const int32_t* prev_i = state ? st_i.prev_ids : nullptr;
    // with e4m3 weights the gather writes the piece's codes and scales where it can (as engram_forward)
    uint8_t* e8_i = codes ? ws.e8 + t0 * plan->d_mem : nullptr;
    float* es_i = codes ? ws.e_scale + t0 : nullptr;
    const cudaError_t ga =
        codes ? engram::launch_hash_gather_e4m3(plan, ids + t0, nb, T, proj, V, prev_i, tab, e8_i, es_i, sa, host)
        : cache ? engram::launch_hash_gather_cached(plan, ids + t0, nb, T, proj, V, prev_i, cache->table,
                                                    static_cast<const uint16_t*>(sc), e_i, cache->slot, cache->rows,
                                                    cache->stats, sa, cache->table_on_host)
                : engram::launch_hash_gather(plan, ids + t0, nb, T, proj, V, prev_i, tab,
                                             static_cast<const uint16_t*>(sc), e_i, sa, host);
    if (ga != cudaSuccess || !order(sa, sb, engram::split_event(split, 1 + i))) {
      status = ENGRAM_ERR_CUDA;
      break;
    }
    status = run_stage_b(plan, ws, codes ? nullptr : e_i, ids + t0, proj, V, nb, T, w,
                         static_cast<char*>(H) + t0 * h_row, state ? &st_i : nullptr, sb, e8_i, es_i);
  }
  // `stream` waits for both groups, also after an error, so that no work of this call is left unordered
  if (!order(sa, s, engram::split_event(split, n_pieces + 1)) || !order(sb, s, engram::split_event(split, n_pieces + 2)))
    return ENGRAM_ERR_CUDA;
  return status;
}

engram_status_t engram_cache_stats(const engram_cache_t* c, engram_stream_t stream, int reset,
                                   uint64_t* rows_looked_up, uint64_t* rows_from_hbm, uint64_t* rows_over_link,
                                   int64_t* cached_rows) {
  if (!c) return ENGRAM_ERR_INVALID_ARG;
  if (cudaStreamSynchronize((cudaStream_t)stream) != cudaSuccess) return ENGRAM_ERR_CUDA;
  unsigned long long st[4] = {0, 0, 0, 0};
  if (cudaMemcpy(st, c->stats, sizeof(st), cudaMemcpyDeviceToHost) != cudaSuccess) return ENGRAM_ERR_CUDA;
  if (reset && (cudaMemset(c->stats, 0, 2 * sizeof(unsigned long long)) != cudaSuccess ||
                cudaMemset(c->stats + 3, 0, sizeof(unsigned long long)) != cudaSuccess))
    return ENGRAM_ERR_CUDA;
  if (rows_looked_up) *rows_looked_up = st[0];
  if (rows_from_hbm) *rows_from_hbm = st[1];
  if (rows_over_link) *rows_over_link = (st[0] - st[1]) + st[3];
  if (cached_rows) *cached_rows = c->cached;
  return ENGRAM_OK;
}

engram_status_t engram_quantize_fp8(const engram_plan_t* plan, const void* x, int64_t rows, int cols, uint8_t* q,
                                    float* scale, engram_stream_t stream) {
  NvtxRange nvtx_range("engram_quantize_fp8");
  if (!plan || !x || !q || !scale || rows < 0 || cols <= 0 || cols % 16) return ENGRAM_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(q) || !aligned16(scale)) return ENGRAM_ERR_INVALID_ARG;
  if (rows == 0) return ENGRAM_OK;
  return cuda_status(engram::launch_quantize_rows_e4m3(x, rows, cols, q, scale, plan->num_sms, (cudaStream_t)stream));
}

engram_status_t engram_plan_set_fused_stage_b(engram_plan_t* plan, int enable) {
  if (!plan || (enable != 0 && enable != 1)) return ENGRAM_ERR_INVALID_ARG;
  plan->fused_stage_b = enable != 0;
  return ENGRAM_OK;
}

engram_status_t engram_plan_set_sm_limit(engram_plan_t* plan, int n_sms) {
  if (!plan || n_sms < 0) return ENGRAM_ERR_INVALID_ARG;
  plan->sm_limit = n_sms;
  return ENGRAM_OK;
}

int engram_plan_host_gather_sms(const engram_plan_t* plan) {
  return plan ? engram::hostgrid_sms(plan) : 0;
}

engram_status_t engram_plan_set_host_gather_sms(engram_plan_t* plan, int n_sms) {
  if (!plan || n_sms < 0) return ENGRAM_ERR_INVALID_ARG;
  plan->host_sms = n_sms;
  return ENGRAM_OK;
}

engram_status_t engram_plan_set_fused_decode(engram_plan_t* plan, int enable) {
  if (!plan || (enable != 0 && enable != 1)) return ENGRAM_ERR_INVALID_ARG;
  plan->fused_decode = enable != 0;
  return ENGRAM_OK;
}

engram_status_t engram_plan_set_cta_pairs(engram_plan_t* plan, int enable) {
  if (!plan || (enable != 0 && enable != 1)) return ENGRAM_ERR_INVALID_ARG;
  plan->cta_pairs = enable != 0;
  return ENGRAM_OK;
}

engram_status_t engram_plan_set_timing(engram_plan_t* plan, int enable) {
  if (!plan) return ENGRAM_ERR_INVALID_ARG;
  if (enable && !plan->timing) {
    for (int i = 0; i < engram_plan::kMaxMarks; ++i) {
      if (cudaEventCreate(&plan->marks[i]) != cudaSuccess) {
        for (int j = 0; j < i; ++j) cudaEventDestroy(plan->marks[j]);
        return ENGRAM_ERR_CUDA;
      }
    }
    plan->timing = true;
  } else if (!enable && plan->timing) {
    for (int i = 0; i < engram_plan::kMaxMarks; ++i) cudaEventDestroy(plan->marks[i]);
    plan->timing = false;
  }
  plan->n_marks = 0;
  return ENGRAM_OK;
}

engram_status_t engram_plan_kernel_times(const engram_plan_t* plan, float* ms_out, int max_out, int* count) {
  if (!plan || !count || (max_out > 0 && !ms_out)) return ENGRAM_ERR_INVALID_ARG;
  *count = 0;
  if (!plan->timing || plan->n_marks < 2) return ENGRAM_OK;
  if (cudaEventSynchronize(plan->marks[plan->n_marks - 1]) != cudaSuccess) return ENGRAM_ERR_CUDA;
  const int n = plan->n_marks - 1;
  for (int i = 0; i < n && i < max_out; ++i) {
    if (cudaEventElapsedTime(&ms_out[i], plan->marks[i], plan->marks[i + 1]) != cudaSuccess) return ENGRAM_ERR_CUDA;
  }
  *count = n < max_out ? n : max_out;
  return ENGRAM_OK;
}

engram_status_t engram_get_error(const engram_plan_t* plan, engram_stream_t stream, uint32_t* flags_out) {
  if (!plan) return ENGRAM_ERR_INVALID_ARG;
  if (cudaStreamSynchronize((cudaStream_t)stream) != cudaSuccess) return ENGRAM_ERR_CUDA;
  uint32_t bits = 0;
  if (cudaMemcpy(&bits, &plan->dev->err, sizeof(bits), cudaMemcpyDeviceToHost) != cudaSuccess)
    return ENGRAM_ERR_CUDA;
  const uint32_t zero = 0;
  if (cudaMemcpy(&plan->dev->err, &zero, sizeof(zero), cudaMemcpyHostToDevice) != cudaSuccess)
    return ENGRAM_ERR_CUDA;
  if (flags_out) *flags_out = bits;
  if (bits & engram::kErrTimeout) return ENGRAM_ERR_TIMEOUT;
  if (bits & engram::kErrIndexRange) return ENGRAM_ERR_INDEX_RANGE;
  return ENGRAM_OK;
}

}  // extern "C"
