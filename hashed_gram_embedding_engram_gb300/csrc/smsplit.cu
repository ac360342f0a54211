// Host side of an SM split: the device's SMs in two disjoint sets, each a
// green context of the driver with one non-blocking stream, so that work on
// one stream never takes an SM of the other.  Kernels launched into these
// streams by the runtime run in the primary context's address space (the
// driver reports the primary context as the context of a green context's
// stream), on their set's SMs only.  The driver calls are reached through the
// runtime's entry-point query, as the tensor-map encoder is.
#include <cuda.h>
#include <cuda_runtime.h>

#include <mutex>
#include <new>

#include "engram.h"
#include "engram_internal.h"

struct engram_sm_split {
  CUgreenCtx ctx[2];
  CUstream stream[2];
  int sms[2];
  cudaEvent_t ev[engram::kSplitEvents];   // ordering events for engram_forward_split
};

namespace {

struct GreenFns {
  CUresult (*device_get)(CUdevice*, int) = nullptr;
  CUresult (*get_resource)(CUdevice, CUdevResource*, CUdevResourceType) = nullptr;
  CUresult (*split)(CUdevResource*, unsigned int*, const CUdevResource*, CUdevResource*, unsigned int,
                    unsigned int) = nullptr;
  CUresult (*gen_desc)(CUdevResourceDesc*, CUdevResource*, unsigned int) = nullptr;
  CUresult (*ctx_create)(CUgreenCtx*, CUdevResourceDesc, CUdevice, unsigned int) = nullptr;
  CUresult (*ctx_destroy)(CUgreenCtx) = nullptr;
  CUresult (*stream_create)(CUstream*, CUgreenCtx, unsigned int, int) = nullptr;
  CUresult (*stream_destroy)(CUstream) = nullptr;
  bool ok = false;
};

template <typename F>
bool entry(const char* name, F& fn) {
  void* p = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion(name, &p, 12050, cudaEnableDefault, &q) != cudaSuccess ||
      q != cudaDriverEntryPointSuccess || p == nullptr)
    return false;
  fn = reinterpret_cast<F>(p);
  return true;
}

const GreenFns& green_fns() {
  static GreenFns f;
  static std::once_flag once;
  std::call_once(once, [] {
    f.ok = entry("cuDeviceGet", f.device_get) && entry("cuDeviceGetDevResource", f.get_resource) &&
           entry("cuDevSmResourceSplitByCount", f.split) && entry("cuDevResourceGenerateDesc", f.gen_desc) &&
           entry("cuGreenCtxCreate", f.ctx_create) && entry("cuGreenCtxDestroy", f.ctx_destroy) &&
           entry("cuGreenCtxStreamCreate", f.stream_create) && entry("cuStreamDestroy", f.stream_destroy);
  });
  return f;
}

void release(const GreenFns& f, engram_sm_split* sp) {
  for (cudaEvent_t& e : sp->ev)
    if (e) cudaEventDestroy(e);
  for (int g = 0; g < 2; ++g) {
    if (sp->stream[g]) f.stream_destroy(sp->stream[g]);
    if (sp->ctx[g]) f.ctx_destroy(sp->ctx[g]);
  }
  delete sp;
}

}  // namespace

namespace engram {
cudaStream_t split_stream(const engram_sm_split* sp, int group) { return sp->stream[group]; }
int split_sms(const engram_sm_split* sp, int group) { return sp->sms[group]; }
cudaEvent_t split_event(const engram_sm_split* sp, int i) { return sp->ev[i]; }
}  // namespace engram

extern "C" {

engram_status_t engram_sm_split_create(int device, int n_sms, engram_sm_split_t** out) {
  if (!out || n_sms <= 0) return ENGRAM_ERR_INVALID_ARG;
  *out = nullptr;
  const GreenFns& f = green_fns();
  if (!f.ok) return ENGRAM_ERR_UNSUPPORTED;
  // the primary context first: green contexts retain it
  if (cudaSetDevice(device) != cudaSuccess || cudaFree(nullptr) != cudaSuccess) return ENGRAM_ERR_CUDA;
  CUdevice dev;
  CUdevResource all{};
  if (f.device_get(&dev, device) != CUDA_SUCCESS || f.get_resource(dev, &all, CU_DEV_RESOURCE_TYPE_SM) != CUDA_SUCCESS)
    return ENGRAM_ERR_CUDA;
  if (static_cast<unsigned>(n_sms) >= all.sm.smCount) return ENGRAM_ERR_INVALID_ARG;
  CUdevResource part[2] = {};
  unsigned int groups = 1;
  if (f.split(&part[0], &groups, &all, &part[1], 0, static_cast<unsigned>(n_sms)) != CUDA_SUCCESS || groups != 1 ||
      part[1].sm.smCount == 0)
    return ENGRAM_ERR_UNSUPPORTED;
  auto* sp = new (std::nothrow) engram_sm_split{};
  if (!sp) return ENGRAM_ERR_CUDA;
  for (int g = 0; g < 2; ++g) {
    CUdevResourceDesc desc;
    if (f.gen_desc(&desc, &part[g], 1) != CUDA_SUCCESS ||
        f.ctx_create(&sp->ctx[g], desc, dev, CU_GREEN_CTX_DEFAULT_STREAM) != CUDA_SUCCESS ||
        f.stream_create(&sp->stream[g], sp->ctx[g], CU_STREAM_NON_BLOCKING, 0) != CUDA_SUCCESS) {
      release(f, sp);
      return ENGRAM_ERR_CUDA;
    }
    sp->sms[g] = static_cast<int>(part[g].sm.smCount);
  }
  for (cudaEvent_t& e : sp->ev) {
    if (cudaEventCreateWithFlags(&e, cudaEventDisableTiming) != cudaSuccess) {
      e = nullptr;
      release(f, sp);
      return ENGRAM_ERR_CUDA;
    }
  }
  *out = sp;
  return ENGRAM_OK;
}

int engram_sm_split_sms(const engram_sm_split_t* split, int group) {
  return split && (group == 0 || group == 1) ? split->sms[group] : 0;
}

void* engram_sm_split_stream(const engram_sm_split_t* split, int group) {
  return split && (group == 0 || group == 1) ? static_cast<void*>(split->stream[group]) : nullptr;
}

engram_status_t engram_sm_split_destroy(engram_sm_split_t* split) {
  if (!split) return ENGRAM_OK;
  const GreenFns& f = green_fns();
  if (!f.ok) return ENGRAM_ERR_UNSUPPORTED;
  release(f, split);
  return ENGRAM_OK;
}

}  // extern "C"
