// Per-row e4m3 quantisation for the FP8 K/V projection.  The section
// "多分支 backbone 上的变体" of "DeepSeek Engram 系列导读" suggests running the
// fused [W_V; W_K^(1..M)] projection as one FP8 GEMM; it fixes no scaling, so
// this build scales per row: for the activations e one scale per token, for
// W_kv one per output row, s = amax / 448 (448 = the largest finite e4m3
// value) and q = e4m3(x * (448 / amax)) rounded to nearest even, saturating
// to +-448.  Both quotients are IEEE binary32 divisions and the product one
// binary32 multiply, so the codes are a function of the bf16 inputs alone.
// An all-zero row gets s = 1 and zero codes.
//
// One warp per row: a pass for the row's absolute maximum (a warp max), a
// second pass that converts 16 elements per lane and step into one 16-byte
// store.  The second pass re-reads the row from L1/L2.
#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>

#include "e4m3.cuh"
#include "engram_internal.h"
#include "ptx.cuh"

namespace engram {
namespace {

using e4m3::amax8;
using e4m3::quant8;

__global__ void __launch_bounds__(256) quantize_rows_kernel(const __nv_bfloat16* __restrict__ x, int64_t rows, int cols,
                                                            uint8_t* __restrict__ q, float* __restrict__ scale) {
  ptx::grid_dep_wait();
  ptx::grid_dep_launch();
  const int lane = threadIdx.x & 31;
  const int64_t n_warps = static_cast<int64_t>(gridDim.x) * (blockDim.x >> 5);
  const int n8 = cols / 8;                          // 16-byte groups of 8 bf16
  for (int64_t row = static_cast<int64_t>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5); row < rows;
       row += n_warps) {
    const uint4* xr = reinterpret_cast<const uint4*>(x + row * cols);
    float amax = 0.f;
    for (int i = lane; i < n8; i += 32) amax = amax8(xr[i], amax);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, o));
    const float inv = e4m3::inv_of(amax);
    if (lane == 0) scale[row] = e4m3::scale_of(amax);
    uint4* qr = reinterpret_cast<uint4*>(q + row * cols);
    for (int i = lane; i < n8 / 2; i += 32) {
      const uint2 a = quant8(xr[2 * i], inv);
      const uint2 b = quant8(xr[2 * i + 1], inv);
      qr[i] = make_uint4(a.x, a.y, b.x, b.y);
    }
  }
}

}  // namespace

cudaError_t launch_quantize_rows_e4m3(const void* x, int64_t rows, int cols, uint8_t* q, float* scale, int num_sms,
                                      cudaStream_t s) {
  if (rows <= 0 || cols <= 0 || cols % 16) return cudaErrorInvalidValue;
  int64_t blocks = (rows + 7) / 8;
  const int64_t cap = static_cast<int64_t>(num_sms) * 8;
  if (blocks > cap) blocks = cap;
  return launch_pdl(quantize_rows_kernel, dim3(static_cast<unsigned>(blocks)), dim3(256), 0, s,
                    static_cast<const __nv_bfloat16*>(x), rows, cols, q, scale);
}

}  // namespace engram
