// Host-side preparation of the conv (tile shape, shared-memory layout, tensor
// maps), shared by the conv launch (fusion.cu) and the fused Stage-B kernel
// (stage_b.cu).
#pragma once

#include "conv_parts.cuh"
#include "engram_internal.h"

namespace engram {

// Arguments of launch_conv_residual; fills the kernel arguments, the three
// tensor maps (v, H, sa or the partials) and the dynamic shared memory, which
// the tile shape keeps within smem_cap bytes (1024-byte alignment included).
cudaError_t conv_prepare(const engram_plan* p, const float* v, int64_t sv, const float* sa, int B, int T,
                         const float* g_c, const float* conv, void* H, const engram_state_t* state, const float* part,
                         float* sa_out, cv::ConvArgs* out, CUtensorMap* tv_out, CUtensorMap* th_out,
                         CUtensorMap* ts_out, size_t* smem_out, size_t smem_cap);

}  // namespace engram
