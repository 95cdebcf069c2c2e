// eg_gated.h -- launcher of the gated-unit combine kernel (INT8 and
// Block_FP8 gated units, which run as the fused kernel's accumulator output
// over all 2N weight rows followed by this kernel).
#pragma once
#include <cstdint>
#include <cuda_runtime.h>

namespace eg {

// acc: [M][2N] accumulator words from the fused kernel's accumulator output
// (INT8: exact int32 sums; block scales: the promoted float32 sums), gate
// half in columns [0, N), up half in [N, 2N).  s_a [M] and s_w [2N] (INT8
// only, else unused), bias [2N] bf16 (flags & 1), R [M][ldr] bf16 (flags &
// 2), Y [M][ldy] in the output format `out` (0 bf16, 1 fp16, 2 E4M3 codes of
// y / s_y).  pdl: launch as a programmatic dependent of the previous kernel.
cudaError_t launch_gated_combine(const uint32_t* acc, int64_t M, int64_t N, bool int8,
                                 const float* s_a, const float* s_w, const void* bias,
                                 const void* R, int64_t ldr, void* Y, int64_t ldy, int act,
                                 uint32_t flags, int out, const float* s_y, cudaStream_t st,
                                 bool pdl);

}  // namespace eg
