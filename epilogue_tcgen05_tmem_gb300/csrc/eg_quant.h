// eg_quant.h -- launcher of the per-token activation quantisation kernel.
#pragma once
#include <cstdint>
#include <cuda_runtime.h>

namespace eg {

// x: bf16 [M][ldx]; q: codes [M][ldq] (E4M3 when e4m3, else int8); s: [M].
// pdl: launch as a programmatic dependent of the previous kernel on st.
cudaError_t launch_quant_rows(const void* x, int64_t M, int64_t K, int64_t ldx, bool e4m3,
                              void* q, int64_t ldq, float* s, cudaStream_t st, bool pdl);

}  // namespace eg
