// eg_quant.cu -- dynamic per-token activation quantisation, the prologue
// transform in front of the FP8_Dynamic and W8A8_INT8 layers ("Helion linear
// backend in vLLM", section "One kernel instead of three": per-token
// activation scales; "Helion + TorchInductor co-operation: operator fusion",
// section on prologue fusion).  One CTA per row: amax over the row, s =
// amax / 448 (E4M3) or amax / 127 (INT8), s = 1 for an all-zero row, then
// code = round-to-nearest-even(x / s), saturated (E4M3: +-448; INT8: +-127).
// It runs as its own small kernel just before the GEMM, in the same stream
// (and graph); the GEMM, launched as its programmatic dependent, streams its
// weights while this runs.
#include <cuda_bf16.h>
#include <cuda_fp8.h>

#include "eg_ptx.cuh"
#include "eg_quant.h"

namespace eg {

namespace {

constexpr int kQuantThreads = 512;

__device__ __forceinline__ float block_max(float v, float* red) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (lane == 0) red[warp] = v;
  __syncthreads();
  if (warp == 0) {
    v = lane < kQuantThreads / 32 ? red[lane] : 0.0f;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    if (lane == 0) red[0] = v;
  }
  __syncthreads();
  return red[0];
}

template <bool E4M3>
__device__ __forceinline__ uint8_t quant_code(float x, float s) {
  const float t = __fdiv_rn(x, s);  // IEEE division, as the definition states
  if constexpr (E4M3) {
    return static_cast<uint8_t>(__nv_cvt_float_to_fp8(t, __NV_SATFINITE, __NV_E4M3));
  } else {
    int r = __float2int_rn(t);  // ties to even
    r = r > 127 ? 127 : (r < -127 ? -127 : r);
    return static_cast<uint8_t>(static_cast<int8_t>(r));
  }
}

// vec: x rows and q rows 16-byte aligned and K % 8 == 0 (8 elements a step);
// with vec and K <= kQuantThreads * 8 * kRegVec the row is read once and
// kept in registers.
constexpr int kRegVec = 4;

template <bool E4M3>
__global__ void __launch_bounds__(kQuantThreads)
    quant_rows_kernel(const __nv_bfloat16* __restrict__ x, int64_t K, int64_t ldx,
                      uint8_t* __restrict__ q, int64_t ldq, float* __restrict__ s, int vec) {
  // the dependent GEMM may start (and stream its weights) right away; it
  // waits for this grid to finish before it reads the codes and scales
  griddep_launch_dependents();
  // x may be written by the previous kernel (when launched as its dependent)
  griddep_wait();
  __shared__ float red[kQuantThreads / 32];
  const int64_t m = blockIdx.x;
  const __nv_bfloat16* row = x + m * ldx;
  uint8_t* qrow = q + m * ldq;
  const bool in_regs = vec && K <= static_cast<int64_t>(kQuantThreads) * 8 * kRegVec;
  uint4 v[kRegVec];
  float amax = 0.0f;
  if (in_regs) {
#pragma unroll
    for (int i = 0; i < kRegVec; ++i) {
      const int64_t k = (static_cast<int64_t>(i) * kQuantThreads + threadIdx.x) * 8;
      v[i] = k < K ? *reinterpret_cast<const uint4*>(row + k) : make_uint4(0, 0, 0, 0);
      const uint32_t w[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        amax = fmaxf(amax, fabsf(__uint_as_float(w[j] << 16)));
        amax = fmaxf(amax, fabsf(__uint_as_float(w[j] & 0xFFFF0000u)));
      }
    }
  } else if (vec) {
    for (int64_t k = static_cast<int64_t>(threadIdx.x) * 8; k < K; k += kQuantThreads * 8) {
      const uint4 u = *reinterpret_cast<const uint4*>(row + k);
      const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        amax = fmaxf(amax, fabsf(__uint_as_float(w[j] << 16)));
        amax = fmaxf(amax, fabsf(__uint_as_float(w[j] & 0xFFFF0000u)));
      }
    }
  } else {
    for (int64_t k = threadIdx.x; k < K; k += kQuantThreads)
      amax = fmaxf(amax, fabsf(__bfloat162float(row[k])));
  }
  amax = block_max(amax, red);
  const float sm = amax > 0.0f ? __fdiv_rn(amax, E4M3 ? 448.0f : 127.0f) : 1.0f;
  if (threadIdx.x == 0) s[m] = sm;
  auto quant8 = [&](const uint4& u) {
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
    uint32_t out[2] = {0u, 0u};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const uint32_t lo = quant_code<E4M3>(__uint_as_float(w[j] << 16), sm);
      const uint32_t hi = quant_code<E4M3>(__uint_as_float(w[j] & 0xFFFF0000u), sm);
      out[j >> 1] |= (lo | (hi << 8)) << (16 * (j & 1));
    }
    return make_uint2(out[0], out[1]);
  };
  if (in_regs) {
#pragma unroll
    for (int i = 0; i < kRegVec; ++i) {
      const int64_t k = (static_cast<int64_t>(i) * kQuantThreads + threadIdx.x) * 8;
      if (k < K) *reinterpret_cast<uint2*>(qrow + k) = quant8(v[i]);
    }
  } else if (vec) {
    for (int64_t k = static_cast<int64_t>(threadIdx.x) * 8; k < K; k += kQuantThreads * 8)
      *reinterpret_cast<uint2*>(qrow + k) = quant8(*reinterpret_cast<const uint4*>(row + k));
  } else {
    for (int64_t k = threadIdx.x; k < K; k += kQuantThreads)
      qrow[k] = quant_code<E4M3>(__bfloat162float(row[k]), sm);
  }
}

}  // namespace

cudaError_t launch_quant_rows(const void* x, int64_t M, int64_t K, int64_t ldx, bool e4m3,
                              void* q, int64_t ldq, float* s, cudaStream_t st, bool pdl) {
  if (M == 0) return cudaSuccess;
  const int vec = (reinterpret_cast<uintptr_t>(x) % 16 == 0) && (ldx * 2) % 16 == 0 &&
                  (reinterpret_cast<uintptr_t>(q) % 8 == 0) && ldq % 8 == 0 && K % 8 == 0;
  const auto* xb = static_cast<const __nv_bfloat16*>(x);
  auto* qb = static_cast<uint8_t*>(q);
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(static_cast<unsigned>(M));
  cfg.blockDim = dim3(kQuantThreads);
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  if (e4m3) return cudaLaunchKernelEx(&cfg, quant_rows_kernel<true>, xb, K, ldx, qb, ldq, s, vec);
  return cudaLaunchKernelEx(&cfg, quant_rows_kernel<false>, xb, K, ldx, qb, ldq, s, vec);
}

}  // namespace eg
