// eg_gated.cu -- the combine step of the INT8 and Block_FP8 gated units
// (SwiGLU with SiLU; "two W halves -> act(g) * u" in the PluS model-drift
// discussion of gated MLP epilogues).  The fused kernel writes the raw
// accumulators of all 2N weight rows (the gate half, then the up half) for
// each token; per output (m, n) this kernel forms
//   g = scale(acc[m][n]) + bias[n],  u = scale(acc[m][N + n]) + bias[N + n],
//   y = act(g) * u (+ R[m][n]),  one narrowing to the output format,
// where scale() is s_a[m] * s_w[row] for INT8 (the exact int32 sum times the
// two scales formed as a float pair, then rounded once to float) and nothing
// for block scales (the promoted sums already carry them).
#include "eg_kernel.cuh"
#include "eg_gated.h"

namespace eg {

namespace {

template <int ACT>
__global__ void __launch_bounds__(256) gated_combine_kernel(
    const uint32_t* __restrict__ acc, int64_t M, int64_t N, int int8, const float* __restrict__ s_a,
    const float* __restrict__ s_w, const __nv_bfloat16* __restrict__ bias,
    const __nv_bfloat16* __restrict__ R, int64_t ldr, void* Y, int64_t ldy, uint32_t flags, int out,
    const float* __restrict__ s_y) {
  // a programmatic dependent of the GEMM: its accumulators are complete and
  // visible once this returns
  griddep_wait();
  const float inv_sy = out == OUT_E4M3 ? __frcp_rn(__ldg(s_y)) : 1.0f;
  const bool has_bias = (flags & F_BIAS) != 0;
  const bool has_res = (flags & F_RES) != 0;
  for (int64_t m = blockIdx.y; m < M; m += gridDim.y) {
    const uint32_t* arow = acc + m * 2 * N;
    const float sa = int8 ? __ldg(s_a + m) : 1.0f;
    for (int64_t n = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; n < N;
         n += static_cast<int64_t>(gridDim.x) * blockDim.x) {
      const uint32_t ga = __ldg(arow + n), ua = __ldg(arow + N + n);
      float g, u;
      if (int8) {
        const DF dg = df_scale_int(static_cast<int32_t>(ga), sa, __ldg(s_w + n));
        const DF du = df_scale_int(static_cast<int32_t>(ua), sa, __ldg(s_w + N + n));
        g = __fadd_rn(dg.hi, dg.lo);
        u = __fadd_rn(du.hi, du.lo);
      } else {
        g = __uint_as_float(ga);
        u = __uint_as_float(ua);
      }
      if (has_bias) {
        g += __bfloat162float(bias[n]);
        u += __bfloat162float(bias[N + n]);
      }
      float y = act_c<ACT>(g) * u;
      if (has_res) y += __bfloat162float(R[m * ldr + n]);
      const uint16_t o = out_bits(y, out, inv_sy);
      if (out == OUT_E4M3)
        static_cast<uint8_t*>(Y)[m * ldy + n] = static_cast<uint8_t>(o);
      else
        static_cast<uint16_t*>(Y)[m * ldy + n] = o;
    }
  }
}

template <int ACT>
cudaError_t launch_act(const cudaLaunchConfig_t& cfg, const uint32_t* acc, int64_t M, int64_t N, int int8,
                       const float* s_a, const float* s_w, const void* bias, const void* R, int64_t ldr,
                       void* Y, int64_t ldy, uint32_t flags, int out, const float* s_y) {
  return cudaLaunchKernelEx(&cfg, gated_combine_kernel<ACT>, acc, M, N, int8, s_a, s_w,
                            static_cast<const __nv_bfloat16*>(bias), static_cast<const __nv_bfloat16*>(R),
                            ldr, Y, ldy, flags, out, s_y);
}

}  // namespace

cudaError_t launch_gated_combine(const uint32_t* acc, int64_t M, int64_t N, bool int8,
                                 const float* s_a, const float* s_w, const void* bias,
                                 const void* R, int64_t ldr, void* Y, int64_t ldy, int act,
                                 uint32_t flags, int out, const float* s_y, cudaStream_t st,
                                 bool pdl) {
  if (M == 0 || N == 0) return cudaSuccess;
  constexpr int kThreads = 256;
  const int64_t bx = (N + kThreads - 1) / kThreads;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(static_cast<unsigned>(bx < 1024 ? bx : 1024),
                     static_cast<unsigned>(M < 65535 ? M : 65535));
  cfg.blockDim = dim3(kThreads);
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  const int i8 = int8 ? 1 : 0;
  switch (act) {
    case ACT_RELU: return launch_act<ACT_RELU>(cfg, acc, M, N, i8, s_a, s_w, bias, R, ldr, Y, ldy, flags, out, s_y);
    case ACT_GELU_ERF:
      return launch_act<ACT_GELU_ERF>(cfg, acc, M, N, i8, s_a, s_w, bias, R, ldr, Y, ldy, flags, out, s_y);
    case ACT_GELU_TANH:
      return launch_act<ACT_GELU_TANH>(cfg, acc, M, N, i8, s_a, s_w, bias, R, ldr, Y, ldy, flags, out, s_y);
    case ACT_SILU: return launch_act<ACT_SILU>(cfg, acc, M, N, i8, s_a, s_w, bias, R, ldr, Y, ldy, flags, out, s_y);
    default: return launch_act<ACT_NONE>(cfg, acc, M, N, i8, s_a, s_w, bias, R, ldr, Y, ldy, flags, out, s_y);
  }
}

}  // namespace eg
