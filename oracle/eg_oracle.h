/*
 * CPU oracle for the fused scaled linear layer -- TEST INFRASTRUCTURE ONLY.
 *
 * Only the tests, the smoke check and the bench's CPU-baseline leg may call
 * this library.  It shares no code, header or constant with the CUDA path.
 *
 * It computes, in float64, the plain definition of what the fused kernel
 * reaches (fusion, tiling, split-K and swap-AB change only the rounding
 * points):
 *
 *   acc[m][n] = sum_k a[m][k] * w[n][k]                  (ascending k)
 *   block scaling:  acc = sum_kb sa[m][kb] * sw[n/128][kb] * (sum_{k in kb} a*w)
 *   token/channel:  v = acc * (sa[m] * sw[n]);  otherwise v = acc
 *   v += bias[n]                                        (if BIAS)
 *   default order:  v = act(v); v += R[m][n]            (if RESIDUAL)
 *   pre-act order:  v += R[m][n]; v = act(v)            (if RESIDUAL_PRE_ACT)
 *   Y[m][n] = bf16 round-to-nearest-even of v, rounded directly from float64
 *   (or fp16, or the E4M3 code of v / s_y: ORC_OUT_F16, ORC_OUT_E4M3; the
 *   uint16 output then holds the fp16 bits or the code in its low byte).
 *
 * Sources: "Helion + TorchInductor co-operation: operator fusion", section
 * "Designing extensible epilogues in Helion" (bias broadcast over rows, ReLU,
 * tanh-GELU with its constants, masked tails), and the section on prologue
 * and epilogue fusion strategies (scale, bias, residual, GELU/SiLU, narrowing
 * before the store); "Helion linear backend in vLLM", section "One kernel
 * instead of three" (the FP8_Dynamic, W8A8_INT8 and Block_FP8 scale formats).
 *
 * Data: A is [M][K] and W is [N][K], both row-major (K contiguous).  Element
 * codes: bf16 bit patterns (uint16), OCP FP8 E4M3 codes (uint8) or int8.
 * Scales are float32: sa[M], sw[N] (token/channel) or sa[M][K/128],
 * sw[ceil(N/128)][K/128] (block).  bias[N] and R[M][N] are bf16 bits.
 */
#ifndef EG_ORACLE_H
#define EG_ORACLE_H
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define ORC_IN_BF16 0
#define ORC_IN_E4M3 1
#define ORC_IN_INT8 2

#define ORC_SCALE_NONE 0
#define ORC_SCALE_TOKEN_CHANNEL 1
#define ORC_SCALE_BLOCK 2

#define ORC_ACT_NONE 0
#define ORC_ACT_RELU 1
#define ORC_ACT_GELU_ERF 2
#define ORC_ACT_GELU_TANH 3
#define ORC_ACT_SILU 4

#define ORC_BIAS 1u
#define ORC_RESIDUAL 2u
#define ORC_RESIDUAL_PRE_ACT 4u
/* Output narrowing ("Helion + TorchInductor co-operation: operator fusion":
 * the FP32 -> narrow conversion right before the store, fp16 on that page's
 * own kernel): without these flags Y is bf16; ORC_OUT_F16 rounds v to IEEE
 * binary16 (nearest even, overflow to infinity); ORC_OUT_E4M3 writes the
 * E4M3 code of v / s_y (float64 division, nearest even, saturating). */
#define ORC_OUT_F16 8u
#define ORC_OUT_E4M3 16u

typedef struct {
  int64_t M, N, K;
  int32_t dtype, scale, act;
  uint32_t flags;
  float s_y; /* output scale, ORC_OUT_E4M3 only */
} orc_problem;

/* Element codecs. */
double orc_bf16_to_double(uint16_t bits);
double orc_e4m3_to_double(uint8_t code);
uint16_t orc_bf16_from_double(double v);
double orc_act(int32_t act, double v);

/* Full problem.  Y (bf16 bits, [M][N]) may be NULL.  acc ([M][N] float64:
 * the value of `acc` above, before scaling) may be NULL.  acc_i64 ([M][N])
 * is filled for INT8 only and may be NULL.  nthreads <= 0 uses every core
 * in the affinity mask.  Returns 0, or -1 on a bad argument. */
int orc_linear(const orc_problem* p, const void* A, const void* W,
               const float* sa, const float* sw, const uint16_t* bias,
               const uint16_t* R, uint16_t* Y, double* acc, int64_t* acc_i64,
               int nthreads);

/* The same definition as a single-threaded triple loop with on-the-fly
 * decoding (brute force for tiny shapes). */
int orc_linear_naive(const orc_problem* p, const void* A, const void* W,
                     const float* sa, const float* sw, const uint16_t* bias,
                     const uint16_t* R, uint16_t* Y, double* acc,
                     int64_t* acc_i64);

/* Selected outputs only: for each i < npts, Y[i] and acc[i] at
 * (ms[i], ns[i]).  Used for sampled checks at full size. */
int orc_linear_points(const orc_problem* p, const void* A, const void* W,
                      const float* sa, const float* sw, const uint16_t* bias,
                      const uint16_t* R, const int64_t* ms, const int64_t* ns,
                      int64_t npts, uint16_t* Y, double* acc, int nthreads);

/* Split-K decomposition of the accumulator: the K range is cut into S
 * parts [s*T/S, (s+1)*T/S) of T = ceil(K/kunit) units of kunit columns,
 * each part is summed on its own and the parts are added in order
 * s = 0..S-1.  acc is [M][N] float64, acc_i64 (INT8) may be NULL. */
int orc_accum_splitk(const orc_problem* p, const void* A, const void* W,
                     const float* sa, const float* sw, int64_t S,
                     int64_t kunit, double* acc, int64_t* acc_i64);

/* Number of worker threads orc_linear uses for nthreads <= 0. */
int orc_default_threads(void);

/* Gated linear unit (the SwiGLU epilogue when act is SiLU): W holds 2N rows,
 * the gate half [0, N) and the up half [N, 2N) ("two W halves"); s_w (token/
 * channel) has 2N entries, or 2N/128 block rows (block scaling); bias has 2N
 * entries.  With acc = A . W^T over all 2N rows (the accumulation of
 * orc_linear), per output (m, n), n < N:
 *   g = scale(acc[m][n]) + bias[n],  u = scale(acc[m][N + n]) + bias[N + n]
 *   y = act(g) * u;  y += R[m][n] (ORC_RESIDUAL);  Y[m][n] = round(y)
 * where scale() is the token/channel scaling (sa[m] * sw[row]) or nothing
 * (bf16, block: already scaled), and round() follows the output flags.
 * ORC_RESIDUAL_PRE_ACT is rejected.  Returns 0 or -1. */
int orc_linear_gated(const orc_problem* p, const void* A, const void* W, const float* sa,
                     const float* sw, const uint16_t* bias, const uint16_t* R, uint16_t* Y,
                     int nthreads);

/* Dynamic per-token quantisation of activations (the prologue transform
 * that precedes the FP8_Dynamic and W8A8_INT8 layers; "Helion linear backend
 * in vLLM", section "One kernel instead of three", scale formats, and
 * "Helion + TorchInductor co-operation: operator fusion", section on
 * prologue fusion).  For each row m of the bf16 matrix x [M][ldx]:
 *   amax = max_k |x[m][k]|                           (float32, exact)
 *   s[m] = amax / 448 (E4M3) or amax / 127 (INT8)    (float32 division)
 *          and s[m] = 1 when amax = 0
 *   E4M3: q = E4M3 code of (x / s[m]) rounded to nearest even, saturated
 *         to +-448 (float32 division)
 *   INT8: q = clamp(round-half-even(x / s[m]), -127, 127)
 * q is written to q[M][ldq] (bytes).  dtype is ORC_IN_E4M3 or ORC_IN_INT8.
 * Returns 0, or -1 for bad arguments. */
int orc_quant_rows(const uint16_t* x, int64_t M, int64_t K, int64_t ldx, int32_t dtype,
                   uint8_t* q, int64_t ldq, float* s);

/* OCP FP8 E4M3 code of a float: round to nearest, ties to even, finite
 * values saturate to +-448, NaN -> 0x7F (sign kept). */
uint8_t orc_e4m3_from_float(float v);
uint8_t orc_e4m3_from_double(double v);

/* IEEE binary16: decode, and round a float64 to nearest even in one step
 * (subnormals on the 2^-24 grid; magnitudes that round past 65504 become
 * infinity). */
double orc_f16_to_double(uint16_t bits);
uint16_t orc_f16_from_double(double v);

#ifdef __cplusplus
}
#endif
#endif
