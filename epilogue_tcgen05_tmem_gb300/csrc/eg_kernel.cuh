// eg_kernel.cuh -- the fused scaled linear-layer kernel for sm_103a.
//
// One kernel computes Y = epilogue(A . W^T) and stores each output once.
// The method follows "Helion + TorchInductor co-operation: operator fusion"
// (sections on prologue/epilogue fusion strategies and on extensible
// epilogues: fp32 accumulator; bias broadcast over rows; ReLU/GELU; masked
// tails read as zero; narrowing right before the single store) and "Helion
// linear backend in vLLM" (section "One kernel instead of three": the
// FP8_Dynamic / W8A8_INT8 / Block_FP8 scale formats; split_k and swap_ab as
// tunables of the one kernel).  The Hopper/A100 tile kernels described
// there keep the accumulator in registers; on sm_103a it lives in tensor
// memory (TMEM) and the epilogue reads it back with tcgen05.ld.
//
// Roles inside a CTA (one work unit = one 128 x BN output tile and one
// K-split):
//   warp 0      TMA producer: 2-D bulk-tensor loads of the row operand P and
//               the column operand Q into a `stages`-deep shared-memory ring
//               (128-byte swizzle, zero fill outside the tensor).
//   warp 1      allocates TMEM; lane 0 issues tcgen05.mma (UMMA 128 x BN) and
//               tcgen05.commit; frees TMEM at the end.
//   warps 2..5  epilogue: tcgen05.ld of the accumulator (lane quarter
//               warp%4), per-element scale, bias, activation, residual,
//               bf16 rounding and the single store; split-K partials go
//               through an fp32 workspace, the last CTA of a tile to arrive
//               reduces them in split order and runs the epilogue.
//   warps 6..9  (INT8 only) prologue transform, exact: the int8 P tile ->
//               fp16 in tensor memory (the UMMA reads its A operand there),
//               the int8 Q tile -> fp16 in shared memory (UMMA layout).
// Rows of the UMMA are M (P = A, Q = W) or, with swap-AB, N (P = W, Q = A),
// so TMEM lane = row and column = the other dimension.
//
// Promotion: for Block_FP8 each 128-wide K block is accumulated into one of
// two TMEM buffers and the epilogue warps add s_a[m][kb] * s_w[n/128][kb] *
// block into fp32 registers while UMMA fills the other buffer.  INT8 uses
// the same double-buffered rhythm: each 128-wide K chunk of the fp16 UMMA
// is an exact integer below 2^21 in fp32 and is added into int32 registers,
// so the int32 accumulator is exact.
#pragma once
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include "eg_ptx.cuh"

namespace eg {

enum : int { IN_BF16 = 0, IN_E4M3 = 1, IN_INT8 = 2 };
enum : int { SC_NONE = 0, SC_TC = 1, SC_BLOCK = 2 };
enum : int { ACT_NONE = 0, ACT_RELU = 1, ACT_GELU_ERF = 2, ACT_GELU_TANH = 3, ACT_SILU = 4 };
enum : uint32_t { F_BIAS = 1, F_RES = 2, F_RES_PRE = 4, F_DEBUG = 8 };
// (gated units are a compile-time variant of the kernel, G below)
// Output element formats: bf16, fp16, or the E4M3 code of v / s_y.
enum : int { OUT_BF16 = 0, OUT_F16 = 1, OUT_E4M3 = 2 };
// Device status codes (first failure wins).
enum : int { ST_TIMEOUT_PRODUCER = 1, ST_TIMEOUT_MMA = 2, ST_TIMEOUT_EPILOGUE = 3,
             ST_TIMEOUT_CONVERT = 4, ST_TIMEOUT_TEARDOWN = 5 };

struct KParams {
  int32_t M, N, K;
  int32_t rows, cols;             // extents along UMMA rows / columns
  int32_t tiles_rows, tiles_cols;
  int32_t k_tiles;                // K tiles of 128 bytes of the input type
  int32_t split_k;
  int32_t stages;
  int32_t act;
  uint32_t flags;
  int32_t kb_count;               // K / 128 (block scales)
  const float* s_a;
  const float* s_w;
  const __nv_bfloat16* bias;
  const __nv_bfloat16* R;
  int64_t ldr;
  void* Y;
  int64_t ldy;
  float* ws;                      // split-K partials (fp32 or int32 bits)
  int* counters;                  // per-tile arrival counters
  int* status;                    // device status word
  uint64_t wait_limit_ns;
  int32_t stall_producer;         // failure-detection test hook: 1 every CTA's load
                                  // warp issues nothing, 2 only odd-numbered CTAs'
                                  // (the others finish and count their split-K
                                  // arrivals)
  int32_t evict_first_p;          // L2 evict-first hint on the P operand
  int32_t evict_first_q;          // ... on the Q operand
  int32_t vec_ok;                 // Y (and R) rows 16-byte aligned: vector path
  int32_t pdl;                    // launched as a programmatic dependent
  int32_t l2_prefetch;            // ... and prefetches its weight range into L2
  int32_t commit_group;           // ring stages released per UMMA commit (divides stages)
  int32_t acc_release;            // promotion: the per-K-block accumulator commit also
                                  // frees the block's ring stage (block scales, stages
                                  // <= accumulator buffers) or INT8 operand slot
  uint64_t* trace;                // per-CTA timeline (nullable), kTracePoints each
  int32_t trace_ctas;             // CTAs the trace buffer holds
  int32_t stream_k;               // balanced split-K over the grid (else split_k)
  int32_t max_contrib;            // workspace slots per tile
  int32_t cluster_reduce;         // split-K through distributed shared memory
  int32_t out;                    // OUT_BF16 / OUT_F16 / OUT_E4M3
  const float* s_y;               // per-tensor output scale (OUT_E4M3)
  int32_t tma_store;              // rows over M, 2-byte outputs: staged TMA stores of Y
  uint32_t out_stage_off;         // shared-memory offset of the staging boxes
};

constexpr int kTracePoints = 16;
enum : int { TR_START = 0, TR_SETUP = 1, TR_FIRST_TMA = 2, TR_FIRST_OPERANDS = 3,
             TR_LAST_COMMIT = 4, TR_FIRST_ACC = 5, TR_EPI_DONE = 6, TR_END = 7,
             // producer: first-unit weight loads (and L2 prefetches) issued,
             // before the wait on the previous kernel; last load issued
             TR_PRE_ISSUED = 8, TR_LAST_LOAD = 9,
             // epilogue (first epilogue thread, the CTA's last unit):
             // accumulator final; split-K partial stored or sent; arrival
             // counted (workspace) or all partials received (cluster); the
             // last arriver's first chunk reduced (tensor-memory accumulator
             // path); output stores begin.  Point 15 is not recorded.
             TR_LAST_ACC = 10, TR_PARTIAL_OUT = 11, TR_ARRIVED = 12, TR_REDUCED = 13,
             TR_STORE_BEGIN = 14 };

__device__ __forceinline__ void trace_point(const KParams& p, int point) {
  if (p.trace != nullptr && static_cast<int>(blockIdx.x) < p.trace_ctas)
    p.trace[static_cast<int64_t>(blockIdx.x) * kTracePoints + point] = global_timer_ns();
}

// G: gated linear unit (SwiGLU with SiLU).  W holds 2N rows, the gate half
// then the up half; each stage also carries the up half's weight tile and
// UMMA fills two accumulators per unit, gate in columns [0, BN) and up in
// [BN, 2 BN).
// PR: CTA pair.  Two CTAs of a cluster compute one 256 x BN tile with pair
// UMMAs (M = 256): each holds its 128 activation rows and half of the
// weight tile (BN/2 rows) per stage, and its 128 output rows in tensor
// memory; the even CTA issues the UMMAs.
template <int IN, int SC, bool SWAP, int BN, bool G = false, bool PR = false>
struct Cfg {
  static constexpr bool kConvert = (IN == IN_INT8);
  static constexpr bool kPromote = (SC == SC_BLOCK) || kConvert;
  static constexpr int kAtoms = kConvert ? 2 : 1;          // 128-byte K atoms per UMMA stage
  static constexpr int kElemsPerStage = (IN == IN_BF16) ? 64 : 128;
  static constexpr uint32_t kPBytes = 128u * 128u * kAtoms; // UMMA operand P per stage
  static constexpr uint32_t kQBytes = uint32_t(PR ? BN / 2 : BN) * 128u * kAtoms;
  static constexpr uint32_t kP8Bytes = kConvert ? 128u * 128u : 0u;  // int8 staging
  static constexpr uint32_t kQ8Bytes = kConvert ? uint32_t(BN) * 128u : 0u;
  // TMA ring stage: the UMMA operands, or (INT8) the int8 staging tiles.
  // INT8 converts P (128 rows) into fp16 in tensor memory (the UMMA's A
  // operand, two buffers of 64 columns) and Q into fp16 in a 2-slot shared
  // ring, so the int8 ring can be deep while the fp16 operands stay small
  // and shared memory carries the conversion's traffic for Q only.
  static constexpr uint32_t kWBytes = SWAP ? kPBytes : kQBytes;  // one weight operand tile
  static constexpr uint32_t kStageBytes =
      kConvert ? kP8Bytes + kQ8Bytes : kPBytes + kQBytes + (G ? kWBytes : 0u);
  // INT8 fp16 operand slots (P in tensor memory, Q in shared memory): the
  // transform of K tile g waits for the UMMAs of tile g - kOpSlots, so
  // three slots keep two tiles of slack between the transform warps and the
  // UMMA issuer (at most the accumulator buffers, for the release by the
  // accumulator commit; 64 + 64 x 3 tensor-memory columns at tile_n 16).
  // Two at tile_n 32, so that 4 x 32 + 2 x 64 columns leave room for a
  // second CTA on the SM.
  static constexpr int kOpSlots = kConvert ? (BN == 32 ? 2 : 3) : 2;
  static constexpr uint32_t kOpBytes = kConvert ? kOpSlots * kQBytes : 0u;
  static constexpr uint32_t kTxBytes =  // bytes one stage's TMA delivers (PR: to both CTAs)
      PR ? 2u * (128u + BN / 2) * 128u
         : (128u + BN) * 128u + (G ? (SWAP ? 128u : uint32_t(BN)) * 128u : 0u);
  // Epilogue warps: 4 (one per TMEM lane quarter), or 8 (two column halves
  // per quarter) for block-scale promotion of wide tiles, so each thread
  // keeps BN/2 running sums and the promotion keeps up with UMMA, and for
  // wide large-M tiles, so two warps per SM sub-partition hide the TMEM,
  // residual-load and activation latencies of a 128 x 128..256 epilogue.
  static constexpr int kEpiWarps =
      ((kPromote && !kConvert && BN >= 64) || (!SWAP && !kPromote && !G && BN >= 128)) ? 8 : 4;
  static constexpr int kEpiThreads = kEpiWarps * 32;
  static constexpr int kColsPerThread = BN / (kEpiWarps / 4);
  // Wide block-scale promotion (tile_n above 128): each epilogue thread
  // keeps 128 running sums.  The epilogue warps then form their own two
  // warpgroups (warps 4..11; warps 2 and 3 stay idle) so that the first
  // warpgroup (producer, UMMA issuer) can hand registers over to them with
  // setmaxnreg: kRegsLow per thread there, kRegsHigh in the epilogue.
  static constexpr bool kWidePromote = kPromote && !kConvert && BN > 128;
  static constexpr int kEpiWarp0 = kWidePromote ? 4 : 2;   // first epilogue warp
  static constexpr int kThreads = 32 * kEpiWarp0 + kEpiThreads + (kConvert ? 128 : 0);
  static constexpr int kRegsLow = 64, kRegsHigh = 216;
  // registers the split needs from the block's launch allocation
  static constexpr int kRegSplitNeed = kWidePromote ? 128 * kRegsLow + kEpiThreads * kRegsHigh : 0;
  // Small tiles (decode) are meant to run two CTAs per SM; cap registers so
  // two fit.  Promotion with wide tiles keeps BN accumulators per thread.
  // Decode tiles (BN 16) keep a third slot per SM free so that the next
  // call's CTAs (programmatic dependents) become resident while this grid
  // still runs.
  // Gated units hold twice the accumulator values in the epilogue: two
  // CTAs per SM for decode tiles.
  static constexpr int kMinBlocks =
      G ? (BN <= 32 ? 2 : 1)
        : kConvert ? (BN <= 32 ? 2 : 1)
                   : ((kPromote && BN >= 64) || BN >= 128) ? 1 : (BN <= 32 ? 3 : 2);
  // Register cap per thread for that residency.  The SM's 64K registers are
  // split over its 4 sub-partitions (16K each) and warps are spread over
  // them, so the busiest sub-partition holds ceil(warps / 4) warps of
  // 32 threads: at most 512 / ceil(warps / 4) registers per thread
  // (allocated in units of 8).
  static constexpr int kWarpsPerSmsp = (kMinBlocks * (kThreads / 32) + 3) / 4;
  static constexpr int kMaxRegs =
      (512 / kWarpsPerSmsp) / 8 * 8 > 255 ? 255 : (512 / kWarpsPerSmsp) / 8 * 8;
  // TMEM load chunk (columns): 32, or 16 where a thread's share of a wide
  // tile is not a multiple of 32 (tile_n 224 over two column halves)
  static constexpr int kCW = BN < 32 ? BN : (kColsPerThread % 32 != 0 ? 16 : 32);
  // TMEM accumulator buffers: 2 (one unit drains while the next fills), or
  // 4 when promoting K blocks so UMMA runs further ahead of the epilogue
  static constexpr int kAccBufs = (kPromote && 4 * BN <= 512) ? 4 : 2;
  static constexpr int kAccN = G ? 2 * BN : BN;  // accumulator columns of one unit
  // TMEM columns between accumulator buffers: a unit's columns, rounded up
  // to 256 for tiles between 128 and 256 columns (192, 224) so every buffer
  // starts at column 0 or 256
  static constexpr int kAccStride = (kAccN > 128 && kAccN < 256) ? 256 : kAccN;
  static constexpr uint32_t kAccCols = kAccBufs * kAccStride;
  static constexpr uint32_t kTmemACols = kConvert ? kOpSlots * 64u : 0u;  // fp16 P, 128 K each
  static constexpr uint32_t kTmemUsed = kAccCols + kTmemACols;
  static constexpr uint32_t kTmemCols =
      kTmemUsed <= 32 ? 32 : kTmemUsed <= 64 ? 64 : kTmemUsed <= 128 ? 128 : kTmemUsed <= 256 ? 256 : 512;
  static constexpr uint32_t kUmmaM = PR ? 256u : 128u;
  static constexpr uint32_t kIdesc =
      (IN == IN_BF16) ? idesc_f32acc(1, 1, kUmmaM, BN)
                      : idesc_f32acc(0, 0, kUmmaM, BN);  // e4m3 (f8f6f4) or f16 (converted int8)
  static_assert(BN % 16 == 0 && BN >= 16 && BN <= 256, "UMMA N for M=128");
  static_assert(!kPromote || BN <= 128 || (kWidePromote && BN == 256 && !SWAP && !G),
                "wide promotion: block scales, tile_n 256, rows over M");
  static_assert(!kWidePromote || kColsPerThread == 128, "128 running sums per epilogue thread");
  static_assert(!kWidePromote || 128 * kRegsLow + kEpiThreads * kRegsHigh <= kThreads * kMaxRegs,
                "register split within the launch allocation");
  static_assert(kTmemUsed <= 512, "tensor memory holds 512 columns");
  static_assert(!kConvert || kOpSlots <= kAccBufs,
                "an operand slot is released by the accumulator commit of its K tile");
  static_assert(!G || !kPromote, "gated units use the tensor-memory accumulator path");
  static_assert(!PR || (!SWAP && !G && (BN == 128 || BN == 256) && (!kPromote || kWidePromote)),
                "CTA pairs: tiles of 256 x 128 or 256 x 256 (per-token/channel or bf16), or "
                "256 x 256 with block-scale promotion");
};

template <int IN, int SC, bool SWAP, int BN, bool G = false, bool PR = false>
constexpr uint32_t smem_bytes_for(int stages) {
  using C = Cfg<IN, SC, SWAP, BN, G, PR>;
  return 1024u + uint32_t(stages) * C::kStageBytes + C::kOpBytes + 512u;
}

// ------------------------------------------------------------- helpers ----

__device__ __forceinline__ void record_status(int* status, int code) {
  if (status) atomicCAS(status, 0, code);
}

// Named barrier 1 among the epilogue warps only.
__device__ __forceinline__ void epi_bar_sync(int nthreads) {
  asm volatile("bar.sync 1, %0;" ::"r"(nthreads) : "memory");
}

__device__ __forceinline__ float tanh_fast(float x) {
  float y;
  asm("tanh.approx.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ float act_apply(int act, float v) {
  switch (act) {
    case ACT_RELU: return fmaxf(v, 0.0f);
    case ACT_GELU_ERF: return 0.5f * v * (1.0f + erff(v * 0.70710678118654752f));
    case ACT_GELU_TANH: {
      const float u = 0.7978845608028654f * (v + 0.044715f * v * v * v);
      return 0.5f * v * (1.0f + tanh_fast(u));
    }
    case ACT_SILU: return __fdividef(v, 1.0f + __expf(-v));
    default: return v;
  }
}

// The activation as a compile-time choice.  The epilogue code is
// instantiated per activation and selected once per chunk (EG_ACT_DISPATCH):
// a runtime switch inside the per-element code would be repeated for every
// unrolled element, spreading the path actually taken over a large stretch
// of code that the instruction cache cannot hold.
template <int ACT>
__device__ __forceinline__ float act_c(float v) {
  if constexpr (ACT == ACT_RELU) return fmaxf(v, 0.0f);
  if constexpr (ACT == ACT_GELU_ERF) return 0.5f * v * (1.0f + erff(v * 0.70710678118654752f));
  if constexpr (ACT == ACT_GELU_TANH) {
    const float u = 0.7978845608028654f * (v + 0.044715f * v * v * v);
    return 0.5f * v * (1.0f + tanh_fast(u));
  }
  if constexpr (ACT == ACT_SILU) return __fdividef(v, 1.0f + __expf(-v));
  return v;
}

// Runs CALL (an expression that names the activation as A_) with A_ bound to
// the compile-time value of `act`.
#define EG_ACT_DISPATCH(act, CALL)                                   \
  switch (act) {                                                     \
    case ACT_RELU: {                                                 \
      constexpr int A_ = ACT_RELU;                                   \
      CALL;                                                          \
    } break;                                                         \
    case ACT_GELU_ERF: {                                             \
      constexpr int A_ = ACT_GELU_ERF;                               \
      CALL;                                                          \
    } break;                                                         \
    case ACT_GELU_TANH: {                                            \
      constexpr int A_ = ACT_GELU_TANH;                              \
      CALL;                                                          \
    } break;                                                         \
    case ACT_SILU: {                                                 \
      constexpr int A_ = ACT_SILU;                                   \
      CALL;                                                          \
    } break;                                                         \
    default: {                                                       \
      constexpr int A_ = ACT_NONE;                                   \
      CALL;                                                          \
    } break;                                                         \
  }

// Float pair (hi + lo) arithmetic for the INT8 epilogue, so that
// acc * s_a * s_w + R is formed to ~2^-44 relative before the single bf16
// rounding (the oracle forms it in float64).
struct DF {
  float hi, lo;
};
__device__ __forceinline__ DF two_sum(float a, float b) {
  const float s = __fadd_rn(a, b);
  const float bb = __fsub_rn(s, a);
  const float e = __fadd_rn(__fsub_rn(a, __fsub_rn(s, bb)), __fsub_rn(b, bb));
  return {s, e};
}
__device__ __forceinline__ DF two_prod(float a, float b) {
  const float p = __fmul_rn(a, b);
  return {p, __fmaf_rn(a, b, -p)};
}
__device__ __forceinline__ DF df_add(DF x, float b) {
  const DF s = two_sum(x.hi, b);
  return two_sum(s.hi, __fadd_rn(s.lo, x.lo));
}
// Exact-input product acc * (sa * sw) as a float pair.
__device__ __forceinline__ DF df_scale_int(int32_t acc, float sa, float sw) {
  const DF s = two_prod(sa, sw);                 // exact
  const int32_t a0i = acc & 0xFFF;               // 0..4095
  const int32_t a1i = acc - a0i;                 // multiple of 4096: exact in fp32
  const float a1 = static_cast<float>(a1i), a0 = static_cast<float>(a0i);
  const DF p = two_prod(a1, s.hi);
  const DF q = two_prod(a0, s.hi);
  const float t = __fmaf_rn(a1, s.lo, __fmul_rn(a0, s.lo));
  const DF r = two_sum(p.hi, q.hi);
  const float tail = __fadd_rn(__fadd_rn(p.lo, q.lo), __fadd_rn(t, r.lo));
  return two_sum(r.hi, tail);
}
// Round hi + lo to bf16, nearest even, deciding exact ties of hi by lo.
__device__ __forceinline__ uint16_t bf16_bits_from_df(DF v) {
  const uint32_t u = __float_as_uint(v.hi);
  if ((u & 0x7F800000u) == 0x7F800000u)
    return __bfloat16_as_ushort(__float2bfloat16_rn(v.hi));
  const uint32_t rem = u & 0xFFFFu;
  const uint32_t base = u >> 16;
  bool up;
  if (rem > 0x8000u)
    up = true;
  else if (rem < 0x8000u)
    up = false;
  else if (v.lo == 0.0f)
    up = (base & 1u) != 0;
  else
    up = (v.lo > 0.0f) == (v.hi > 0.0f);
  return static_cast<uint16_t>(base + (up ? 1u : 0u));
}

__device__ __forceinline__ float bf16_to_f(uint16_t b) {
  return __uint_as_float(static_cast<uint32_t>(b) << 16);
}

// The single narrowing of an epilogue value to the output format: bf16 or
// fp16 bits, or (E4M3) the code of v * (1 / s_y), saturated to +-448, in the
// low byte.  All round to nearest even.  Each is one or two instructions,
// so the per-element code stays compact whatever the format.
__device__ __forceinline__ uint16_t out_bits(float v, int out, float inv_sy) {
  if (out == OUT_F16) return __half_as_ushort(__float2half_rn(v));
  if (out == OUT_E4M3)
    return static_cast<uint16_t>(
        __nv_cvt_float_to_fp8(__fmul_rn(v, inv_sy), __NV_SATFINITE, __NV_E4M3));
  return __bfloat16_as_ushort(__float2bfloat16_rn(v));
}

// 1 / s_y for E4M3 outputs (the multiply may differ from the division by
// one float32 ulp of v / s_y, far below the E4M3 step).
__device__ __forceinline__ float out_scale(const KParams& p) {
  return p.out == OUT_E4M3 ? __frcp_rn(__ldg(p.s_y)) : 1.0f;
}

// Store one output element at element index i of Y.
__device__ __forceinline__ void store_out(const KParams& p, int64_t i, uint16_t bits) {
  if (p.out == OUT_E4M3)
    reinterpret_cast<uint8_t*>(p.Y)[i] = static_cast<uint8_t>(bits);
  else
    reinterpret_cast<uint16_t*>(p.Y)[i] = bits;
}

// Store 8 consecutive output elements at element index i (vector path: Y
// rows 16-byte aligned, i a multiple of 8).
__device__ __forceinline__ void store_out8(const KParams& p, int64_t i, const uint16_t (&o)[8]) {
  if (p.out == OUT_E4M3) {
    uint32_t w[2];
#pragma unroll
    for (int h = 0; h < 2; ++h)
      w[h] = static_cast<uint32_t>(o[4 * h] & 0xFF) | (static_cast<uint32_t>(o[4 * h + 1] & 0xFF) << 8) |
             (static_cast<uint32_t>(o[4 * h + 2] & 0xFF) << 16) |
             (static_cast<uint32_t>(o[4 * h + 3] & 0xFF) << 24);
    *reinterpret_cast<uint2*>(reinterpret_cast<uint8_t*>(p.Y) + i) = make_uint2(w[0], w[1]);
  } else {
    uint32_t w[4];
#pragma unroll
    for (int h = 0; h < 4; ++h)
      w[h] = static_cast<uint32_t>(o[2 * h]) | (static_cast<uint32_t>(o[2 * h + 1]) << 16);
    *reinterpret_cast<uint4*>(reinterpret_cast<uint16_t*>(p.Y) + i) = make_uint4(w[0], w[1], w[2], w[3]);
  }
}

// One output element of the epilogue (float path).  `bias` and `r` are the
// bf16 inputs already widened; unused ones are ignored by the flags.
template <int ACT>
__device__ __forceinline__ float epi_value(float v, float scale, float bias, float r,
                                           uint32_t flags) {
  v = v * scale;
  if (flags & F_BIAS) v += bias;
  if (flags & F_RES_PRE) {
    v += r;
    v = act_c<ACT>(v);
  } else {
    v = act_c<ACT>(v);
    if (flags & F_RES) v += r;
  }
  return v;
}

// INT8 epilogue element: exact int32 accumulator -> output bits (bf16 from
// the float pair directly; fp16 and E4M3 from its float sum).
template <int ACT>
__device__ __forceinline__ uint16_t epi_int8(int32_t acc, float sa, float sw, float bias, float r,
                                             uint32_t flags, int out, float inv_sy) {
  constexpr int kAct = ACT;
  DF v = df_scale_int(acc, sa, sw);
  if (flags & F_BIAS) v = df_add(v, bias);
  if (flags & F_RES_PRE) {
    v = df_add(v, r);
    if (kAct != ACT_NONE) v = DF{act_c<kAct>(__fadd_rn(v.hi, v.lo)), 0.0f};
  } else {
    if (kAct != ACT_NONE) v = DF{act_c<kAct>(__fadd_rn(v.hi, v.lo)), 0.0f};
    if (flags & F_RES) v = df_add(v, r);
  }
  if (out == OUT_BF16) return bf16_bits_from_df(v);
  return out_bits(__fadd_rn(v.hi, v.lo), out, inv_sy);
}

// ------------------------------------------------------------ epilogue ----

// Swap-AB epilogue inputs of one TMEM lane (output channel n) and CW tokens
// col0..col0+CW-1.  None depends on the accumulator, so the decode path loads
// them before it waits for the mainloop; every load is independent and
// predicated, so their latencies overlap.
template <int CW>
struct SwapIn {
  float b, sw;
};

template <int SC, int CW>
__device__ __forceinline__ void load_swap_inputs(const KParams& p, int n, int col0, SwapIn<CW>& in) {
  const bool nv = n < p.N;
  const bool has_bias = (p.flags & F_BIAS) != 0;
  in.b = (has_bias && nv) ? __bfloat162float(p.bias[n]) : 0.0f;
  in.sw = (SC == SC_TC && nv) ? __ldg(p.s_w + n) : 1.0f;
  if constexpr (SC == SC_TC) {
    // the token scales are the same for every lane: touch them now so the
    // epilogue finds them in L1
    if (nv && (threadIdx.x & 31) == 0 && col0 < p.M) (void)__ldg(p.s_a + col0);
  }
}

// Swap-AB epilogue compute and store: lanes of a warp hold consecutive n, so
// each token's residual loads and Y stores are coalesced across the warp.
// This path runs once per output tile, in split-K by whichever CTA of the
// tile arrives last, so its code is usually not in that SM's instruction
// cache (nor, for a call on its own, in L2): it is kept compact.  A runtime
// loop walks the chunk's valid tokens four at a time (their loads first,
// then their arithmetic), the activation is a compile-time choice made once
// per chunk, and the output format is chosen per element.
template <int CW>
__device__ __forceinline__ uint32_t pick(const uint32_t (&v)[CW], int j) {
  uint32_t x = v[0];
#pragma unroll
  for (int k = 1; k < CW; ++k) x = (j == k) ? v[k] : x;
  return x;
}

template <int IN, int SC, int CW, int ACT, int OF = -1>
__device__ __forceinline__ void store_swap(const KParams& p, int n, int col0,
                                           const uint32_t (&vals)[CW], const SwapIn<CW>& in) {
  if (n >= p.N) return;
  const bool has_res = (p.flags & (F_RES | F_RES_PRE)) != 0;
  const float sy = out_scale(p);
  const int count = min(CW, p.M - col0);
#pragma unroll 1
  for (int j0 = 0; j0 < count; j0 += 4) {
    float r[4], sa[4];
    uint32_t v[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int m = col0 + j0 + q;
      const bool ok = j0 + q < count;
      v[q] = pick<CW>(vals, j0 + q);
      r[q] = (has_res && ok) ? __bfloat162float(p.R[static_cast<int64_t>(m) * p.ldr + n]) : 0.0f;
      sa[q] = (SC == SC_TC && ok) ? __ldg(p.s_a + m) : 1.0f;
    }
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      if (j0 + q < count) {
        uint16_t o;
        if (IN == IN_INT8) {
          o = epi_int8<ACT>(static_cast<int32_t>(v[q]), sa[q], in.sw, in.b, r[q], p.flags, p.out, sy);
        } else {
          const float y = epi_value<ACT>(__uint_as_float(v[q]), (SC == SC_TC) ? sa[q] * in.sw : 1.0f,
                                         in.b, r[q], p.flags);
          o = (OF == OUT_BF16) ? __bfloat16_as_ushort(__float2bfloat16_rn(y)) : out_bits(y, p.out, sy);
        }
        const int64_t at = static_cast<int64_t>(col0 + j0 + q) * p.ldy + n;
        if (OF == OUT_BF16)
          reinterpret_cast<uint16_t*>(p.Y)[at] = o;
        else
          store_out(p, at, o);
      }
    }
  }
}

// Output bits of CW consecutive columns col0 .. col0 + CW - 1 of row m (rows
// over M, m < M), the fused epilogue applied to the accumulator values
// `vals` (fp32 bits, or int32 for INT8); columns at or beyond N give 0.
template <int IN, int SC, int CW, int ACT>
__device__ __forceinline__ void epi_row_values(const KParams& p, int m, int col0,
                                               const uint32_t (&vals)[CW], uint16_t (&out)[CW]) {
  const bool has_bias = (p.flags & F_BIAS) != 0;
  const bool has_res = (p.flags & (F_RES | F_RES_PRE)) != 0;
  const float sa = (SC == SC_TC) ? __ldg(p.s_a + m) : 1.0f;
  const float sy = out_scale(p);
  const __nv_bfloat16* rrow = has_res ? p.R + static_cast<int64_t>(m) * p.ldr : nullptr;
  if (p.vec_ok && col0 + CW <= p.N) {
    // full chunk: 16-byte vector loads of bias / R / s_w
#pragma unroll
    for (int g = 0; g < CW / 8; ++g) {
      uint4 bv = make_uint4(0, 0, 0, 0), rv = make_uint4(0, 0, 0, 0);
      if (has_bias) bv = __ldg(reinterpret_cast<const uint4*>(p.bias + col0) + g);
      if (has_res) rv = __ldg(reinterpret_cast<const uint4*>(rrow + col0) + g);
      float4 sw0 = make_float4(1, 1, 1, 1), sw1 = make_float4(1, 1, 1, 1);
      if (SC == SC_TC) {
        sw0 = __ldg(reinterpret_cast<const float4*>(p.s_w + col0) + 2 * g);
        sw1 = __ldg(reinterpret_cast<const float4*>(p.s_w + col0) + 2 * g + 1);
      }
      const uint32_t bw[4] = {bv.x, bv.y, bv.z, bv.w};
      const uint32_t rw[4] = {rv.x, rv.y, rv.z, rv.w};
      const float sws[8] = {sw0.x, sw0.y, sw0.z, sw0.w, sw1.x, sw1.y, sw1.z, sw1.w};
#pragma unroll
      for (int h = 0; h < 4; ++h) {
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int j = g * 8 + h * 2 + e;
          const float b = bf16_to_f(static_cast<uint16_t>(bw[h] >> (16 * e)));
          const float r = bf16_to_f(static_cast<uint16_t>(rw[h] >> (16 * e)));
          if (IN == IN_INT8) {
            out[j] = epi_int8<ACT>(static_cast<int32_t>(vals[j]), sa, sws[h * 2 + e], b, r, p.flags,
                                   p.out, sy);
          } else {
            const float sc = (SC == SC_TC) ? sa * sws[h * 2 + e] : 1.0f;
            out[j] = out_bits(epi_value<ACT>(__uint_as_float(vals[j]), sc, b, r, p.flags), p.out, sy);
          }
        }
      }
    }
  } else {
#pragma unroll
    for (int j = 0; j < CW; ++j) {
      const int n = col0 + j;
      out[j] = 0;
      if (n < p.N) {
        const float b = has_bias ? __bfloat162float(p.bias[n]) : 0.0f;
        const float r = has_res ? __bfloat162float(rrow[n]) : 0.0f;
        const float sw = (SC == SC_TC) ? __ldg(p.s_w + n) : 1.0f;
        if (IN == IN_INT8)
          out[j] = epi_int8<ACT>(static_cast<int32_t>(vals[j]), sa, sw, b, r, p.flags, p.out, sy);
        else
          out[j] = out_bits(epi_value<ACT>(__uint_as_float(vals[j]), (SC == SC_TC) ? sa * sw : 1.0f,
                                           b, r, p.flags),
                            p.out, sy);
      }
    }
  }
}

// The same for 16-bit outputs (bf16 or fp16), packed two per word: the float
// path forms every value of the chunk first and then narrows pairs with one
// conversion each (the format chosen once per chunk, not per element); the
// rounding of each value is the same as the single-element narrowing.
template <int IN, int SC, int CW, int ACT>
__device__ __forceinline__ void epi_row_words(const KParams& p, int m, int col0,
                                              const uint32_t (&vals)[CW], uint32_t (&wd)[CW / 2]) {
  if constexpr (IN == IN_INT8) {
    uint16_t o[CW];
    epi_row_values<IN, SC, CW, ACT>(p, m, col0, vals, o);
#pragma unroll
    for (int j = 0; j < CW / 2; ++j)
      wd[j] = static_cast<uint32_t>(o[2 * j]) | (static_cast<uint32_t>(o[2 * j + 1]) << 16);
  } else {
    const uint32_t flags = p.flags;
    const bool has_bias = (flags & F_BIAS) != 0;
    const bool has_res = (flags & (F_RES | F_RES_PRE)) != 0;
    const float sa = (SC == SC_TC) ? __ldg(p.s_a + m) : 1.0f;
    const __nv_bfloat16* rrow = has_res ? p.R + static_cast<int64_t>(m) * p.ldr : nullptr;
    float v[CW];
    if (p.vec_ok && col0 + CW <= p.N && !has_bias && !has_res) {
      // no bias or residual: the scaled, activated accumulator (epi_value's
      // arithmetic with no epilogue terms), the flag tests out of the loop
#pragma unroll
      for (int g = 0; g < CW / 8; ++g) {
        float4 sw0 = make_float4(1, 1, 1, 1), sw1 = make_float4(1, 1, 1, 1);
        if (SC == SC_TC) {
          sw0 = __ldg(reinterpret_cast<const float4*>(p.s_w + col0) + 2 * g);
          sw1 = __ldg(reinterpret_cast<const float4*>(p.s_w + col0) + 2 * g + 1);
        }
        const float sws[8] = {sw0.x, sw0.y, sw0.z, sw0.w, sw1.x, sw1.y, sw1.z, sw1.w};
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const float sc = (SC == SC_TC) ? sa * sws[e] : 1.0f;
          v[g * 8 + e] = act_c<ACT>(__uint_as_float(vals[g * 8 + e]) * sc);
        }
      }
    } else if (p.vec_ok && col0 + CW <= p.N) {
#pragma unroll
      for (int g = 0; g < CW / 8; ++g) {
        uint4 bv = make_uint4(0, 0, 0, 0), rv = make_uint4(0, 0, 0, 0);
        if (has_bias) bv = __ldg(reinterpret_cast<const uint4*>(p.bias + col0) + g);
        if (has_res) rv = __ldg(reinterpret_cast<const uint4*>(rrow + col0) + g);
        float4 sw0 = make_float4(1, 1, 1, 1), sw1 = make_float4(1, 1, 1, 1);
        if (SC == SC_TC) {
          sw0 = __ldg(reinterpret_cast<const float4*>(p.s_w + col0) + 2 * g);
          sw1 = __ldg(reinterpret_cast<const float4*>(p.s_w + col0) + 2 * g + 1);
        }
        const uint32_t bw[4] = {bv.x, bv.y, bv.z, bv.w};
        const uint32_t rw[4] = {rv.x, rv.y, rv.z, rv.w};
        const float sws[8] = {sw0.x, sw0.y, sw0.z, sw0.w, sw1.x, sw1.y, sw1.z, sw1.w};
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const float b = bf16_to_f(static_cast<uint16_t>(bw[e >> 1] >> (16 * (e & 1))));
          const float r = bf16_to_f(static_cast<uint16_t>(rw[e >> 1] >> (16 * (e & 1))));
          const float sc = (SC == SC_TC) ? sa * sws[e] : 1.0f;
          v[g * 8 + e] = epi_value<ACT>(__uint_as_float(vals[g * 8 + e]), sc, b, r, flags);
        }
      }
    } else {
#pragma unroll
      for (int j = 0; j < CW; ++j) {
        const int n = col0 + j;
        v[j] = 0.0f;
        if (n < p.N) {
          const float b = has_bias ? __bfloat162float(p.bias[n]) : 0.0f;
          const float r = has_res ? __bfloat162float(rrow[n]) : 0.0f;
          const float sw = (SC == SC_TC) ? __ldg(p.s_w + n) : 1.0f;
          v[j] = epi_value<ACT>(__uint_as_float(vals[j]), (SC == SC_TC) ? sa * sw : 1.0f, b, r, flags);
        }
      }
    }
    if (p.out == OUT_F16) {
#pragma unroll
      for (int j = 0; j < CW / 2; ++j) {
        const __half2 h = __floats2half2_rn(v[2 * j], v[2 * j + 1]);
        wd[j] = *reinterpret_cast<const uint32_t*>(&h);
      }
    } else {
#pragma unroll
      for (int j = 0; j < CW / 2; ++j) {
        const __nv_bfloat162 h = __floats2bfloat162_rn(v[2 * j], v[2 * j + 1]);
        wd[j] = *reinterpret_cast<const uint32_t*>(&h);
      }
    }
  }
}

// Apply the epilogue to CW consecutive accumulator columns of one TMEM lane
// (= one UMMA row) and store them.  `vals` holds fp32 bits, or int32 for
// INT8.  row = tile row index + lane row; c0 = first column of the chunk.
template <int IN, int SC, bool SWAP, int CW, int ACT>
__device__ __forceinline__ void epilogue_chunk_a(const KParams& p, int row, int col0,
                                                 const uint32_t (&vals)[CW]) {
  const bool debug = (p.flags & F_DEBUG) != 0;
  if (!SWAP) {
    // row = m, columns = n: a thread owns CW consecutive outputs of one row.
    const int m = row;
    if (m >= p.M) return;
    if (debug) {
      uint32_t* y = reinterpret_cast<uint32_t*>(p.Y) + static_cast<int64_t>(m) * p.ldy;
#pragma unroll
      for (int j = 0; j < CW; ++j)
        if (col0 + j < p.N) y[col0 + j] = vals[j];
      return;
    }
    uint16_t out[CW];
    epi_row_values<IN, SC, CW, ACT>(p, m, col0, vals, out);
    const int64_t yrow = static_cast<int64_t>(m) * p.ldy;  // element index of row m
    if (p.vec_ok && col0 + CW <= p.N) {
#pragma unroll
      for (int g = 0; g < CW / 8; ++g) {
        uint16_t o8[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) o8[e] = out[g * 8 + e];
        store_out8(p, yrow + col0 + g * 8, o8);
      }
    } else {
#pragma unroll
      for (int j = 0; j < CW; ++j)
        if (col0 + j < p.N) store_out(p, yrow + col0 + j, out[j]);
    }
  } else {
    // row = n, columns = m: lanes of a warp hold consecutive n, so each
    // column's loads of R and stores of Y are coalesced across the warp.
    const int n = row;
    if (n >= p.N) return;
    if (debug) {
      uint32_t* y = reinterpret_cast<uint32_t*>(p.Y);
#pragma unroll
      for (int j = 0; j < CW; ++j) {
        const int m = col0 + j;
        if (m < p.M) y[static_cast<int64_t>(m) * p.ldy + n] = vals[j];
      }
      return;
    }
    SwapIn<CW> in;
    load_swap_inputs<SC, CW>(p, n, col0, in);
    store_swap<IN, SC, CW, ACT>(p, n, col0, vals, in);
  }
}

// ---------------------------------------------------- staged TMA stores ----
//
// Rows over M: a thread holds CW consecutive outputs of one row, so a warp's
// direct stores touch 32 rows per instruction.  Instead each warp writes its
// 32 rows x CW columns (2-byte outputs) into a shared-memory staging box in
// the layout a bulk-tensor store with 64-byte (CW = 32) or 32-byte (CW = 16)
// swizzle reads, and one lane stores the box with one TMA store (rows and
// columns outside Y are not written).  Two boxes per warp alternate, so the
// next chunk is computed while the previous box is read out.

// Bytes of one warp's staging box.
template <int CW>
__host__ __device__ constexpr uint32_t stage_box_bytes() { return 32u * CW * 2u; }

// Write row r's CW outputs (2 bytes each, packed two per word) into the
// swizzled box.
template <int CW>
__device__ __forceinline__ void stage_row(uint8_t* box, int r, const uint32_t (&wd)[CW / 2]) {
  static_assert(CW == 32 || CW == 16, "64- or 32-byte box rows");
#pragma unroll
  for (int c = 0; c < CW / 8; ++c) {
    const int pc = (CW == 32) ? (c ^ ((r >> 1) & 3)) : (c ^ ((r >> 2) & 1));
    *reinterpret_cast<uint4*>(box + r * (CW * 2) + pc * 16) =
        make_uint4(wd[4 * c], wd[4 * c + 1], wd[4 * c + 2], wd[4 * c + 3]);
  }
}

// The epilogue of one chunk through a staging box: every lane of the warp
// calls this (row = the lane's row, row_base = the warp's first row).  The
// box was last used two chunks ago; lane 0 waits until that store has read
// it.
template <int IN, int SC, int CW, int ACT>
__device__ __forceinline__ void epilogue_chunk_staged(const KParams& p, const CUtensorMap* tmY, int row,
                                                      int row_base, int col0,
                                                      const uint32_t (&vals)[CW], uint8_t* box,
                                                      int lane) {
  if (lane == 0) bulk_wait_group_read<1>();
  __syncwarp();
  uint32_t wd[CW / 2];
  if (row < p.M) {
    epi_row_words<IN, SC, CW, ACT>(p, row, col0, vals, wd);
  } else {
#pragma unroll
    for (int j = 0; j < CW / 2; ++j) wd[j] = 0u;
  }
  stage_row<CW>(box, lane, wd);
  fence_proxy_async_smem();
  __syncwarp();
  if (lane == 0) {
    tma_store_2d(tmY, box, col0, row_base);
    bulk_commit_group();
  }
}

template <int IN, int SC, bool SWAP, int CW>
__device__ __forceinline__ void epilogue_chunk(const KParams& p, int row, int col0,
                                               const uint32_t (&vals)[CW]) {
  EG_ACT_DISPATCH(p.act, (epilogue_chunk_a<IN, SC, SWAP, CW, A_>(p, row, col0, vals)))
}

// The epilogue of a thread's CPT promoted accumulators (columns col0 ..
// col0 + CPT - 1 of its row), CW columns at a time, with the activation a
// compile-time choice made once for all of them (the chunk loop unrolls and
// the accumulators stay in registers).
// Chunk `idx` (CW values) of a thread's CPT accumulators, picked with
// selects so that the accumulators stay in registers while the chunk loop
// itself is not unrolled.
template <int CW, int CPT>
__device__ __forceinline__ void pick_chunk(const uint32_t (&acc)[CPT], int idx, uint32_t (&r)[CW]) {
#pragma unroll
  for (int j = 0; j < CW; ++j) r[j] = acc[j];
#pragma unroll
  for (int k = 1; k < CPT / CW; ++k)
#pragma unroll
    for (int j = 0; j < CW; ++j) r[j] = (idx == k) ? acc[k * CW + j] : r[j];
}

// The promoted store runs once per output tile, between two tiles' K loops,
// so its code is usually not in the instruction cache when it starts: the
// chunk loop is a runtime loop (one copy of the chunk code per activation).
template <int IN, int SC, bool SWAP, int CW, int CPT, int ACT>
__device__ __forceinline__ void promoted_store(const KParams& p, int row, int col0,
                                               const uint32_t (&acc)[CPT]) {
#pragma unroll 1
  for (int q = 0; q < CPT / CW; ++q) {
    uint32_t r[CW];
    pick_chunk<CW, CPT>(acc, q, r);
    epilogue_chunk_a<IN, SC, SWAP, CW, ACT>(p, row, col0 + q * CW, r);
  }
}

// The same through staging boxes and TMA stores (rows over M); `nbox`
// counts the warp's boxes used so far (they alternate).  Here the chunk loop
// is unrolled: with rows over M the store runs once per large tile, and the
// selects a runtime chunk index needs (three per value) cost the epilogue
// warps more than the unrolled code's instruction fetches (Block_FP8, 2048
// tokens: 307 -> 299 us).
template <int IN, int SC, int CW, int CPT, int ACT>
__device__ __forceinline__ void promoted_store_staged(const KParams& p, const CUtensorMap* tmY, int row,
                                                      int row_base, int col0, const uint32_t (&acc)[CPT],
                                                      uint8_t* boxes, uint32_t& nbox, int lane) {
#pragma unroll
  for (int q = 0; q < CPT / CW; ++q) {
    uint32_t r[CW];
    pick_chunk<CW, CPT>(acc, q, r);
    epilogue_chunk_staged<IN, SC, CW, ACT>(p, tmY, row, row_base, col0 + q * CW, r,
                                           boxes + (nbox & 1u) * stage_box_bytes<CW>(), lane);
    ++nbox;
  }
}

// Gated unit epilogue of CW consecutive accumulator columns of one TMEM lane:
// gate values g and up values u (fp32 bits).  Per output (m, n):
// gate = scale(g) + bias[n], up = scale(u) + bias[N + n] (scale: s_a[m] *
// s_w[n] and s_a[m] * s_w[N + n]), y = act(gate) * up (+ R[m][n]), one
// narrowing, one store.  Rows over N (swap-AB: row = n, columns = tokens)
// or over M (row = m, columns = n).
template <int SC, bool SWAP, int CW, int ACT>
__device__ __forceinline__ void epilogue_gated_a(const KParams& p, int row, int col0,
                                                 const uint32_t (&g)[CW], const uint32_t (&u)[CW]) {
  const bool has_bias = (p.flags & F_BIAS) != 0;
  const bool has_res = (p.flags & F_RES) != 0;
  const float sy = out_scale(p);
  if (SWAP ? row >= p.N : row >= p.M) return;
  float rsg = 1.0f, rsu = 1.0f, rbg = 0.0f, rbu = 0.0f;  // per-row inputs
  if (SWAP) {
    if (SC == SC_TC) { rsg = __ldg(p.s_w + row); rsu = __ldg(p.s_w + p.N + row); }
    if (has_bias) { rbg = __bfloat162float(p.bias[row]); rbu = __bfloat162float(p.bias[p.N + row]); }
  } else if (SC == SC_TC) {
    rsg = rsu = __ldg(p.s_a + row);
  }
  constexpr int GR = CW < 8 ? CW : 8;
#pragma unroll
  for (int c0 = 0; c0 < CW; c0 += GR) {
    float sg[GR], su[GR], bg[GR], bu[GR], rr[GR];
#pragma unroll
    for (int j = 0; j < GR; ++j) {
      const int col = col0 + c0 + j;
      const bool ok = SWAP ? col < p.M : col < p.N;
      const int m = SWAP ? col : row, n = SWAP ? row : col;
      sg[j] = su[j] = 1.0f;
      bg[j] = rbg;
      bu[j] = rbu;
      if (ok && SC == SC_TC) {
        if (SWAP) {
          const float sa = __ldg(p.s_a + col);
          sg[j] = sa * rsg;
          su[j] = sa * rsu;
        } else {
          sg[j] = rsg * __ldg(p.s_w + col);
          su[j] = rsu * __ldg(p.s_w + p.N + col);
        }
      }
      if (ok && !SWAP && has_bias) {
        bg[j] = __bfloat162float(p.bias[col]);
        bu[j] = __bfloat162float(p.bias[p.N + col]);
      }
      rr[j] = (ok && has_res) ? __bfloat162float(p.R[static_cast<int64_t>(m) * p.ldr + n]) : 0.0f;
    }
#pragma unroll
    for (int j = 0; j < GR; ++j) {
      const int col = col0 + c0 + j;
      if (SWAP ? col >= p.M : col >= p.N) break;
      const int m = SWAP ? col : row, n = SWAP ? row : col;
      float gv = __uint_as_float(g[c0 + j]) * sg[j];
      float uv = __uint_as_float(u[c0 + j]) * su[j];
      if (has_bias) {
        gv += bg[j];
        uv += bu[j];
      }
      float y = act_c<ACT>(gv) * uv;
      if (has_res) y += rr[j];
      store_out(p, static_cast<int64_t>(m) * p.ldy + n, out_bits(y, p.out, sy));
    }
  }
}

template <int SC, bool SWAP, int CW>
__device__ __forceinline__ void epilogue_gated(const KParams& p, int row, int col0,
                                               const uint32_t (&g)[CW], const uint32_t (&u)[CW]) {
  EG_ACT_DISPATCH(p.act, (epilogue_gated_a<SC, SWAP, CW, A_>(p, row, col0, g, u)))
}

template <int CW>
__device__ __forceinline__ void tmem_load_chunk_p(uint32_t taddr, uint32_t* r) {
  if constexpr (CW == 32) {
    tmem_ld32p(taddr, r);
  } else {
    tmem_ld16(taddr, r);
  }
}

template <int CW>
__device__ __forceinline__ void tmem_load_chunk(uint32_t taddr, uint32_t (&r)[CW]) {
  if constexpr (CW == 32) {
    tmem_ld32(taddr, r);
  } else {
    tmem_ld16(taddr, r);
  }
}

// Split-K: store this split's partial for (tile, split); valid entries only.
// Layout: [split][tile][column][128 lanes] so a warp's stores coalesce.
template <int BN>
__device__ __forceinline__ uint32_t* ws_slot(const KParams& p, int split, int tile, int col,
                                             int lane_row) {
  const int64_t tiles = static_cast<int64_t>(p.tiles_rows) * p.tiles_cols;
  return reinterpret_cast<uint32_t*>(p.ws) +
         ((static_cast<int64_t>(split) * tiles + tile) * BN + col) * 128 + lane_row;
}

// ---------------------------------------------------------------- kernel ---

// INT8 prologue transform of one ring stage: the int8 staging tiles (TMA,
// 128-byte swizzled rows of 128 codes) become fp16 tiles in the UMMA layout
// (two 128-byte K atoms per tile).  Exact: every int8 value is an fp16 value.
// Convert the int8 tile of `rows` rows (128 codes each) at src to fp16 at dst.
// The 128 transform threads own 16-byte chunks q = ct + 128 k: one chunk
// column j = ct % 8 and rows ct/8 + 16 k, so the swizzle phase (row % 8) is
// the same for all of a thread's chunks.  All loads are issued first, then
// the arithmetic, then the stores.
template <int NCH>
__device__ __forceinline__ void convert_tile(const uint8_t* src, uint8_t* dst, int rows, int ct) {
  const int j = ct & 7;
  const int r0 = ct >> 3;
  const int sw = r0 & 7;                  // == (r0 + 16 k) & 7
  const uint32_t src_off = static_cast<uint32_t>(r0) * 128u + (static_cast<uint32_t>(j ^ sw) << 4);
  uint4 v[NCH];
#pragma unroll
  for (int k = 0; k < NCH; ++k)
    v[k] = *reinterpret_cast<const uint4*>(src + src_off + static_cast<uint32_t>(k) * 16u * 128u);
  // 16 fp16 values = two 16-byte chunks of fp16 atom j/4: chunks 2(j%4), +1
  uint8_t* atom = dst + static_cast<uint32_t>(j >> 2) * static_cast<uint32_t>(rows) * 128u;
  const int c0 = 2 * (j & 3);
  const uint32_t d0 = static_cast<uint32_t>(r0) * 128u + (static_cast<uint32_t>(c0 ^ sw) << 4);
  const uint32_t d1 = static_cast<uint32_t>(r0) * 128u + (static_cast<uint32_t>((c0 + 1) ^ sw) << 4);
  const __half2 bias2 = __floats2half2_rn(1152.0f, 1152.0f);
#pragma unroll
  for (int k = 0; k < NCH; ++k) {
    const uint32_t w4[4] = {v[k].x, v[k].y, v[k].z, v[k].w};
    uint32_t h[8];
#pragma unroll
    for (int t = 0; t < 4; ++t) {
      const uint32_t x = w4[t] ^ 0x80808080u;  // byte b -> b + 128 (unsigned)
      uint32_t lo, hi;
      asm("prmt.b32 %0, %1, %2, 0x4140;" : "=r"(lo) : "r"(x), "r"(0x64646464u));
      asm("prmt.b32 %0, %1, %2, 0x4342;" : "=r"(hi) : "r"(x), "r"(0x64646464u));
      // fp16 0x64XX = 1024 + XX; subtracting 1152 = 1024 + 128 gives b exactly
      __half2 l2 = __hsub2(*reinterpret_cast<__half2*>(&lo), bias2);
      __half2 h2 = __hsub2(*reinterpret_cast<__half2*>(&hi), bias2);
      h[2 * t] = *reinterpret_cast<uint32_t*>(&l2);
      h[2 * t + 1] = *reinterpret_cast<uint32_t*>(&h2);
    }
    const uint32_t rk = static_cast<uint32_t>(k) * 16u * 128u;
    *reinterpret_cast<uint4*>(atom + d0 + rk) = make_uint4(h[0], h[1], h[2], h[3]);
    *reinterpret_cast<uint4*>(atom + d1 + rk) = make_uint4(h[4], h[5], h[6], h[7]);
  }
}

// INT8 prologue transform of P, one row per thread: row r (TMEM lane r) of
// the int8 staging tile (128 codes, 128-byte swizzled) becomes 64 columns of
// fp16 pairs in tensor memory at t_row (the warp's lane quarter and the
// buffer's first column), in K order, with two 32-column stores.
__device__ __forceinline__ void convert_row_to_tmem(const uint8_t* src, uint32_t t_row, int r) {
  const int sw = r & 7;
  const uint8_t* row = src + r * 128;
  const __half2 bias2 = __floats2half2_rn(1152.0f, 1152.0f);
#pragma unroll
  for (int half = 0; half < 2; ++half) {
    uint32_t h[32];
#pragma unroll
    for (int jj = 0; jj < 4; ++jj) {
      const int j = half * 4 + jj;  // 16-byte chunk: codes 16 j .. 16 j + 15
      const uint4 v = *reinterpret_cast<const uint4*>(row + ((j ^ sw) << 4));
      const uint32_t w4[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int t = 0; t < 4; ++t) {
        const uint32_t x = w4[t] ^ 0x80808080u;  // byte b -> b + 128 (unsigned)
        uint32_t lo, hi;
        asm("prmt.b32 %0, %1, %2, 0x4140;" : "=r"(lo) : "r"(x), "r"(0x64646464u));
        asm("prmt.b32 %0, %1, %2, 0x4342;" : "=r"(hi) : "r"(x), "r"(0x64646464u));
        // fp16 0x64XX = 1024 + XX; subtracting 1152 = 1024 + 128 gives b exactly
        __half2 l2 = __hsub2(*reinterpret_cast<__half2*>(&lo), bias2);
        __half2 h2 = __hsub2(*reinterpret_cast<__half2*>(&hi), bias2);
        h[jj * 8 + 2 * t] = *reinterpret_cast<uint32_t*>(&l2);
        h[jj * 8 + 2 * t + 1] = *reinterpret_cast<uint32_t*>(&h2);
      }
    }
    tmem_st32(t_row + static_cast<uint32_t>(half * 32), h);
  }
}

// One work unit = one 128 x BN output tile and one K split.
// A work unit: K tiles [kt0, kt0 + nk) of one 128 x BN output tile.  The
// tile's K range is cut into `contrib` parts; this is part `j` (parts reduce
// in the order j = 0..contrib-1).
struct Unit {
  int j, contrib, tile, tile_r, tile_c, row0, col0, kt0, nk;
};

// PR: tiles are 256 rows high (tiles_rows counts them); the odd CTA of the
// pair owns the tile's second 128 rows.
template <bool PR = false>
__device__ __forceinline__ void unit_tile(const KParams& p, int tile, int bn, Unit& w) {
  w.tile = tile;
  w.tile_r = tile % p.tiles_rows;
  w.tile_c = tile / p.tiles_rows;
  w.row0 = PR ? w.tile_r * 256 + static_cast<int>(blockIdx.x & 1u) * 128 : w.tile_r * 128;
  w.col0 = w.tile_c * bn;
}

// The work slot of this CTA and the number of slots: one per CTA, or (PR)
// one per CTA pair, both CTAs of a pair walking the same units.
template <bool PR>
__device__ __forceinline__ int work_slot() {
  return PR ? static_cast<int>(blockIdx.x >> 1) : static_cast<int>(blockIdx.x);
}
template <bool PR>
__device__ __forceinline__ int work_slots() {
  return PR ? static_cast<int>(gridDim.x >> 1) : static_cast<int>(gridDim.x);
}

// Work assignment of this CTA.  Split-K: units u = blockIdx.x, +gridDim.x,
// ... each one (tile, split) with even K splits.  Balanced split-K (stream
// K), over T tiles and G CTAs: the first stream_dp_tiles() tiles are whole
// units handed out data-parallel (tile c, c + G, ...: concurrently running
// CTAs work on neighbouring tiles, so each weight tile is fetched from DRAM
// once and shared through L2); the remaining tiles' tiles x K-tiles
// iterations are cut into G equal contiguous ranges, CTA c owning
// [floor(c I / G), floor((c+1) I / G)) and walking it tile by tile, so a
// tile's K range is shared by the CTAs whose ranges overlap it.
// 32-bit positions (the host keeps tiles x max(split_k, K tiles) within
// int32): the iterator lives in registers of all three roles.
struct WorkIter {
  int pos, end;      // stream-K iterations (relative to the split tiles), or units
  int dp, dp_tiles;  // next data-parallel tile; tiles before the split ones
};

// Whole-tile waves before the split tail: all but the last full wave, so the
// split part covers between one and two waves of tiles.
__host__ __device__ __forceinline__ int64_t stream_dp_tiles(int64_t T, int64_t G) {
  return T / G >= 2 ? (T / G - 1) * G : 0;
}

template <bool PR = false>
__device__ __forceinline__ WorkIter work_begin(const KParams& p) {
  WorkIter it;
  const int T = p.tiles_rows * p.tiles_cols;
  const int c = work_slot<PR>(), G = work_slots<PR>();
  if (p.stream_k) {
    it.dp_tiles = static_cast<int>(stream_dp_tiles(T, G));
    it.dp = c;
    const int64_t I = static_cast<int64_t>(T - it.dp_tiles) * p.k_tiles;
    it.pos = static_cast<int>(I * c / G);
    it.end = static_cast<int>(I * (c + 1) / G);
  } else {
    it.dp = it.dp_tiles = 0;
    it.pos = c;
    it.end = T * p.split_k;
  }
  return it;
}

template <bool PR = false>
__device__ __forceinline__ bool work_next(const KParams& p, int bn, WorkIter& it, Unit& w) {
  if (p.stream_k && it.dp < it.dp_tiles) {
    // a whole tile, data-parallel
    unit_tile<PR>(p, it.dp, bn, w);
    it.dp += work_slots<PR>();
    w.j = 0;
    w.contrib = 1;
    w.kt0 = 0;
    w.nk = p.k_tiles;
    return true;
  }
  if (it.pos >= it.end) return false;
  if (!p.stream_k) {
    const int u = it.pos;
    it.pos += work_slots<PR>();
    w.j = u % p.split_k;
    w.contrib = p.split_k;
    unit_tile<PR>(p, u / p.split_k, bn, w);
    w.kt0 = static_cast<int>(static_cast<int64_t>(w.j) * p.k_tiles / p.split_k);
    w.nk = static_cast<int>(static_cast<int64_t>(w.j + 1) * p.k_tiles / p.split_k) - w.kt0;
    return true;
  }
  const int KT = p.k_tiles;
  const int T = p.tiles_rows * p.tiles_cols;
  const int64_t I = static_cast<int64_t>(T - it.dp_tiles) * KT;
  const int64_t G = work_slots<PR>();
  const int rt = it.pos / KT;  // tile within the split part
  const int tile_begin = rt * KT, tile_end = tile_begin + KT;
  const int seg_end = it.end < tile_end ? it.end : tile_end;
  unit_tile<PR>(p, it.dp_tiles + rt, bn, w);
  w.kt0 = it.pos - tile_begin;
  w.nk = seg_end - it.pos;
  // owner of iteration i: the CTA c with floor(c I/G) <= i < floor((c+1) I/G)
  const int first = static_cast<int>(((tile_begin + 1) * G - 1) / I);
  const int last = static_cast<int>((static_cast<int64_t>(tile_end) * G - 1) / I);
  w.contrib = last - first + 1;
  w.j = work_slot<PR>() - first;
  it.pos = seg_end;
  return true;
}

// Split-K arrival: after this CTA's partial is in the workspace, count it;
// true for the last of the tile's splits to arrive (which then reduces).
// The CTA barrier orders every epilogue thread's partial stores before one
// thread's release-acquire increment at GPU scope; the last CTA's acquire,
// followed by the barrier, orders its reads of the other partials after
// them (the semaphore pattern of split-K GEMMs).
__device__ __forceinline__ void red_add_s32(int* addr, int v) {
  asm volatile("red.relaxed.gpu.global.add.s32 [%0], %1;" ::"l"(addr), "r"(v) : "memory");
}

__device__ __forceinline__ int atom_add_acq_rel_gpu(int* addr, int v) {
  int old;
  asm volatile("atom.add.acq_rel.gpu.global.s32 %0, [%1], %2;"
               : "=r"(old)
               : "l"(addr), "r"(v)
               : "memory");
  return old;
}

__device__ __forceinline__ bool split_arrive_last(const KParams& p, int tile, int contrib, int ept,
                                                  int nthreads, int* last_flag) {
  epi_bar_sync(nthreads);
  if (ept == 0) {
    const int prev = atom_add_acq_rel_gpu(p.counters + tile, 1);
    const int last = (prev == contrib - 1);
    if (last) p.counters[tile] = 0;  // ready for the next call (stream-ordered)
    *last_flag = last;
  }
  epi_bar_sync(nthreads);
  const bool last = *last_flag != 0;
  epi_bar_sync(nthreads);  // the flag is rewritten by the next unit
  return last;
}

// The last CTA of a tile sums the tile's partials (its own one included, read
// back from the workspace) for NV consecutive columns starting at col_first,
// in contributor order 0..contrib-1, so the result is the same whichever CTA
// arrives last.  G contributors' loads are issued per round, so the latency
// is paid once per G contributors, not once per contributor.
template <int IN, int BN, int NV, int GMAX = 8>
__device__ __forceinline__ void reduce_partials(const KParams& p, int tile, int contrib,
                                                int col_first, int lane_row, bool row_valid,
                                                int cols_left, uint32_t (&acc)[NV]) {
  constexpr int G0 = (32 / NV) < 1 ? 1 : ((32 / NV) > 8 ? 8 : (32 / NV));
  constexpr int G = G0 > GMAX ? GMAX : G0;
  for (int s0 = 0; s0 < contrib; s0 += G) {
    uint32_t v[G][NV];
#pragma unroll
    for (int u = 0; u < G; ++u) {
      const bool su = s0 + u < contrib;
      const uint32_t* wsb = ws_slot<BN>(p, su ? s0 + u : 0, tile, col_first, lane_row);
#pragma unroll
      for (int c = 0; c < NV; ++c)
        v[u][c] = (su && row_valid && c < cols_left) ? __ldcg(wsb + c * 128) : 0u;
    }
#pragma unroll
    for (int u = 0; u < G; ++u) {
      if (s0 + u < contrib) {
#pragma unroll
        for (int c = 0; c < NV; ++c) {
          if (s0 + u == 0)
            acc[c] = v[u][c];
          else if (IN == IN_INT8)
            acc[c] = static_cast<uint32_t>(static_cast<int32_t>(acc[c]) + static_cast<int32_t>(v[u][c]));
          else
            acc[c] = __float_as_uint(__fadd_rn(__uint_as_float(acc[c]), __uint_as_float(v[u][c])));
        }
      }
    }
  }
}

// Row stride (floats) of a unit's staged block scales: nk rounded up to a
// multiple of 4, plus 4 (16-byte aligned rows for vector copies).
__host__ __device__ constexpr int scale_row_stride(int nk) { return (nk + 3) / 4 * 4 + 4; }

// Block scales of one unit into a shared-memory buffer, with asynchronous
// copies (the caller commits and waits): sc_a[t][i] = s_a of tile row t at
// K block kt0 + i, row stride scale_row_stride(nk), zero beyond M; with
// swap-AB (t a tile column, i.e. a token) K-block-major instead,
// sc_a[i][t] (row length BN), so that a thread reads a K block's token
// scales as 16-byte vectors; then sc_w[i] of the tile's weight block row.
// 16-byte copies when the rows' pieces are 16-byte aligned.
template <bool SWAP, int BN, int NT>
__device__ __forceinline__ void stage_block_scales(const KParams& p, const Unit& w, float* buf,
                                                   int ept) {
  const int T = SWAP ? BN : 128;
  const int base = SWAP ? w.col0 : w.row0;
  const int ss = scale_row_stride(w.nk);
  float* sc_a = buf;
  float* sc_w = buf + T * ss;
  if constexpr (SWAP) {
    for (int idx = ept; idx < T * w.nk; idx += NT) {
      const int i = idx / T, t = idx - i * T;
      const int m = base + t;
      const bool ok = m < p.M;
      const float* src = p.s_a + (ok ? static_cast<int64_t>(m) * p.kb_count + w.kt0 + i : 0);
      cp_async_4(sc_a + i * T + t, src, ok ? 4u : 0u);
    }
  } else if ((p.kb_count & 3) == 0 && (w.kt0 & 3) == 0 && (w.nk & 3) == 0) {
    const int q = w.nk >> 2;
    for (int idx = ept; idx < T * q; idx += NT) {
      const int t = idx / q, c = idx - t * q;
      const int m = base + t;
      const bool ok = m < p.M;
      const float* src = p.s_a + (ok ? static_cast<int64_t>(m) * p.kb_count + w.kt0 + 4 * c : 0);
      cp_async_16(sc_a + t * ss + 4 * c, src, ok ? 16u : 0u);
    }
  } else {
    for (int idx = ept; idx < T * w.nk; idx += NT) {
      const int t = idx / w.nk, i = idx - t * w.nk;
      const int m = base + t;
      const bool ok = m < p.M;
      const float* src = p.s_a + (ok ? static_cast<int64_t>(m) * p.kb_count + w.kt0 + i : 0);
      cp_async_4(sc_a + t * ss + i, src, ok ? 4u : 0u);
    }
  }
  // the tile's weight block rows: one, or (rows over M, tiles wider than
  // 128) one per 128 columns, row h at sc_w + h ss; rows past N read zero
  constexpr int WR = (!SWAP && BN > 128) ? BN / 128 : 1;
  const int wrow = SWAP ? w.tile_r : (w.col0 / 128);
  const int wrows = (p.N + 127) / 128;
  for (int idx = ept; idx < WR * w.nk; idx += NT) {
    const int h = idx / w.nk, i = idx - h * w.nk;
    const bool ok = SWAP || wrow + h < wrows;
    const float* src = p.s_w + (ok ? static_cast<int64_t>(wrow + h) * p.kb_count + w.kt0 + i : 0);
    cp_async_4(sc_w + h * ss + i, src, ok ? 4u : 0u);
  }
}

// ------------------------------------------- split-K inside a cluster ----
//
// The S = split_k CTAs of a tile form one thread-block cluster (cluster rank
// = split index j).  Rank o owns the tile's rows [o R, (o+1) R), R = 128 / S.
// The exchange buffer of a CTA, [j][row - o R][BN + 4] fp32 words (rows
// padded so that 16-byte reads of consecutive rows hit distinct banks), lies
// over its operand ring, which is idle once the CTA's last UMMA completed.
// All traffic is asynchronous remote stores that complete transaction bytes
// on the receiving CTA's mbarrier, so no fences are needed:
//   1. once its accumulator is final, CTA o writes one word into every CTA
//      of the cluster (red_ready of each expects 4 S bytes): "my buffer is
//      free";
//   2. when red_ready completes, each epilogue thread sends the BN partial
//      sums of its row to the row's owner (red_full of the owner expects
//      S x its valid rows x BN x 4 bytes);
//   3. the owner sums the S partials of each of its elements in split order
//      j = 0..S-1 (the workspace path's order, so the results are the same)
//      and runs the epilogue.

__host__ __device__ constexpr int red_row_words(int bn) { return bn + 4; }

// Bytes CTA `rank` of the cluster of unit w receives in step 2.
__device__ __forceinline__ uint32_t cluster_bytes_expected(const KParams& p, int row0, int rank,
                                                           int bn) {
  const int R = 128 / p.split_k;
  int rows = p.rows - (row0 + rank * R);
  rows = rows < 0 ? 0 : (rows > R ? R : rows);
  return static_cast<uint32_t>(p.split_k * rows * bn * 4);
}

// Step 1: thread o < S of the epilogue writes CTA o's flag word.
__device__ __forceinline__ void cluster_signal_ready(const KParams& p, uint64_t* red_ready,
                                                     uint32_t* flags, int ept) {
  if (ept < p.split_k) {
    const uint32_t o = static_cast<uint32_t>(ept);
    const uint32_t me = cluster_ctarank();
    st_async_u32(cluster_map(smem_u32(flags + me), o), me, cluster_map(smem_u32(red_ready), o));
  }
}

// Step 2 for NV consecutive columns starting at col_first of this thread's
// row (NV a multiple of 4).
template <int BN, int NV>
__device__ __forceinline__ void cluster_send(const KParams& p, uint32_t red_base, uint64_t* red_full,
                                             const Unit& w, int lane_row, int col_first,
                                             const uint32_t* vals) {
  static_assert(NV % 4 == 0, "16-byte pieces");
  const int R = 128 / p.split_k;
  if (w.row0 + lane_row >= p.rows) return;
  const uint32_t owner = static_cast<uint32_t>(lane_row / R);
  const int lr = lane_row - static_cast<int>(owner) * R;
  const uint32_t dst = cluster_map(red_base, owner) +
                       static_cast<uint32_t>(((w.j * R + lr) * red_row_words(BN) + col_first) * 4);
  const uint32_t bar = cluster_map(smem_u32(red_full), owner);
#pragma unroll
  for (int c = 0; c < NV; c += 4)
    st_async_v4(dst + static_cast<uint32_t>(c * 4), vals[c], vals[c + 1], vals[c + 2], vals[c + 3], bar);
}

// Epilogue inputs that depend only on an owner thread's row (it keeps one
// row): bias and weight scale (rows over N) or token scale (rows over M).
// Loaded before the thread waits for the partial sums.
struct RowIn {
  float b, s;
};

template <int SC, bool SWAP>
__device__ __forceinline__ RowIn cluster_row_inputs(const KParams& p, int row) {
  RowIn in{0.0f, 1.0f};
  if (row >= p.rows || (p.flags & F_DEBUG)) return in;
  if (SWAP) {
    if (p.flags & F_BIAS) in.b = __bfloat162float(p.bias[row]);
    if (SC == SC_TC) in.s = __ldg(p.s_w + row);
  } else {
    if (SC == SC_TC) in.s = __ldg(p.s_a + row);
  }
  return in;
}

// Step 3.  Thread e keeps row e % R of the owned slice and handles the
// 4-column groups e / R, + T / R, ... (T = epilogue threads, a multiple of
// R): the group's global loads and S 16-byte partial reads first, then its
// arithmetic and stores.  False on timeout.
template <int IN, int SC, bool SWAP, int BN, int T, int ACT, int OF = -1>
__device__ __forceinline__ bool cluster_reduce_store(const KParams& p, const uint32_t* red,
                                                     uint64_t* red_full, const Unit& w, int ept,
                                                     const RowIn& in) {
  const int S = p.split_k;
  const int R = 128 / S;
  if (!mbar_wait_cluster(red_full, 0, p.wait_limit_ns)) return false;
  if (ept == 0) trace_point(p, TR_ARRIVED);
  const int rr = ept % R;
  const int row = w.row0 + static_cast<int>(cluster_ctarank()) * R + rr;
  if (row >= p.rows) return true;
  const int cv = min(BN, p.cols - w.col0);
  const int step = 4 * (T / R);
  const bool debug = (p.flags & F_DEBUG) != 0;
  const bool has_res = (p.flags & (F_RES | F_RES_PRE)) != 0;
  const bool has_bias = (p.flags & F_BIAS) != 0;
  const float sy = out_scale(p);
  constexpr int W = red_row_words(BN);
  for (int c0 = 4 * (ept / R); c0 < cv; c0 += step) {
    float rv[4], cs[4], cb[4];
#pragma unroll
    for (int g = 0; g < 4; ++g) {
      const bool ok = c0 + g < cv && !debug;
      const int col = w.col0 + c0 + g;
      const int m = SWAP ? col : row, n = SWAP ? row : col;
      rv[g] = (ok && has_res) ? __bfloat162float(p.R[static_cast<int64_t>(m) * p.ldr + n]) : 0.0f;
      cs[g] = (ok && SC == SC_TC) ? __ldg(SWAP ? p.s_a + col : p.s_w + col) : 1.0f;
      cb[g] = (ok && !SWAP && has_bias) ? __bfloat162float(p.bias[col]) : 0.0f;
    }
    uint4 v = *reinterpret_cast<const uint4*>(red + rr * W + c0);
    for (int j = 1; j < S; ++j) {
      const uint4 x = *reinterpret_cast<const uint4*>(red + (j * R + rr) * W + c0);
      if (IN == IN_INT8) {
        v.x = static_cast<uint32_t>(static_cast<int32_t>(v.x) + static_cast<int32_t>(x.x));
        v.y = static_cast<uint32_t>(static_cast<int32_t>(v.y) + static_cast<int32_t>(x.y));
        v.z = static_cast<uint32_t>(static_cast<int32_t>(v.z) + static_cast<int32_t>(x.z));
        v.w = static_cast<uint32_t>(static_cast<int32_t>(v.w) + static_cast<int32_t>(x.w));
      } else {
        v.x = __float_as_uint(__fadd_rn(__uint_as_float(v.x), __uint_as_float(x.x)));
        v.y = __float_as_uint(__fadd_rn(__uint_as_float(v.y), __uint_as_float(x.y)));
        v.z = __float_as_uint(__fadd_rn(__uint_as_float(v.z), __uint_as_float(x.z)));
        v.w = __float_as_uint(__fadd_rn(__uint_as_float(v.w), __uint_as_float(x.w)));
      }
    }
    const uint32_t acc[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int g = 0; g < 4; ++g) {
      if (c0 + g >= cv) break;
      const int col = w.col0 + c0 + g;
      const int m = SWAP ? col : row, n = SWAP ? row : col;
      const int64_t at = static_cast<int64_t>(m) * p.ldy + n;
      if (debug) {
        reinterpret_cast<uint32_t*>(p.Y)[at] = acc[g];
        continue;
      }
      // the scale is s_a[m] * s_w[n] in that order, as in the other paths
      const float sa = SWAP ? cs[g] : in.s, sw = SWAP ? in.s : cs[g];
      const float bias = SWAP ? in.b : cb[g];
      uint16_t o;
      if (IN == IN_INT8) {
        o = epi_int8<ACT>(static_cast<int32_t>(acc[g]), sa, sw, bias, rv[g], p.flags, p.out, sy);
      } else {
        const float y = epi_value<ACT>(__uint_as_float(acc[g]), (SC == SC_TC) ? sa * sw : 1.0f,
                                       bias, rv[g], p.flags);
        o = (OF == OUT_BF16) ? __bfloat16_as_ushort(__float2bfloat16_rn(y)) : out_bits(y, p.out, sy);
      }
      if (OF == OUT_BF16)
        reinterpret_cast<uint16_t*>(p.Y)[at] = o;
      else
        store_out(p, at, o);
    }
  }
  return true;
}

// ---------------------------------------------------------------- kernel ---
//
// Persistent: CTA b handles work units b, b + gridDim.x, ...  Ring stages,
// TMEM accumulator buffers and promotion buffers carry their phases across
// units, so the epilogue of one unit overlaps the UMMA mainloop of the next.

// Position in the ring of S stages whose stages are released in groups of CG
// (NG = S / CG group slots): stage and the parity of its current use, index
// within the group, group slot and the parity of its current use.  Kept as
// counters: the producer and the UMMA issuer are single threads whose
// per-stage instruction latency sits on the tensor pipe's critical path,
// and a division by a runtime ring depth costs it a few hundred cycles.
struct RingPos {
  int s;
  uint32_t ph;
  int gi, gs;
  uint32_t gph;
};

__device__ __forceinline__ void ring_next(RingPos& r, int S, int CG, int NG) {
  if (++r.s == S) {
    r.s = 0;
    r.ph ^= 1u;
  }
  if (++r.gi == CG) {
    r.gi = 0;
    if (++r.gs == NG) {
      r.gs = 0;
      r.gph ^= 1u;
    }
  }
}

template <int IN, int SC, bool SWAP, int BN, bool G = false, bool PR = false>
__global__ void __launch_bounds__(Cfg<IN, SC, SWAP, BN, G, PR>::kThreads)
    __maxnreg__((Cfg<IN, SC, SWAP, BN, G, PR>::kMaxRegs))
    fused_linear_kernel(const __grid_constant__ CUtensorMap tmP,
                        const __grid_constant__ CUtensorMap tmQ,
                        const __grid_constant__ CUtensorMap tmY, const KParams p) {
  using C = Cfg<IN, SC, SWAP, BN, G, PR>;
  constexpr int CW = C::kCW;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const int S = p.stages;
  const int CG = p.commit_group > 0 ? p.commit_group : 1;  // divides S (host)
  const int NG = S / CG;
  // Shared memory: [TMA ring: S stages of (P | Q), or (P8 | Q8) for INT8]
  // [INT8: 2 fp16 operand slots of (P | Q)] [barriers, 512 B] [block scales].
  // Every tile part is a multiple of 1 KB, so 1024-byte alignment holds.
  auto stage_base = [&](int s) { return smem + static_cast<uint32_t>(s) * C::kStageBytes; };
  uint8_t* op_area = smem + static_cast<uint32_t>(S) * C::kStageBytes;
  // UMMA operands of ring iteration g: the ring stage itself, or (INT8) the
  // fp16 slot the transform warps wrote
  auto op_base = [&](uint32_t g, int s) {
    return C::kConvert ? op_area + (g % C::kOpSlots) * C::kQBytes : stage_base(s);
  };
  uint64_t* bars = reinterpret_cast<uint64_t*>(op_area + C::kOpBytes);
  uint64_t* full = bars;              // [S] TMA landed (expect_tx)
  uint64_t* empty = bars + S;         // [S] ring stage free (UMMA commit, or converter)
  uint64_t* bfull = bars + 2 * S;     // [kOpSlots] fp16 operands ready (INT8)
  uint64_t* bempty = bfull + C::kOpSlots;  // [kOpSlots] fp16 operands consumed (INT8)
  constexpr int NB = C::kAccBufs;
  uint64_t* tfull = bempty + C::kOpSlots;  // [NB] TMEM buffer holds a finished K block / tile
  uint64_t* tempty = tfull + NB;      // [NB] TMEM buffer drained by the epilogue
  uint64_t* mma_done = tempty + NB;
  uint64_t* red_full = mma_done + 1;  // cluster split-K: this CTA's rows have all partials
  uint64_t* red_ready = red_full + 1; // cluster split-K: every CTA's exchange buffer is free
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(red_ready + 1);
  int* last_flag = reinterpret_cast<int*>(tmem_slot + 1);
  uint32_t* red_flags = reinterpret_cast<uint32_t*>(last_flag + 1);  // [split_k] words
  // block scales of the current unit (block scaling only; sized by the host)
  float* scale_smem = reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(bars) + 512u);
  // cluster split-K exchange buffer [split][128 / split][BN + 4]: over the
  // operand ring, once the ring is idle (the host checks that it fits)
  uint32_t* red_buf = reinterpret_cast<uint32_t*>(smem);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint64_t lim = p.wait_limit_ns;
  const bool has_work = p.k_tiles > 0;
  // CTA pair: the even CTA issues the UMMAs; stage barriers and the
  // accumulator-free barriers that count are the even CTA's
  const bool pair_leader = !PR || (blockIdx.x & 1u) == 0;

  if (threadIdx.x == 0) trace_point(p, TR_START);
  if (warp == 0 && lane == 0 && has_work) {
    tma_prefetch_desc(&tmP);
    tma_prefetch_desc(&tmQ);
  }
  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], C::kConvert ? 128 : 1);
    }
    for (int o = 0; o < C::kOpSlots; ++o) {
      mbar_init(&bfull[o], 128);
      mbar_init(&bempty[o], 1);
    }
    for (int b = 0; b < NB; ++b) {
      mbar_init(&tfull[b], 1);
      // per epilogue thread; CTA pairs: one arrival per CTA of the pair per
      // unit, or (promotion, per K block) one per epilogue warp of both CTAs
      mbar_init(&tempty[b], PR ? (C::kPromote ? 2 * C::kEpiWarps : 2) : C::kEpiThreads);
    }
    mbar_init(mma_done, 1);
    mbar_init(red_full, 1);
    mbar_init(red_ready, 1);
    fence_mbar_init();
    if (p.cluster_reduce) {
      // one unit per CTA: what this CTA will receive is known now, before
      // any CTA of the cluster can send (they all pass the cluster barrier
      // below first)
      mbar_arrive_expect_tx(red_ready, 4u * static_cast<uint32_t>(p.split_k));
      const int tile = static_cast<int>(blockIdx.x) / p.split_k;
      mbar_arrive_expect_tx(red_full, cluster_bytes_expected(p, (tile % p.tiles_rows) * 128,
                                                             static_cast<int>(cluster_ctarank()), BN));
    }
  }
  if (warp == 1) {
    if constexpr (PR) {
      tmem_alloc_pair(tmem_slot, C::kTmemCols);
      tmem_relinquish_pair();
    } else {
      tmem_alloc(tmem_slot, C::kTmemCols);
      tmem_relinquish();
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  // cluster split-K and CTA pairs: every CTA's barriers are initialised
  // before any remote arrival
  if (PR || p.cluster_reduce) cluster_sync_all();
  const uint32_t tmem_base = *tmem_slot;
  if (p.pdl && threadIdx.x == 0) griddep_launch_dependents();
  if (threadIdx.x == 0) trace_point(p, TR_SETUP);

  // Roles: producer (warp 0), UMMA issuer (warp 1), INT8 converters (the
  // last four warps), epilogue (the rest from kEpiWarp0 on).  Wide
  // promotion tiles: warpgroup 0 (producer, issuer and two idle warps) hands
  // registers to the two epilogue warpgroups with setmaxnreg, each
  // warpgroup executing one and the same instruction at the top of its
  // branch (the host checked that the split fits the launch allocation).
  const bool epi_warp =
      warp >= C::kEpiWarp0 && !(C::kConvert && warp >= C::kEpiWarp0 + C::kEpiWarps);
  if (!epi_warp) {
  if constexpr (C::kWidePromote) setmaxnreg_dec<C::kRegsLow>();
  if (warp == 0) {
    // ------------------------------------------------ TMA producer ----
    const bool stalled = p.stall_producer == 1 || (p.stall_producer == 2 && (blockIdx.x & 1u));
    if (lane == 0 && !stalled && has_work) {
      const uint64_t pol_first = policy_evict_first();
      // The weight operand (P with swap-AB, else Q) is constant across calls;
      // the activation operand may be written by the previous kernel.
      // PR: loads complete on the even CTA's stage barrier; this CTA's half
      // of the weight tile starts BN/2 rows further for the odd CTA
      const uint32_t full_pair0 = PR ? cluster_map(smem_u32(&full[0]), 0) : 0u;
      const int q_off = PR ? static_cast<int>(blockIdx.x & 1u) * (BN / 2) : 0;
      auto load_op = [&](bool weight, const Unit& w, int i, int s) {
        uint8_t* base = stage_base(s);
        const bool isP = (weight == SWAP);
        uint8_t* dst = base + (isP ? 0u : (C::kConvert ? C::kP8Bytes : C::kPBytes));
        const int kx = (w.kt0 + i) * C::kElemsPerStage;
        const CUtensorMap* map = isP ? &tmP : &tmQ;
        const int y = isP ? w.row0 : w.col0 + q_off;
        if constexpr (PR) {
          const uint32_t cbar = full_pair0 + static_cast<uint32_t>(s) * 8u;
          if (isP ? p.evict_first_p : p.evict_first_q)
            tma_load_2d_pair_hint(dst, map, cbar, kx, y, pol_first);
          else
            tma_load_2d_pair(dst, map, cbar, kx, y);
          return;
        }
        if (isP ? p.evict_first_p : p.evict_first_q)
          tma_load_2d_hint(dst, map, &full[s], kx, y, pol_first);
        else
          tma_load_2d(dst, map, &full[s], kx, y);
        if constexpr (G) {
          // gated: the up half's tile, N weight rows further, after P and Q
          if (weight) {
            uint8_t* dst2 = base + C::kPBytes + C::kQBytes;
            if (isP ? p.evict_first_p : p.evict_first_q)
              tma_load_2d_hint(dst2, map, &full[s], kx, y + p.N, pol_first);
            else
              tma_load_2d(dst2, map, &full[s], kx, y + p.N);
          }
        }
      };
      RingPos rp = {0, 0u, 0, 0, 0u};  // ring position across units
      uint32_t gp = 0;                 // ring iteration (= K block when promoting)
      // block scales: a stage is free once the accumulator commit of the K
      // block that used it (S iterations back) has arrived
      const bool stage_by_acc = C::kPromote && !C::kConvert && p.acc_release;
      bool first = true;
      bool ok = true;
      WorkIter it = work_begin<PR>(p);
      Unit w;
      while (ok && work_next<PR>(p, BN, it, w)) {
        int i0 = 0;
        if (first) {
          first = false;
          // As a programmatic dependent: stream the first ring of weight
          // tiles, and send the rest of this unit's weight range to L2, while
          // the previous kernel finishes; then wait for its results.
          const int pre = p.pdl ? (w.nk < S ? w.nk : S) : 0;
          for (int i = 0; i < pre; ++i) {
            if (pair_leader) mbar_arrive_expect_tx(&full[i], C::kTxBytes);
            load_op(true, w, i, i);
          }
          if (p.pdl && p.l2_prefetch) {
            const CUtensorMap* wmap = SWAP ? &tmP : &tmQ;
            const int wy = SWAP ? w.row0 : w.col0 + q_off;
            for (int i = pre; i < w.nk; ++i) {
              tma_prefetch_l2_2d(wmap, (w.kt0 + i) * C::kElemsPerStage, wy);
              if constexpr (G) tma_prefetch_l2_2d(wmap, (w.kt0 + i) * C::kElemsPerStage, wy + p.N);
            }
            // weights read once per call (decode, rows over N): this CTA's
            // later units too, so the whole of its weight range streams
            // into L2 while the previous kernel finishes
            if (SWAP && p.evict_first_p) {
              WorkIter it2 = it;
              Unit w2;
              while (work_next<PR>(p, BN, it2, w2))
                for (int i = 0; i < w2.nk; ++i) {
                  tma_prefetch_l2_2d(wmap, (w2.kt0 + i) * C::kElemsPerStage, w2.row0);
                  if constexpr (G) tma_prefetch_l2_2d(wmap, (w2.kt0 + i) * C::kElemsPerStage, w2.row0 + p.N);
                }
            }
          }
          trace_point(p, TR_PRE_ISSUED);
          griddep_wait();
          for (int i = 0; i < pre; ++i) load_op(false, w, i, i);
          trace_point(p, TR_FIRST_TMA);
          i0 = pre;
          for (int i = 0; i < pre; ++i) ring_next(rp, S, CG, NG);
          gp = static_cast<uint32_t>(pre);
        }
        for (int i = i0; i < w.nk; ++i) {
          const int s = rp.s;
          // stages are released in groups of CG by one commit on the
          // group's barrier: wait for the previous use of this group slot
          bool free_ok;
          if (stage_by_acc) {
            const uint32_t j = gp - static_cast<uint32_t>(S);  // used only when gp >= S
            free_ok = gp < static_cast<uint32_t>(S) || mbar_wait(&tfull[j % NB], (j / NB) & 1u, lim);
          } else {
            free_ok = mbar_wait(&empty[rp.gs], rp.gph ^ 1u, lim);
          }
          if (!free_ok) {
            record_status(p.status, ST_TIMEOUT_PRODUCER);
            ok = false;
            break;
          }
          if (pair_leader) mbar_arrive_expect_tx(&full[s], C::kTxBytes);
          load_op(true, w, i, s);
          load_op(false, w, i, s);
          ring_next(rp, S, CG, NG);
          ++gp;
        }
      }
      trace_point(p, TR_LAST_LOAD);
      // Wind-down: wait (bounded) until every stage this thread armed has
      // received all of its bytes, so that no bulk copy is still landing in
      // shared memory when the CTA leaves after some role gave up on a wait.
      // Stage s was armed n_s times; its last armed phase is n_s - 1, and a
      // phase is only armed once the one before it has completed, so its
      // parity identifies it.  On the normal path the UMMA issuer (or the
      // INT8 converters) already consumed every phase and these return at
      // once.  CTA pairs: the even CTA's stage barriers count both CTAs'
      // bytes, and the odd CTA leaves only after the cluster barrier of the
      // teardown, which the even CTA reaches after this wait.
      if (pair_leader) {
        const uint32_t su = static_cast<uint32_t>(S);
        for (int s = 0; s < S; ++s) {
          const uint32_t n = gp / su + (static_cast<uint32_t>(s) < gp % su ? 1u : 0u);
          if (n > 0 && !mbar_wait(&full[s], (n - 1u) & 1u, lim)) {
            record_status(p.status, ST_TIMEOUT_PRODUCER);
            break;
          }
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------- UMMA issuer ----
    // (PR: the even CTA's thread issues for the pair)
    if (lane == 0 && has_work && pair_leader) {
      uint32_t g = 0;     // ring iteration (INT8 operand slots: g mod 2)
      RingPos rm = {0, 0u, 0, 0, 0u};  // ring position of iteration g
      uint32_t blk = 0;   // TMEM buffer use (per K block when promoting, else per unit)
      bool ok = true;
      WorkIter it = work_begin<PR>(p);
      Unit w;
      while (ok && work_next<PR>(p, BN, it, w)) {
        if (!C::kPromote) {
          // one TMEM buffer per unit; wait until the epilogue drained it
          // (PR: both CTAs' epilogues, the odd one's arrival remote)
          const int b = blk % NB;
          const uint32_t tph = ((blk / NB) & 1u) ^ 1u;
          if (!(PR ? mbar_wait_cluster(&tempty[b], tph, lim) : mbar_wait(&tempty[b], tph, lim))) {
            record_status(p.status, ST_TIMEOUT_MMA);
            ok = false;
            break;
          }
          // the epilogue's tensor-memory reads of buffer b are ordered
          // before this unit's UMMAs overwrite it
          tc_fence_after();
        }
        for (int i = 0; i < w.nk; ++i, ++g, ring_next(rm, S, CG, NG)) {
          const int s = rm.s;
          const uint32_t ph = rm.ph;
          const int b = blk % NB;
          if (C::kPromote) {
            const uint32_t tph = ((blk / NB) & 1u) ^ 1u;
            if (!(PR ? mbar_wait_cluster(&tempty[b], tph, lim) : mbar_wait(&tempty[b], tph, lim))) {
              record_status(p.status, ST_TIMEOUT_MMA);
              ok = false;
              break;
            }
            tc_fence_after();  // as above, per K block
          }
          // INT8: fp16 operand slot g%2 (its own phase); else the ring stage
          const int os = static_cast<int>(g % C::kOpSlots);
          const uint32_t oph = (g / C::kOpSlots) & 1u;
          if (!mbar_wait(C::kConvert ? &bfull[os] : &full[s], C::kConvert ? oph : ph, lim)) {
            record_status(p.status, ST_TIMEOUT_MMA);
            ok = false;
            break;
          }
          // INT8: the converting threads wrote the A operand into tensor
          // memory (tcgen05.st) before their arrival, so their tcgen05 ops
          // are ordered before these UMMAs.  TMA-loaded stages need no
          // tcgen05 fence: the stage barrier's transaction count makes the
          // bulk copies visible to the UMMAs.
          if constexpr (C::kConvert) tc_fence_after();
          if (g == 0) trace_point(p, TR_FIRST_OPERANDS);
          const uint32_t d = tmem_base + static_cast<uint32_t>(b * C::kAccStride);
          const uint32_t pa = smem_u32(op_base(g, s));
          const uint32_t qa = C::kConvert ? pa : pa + C::kPBytes;
          // INT8: P is in tensor memory, buffer os, 8 columns per K step of 16
          const uint32_t pt = tmem_base + C::kAccCols + static_cast<uint32_t>(os) * 64u;
#pragma unroll
          for (int a = 0; a < C::kAtoms; ++a) {
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              const uint64_t bd = sdesc_k_sw128(qa + static_cast<uint32_t>(a) * BN * 128u + 32u * k);
              const uint32_t accum = C::kPromote ? ((a | k) != 0) : ((i | a | k) != 0);
              if constexpr (C::kConvert) {
                umma_f16_ts(d, pt + static_cast<uint32_t>(a * 4 + k) * 8u, bd, C::kIdesc, accum);
              } else {
                const uint64_t ad = sdesc_k_sw128(pa + static_cast<uint32_t>(a) * 128u * 128u + 32u * k);
                if constexpr (PR) {
                  if (IN == IN_E4M3)
                    umma_f8_pair(d, ad, bd, C::kIdesc, accum);
                  else
                    umma_f16_pair(d, ad, bd, C::kIdesc, accum);
                } else if (IN == IN_E4M3) {
                  umma_f8(d, ad, bd, C::kIdesc, accum);
                } else {
                  umma_f16(d, ad, bd, C::kIdesc, accum);
                }
                if constexpr (G) {
                  // up half: its weight tile replaces the gate's, same
                  // activation tile, accumulator columns [BN, 2 BN)
                  const uint32_t wa = pa + C::kPBytes + C::kQBytes;
                  const uint64_t ad2 = SWAP ? sdesc_k_sw128(wa + 32u * k) : ad;
                  const uint64_t bd2 = SWAP ? bd : sdesc_k_sw128(wa + 32u * k);
                  if (IN == IN_E4M3)
                    umma_f8(d + BN, ad2, bd2, C::kIdesc, accum);
                  else
                    umma_f16(d + BN, ad2, bd2, C::kIdesc, accum);
                }
              }
            }
          }
          // one commit per group of CG stages: a commit costs the tensor
          // pipe a bubble of a few hundred cycles unless enough UMMAs
          // follow it, so every-stage commits of 4 UMMAs run at ~60% rate
          if (C::kConvert) {
            if (!p.acc_release) umma_commit(&bempty[os]);
          } else if (C::kPromote && p.acc_release) {
            // the stage is freed by the accumulator commit below
          } else if (rm.gi == CG - 1) {
            uint64_t* eb = &empty[rm.gs];  // the last stage of this group is done
            if constexpr (PR)
              umma_commit_pair(eb);  // frees the stages in both CTAs
            else
              umma_commit(eb);
          }
          if (C::kPromote) {
            if constexpr (PR)
              umma_commit_pair(&tfull[b]);  // both CTAs' accumulators of the K block
            else
              umma_commit(&tfull[b]);
            ++blk;
          }
        }
        if (!C::kPromote && ok) {
          if (w.nk > 0) {
            if constexpr (PR)
              umma_commit_pair(&tfull[blk % NB]);
            else
              umma_commit(&tfull[blk % NB]);
          }
          ++blk;
        }
      }
      trace_point(p, TR_LAST_COMMIT);
      if constexpr (PR)
        umma_commit_pair(mma_done);
      else
        umma_commit(mma_done);
    }
  } else if (C::kConvert && warp >= C::kEpiWarp0 + C::kEpiWarps) {
    // ---------------------------------- INT8 -> fp16 prologue transform ----
    if constexpr (C::kConvert) {
      const int ct = threadIdx.x - 192;  // 0..127
      // the row this thread converts into tensor memory: its warp's lane
      // quarter (warp % 4) and its lane
      const int conv_row = (warp & 3) * 32 + lane;
      const uint32_t t_conv = tmem_base + (static_cast<uint32_t>((warp & 3) * 32) << 16) + C::kAccCols;
      uint32_t g = 0;
      RingPos rc = {0, 0u, 0, 0, 0u};
      bool ok = true;
      WorkIter it = work_begin<PR>(p);
      Unit w;
      while (ok && work_next<PR>(p, BN, it, w)) {
        for (int i = 0; i < w.nk; ++i, ++g, ring_next(rc, S, 1, S)) {
          const int s = rc.s;                               // int8 ring stage
          const uint32_t ph = rc.ph;
          const int os = static_cast<int>(g % C::kOpSlots);  // fp16 operand slot
          const uint32_t oph = (g / C::kOpSlots) & 1u;
          // the fp16 slot os was last read by the UMMAs of K block g - 2: its
          // accumulator commit (or the slot's own commit) says they are done
          const bool slot_ok =
              p.acc_release
                  ? (g < static_cast<uint32_t>(C::kOpSlots) ||
                     mbar_wait(&tfull[(g - C::kOpSlots) % NB], ((g - C::kOpSlots) / NB) & 1u, lim))
                  : mbar_wait(&bempty[os], oph ^ 1u, lim);
          if (!mbar_wait(&full[s], ph, lim) || !slot_ok) {
            record_status(p.status, ST_TIMEOUT_CONVERT);
            ok = false;
            break;
          }
          tc_fence_after();  // the UMMAs that read buffer os have completed
          // P row -> tensor memory (buffer os); Q -> fp16 shared slot os
          convert_row_to_tmem(stage_base(s), t_conv + static_cast<uint32_t>(os) * 64u, conv_row);
          static_assert(BN % 16 == 0, "Q tile rows come in groups of 16");
          convert_tile<BN / 16>(stage_base(s) + C::kP8Bytes, op_base(g, s), BN, ct);
          tmem_st_wait();
          tc_fence_before();
          fence_proxy_async_smem();
          mbar_arrive(&empty[s]);
          mbar_arrive(&bfull[os]);
        }
      }
    }
  }
  } else {
    // ----------------------------------------------------- epilogue ----
    if constexpr (C::kWidePromote) setmaxnreg_inc<C::kRegsHigh>();
    const int quarter = warp & 3;
    const int lane_row = quarter * 32 + lane;
    constexpr int CPT = C::kColsPerThread;
    static_assert(CPT % C::kCW == 0, "whole TMEM load chunks per thread");
    static_assert(!G || CPT == BN, "gated units use 4 epilogue warps");
    // this thread's first column in the tile
    const int cbeg = (C::kEpiWarps == 4) ? 0 : ((warp - C::kEpiWarp0) >> 2) * CPT;
    const uint32_t t_lane = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) +
                            static_cast<uint32_t>(cbeg);
    const int ept = threadIdx.x - 32 * C::kEpiWarp0;  // 0 .. kEpiThreads-1
    // staged TMA stores of Y (rows over M): two boxes per epilogue warp
    const bool tstore = !SWAP && !G && p.tma_store != 0;
    uint8_t* boxes = smem + p.out_stage_off +
                     static_cast<uint32_t>(warp - C::kEpiWarp0) * 2u * stage_box_bytes<CW>();
    uint32_t nbox = 0;
    griddep_wait();
    uint32_t blk = 0;
    bool ok = true;
    WorkIter it = work_begin<PR>(p);
    Unit w;
    // Block scales: without swap-AB (large M, many units per CTA) they are
    // staged one unit ahead, into the other of two buffers, so their global
    // latency overlaps the current unit; with swap-AB (decode, about one unit
    // per CTA) each unit stages its own, all copies in flight at once.
    constexpr int kScaleRows = SWAP ? BN : 128;
    constexpr int kWRows = (!SWAP && BN > 128) ? BN / 128 : 1;  // weight block rows per tile
    constexpr bool kAhead = (SC == SC_BLOCK) && !SWAP;
    const int scale_buf_floats = (kScaleRows + kWRows) * scale_row_stride(p.k_tiles);
    WorkIter it_pf = it;
    uint32_t su = 0;
    if constexpr (kAhead) {
      Unit w0;
      if (work_next<PR>(p, BN, it_pf, w0))
        stage_block_scales<SWAP, BN, C::kEpiThreads>(p, w0, scale_smem, ept);
      cp_async_commit();
    }
    while (ok && work_next<PR>(p, BN, it, w)) {
      const int row = w.row0 + lane_row;
      const uint32_t cur = su++;
      if constexpr (C::kPromote) {
        // ---- promotion: per 128-K block, TMEM buffer -> registers ----
        uint32_t acc[CPT];
#pragma unroll
        for (int c = 0; c < CPT; ++c) acc[c] = 0u;  // +0.0f or int 0
        // this unit's block scales (staged one unit ahead; layout in
        // stage_block_scales)
        float* sc_a = scale_smem + (kAhead ? (cur & 1u) * scale_buf_floats : 0);
        const int ss = scale_row_stride(w.nk);
        float* sc_w = sc_a + kScaleRows * ss;
        if constexpr (kAhead) {
          // every thread is done with the other buffer (the previous unit's)
          epi_bar_sync(C::kEpiThreads);
          Unit wn;
          if (work_next<PR>(p, BN, it_pf, wn))
            stage_block_scales<SWAP, BN, C::kEpiThreads>(
                p, wn, scale_smem + ((cur + 1u) & 1u) * scale_buf_floats, ept);
          cp_async_commit();
          cp_async_wait<1>();            // this thread's copies for this unit landed
          epi_bar_sync(C::kEpiThreads);  // ... and every thread's
        } else if constexpr (SC == SC_BLOCK) {
          epi_bar_sync(C::kEpiThreads);  // the previous unit's reads of this buffer are done
          stage_block_scales<SWAP, BN, C::kEpiThreads>(p, w, sc_a, ept);
          cp_async_commit();
          cp_async_wait<0>();
          epi_bar_sync(C::kEpiThreads);
          if constexpr (SWAP) {
            // the tile's weight block row is one scale per K block: fold it
            // in, sc_a[i][t] = s_w[i] * s_a[t][i] (the product the promotion
            // applies), so a K block's promotion reads one vector per 4 tokens
            for (int idx = ept; idx < BN * w.nk; idx += C::kEpiThreads)
              sc_a[idx] = sc_w[idx / BN] * sc_a[idx];
            epi_bar_sync(C::kEpiThreads);
          }
        }
        if constexpr (C::kWidePromote) {
          // 128 running sums per thread: one row (m) and the 128 columns of
          // one weight block (n / 128), so one s_a and one s_w per K block
          // (staged in shared memory one unit ahead).  Per K block the
          // buffer is read in four 32-column pieces, each piece's load in
          // flight while the previous piece is added (two pieces in
          // registers at a time).
          const float* sa_row = sc_a + lane_row * ss;
          const float* sw_row = sc_w + (cbeg >> 7) * ss;
          for (int i = 0; i < w.nk; ++i, ++blk) {
            const int b = blk % NB;
            const uint32_t bph = (blk / NB) & 1u;
            const float srow = sa_row[i] * sw_row[i];
            if (!mbar_wait(&tfull[b], bph, lim)) {
              record_status(p.status, ST_TIMEOUT_EPILOGUE);
              ok = false;
              break;
            }
            tc_fence_after();
            if (blk == 0 && ept == 0) trace_point(p, TR_FIRST_ACC);
            const uint32_t tb = t_lane + static_cast<uint32_t>(b * BN);
            // two halves of 64 columns: each half's four loads in flight
            // together, one wait, then its 64 FMAs (two waits per K block)
            uint32_t rh[64];
#pragma unroll
            for (int h = 0; h < CPT / 64; ++h) {
              tmem_ld32p(tb + static_cast<uint32_t>(64 * h), rh);
              tmem_ld32p(tb + static_cast<uint32_t>(64 * h + 32), rh + 32);
              tmem_ld_wait();
              reg_fence<64>(rh);
              if (h + 1 == CPT / 64) {
                // the buffer is free once all of it is in registers (CTA
                // pairs: each warp's arrival on the even CTA's barrier)
                tc_fence_before();
                if constexpr (PR) {
                  __syncwarp();
                  if (lane == 0) mbar_arrive_cluster(cluster_map(smem_u32(&tempty[b]), 0));
                } else {
                  mbar_arrive(&tempty[b]);
                }
              }
#pragma unroll
              for (int j = 0; j < 64; ++j)
                acc[64 * h + j] = __float_as_uint(__fmaf_rn(srow, __uint_as_float(rh[j]),
                                                            __uint_as_float(acc[64 * h + j])));
            }
          }
        } else
        for (int i = 0; i < w.nk; ++i, ++blk) {
          const int b = blk % NB;
          const uint32_t bph = (blk / NB) & 1u;
          float srow = 1.0f;  // scale shared by the thread's row (block scaling)
          if constexpr (SC == SC_BLOCK) {
            srow = SWAP ? sc_w[i] : sc_a[lane_row * ss + i] * sc_w[i];
          }
          if (!mbar_wait(&tfull[b], bph, lim)) {
            record_status(p.status, ST_TIMEOUT_EPILOGUE);
            ok = false;
            break;
          }
          tc_fence_after();
          if (blk == 0 && ept == 0) trace_point(p, TR_FIRST_ACC);
          // all of this thread's columns of the block, then one wait
          uint32_t r[CPT];
#pragma unroll
          for (int c = 0; c < CPT; c += CW)
            tmem_load_chunk_p<CW>(t_lane + static_cast<uint32_t>(b * BN + c), r + c);
          tmem_ld_wait();
          tc_fence_before();
          mbar_arrive(&tempty[b]);  // the buffer is free once the values are in registers
          if constexpr (SC == SC_BLOCK && SWAP) {
            // s_w[i] * s_a[token][i] of this thread's tokens (0 beyond M),
            // four per 16-byte read
            const float4* sp = reinterpret_cast<const float4*>(sc_a + i * BN + cbeg);
#pragma unroll
            for (int c4 = 0; c4 < CPT / 4; ++c4) {
              const float4 s = sp[c4];
              const float sv[4] = {s.x, s.y, s.z, s.w};
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                const int c = 4 * c4 + e;
                acc[c] = __float_as_uint(__fmaf_rn(sv[e], __uint_as_float(r[c]), __uint_as_float(acc[c])));
              }
            }
          } else {
#pragma unroll
            for (int c = 0; c < CPT; ++c) {
              if constexpr (SC == SC_BLOCK) {
                acc[c] = __float_as_uint(__fmaf_rn(srow, __uint_as_float(r[c]), __uint_as_float(acc[c])));
              } else {
                acc[c] = static_cast<uint32_t>(static_cast<int32_t>(acc[c]) +
                                               __float2int_rn(__uint_as_float(r[c])));
              }
            }
          }
        }
        if (!ok) break;
        if (ept == 0) trace_point(p, TR_LAST_ACC);
        // (wide tiles take split-K through the workspace only)
        if constexpr (!C::kWidePromote) {
        if (p.cluster_reduce) {
          // every UMMA of the unit has completed (its last buffer was full),
          // so this CTA's operand ring is idle
          cluster_signal_ready(p, red_ready, red_flags, ept);
          const RowIn rin = cluster_row_inputs<SC, SWAP>(
              p, w.row0 + static_cast<int>(cluster_ctarank()) * (128 / p.split_k) + ept % (128 / p.split_k));
          if (!mbar_wait_cluster(red_ready, 0, lim)) {
            record_status(p.status, ST_TIMEOUT_EPILOGUE);
            ok = false;
            break;
          }
#pragma unroll
          for (int c = 0; c < CPT; c += CW)
            cluster_send<BN, CW>(p, smem_u32(red_buf), red_full, w, lane_row, cbeg + c, acc + c);
          bool red_ok = false;
          EG_ACT_DISPATCH(p.act, (red_ok = cluster_reduce_store<IN, SC, SWAP, BN, C::kEpiThreads, A_>(
                                      p, red_buf, red_full, w, ept, rin)))
          if (!red_ok) {
            record_status(p.status, ST_TIMEOUT_EPILOGUE);
            ok = false;
            break;
          }
          continue;
        }
        }
        bool do_epi = true;
        if (w.contrib > 1) {
          if constexpr (IN == IN_INT8) {
            // int32 sums are exact in any order: every contributor adds its
            // partial into the tile's slot 0 (kept at zero between calls);
            // the last one reads the total in one round and re-zeroes it
            uint32_t* wsb = ws_slot<BN>(p, 0, w.tile, cbeg, lane_row);  // column stride 128
#pragma unroll
            for (int c = 0; c < CPT; ++c)
              if (row < p.rows && w.col0 + cbeg + c < p.cols)
                red_add_s32(reinterpret_cast<int*>(wsb + c * 128), static_cast<int32_t>(acc[c]));
            if (ept == 0) trace_point(p, TR_PARTIAL_OUT);
            do_epi = split_arrive_last(p, w.tile, w.contrib, ept, C::kEpiThreads, last_flag);
            if (ept == 0) trace_point(p, TR_ARRIVED);
            if (do_epi) {
#pragma unroll
              for (int c = 0; c < CPT; ++c) {
                const bool okc = row < p.rows && w.col0 + cbeg + c < p.cols;
                acc[c] = okc ? __ldcg(wsb + c * 128) : 0u;
              }
#pragma unroll
              for (int c = 0; c < CPT; ++c)
                if (row < p.rows && w.col0 + cbeg + c < p.cols) __stcg(wsb + c * 128, 0u);
            }
          } else {
            uint32_t* wsb = ws_slot<BN>(p, w.j, w.tile, cbeg, lane_row);  // column stride 128
#pragma unroll
            for (int c = 0; c < CPT; ++c)
              if (row < p.rows && w.col0 + cbeg + c < p.cols) __stcg(wsb + c * 128, acc[c]);
            if (ept == 0) trace_point(p, TR_PARTIAL_OUT);
            do_epi = split_arrive_last(p, w.tile, w.contrib, ept, C::kEpiThreads, last_flag);
            if (ept == 0) trace_point(p, TR_ARRIVED);
            if (do_epi) {
              if constexpr (C::kWidePromote) {
                // 32 columns at a time, so the partials in flight stay small
#pragma unroll
                for (int c = 0; c < CPT; c += 32) {
                  uint32_t part[32];
#pragma unroll
                  for (int j = 0; j < 32; ++j) part[j] = acc[c + j];
                  reduce_partials<IN, BN, 32>(p, w.tile, w.contrib, cbeg + c, lane_row, row < p.rows,
                                              p.cols - (w.col0 + cbeg + c), part);
#pragma unroll
                  for (int j = 0; j < 32; ++j) acc[c + j] = part[j];
                }
              } else {
                reduce_partials<IN, BN, CPT>(p, w.tile, w.contrib, cbeg, lane_row, row < p.rows,
                                             p.cols - (w.col0 + cbeg), acc);
              }
            }
          }
        }
        if (do_epi) {
          if (ept == 0) trace_point(p, TR_STORE_BEGIN);
          if constexpr (!SWAP) {
            if (tstore) {
              EG_ACT_DISPATCH(p.act, (promoted_store_staged<IN, SC, CW, CPT, A_>(
                                         p, &tmY, row, w.row0 + quarter * 32, w.col0 + cbeg, acc, boxes,
                                         nbox, lane)))
            } else {
              EG_ACT_DISPATCH(p.act, (promoted_store<IN, SC, SWAP, CW, CPT, A_>(p, row, w.col0 + cbeg, acc)))
            }
          } else {
            EG_ACT_DISPATCH(p.act, (promoted_store<IN, SC, SWAP, CW, CPT, A_>(p, row, w.col0 + cbeg, acc)))
          }
        }
      } else {
        // ---- accumulator in TMEM buffer blk&1 until the unit is done ----
        const int b = blk % NB;
        const uint32_t tb = t_lane + static_cast<uint32_t>(b * C::kAccStride);
        // swap-AB with one chunk (decode): epilogue inputs load while the
        // mainloop runs
        constexpr bool kPre = SWAP && BN == CW && !G;
        SwapIn<CW> pre;
        if constexpr (kPre) {
          if (!(p.flags & F_DEBUG) && !p.cluster_reduce) load_swap_inputs<SC, CW>(p, row, w.col0, pre);
        }
        if (w.nk > 0) {
          if (!mbar_wait(&tfull[b], (blk / NB) & 1u, lim)) {
            record_status(p.status, ST_TIMEOUT_EPILOGUE);
            ok = false;
            break;
          }
          tc_fence_after();
          if (blk == 0 && ept == 0) trace_point(p, TR_FIRST_ACC);
        }
        if (ept == 0) trace_point(p, TR_LAST_ACC);
        if (p.cluster_reduce) {
          // the accumulator is final, so every UMMA has completed and this
          // CTA's operand ring is idle
          cluster_signal_ready(p, red_ready, red_flags, ept);
          const RowIn rin = cluster_row_inputs<SC, SWAP>(
              p, w.row0 + static_cast<int>(cluster_ctarank()) * (128 / p.split_k) + ept % (128 / p.split_k));
          if (!mbar_wait_cluster(red_ready, 0, lim)) {
            record_status(p.status, ST_TIMEOUT_EPILOGUE);
            ok = false;
            break;
          }
          // this row's partial sums go to the CTA of the cluster owning it
#pragma unroll 1
          for (int c = 0; c < CPT; c += CW) {
            uint32_t r[CW];
            tmem_load_chunk<CW>(tb + static_cast<uint32_t>(c), r);
            tmem_ld_wait();
            cluster_send<BN, CW>(p, smem_u32(red_buf), red_full, w, lane_row, cbeg + c, r);
          }
          if (ept == 0) trace_point(p, TR_PARTIAL_OUT);
          tc_fence_before();
          mbar_arrive(&tempty[b]);
          ++blk;
          bool red_ok = false;
          // decode's usual bf16 output: a narrowing chosen at compile time
          if (SWAP && p.out == OUT_BF16) {
            EG_ACT_DISPATCH(p.act, (red_ok = cluster_reduce_store<IN, SC, SWAP, BN, C::kEpiThreads, A_,
                                                                  OUT_BF16>(p, red_buf, red_full, w, ept, rin)))
          } else {
            EG_ACT_DISPATCH(p.act, (red_ok = cluster_reduce_store<IN, SC, SWAP, BN, C::kEpiThreads, A_>(
                                        p, red_buf, red_full, w, ept, rin)))
          }
          if (!red_ok) {
            record_status(p.status, ST_TIMEOUT_EPILOGUE);
            ok = false;
            break;
          }
          continue;
        }
        bool do_epi = true;
        if (w.contrib > 1) {
          // this thread's accumulator columns of the unit (gated: all of
          // them, gate then up)
#pragma unroll 1
          for (int c = 0; c < (G ? C::kAccN : CPT); c += CW) {
            uint32_t r[CW];
            tmem_load_chunk<CW>(tb + static_cast<uint32_t>(c), r);
            tmem_ld_wait();
            uint32_t* wsb = ws_slot<C::kAccN>(p, w.j, w.tile, cbeg + c, lane_row);  // column stride 128
            const int ct = (cbeg + c) % BN;  // the chunk's first output column in the tile
#pragma unroll
            for (int j = 0; j < CW; ++j)
              if (row < p.rows && w.col0 + ct + j < p.cols) __stcg(wsb + j * 128, r[j]);
          }
          if (ept == 0) trace_point(p, TR_PARTIAL_OUT);
          do_epi = split_arrive_last(p, w.tile, w.contrib, ept, C::kEpiThreads, last_flag);
          if (ept == 0) trace_point(p, TR_ARRIVED);
        }
        if (do_epi) {
          if (ept == 0) trace_point(p, TR_STORE_BEGIN);
#pragma unroll 1
          for (int c = 0; c < CPT; c += CW) {
            // this thread's columns cbeg + c ... (tb already points at cbeg)
            const int cc = cbeg + c;
            uint32_t r[CW];
            if (w.nk > 0) {
              tmem_load_chunk<CW>(tb + static_cast<uint32_t>(c), r);
              tmem_ld_wait();
            } else {
#pragma unroll
              for (int j = 0; j < CW; ++j) r[j] = 0u;
            }
            if (w.contrib > 1) {
              // partials summed in split order 0..S-1 (deterministic; this
              // CTA's own one is read back too); per split, the chunk's loads
              // are independent and overlap
              reduce_partials<IN, C::kAccN, CW>(p, w.tile, w.contrib, cc, lane_row, row < p.rows,
                                                p.cols - (w.col0 + cc), r);
              if (c == 0 && ept == 0) trace_point(p, TR_REDUCED);
            }
            if constexpr (G) {
              // the up half's columns of the same outputs
              uint32_t u[CW];
              if (w.nk > 0) {
                tmem_load_chunk<CW>(tb + static_cast<uint32_t>(BN + c), u);
                tmem_ld_wait();
              } else {
#pragma unroll
                for (int j = 0; j < CW; ++j) u[j] = 0u;
              }
              if (w.contrib > 1)
                reduce_partials<IN, C::kAccN, CW>(p, w.tile, w.contrib, BN + c, lane_row,
                                                  row < p.rows, p.cols - (w.col0 + c), u);
              epilogue_gated<SC, SWAP, CW>(p, row, w.col0 + c, r, u);
              continue;
            }
            if constexpr (kPre) {
              if (!(p.flags & F_DEBUG)) {
                if (p.out == OUT_BF16) {
                  EG_ACT_DISPATCH(p.act, (store_swap<IN, SC, CW, A_, OUT_BF16>(p, row, w.col0, r, pre)))
                } else {
                  EG_ACT_DISPATCH(p.act, (store_swap<IN, SC, CW, A_>(p, row, w.col0, r, pre)))
                }
                continue;
              }
            }
            if constexpr (!SWAP && !G) {
              if (tstore) {
                EG_ACT_DISPATCH(p.act, (epilogue_chunk_staged<IN, SC, CW, A_>(
                                           p, &tmY, row, w.row0 + quarter * 32, w.col0 + cc, r,
                                           boxes + (nbox & 1u) * stage_box_bytes<CW>(), lane)))
                ++nbox;
                continue;
              }
            }
            epilogue_chunk<IN, SC, SWAP, CW>(p, row, w.col0 + cc, r);
          }
        }
        // TMEM buffer b may take the unit after next
        tc_fence_before();
        if constexpr (PR) {
          // every epilogue thread of this CTA is done with buffer b; one
          // arrival on the even CTA's barrier
          epi_bar_sync(C::kEpiThreads);
          if (ept == 0) mbar_arrive_cluster(cluster_map(smem_u32(&tempty[b]), 0));
        } else {
          mbar_arrive(&tempty[b]);
        }
        ++blk;
      }
    }
    // block scales: no copy of this thread may still be landing in shared
    // memory when the CTA leaves (the loop can end early on a timeout)
    if constexpr (SC == SC_BLOCK) cp_async_wait<0>();
    // every staged store of Y has read its box and written Y (the grid's
    // dependents read Y once it completes)
    if (tstore && lane == 0) bulk_wait_group_all();
    if (ept == 0) trace_point(p, TR_EPI_DONE);
  }

  // ------------------------------------------------------------ teardown ---
  tc_fence_before();
  __syncthreads();
  // no CTA of a cluster leaves while another may still write its buffer (or,
  // CTA pairs, still issue UMMAs into its tensor memory)
  if (PR || p.cluster_reduce) cluster_sync_all();
  if (threadIdx.x == 0) trace_point(p, TR_END);
  if (warp == 1) {
    tc_fence_after();
    if (has_work) {
      // every UMMA this CTA issued has completed before TMEM is released.
      // The issuer commits mma_done on every exit path, timeouts included,
      // and UMMAs read only shared and tensor memory, so the commit always
      // arrives; a wait that runs out is recorded and waited again with a
      // limit eight times longer before the columns are freed.
      if (lane == 0 && !mbar_wait(mma_done, 0, lim)) {
        record_status(p.status, ST_TIMEOUT_TEARDOWN);
        (void)mbar_wait(mma_done, 0, 8 * lim);
      }
      __syncwarp();
    }
    __syncwarp();
    if constexpr (PR)
      tmem_dealloc_pair(tmem_base, C::kTmemCols);
    else
      tmem_dealloc(tmem_base, C::kTmemCols);
  }
}

}  // namespace eg
