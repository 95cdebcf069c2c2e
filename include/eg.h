/*
 * eg.h -- C ABI of the fused scaled linear layer for GB300 (sm_103a).
 *
 * One kernel computes  Y = epilogue(A . W^T)  for a dense linear layer and
 * stores Y once, in bf16.  The operation is defined on the pages this
 * library follows:
 *
 *  - "Helion + TorchInductor co-operation: operator fusion", section
 *    "Operator fusion strategies: prologues and epilogues": prologue fusion
 *    applies input transforms (dequantisation, scaling) inside the tile-load
 *    loop; epilogue fusion applies bias, residual, GELU/SiLU and the
 *    FP32->narrow conversion to the accumulator tile right before its store.
 *    Section "Designing extensible epilogues in Helion": an fp32
 *    accumulator, bias broadcast over rows, ReLU or tanh-GELU, masked tails
 *    with zero fill, a single masked store.  Section "Registering the
 *    operator": the op checks that the inner dimensions match and allocates
 *    nothing but its output.
 *  - "Helion linear backend in vLLM", section "One kernel instead of three":
 *    the scale formats FP8_Dynamic (per-token activation scale, per-channel
 *    weight scale), W8A8_INT8 (the same scaling in INT8) and Block_FP8
 *    (1x128 activation blocks, 128x128 weight blocks); split_k (powers of two
 *    up to 256) and swap_ab (A@B computed as (B^T A^T)^T) are tunable
 *    parameters of that one kernel.  Sections "Hybrid dispatch" and "How the
 *    autotuner searches": small token counts (1..32) run a per-shape tuned
 *    configuration under CUDA Graph replay.
 *
 * Per output element (m, n), with acc = sum_k a[m][k] * w[n][k]:
 *
 *   EG_SCALE_TOKEN_CHANNEL:  v = acc * s_a[m] * s_w[n]
 *   EG_SCALE_BLOCK:          v = sum_kb s_a[m][kb] * s_w[n/128][kb] * (sum_{k in kb} a*w)
 *   EG_SCALE_NONE:           v = acc
 *   if EG_EPI_BIAS:              v += bias[n]
 *   if EG_EPI_RESIDUAL_PRE_ACT:  v += R[m][n]; v = act(v)
 *   else:                        v = act(v); if EG_EPI_RESIDUAL: v += R[m][n]
 *   Y[m][n] = bf16_round_nearest_even(v)   (EG_OUT_F16: fp16; EG_OUT_E4M3: the
 *             E4M3 code of v / s_y -- the FP32 -> narrow conversion right
 *             before the store that the fusion page describes)
 *
 * Layouts (all row-major, leading dimensions in ELEMENTS):
 *   A  [M][lda]  activations, K contiguous (bf16, e4m3 or int8 codes)
 *   W  [N][ldw]  weights, K contiguous (same element type as A)
 *   s_a float32: [M] (token/channel) or [M][K/128] (block), contiguous
 *   s_w float32: [N] (token/channel) or [ceil(N/128)][K/128] (block)
 *   bias bf16 [N];  R bf16 [M][ldr];  Y bf16 [M][ldy]
 *   With EG_OUT_DEBUG_ACCUM, Y is [M][ldy] of 4-byte elements instead and
 *   receives the reduced accumulator before the epilogue: int32 for INT8
 *   (exact), float32 otherwise (block mode: already block-scaled).
 *
 * Alignment rules (TMA bulk-tensor loads):
 *   A, W, bias, s_a, s_w are 16-byte aligned; lda*elt and ldw*elt are
 *   multiples of 16 bytes; K*elt is a multiple of 16 bytes.  Y and R need
 *   element alignment and ldy, ldr >= N; when Y, R and their row strides
 *   are 16-byte aligned the epilogue uses 16-byte vector accesses.  Block
 *   scaling needs K % 128 == 0.
 *   INT8 needs K <= 133144 so that |acc| <= 127^2 K fits in int32.
 *
 * Ownership: the caller owns every tensor and keeps it alive until the work
 * queued on the stream has finished.  A plan owns its split-K workspace,
 * its per-tile arrival counters (zeroed at creation and reset by the kernel
 * itself), its device status word, its cached TMA descriptors and its
 * captured graphs; eg_plan_destroy frees them after synchronising the
 * plan's device work.  eg_plan_run allocates nothing, reads no device memory
 * and does not synchronise.  Runs of one plan must not overlap on the GPU
 * (they share the workspace and counters): queue them on one stream.
 *
 * Errors: every call returns an eg_status; eg_last_error_detail() returns a
 * thread-local description of the last failure.  Argument errors are
 * detected before any device work is queued.  A device-side pipeline wait
 * that exceeds its time limit makes the kernel record the failure in the
 * plan's status word and return without hanging; eg_plan_device_status()
 * reports it as EG_ERR_DEVICE_TIMEOUT.
 */
#ifndef EG_H
#define EG_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define EG_API __attribute__((visibility("default")))
#else
#define EG_API
#endif

typedef enum {
  EG_OK = 0,
  EG_ERR_INVALID_ARG = 1,   /* null / misaligned / inconsistent argument */
  EG_ERR_UNSUPPORTED = 2,   /* valid but not supported (device, shape, tuning) */
  EG_ERR_NO_MEMORY = 3,     /* device allocation failed */
  EG_ERR_CUDA = 4,          /* a CUDA runtime or driver call failed */
  EG_ERR_DEVICE_TIMEOUT = 5,/* a device pipeline wait ran past its limit */
  EG_ERR_NOT_TUNED = 6      /* no tuning entry and no default applies */
} eg_status;

typedef enum { EG_IN_BF16 = 0, EG_IN_E4M3 = 1, EG_IN_INT8 = 2 } eg_in_dtype;

typedef enum {
  EG_SCALE_NONE = 0,          /* bf16 inputs only */
  EG_SCALE_TOKEN_CHANNEL = 1, /* FP8_Dynamic / W8A8_INT8: s_a[m] * s_w[n] */
  EG_SCALE_BLOCK = 2          /* Block_FP8: 1x128 activation, 128x128 weight */
} eg_scale_mode;

typedef enum {
  EG_ACT_NONE = 0,
  EG_ACT_RELU = 1,
  EG_ACT_GELU_ERF = 2,   /* 0.5 v (1 + erf(v / sqrt 2)) */
  EG_ACT_GELU_TANH = 3,  /* 0.5 v (1 + tanh(sqrt(2/pi) (v + 0.044715 v^3))) */
  EG_ACT_SILU = 4        /* v / (1 + exp(-v)) */
} eg_act;

enum {
  EG_EPI_BIAS = 1,
  EG_EPI_RESIDUAL = 2,          /* v = act(v) + R */
  EG_EPI_RESIDUAL_PRE_ACT = 4,  /* v = act(v + R)  (excludes EG_EPI_RESIDUAL) */
  EG_OUT_DEBUG_ACCUM = 8,       /* write the raw reduced accumulator */
  EG_RUN_GRAPH = 16,            /* eg_plan_run replays a captured CUDA graph */
  EG_RUN_PDL = 32,              /* launch as a programmatic dependent of the
                                   previous kernel on the stream: the kernel
                                   starts streaming W before that kernel has
                                   finished, and waits for it before reading
                                   A, s_a, R, bias or s_w and before writing.
                                   Requires that the previous kernel does not
                                   write W. */
  EG_RUN_QUANT_A = 64,          /* E4M3 / INT8 with per-token scales only:
                                   eg_args.A holds bf16 activations [M][lda]
                                   (lda in elements); each run first
                                   quantises them per token as
                                   eg_quantize_rows does, into codes and
                                   scales the plan owns (eg_args.s_a is not
                                   read), then runs the GEMM on them as its
                                   programmatic dependent. */
  EG_EPI_GATED = 512,           /* gated linear unit (SwiGLU with SiLU): W is
                                   [2N][ldw], the gate half (rows 0..N-1)
                                   then the up half (rows N..2N-1); s_w and
                                   bias cover the 2N rows; per output (m, n)
                                   gate = scale * acc[m][n] + bias[n],
                                   up = scale * acc[m][N + n] + bias[N + n],
                                   y = act(gate) * up (+ R[m][n]).  bf16 and
                                   E4M3 token/channel inputs: one kernel (no
                                   cluster_reduce).  INT8 token/channel and
                                   E4M3 block scales (N % 128 == 0): two
                                   kernels, the accumulators of all 2N rows
                                   into a buffer the plan owns, then a
                                   combine kernel (eg_plan_run_unfused and
                                   eg_linear_noalloc reject these).  Not with
                                   EG_EPI_RESIDUAL_PRE_ACT or
                                   EG_OUT_DEBUG_ACCUM. */
  EG_OUT_F16 = 128,             /* Y is fp16 [M][ldy] (nearest even) */
  EG_OUT_E4M3 = 256             /* Y is E4M3 codes [M][ldy] (one byte each) of
                                   v / s_y with s_y = *eg_args.s_y (computed
                                   as v times the float32 reciprocal of s_y,
                                   nearest even, saturated to +-448).
                                   EG_OUT_F16, EG_OUT_E4M3 and
                                   EG_OUT_DEBUG_ACCUM exclude each other; the
                                   unfused path writes bf16 only. */
};

typedef struct {
  int64_t M, N, K;
  int32_t dtype;  /* eg_in_dtype */
  int32_t scale;  /* eg_scale_mode */
  int32_t act;    /* eg_act */
  uint32_t flags; /* EG_EPI_* | EG_OUT_DEBUG_ACCUM | EG_RUN_* */
} eg_problem;

/* One point of the kernel's tuning space.  The UMMA tile is 128 rows (256
 * with cta_pair) by tile_n columns; rows run over M, or over N when swap_ab
 * is set. */
typedef struct {
  int32_t tile_n;   /* UMMA N: 16, 32, 64, 128 or 256 */
  int32_t stages;   /* shared-memory ring depth, 2..8 */
  int32_t split_k;  /* 1..256, at most the number of K tiles */
  int32_t swap_ab;  /* 0: rows over M;  1: rows over N (Y^T = W A^T) */
  int32_t stream_k; /* 0: K split evenly split_k ways per tile.  n > 0:
                       balanced split-K: n CTAs per SM share the whole
                       tiles x K-tiles iteration space in equal contiguous
                       ranges (split_k must be 1); a tile's partial sums
                       reduce through the same workspace, in CTA order */
  int32_t cluster_reduce; /* 0: split-K partial sums go through the plan's
                       global workspace and the last CTA of a tile to
                       arrive reduces them.  1: the split_k CTAs of a tile
                       (split_k in {2, 4, 8}, stream_k 0) run as one thread-
                       block cluster and exchange their partial sums through
                       distributed shared memory; each CTA reduces 128 /
                       split_k of the tile's rows (in split order, so the
                       result is the same) and runs their epilogue.  No
                       workspace or arrival counters are used. */
  int32_t cta_pair;  /* 0: one CTA per 128-row tile.  1: CTA pairs: two CTAs
                       of a 2-CTA cluster compute one 256-row tile with
                       pair UMMAs (M = 256, cta_group::2), each holding its
                       128 activation rows and half of the weight tile per
                       stage, so each SM stages half as much of W.  bf16 or
                       E4M3 per-token/channel, swap_ab 0, tile_n 128 or
                       256, split_k 1, stream_k 0, cluster_reduce 0, not
                       gated. */
} eg_tuning;

typedef struct {
  const void* A;
  const void* W;
  const float* s_a;
  const float* s_w;
  const void* bias;      /* bf16 [N], needed with EG_EPI_BIAS */
  const void* residual;  /* bf16 [M][ldr], needed with a residual flag */
  void* Y;
  int64_t lda, ldw, ldr, ldy;
  const float* s_y;      /* device float: output scale, needed with EG_OUT_E4M3 */
} eg_args;

typedef struct eg_plan eg_plan;

/* Validate `problem`, pick a tuning (`tuning` overrides the built-in table;
 * NULL uses the table, then a default rule), allocate the plan's workspace,
 * counters and status word on the current device.  Returns
 * EG_ERR_INVALID_ARG for an inconsistent problem, EG_ERR_UNSUPPORTED for an
 * unsupported device or tuning, EG_ERR_NO_MEMORY / EG_ERR_CUDA on device
 * failures.  On success *out owns a new plan.
 *
 * Environment overrides read at plan creation, for measurements only:
 * EG_PDL_L2_PREFETCH=0 (no L2 prefetch of the weight range as a programmatic
 * dependent), EG_COMMIT_GROUP=n (ring stages released per UMMA commit; n must
 * divide the stages; default two for CTA pairs with 6+ even stages, else
 * one), EG_ACC_RELEASE=0 (promotion kernels release ring stages / INT8
 * operand slots with their own commit instead of the K block's accumulator
 * commit), EG_STAGED_STORE=0 (rows-over-M epilogues store Y directly from
 * registers instead of through shared-memory boxes and TMA stores),
 * EG_WAIT_CAP_MS (bound on any in-kernel wait). */
EG_API eg_status eg_plan_create(const eg_problem* problem, const eg_tuning* tuning,
                         eg_plan** out);

/* Bytes of device scratch the plan holds: the split-K workspace (0 when
 * split_k == 1) and, for INT8 / Block_FP8 gated units, the M x 2N
 * accumulator buffer. */
EG_API eg_status eg_plan_workspace_bytes(const eg_plan* plan, size_t* out);

/* The tuning the plan runs. */
EG_API eg_status eg_plan_get_tuning(const eg_plan* plan, eg_tuning* out);

/* Queue one fused linear-layer call on `stream` (a cudaStream_t; NULL is the
 * legacy default stream).  With EG_RUN_GRAPH the call is captured once per
 * distinct argument set into a CUDA graph and replayed on later calls; the
 * plan keeps the 8 most recently used graphs and destroys older ones. */
EG_API eg_status eg_plan_run(eg_plan* plan, const eg_args* args, void* stream);

/* The unfused comparison path of the same problem: the same GEMM kernel
 * with no epilogue writes bf16 T1 [M][N]; a second kernel writes
 * T2 = T1 + bias (+ R for the pre-activation order); a third writes
 * Y = act(T2) (+ R for the default order).  T1 and T2 are caller-owned bf16
 * [M][N] buffers (row stride N).  Three launches; for measurement only. */
EG_API eg_status eg_plan_run_unfused(eg_plan* plan, const eg_args* args, void* T1,
                              void* T2, void* stream);

/* Synchronise the plan's last queued work and report a device-side wait
 * timeout recorded by its kernels (EG_ERR_DEVICE_TIMEOUT, then cleared).
 * After a timeout the plan's split-K arrival counters and workspace are
 * reset as well (a CTA that gave up leaves its tiles half counted), so the
 * plan's next run is correct. */
EG_API eg_status eg_plan_device_status(eg_plan* plan);

/* Free everything the plan owns.  NULL is accepted. */
EG_API eg_status eg_plan_destroy(eg_plan* plan);

/* Number of kernel launches the last eg_plan_run / eg_plan_run_unfused
 * queued (a graph replay counts the kernels inside it). */
EG_API int32_t eg_plan_last_launch_count(const eg_plan* plan);

/* Testing hook for failure detection: limit every device pipeline wait of
 * this plan to `wait_limit_ns` nanoseconds (0 restores the default of
 * 2 s), and have the load warp issue no loads so that the first wait runs
 * out: `stall_producer` 1 in every CTA, 2 in odd-numbered CTAs only (the
 * others finish their work and count their split-K arrivals, leaving tiles
 * half counted), 0 off; other values are EG_ERR_INVALID_ARG.  No fault,
 * trap or hang results: the kernel records EG_ERR_DEVICE_TIMEOUT and
 * returns. */
EG_API eg_status eg_plan_set_test_stall(eg_plan* plan, uint64_t wait_limit_ns,
                                 int32_t stall_producer);

/* Launch configuration the plan uses: the kernel is persistent, so `grid`
 * CTAs (at most `units`, at most every resident slot of the device) loop
 * over the `units` work units (one 128 x tile_n tile and one K split each). */
typedef struct {
  int32_t grid, block, smem_bytes, units, blocks_per_sm, regs_per_thread;
} eg_launch_info;
EG_API eg_status eg_plan_get_launch(const eg_plan* plan, eg_launch_info* out);

/* Tracing: when `trace` is non-NULL, every later run of this plan records,
 * per CTA, EG_TRACE_POINTS device %globaltimer values (nanoseconds) into
 * trace[cta * EG_TRACE_POINTS + point] for ctas < trace_ctas:
 *   0 CTA start, 1 setup done, 2 first TMA issued (after the wait on the
 *   previous kernel), 3 first UMMA operands ready, 4 last UMMA committed,
 *   5 first accumulator ready in the epilogue, 6 epilogue done, 7 CTA end,
 *   8 first weight loads issued (before the wait on the previous kernel),
 *   9 last load issued, and for the CTA's last work unit, seen by its first
 *   epilogue thread: 10 accumulator final, 11 split-K partial stored or
 *   sent, 12 arrival counted or partials received, 14 output stores (with
 *   the last arriver's reduction) begin, 13 the last arriver's first chunk
 *   reduced (tensor-memory accumulator path).  Point 15, and points a path
 *   does not pass, keep the buffer's value.
 * The buffer is caller-owned device memory of trace_ctas * EG_TRACE_POINTS
 * * 8 bytes.  NULL turns tracing off. */
#define EG_TRACE_POINTS 16
EG_API eg_status eg_plan_set_trace(eg_plan* plan, uint64_t* trace, int32_t trace_ctas);

/* One fused linear-layer call that allocates no device memory.  (The pages
 * this library follows have no counterpart to this call.)
 *
 * For callers that cannot allocate on the path where they run the layer:
 * code living inside a memory pool or arena that owns all of the device's
 * memory, allocators that must not be re-entered from inside a call, or
 * runtimes that forbid cudaMalloc once they are running.  eg_plan_create
 * allocates the split-K workspace, tile counters and a status word; this
 * call instead runs the same kernel with that scratch in one fixed array
 * compiled into the library (4 MiB of split-K partial sums plus 16383 tile
 * counters and the status word), which every device that loads the library
 * holds until the process exits.  The caller still passes inputs and
 * outputs; `problem`, `tuning` (NULL: the built-in table, then the default
 * rule), `args` and `stream` mean what they mean for eg_plan_create and
 * eg_plan_run.  EG_RUN_GRAPH is rejected.
 *
 * The first call on each device looks up the array's device address; make
 * that first call before any stream capture.  The address is kept for the
 * life of the process, so a device reset (cudaDeviceReset) after the first
 * call on that device is not supported.  Every call clears the tile
 * counters and the status word on `stream` before its kernel; the split-K
 * partial sums are written before they are read.  All calls share the one
 * array: calls that overlap on the GPU (other streams, other threads) race
 * and must not be issued.  A problem whose split-K scratch or tile count
 * exceeds the array returns EG_ERR_UNSUPPORTED with the sizes in
 * eg_last_error_detail().  Device-side wait timeouts are not reported. */
EG_API eg_status eg_linear_noalloc(const eg_problem* problem, const eg_tuning* tuning,
                                   const eg_args* args, void* stream);

/* Dynamic per-token quantisation of activations, the prologue transform in
 * front of the FP8_Dynamic and W8A8_INT8 layers ("Helion linear backend in
 * vLLM", section "One kernel instead of three": per-token activation
 * scales; "Helion + TorchInductor co-operation: operator fusion", section
 * on prologue fusion).  For each row m of x (bf16 [M][ldx], device):
 *   s[m] = amax_k |x[m][k]| / 448 (dtype EG_IN_E4M3) or / 127 (EG_IN_INT8),
 *          float32 division; s[m] = 1 when the row is all zero;
 *   q[m][k] = round-to-nearest-even(x[m][k] / s[m]) (float32 division),
 *          saturated to +-448 (E4M3 code) or +-127 (int8).
 * q: device bytes [M][ldq], ldq >= K; s: device float [M].  Enqueued on
 * `stream` (a cudaStream_t, NULL for the default stream); nothing is
 * allocated.  EG_ERR_INVALID_ARG for bad sizes, NULL pointers or another
 * dtype; EG_ERR_CUDA if the launch fails. */
EG_API eg_status eg_quantize_rows(const void* x, int64_t M, int64_t K, int64_t ldx, int32_t dtype,
                                  void* q, int64_t ldq, float* s, void* stream);

EG_API const char* eg_status_string(eg_status s);
EG_API const char* eg_last_error_detail(void);

#ifdef __cplusplus
}
#endif
#endif /* EG_H */
