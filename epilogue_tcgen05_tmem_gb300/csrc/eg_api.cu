// eg_api.cu -- host side of the C ABI declared in include/eg.h: problem and
// argument validation, tuning lookup, TMA descriptor encoding, launches,
// CUDA-graph capture/replay, and the unfused comparison path.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <algorithm>
#include <mutex>
#include <string>
#include <vector>

#include "../../include/eg.h"
#include "eg_kernel.cuh"
#include "eg_registry.h"
#include "eg_gated.h"
#include "eg_quant.h"
#include "eg_tuning.h"

namespace {

thread_local std::string g_detail;

eg_status fail(eg_status s, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  g_detail = buf;
  return s;
}

eg_status cuda_fail(cudaError_t e, const char* what) {
  return fail(e == cudaErrorMemoryAllocation ? EG_ERR_NO_MEMORY : EG_ERR_CUDA, "%s: %s (%s)",
              what, cudaGetErrorName(e), cudaGetErrorString(e));
}

#define EG_CUDA(call, what)                  \
  do {                                       \
    cudaError_t e_ = (call);                 \
    if (e_ != cudaSuccess) return cuda_fail(e_, what); \
  } while (0)

// cuTensorMapEncodeTiled through the runtime's driver entry point, so the
// library needs no link-time dependency on libcuda.
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static std::once_flag once;
  static EncodeTiledFn fn = nullptr;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                        &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

int elt_bytes(int dtype) { return dtype == EG_IN_BF16 ? 2 : 1; }

uint64_t default_wait_limit_ns() {
  const char* e = getenv("EG_WAIT_CAP_MS");
  if (e && *e) {
    const double ms = atof(e);
    if (ms > 0) return static_cast<uint64_t>(ms * 1e6);
  }
  return 2000000000ull;  // 2 s
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Bytes of one Y element for the output flags.
int out_elt_bytes(uint32_t flags) {
  if (flags & EG_OUT_DEBUG_ACCUM) return 4;
  if (flags & EG_OUT_E4M3) return 1;
  return 2;
}

}  // namespace

struct GraphEntry {
  eg_args args;
  cudaGraphExec_t exec;
};

// Captured graphs a plan keeps in EG_RUN_GRAPH mode (one per argument set,
// least recently used dropped first).
constexpr size_t kGraphCache = 8;

struct eg_plan {
  eg_problem prob{};
  eg_tuning tune{};
  int device = -1;
  eg::KernelEntry ke{};
  uint32_t smem = 0;
  int rows = 0, cols = 0, tiles_rows = 0, tiles_cols = 0, k_tiles = 0, grid = 0;
  int kb_count = 0;
  void* ws = nullptr;
  size_t ws_bytes = 0;
  // EG_RUN_QUANT_A: the per-token codes [M][ldq] and scales [M] of A
  void* qa = nullptr;
  float* qs = nullptr;
  int64_t ldq = 0;
  int* counters = nullptr;
  int* status = nullptr;
  uint64_t wait_limit_ns = 0;
  int stall = 0;
  int l2_prefetch = 1;  // EG_PDL_L2_PREFETCH=0 turns the L2 weight prefetch off
  int commit_group = 1; // ring stages released per UMMA commit (see commit_group_for)
  int acc_release = 0;  // promotion frees stages / INT8 slots by the accumulator commit
  int units = 0, blocks_per_sm = 0, regs = 0, max_contrib = 1;
  uint64_t* trace = nullptr;
  int trace_ctas = 0;
  // TMA descriptor cache (re-encoded when A/W or their strides change)
  bool maps_valid = false;
  const void* mapA = nullptr;
  const void* mapW = nullptr;
  int64_t map_lda = 0, map_ldw = 0;
  CUtensorMap tmP{}, tmQ{};
  // staged TMA stores of Y (rows over M, 2-byte outputs): shared-memory
  // offset of the epilogue warps' staging boxes, and the cached tensor map
  // of the Y the last run wrote
  bool stage_ok = false;
  uint32_t out_stage_off = 0;
  CUtensorMap tmY{};
  const void* mapY = nullptr;
  int64_t map_ldy = 0;
  std::vector<GraphEntry> graphs;
  cudaStream_t cap_stream = nullptr;
  int last_launches = 0;
  // Gated units of INT8 and Block_FP8 inputs run in two kernels: the fused
  // kernel's accumulator output over all 2N weight rows into gacc ([M][2N]
  // words), then the combine kernel (act(gate) * up and the epilogue).  prob
  // is then that accumulator GEMM and `user` the caller's problem.
  bool two_pass_gated = false;
  eg_problem user{};
  uint32_t* gacc = nullptr;
};

namespace {

eg_status validate_problem(const eg_problem* p) {
  if (!p) return fail(EG_ERR_INVALID_ARG, "problem is NULL");
  if (p->M < 0 || p->N < 0 || p->K < 0)
    return fail(EG_ERR_INVALID_ARG, "negative dimension (M=%lld N=%lld K=%lld)", (long long)p->M,
                (long long)p->N, (long long)p->K);
  if (p->M > INT32_MAX || p->N > INT32_MAX || p->K > INT32_MAX)
    return fail(EG_ERR_UNSUPPORTED, "dimensions must fit in int32");
  const bool dt_ok = p->dtype == EG_IN_BF16 || p->dtype == EG_IN_E4M3 || p->dtype == EG_IN_INT8;
  if (!dt_ok) return fail(EG_ERR_INVALID_ARG, "unknown dtype %d", p->dtype);
  switch (p->scale) {
    case EG_SCALE_NONE:
      if (p->dtype != EG_IN_BF16)
        return fail(EG_ERR_INVALID_ARG, "8-bit inputs need a scale mode");
      break;
    case EG_SCALE_TOKEN_CHANNEL:
      if (p->dtype == EG_IN_BF16)
        return fail(EG_ERR_INVALID_ARG, "bf16 inputs take EG_SCALE_NONE");
      break;
    case EG_SCALE_BLOCK:
      if (p->dtype != EG_IN_E4M3)
        return fail(EG_ERR_INVALID_ARG, "block scaling is defined for e4m3 inputs");
      if (p->K % 128)
        return fail(EG_ERR_INVALID_ARG, "block scaling needs K %% 128 == 0 (K=%lld)",
                    (long long)p->K);
      break;
    default:
      return fail(EG_ERR_INVALID_ARG, "unknown scale mode %d", p->scale);
  }
  if (p->act < EG_ACT_NONE || p->act > EG_ACT_SILU)
    return fail(EG_ERR_INVALID_ARG, "unknown activation %d", p->act);
  const uint32_t known =
      EG_EPI_BIAS | EG_EPI_RESIDUAL | EG_EPI_RESIDUAL_PRE_ACT | EG_OUT_DEBUG_ACCUM | EG_RUN_GRAPH |
      EG_RUN_PDL | EG_RUN_QUANT_A | EG_OUT_F16 | EG_OUT_E4M3 | EG_EPI_GATED;
  if (p->flags & ~known) return fail(EG_ERR_INVALID_ARG, "unknown flag bits 0x%x", p->flags);
  const uint32_t outs = p->flags & (EG_OUT_F16 | EG_OUT_E4M3 | EG_OUT_DEBUG_ACCUM);
  if (outs & (outs - 1))
    return fail(EG_ERR_INVALID_ARG, "EG_OUT_F16, EG_OUT_E4M3 and EG_OUT_DEBUG_ACCUM exclude each other");
  if (p->flags & EG_EPI_GATED) {
    // block scales: the up half starts on a 128-row weight block
    if (p->scale == EG_SCALE_BLOCK && p->N % 128)
      return fail(EG_ERR_UNSUPPORTED, "gated units with block scales need N %% 128 == 0 (N=%lld)",
                  (long long)p->N);
    if (p->flags & (EG_EPI_RESIDUAL_PRE_ACT | EG_OUT_DEBUG_ACCUM))
      return fail(EG_ERR_INVALID_ARG,
                  "EG_EPI_GATED excludes EG_EPI_RESIDUAL_PRE_ACT and EG_OUT_DEBUG_ACCUM");
    if (p->N > INT32_MAX / 2) return fail(EG_ERR_UNSUPPORTED, "2N must fit in int32");
  }
  if ((p->flags & EG_RUN_QUANT_A) &&
      !((p->dtype == EG_IN_E4M3 || p->dtype == EG_IN_INT8) && p->scale == EG_SCALE_TOKEN_CHANNEL))
    return fail(EG_ERR_INVALID_ARG, "EG_RUN_QUANT_A needs E4M3 or INT8 inputs with per-token scales");
  if ((p->flags & EG_EPI_RESIDUAL) && (p->flags & EG_EPI_RESIDUAL_PRE_ACT))
    return fail(EG_ERR_INVALID_ARG, "EG_EPI_RESIDUAL and EG_EPI_RESIDUAL_PRE_ACT exclude each other");
  if ((p->K * elt_bytes(p->dtype)) % 16)
    return fail(EG_ERR_INVALID_ARG, "K * element size must be a multiple of 16 bytes (K=%lld)",
                (long long)p->K);
  if (p->dtype == EG_IN_INT8 && p->K > 133144)
    return fail(EG_ERR_UNSUPPORTED, "INT8 needs K <= 133144 so the int32 accumulator cannot overflow");
  return EG_OK;
}

bool lookup_kernel(const eg_problem& p, int swap, int bn, int pair, eg::KernelEntry* ke) {
  if (pair) {
    // CTA pairs: plain layers without swap-AB, bf16, FP8 per-token/channel
    // or FP8 block scales
    if (swap || (p.flags & EG_EPI_GATED)) return false;
    if (p.dtype == EG_IN_BF16) return eg::lookup_bf16_pair(bn, ke);
    if (p.dtype == EG_IN_E4M3 && p.scale == EG_SCALE_TOKEN_CHANNEL)
      return eg::lookup_e4m3_tc_pair(bn, ke);
    if (p.dtype == EG_IN_E4M3 && p.scale == EG_SCALE_BLOCK) return eg::lookup_e4m3_block_pair(bn, ke);
    return false;
  }
  if (p.flags & EG_EPI_GATED) {
    if (p.dtype == EG_IN_BF16) return eg::lookup_bf16_gated(swap, bn, ke);
    if (p.dtype == EG_IN_E4M3 && p.scale == EG_SCALE_TOKEN_CHANNEL)
      return eg::lookup_e4m3_tc_gated(swap, bn, ke);
    return false;
  }
  if (p.dtype == EG_IN_BF16) return eg::lookup_bf16(swap, bn, ke);
  if (p.dtype == EG_IN_E4M3 && p.scale == EG_SCALE_TOKEN_CHANNEL)
    return eg::lookup_e4m3_tc(swap, bn, ke);
  if (p.dtype == EG_IN_E4M3 && p.scale == EG_SCALE_BLOCK)
    return eg::lookup_e4m3_block(swap, bn, ke);
  if (p.dtype == EG_IN_INT8) return eg::lookup_int8_tc(swap, bn, ke);
  return false;
}

constexpr uint32_t kMaxSmem = 232448;  // opt-in dynamic shared memory per block on sm_100/103

// Cluster split-K exchange buffer: [split][128 / split rows][tile_n + 4]
// fp32 words, i.e. 128 padded rows whatever the split.  The kernel lays it
// over its operand ring (TMA stages and, for INT8, the fp16 operand slots).
uint64_t red_buffer_bytes(const eg_tuning& t) {
  return t.cluster_reduce ? uint64_t(t.tile_n + 4) * 128u * 4u : 0u;
}

eg_status validate_tuning(const eg_problem& p, const eg_tuning& t, eg::KernelEntry* ke,
                          uint32_t* smem, int* k_tiles) {
  if (t.swap_ab != 0 && t.swap_ab != 1)
    return fail(EG_ERR_INVALID_ARG, "swap_ab must be 0 or 1");
  if (t.cta_pair != 0 && t.cta_pair != 1)
    return fail(EG_ERR_INVALID_ARG, "cta_pair must be 0 or 1");
  if (t.cta_pair && (t.split_k != 1 || t.stream_k != 0 || t.cluster_reduce != 0))
    return fail(EG_ERR_UNSUPPORTED, "cta_pair takes split_k 1, stream_k 0 and cluster_reduce 0");
  if (!lookup_kernel(p, t.swap_ab, t.tile_n, t.cta_pair, ke))
    return fail(EG_ERR_UNSUPPORTED,
                "no kernel for tile_n=%d swap_ab=%d cta_pair=%d with this dtype/scale/epilogue",
                t.tile_n, t.swap_ab, t.cta_pair);
  if (t.stages < 2 || t.stages > 8)
    return fail(EG_ERR_UNSUPPORTED, "stages must be in 2..8 (got %d)", t.stages);
  if (t.cluster_reduce != 0 && t.cluster_reduce != 1)
    return fail(EG_ERR_INVALID_ARG, "cluster_reduce must be 0 or 1");
  if (t.cluster_reduce && (p.flags & EG_EPI_GATED))
    return fail(EG_ERR_UNSUPPORTED, "gated units reduce split-K through the workspace (cluster_reduce 0)");
  if (t.cluster_reduce && p.scale == EG_SCALE_BLOCK && !t.swap_ab && t.tile_n > 128)
    return fail(EG_ERR_UNSUPPORTED,
                "block-scale tiles wider than 128 reduce split-K through the workspace (cluster_reduce 0)");
  if (t.cluster_reduce) {
    if (t.split_k != 2 && t.split_k != 4 && t.split_k != 8)
      return fail(EG_ERR_UNSUPPORTED, "cluster_reduce needs split_k in {2, 4, 8} (got %d)", t.split_k);
    if (t.stream_k != 0)
      return fail(EG_ERR_INVALID_ARG, "cluster_reduce and balanced split-K exclude each other");
  }
  const uint64_t ring = uint64_t(t.stages) * ke->stage_bytes + ke->op_bytes;
  if (red_buffer_bytes(t) > ring)
    return fail(EG_ERR_UNSUPPORTED,
                "cluster_reduce with tile_n=%d needs %llu bytes of operand ring; %d stages give %llu",
                t.tile_n, (unsigned long long)red_buffer_bytes(t), t.stages, (unsigned long long)ring);
  const uint64_t s = ke->fixed_bytes + uint64_t(t.stages) * ke->stage_bytes +
                     eg::block_scale_smem_bytes(p, t.swap_ab, t.tile_n, ke->elems_per_stage);
  if (s > kMaxSmem)
    return fail(EG_ERR_UNSUPPORTED, "%d stages need %llu bytes of shared memory (max %u)", t.stages,
                (unsigned long long)s, kMaxSmem);
  *smem = static_cast<uint32_t>(s);
  const int kt = static_cast<int>((p.K + ke->elems_per_stage - 1) / ke->elems_per_stage);
  *k_tiles = kt;
  {
    // the kernel walks units and K-tile iterations in 32-bit integers
    const int64_t rows = t.swap_ab ? p.N : p.M, cols = t.swap_ab ? p.M : p.N;
    const int64_t tiles = ((rows + 127) / 128) * ((cols + t.tile_n - 1) / t.tile_n);
    if (tiles * std::max<int64_t>(std::max(kt, 1), t.split_k) > INT32_MAX)
      return fail(EG_ERR_UNSUPPORTED, "tiles x K tiles exceeds the kernel's 32-bit work counters");
  }
  if (t.split_k < 1 || t.split_k > 256)
    return fail(EG_ERR_UNSUPPORTED, "split_k must be in 1..256 (got %d)", t.split_k);
  if (t.split_k > (kt > 0 ? kt : 1))
    return fail(EG_ERR_UNSUPPORTED, "split_k=%d exceeds the %d K tiles", t.split_k, kt);
  if (t.stream_k < 0 || t.stream_k > 8)
    return fail(EG_ERR_UNSUPPORTED, "stream_k must be in 0..8 CTAs per SM (got %d)", t.stream_k);
  if (t.stream_k > 0 && t.split_k != 1)
    return fail(EG_ERR_INVALID_ARG, "balanced split-K (stream_k > 0) takes split_k = 1");
  if (t.stream_k > 0 && kt == 0)
    return fail(EG_ERR_UNSUPPORTED, "balanced split-K needs K > 0");
  return EG_OK;
}

// Reserve the epilogue warps' staging boxes for staged TMA stores of Y
// (rows over M, bf16 / fp16 output) when the epilogue can use them and the
// shared memory they take neither exceeds the per-block limit nor lowers the
// number of CTAs an SM holds.  EG_STAGED_STORE=0 turns them off.
void plan_staging(eg_plan* pl, int dev) {
  const eg_problem& p = pl->prob;
  const eg_tuning& t = pl->tune;
  pl->stage_ok = false;
  pl->out_stage_off = 0;
  if (const char* e = getenv("EG_STAGED_STORE"))
    if (atoi(e) == 0) return;
  if (t.swap_ab || t.cluster_reduce || (p.flags & (EG_EPI_GATED | EG_OUT_E4M3 | EG_OUT_DEBUG_ACCUM)))
    return;
  if (pl->ke.cw != 32 && pl->ke.cw != 16) return;
  // boxes after the ring, barriers and block scales, on a 1 KB boundary of
  // the kernel's aligned shared-memory base (pl->smem counts 1 KB of slack)
  const uint32_t off = (pl->smem - 1024u + 1023u) & ~1023u;
  const uint32_t total =
      1024u + off + static_cast<uint32_t>(pl->ke.epi_warps) * 2u * 32u * static_cast<uint32_t>(pl->ke.cw) * 2u;
  if (total > kMaxSmem) return;
  int sm_smem = 0, reserved = 0;
  if (cudaDeviceGetAttribute(&sm_smem, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&reserved, cudaDevAttrReservedSharedMemoryPerBlock, dev) != cudaSuccess)
    return;
  if (sm_smem / static_cast<int>(total + reserved) < sm_smem / static_cast<int>(pl->smem + reserved))
    return;
  pl->stage_ok = true;
  pl->out_stage_off = off;
  pl->smem = total;
}

int sm_count_of(int dev) {
  int n = 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
    n = 148;
  return n;
}

// CTAs of the plan's kernel that fit on one SM: shared memory (with the
// per-block reservation), registers (allocated per warp in units of 256 and
// spread over the SM's 4 sub-partitions), threads, blocks, and the 512 TMEM
// columns.  Also records the kernel's registers per thread.
eg_status residency(eg_plan* pl, int dev, int* per_sm_out) {
  cudaFuncAttributes fa{};
  EG_CUDA(cudaFuncGetAttributes(&fa, pl->ke.fn), "cudaFuncGetAttributes");
  pl->regs = fa.numRegs;
  int sm_smem = 0, reserved = 0, sm_regs = 0, sm_threads = 0, sm_blocks = 0;
  EG_CUDA(cudaDeviceGetAttribute(&sm_smem, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev), "device limits");
  EG_CUDA(cudaDeviceGetAttribute(&reserved, cudaDevAttrReservedSharedMemoryPerBlock, dev), "device limits");
  EG_CUDA(cudaDeviceGetAttribute(&sm_regs, cudaDevAttrMaxRegistersPerMultiprocessor, dev), "device limits");
  EG_CUDA(cudaDeviceGetAttribute(&sm_threads, cudaDevAttrMaxThreadsPerMultiProcessor, dev), "device limits");
  EG_CUDA(cudaDeviceGetAttribute(&sm_blocks, cudaDevAttrMaxBlocksPerMultiprocessor, dev), "device limits");
  const int warps = (pl->ke.threads + 31) / 32;
  const int regs_warp = ((fa.numRegs * 32 + 255) / 256) * 256;
  const int warps_per_smsp = (sm_regs / 4) / std::max(1, regs_warp);
  int per_sm = sm_smem / static_cast<int>(pl->smem + reserved);
  per_sm = std::min(per_sm, (4 * warps_per_smsp) / warps);
  per_sm = std::min(per_sm, sm_threads / pl->ke.threads);
  per_sm = std::min(per_sm, sm_blocks);
  per_sm = std::min(per_sm, 512 / pl->ke.tmem_cols);
  if (per_sm < 1) return fail(EG_ERR_UNSUPPORTED, "the kernel does not fit on an SM");
  // a setmaxnreg split draws on the block's launch allocation (threads x
  // registers per thread): one that does not fit would wait forever
  if (pl->ke.regsplit_need > 0 && fa.numRegs * pl->ke.threads < pl->ke.regsplit_need)
    return fail(EG_ERR_UNSUPPORTED,
                "the kernel's register split needs %d registers; it was built with %d x %d",
                pl->ke.regsplit_need, fa.numRegs, pl->ke.threads);
  *per_sm_out = per_sm;
  return EG_OK;
}

// Launch grid, work units and partial-sum slots per tile of the plan's
// tuning, for `per_sm` resident CTAs on each of `sms` SMs.
void plan_grid(eg_plan* pl, int sms, int per_sm) {
  const eg_tuning& t = pl->tune;
  const long long tiles = static_cast<long long>(pl->tiles_rows) * pl->tiles_cols;
  const long long units = tiles * t.split_k;
  pl->blocks_per_sm = per_sm;
  pl->max_contrib = t.split_k;
  if (t.stream_k > 0) {
    // balanced split-K: whole tiles data-parallel for all but the last full
    // wave, then G CTAs share the remaining I = tiles x K-tiles iterations;
    // CTA c owns [floor(c I/G), floor((c+1) I/G)) of them; a split tile has
    // as many partial sums as CTAs whose ranges overlap it
    long long G = static_cast<long long>(sms) * std::min(per_sm, t.stream_k);
    if (G > tiles * pl->k_tiles) G = tiles * pl->k_tiles;
    const long long dp = G > 0 ? eg::stream_dp_tiles(tiles, G) : 0;
    const long long iters = (tiles - dp) * pl->k_tiles;
    pl->grid = static_cast<int>(G);
    pl->units = static_cast<int>(std::min<long long>(dp + iters, INT32_MAX));
    int mc = 1;
    for (long long tile = 0; tile < tiles - dp && G > 0; ++tile) {
      const long long b = tile * pl->k_tiles, e2 = b + pl->k_tiles;
      const long long first = ((b + 1) * G - 1) / iters, last = (e2 * G - 1) / iters;
      mc = std::max(mc, static_cast<int>(last - first + 1));
    }
    pl->max_contrib = mc;
  } else if (t.cluster_reduce) {
    // one unit per CTA; the split_k CTAs of a tile form one cluster and the
    // partial sums never leave shared memory
    pl->grid = static_cast<int>(units);
    pl->units = static_cast<int>(units);
    pl->max_contrib = 1;
  } else if (t.cta_pair) {
    // persistent CTA pairs: one work slot per 2-CTA cluster
    const long long slots = static_cast<long long>(sms / 2) * per_sm;
    pl->grid = 2 * static_cast<int>(units < slots ? units : slots);
    pl->units = static_cast<int>(units);
  } else {
    const long long slots = static_cast<long long>(sms) * per_sm;
    pl->grid = static_cast<int>(units < slots ? units : slots);
    pl->units = static_cast<int>(units);
  }
}

eg_status encode_map(CUtensorMap* m, const void* base, int dtype, int64_t rows, int64_t K,
                     int64_t ld, int box_k, int box_rows) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return fail(EG_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
  const int eb = elt_bytes(dtype);
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(K), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(ld * eb)};
  cuuint32_t box[2] = {static_cast<cuuint32_t>(box_k), static_cast<cuuint32_t>(box_rows)};
  cuuint32_t estr[2] = {1, 1};
  const CUtensorMapDataType dt =
      dtype == EG_IN_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_UINT8;
  CUresult r = fn(m, dt, 2, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS)
    return fail(EG_ERR_INVALID_ARG, "cuTensorMapEncodeTiled failed (%d) for rows=%lld K=%lld ld=%lld",
                static_cast<int>(r), (long long)rows, (long long)K, (long long)ld);
  return EG_OK;
}

// Tensor map of a 2-byte output Y [M][ldy] for the epilogue's staged
// stores: boxes of `cw` columns x 32 rows, swizzled as the kernel writes its
// staging boxes (64-byte rows for 32 columns, 32-byte rows for 16).
eg_status encode_ymap(CUtensorMap* m, const void* Y, int64_t M, int64_t N, int64_t ldy, int cw) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return fail(EG_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(N), static_cast<cuuint64_t>(M)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(ldy * 2)};
  cuuint32_t box[2] = {static_cast<cuuint32_t>(cw), 32u};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT16, 2, const_cast<void*>(Y), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE,
                  cw == 32 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_32B,
                  CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS)
    return fail(EG_ERR_INVALID_ARG, "cuTensorMapEncodeTiled failed (%d) for Y (M=%lld N=%lld ldy=%lld)",
                static_cast<int>(r), (long long)M, (long long)N, (long long)ldy);
  return EG_OK;
}

bool overlaps(const void* a, size_t an, const void* b, size_t bn) {
  if (!a || !b || an == 0 || bn == 0) return false;
  const uintptr_t a0 = reinterpret_cast<uintptr_t>(a), b0 = reinterpret_cast<uintptr_t>(b);
  return a0 < b0 + bn && b0 < a0 + an;
}

eg_status validate_args_for(const eg_problem& p, const eg_args* a, bool debug_out) {
  if (!a) return fail(EG_ERR_INVALID_ARG, "args is NULL");
  if (p.M == 0 || p.N == 0) return EG_OK;
  const int eb = elt_bytes(p.dtype);
  if (!a->Y) return fail(EG_ERR_INVALID_ARG, "Y is NULL");
  if (p.K > 0 && (!a->A || !a->W)) return fail(EG_ERR_INVALID_ARG, "A or W is NULL");
  const bool quant_a = (p.flags & EG_RUN_QUANT_A) != 0;  // A holds bf16 activations
  if (p.K > 0) {
    if (!aligned16(a->W) || (!quant_a && !aligned16(a->A)))
      return fail(EG_ERR_INVALID_ARG, "A and W must be 16-byte aligned");
    if (quant_a && (reinterpret_cast<uintptr_t>(a->A) & 1u))
      return fail(EG_ERR_INVALID_ARG, "bf16 A must be 2-byte aligned");
    if (a->lda < p.K || a->ldw < p.K)
      return fail(EG_ERR_INVALID_ARG, "lda/ldw must be >= K");
    if ((!quant_a && (a->lda * eb) % 16) || (a->ldw * eb) % 16)
      return fail(EG_ERR_INVALID_ARG, "lda and ldw must be multiples of 16 bytes");
  }
  if (p.scale != EG_SCALE_NONE) {
    if ((!quant_a && !a->s_a) || !a->s_w) return fail(EG_ERR_INVALID_ARG, "scaled modes need s_a and s_w");
    if ((!quant_a && !aligned16(a->s_a)) || !aligned16(a->s_w))
      return fail(EG_ERR_INVALID_ARG, "s_a and s_w must be 16-byte aligned");
  }
  const int esz = out_elt_bytes(p.flags);
  if (reinterpret_cast<uintptr_t>(a->Y) % esz)
    return fail(EG_ERR_INVALID_ARG, "Y must be aligned to its element size");
  if (p.flags & EG_OUT_E4M3) {
    if (!a->s_y || (reinterpret_cast<uintptr_t>(a->s_y) & 3u))
      return fail(EG_ERR_INVALID_ARG, "EG_OUT_E4M3 needs s_y, 4-byte aligned");
  }
  if (a->ldy < p.N) return fail(EG_ERR_INVALID_ARG, "ldy must be >= N");
  if (!debug_out && (p.flags & EG_EPI_BIAS)) {
    if (!a->bias) return fail(EG_ERR_INVALID_ARG, "EG_EPI_BIAS needs bias");
    if (!aligned16(a->bias)) return fail(EG_ERR_INVALID_ARG, "bias must be 16-byte aligned");
  }
  const bool res = (p.flags & (EG_EPI_RESIDUAL | EG_EPI_RESIDUAL_PRE_ACT)) != 0;
  if (!debug_out && res) {
    if (!a->residual) return fail(EG_ERR_INVALID_ARG, "a residual flag needs residual");
    if (reinterpret_cast<uintptr_t>(a->residual) % 2)
      return fail(EG_ERR_INVALID_ARG, "residual must be 2-byte aligned");
    if (a->ldr < p.N) return fail(EG_ERR_INVALID_ARG, "ldr must be >= N");
  }
  const size_t ybytes = size_t(p.M - 1) * size_t(a->ldy) * esz + size_t(p.N) * esz;
  const int ab = quant_a ? 2 : eb;
  if (overlaps(a->Y, ybytes, a->A, size_t(p.M - 1) * a->lda * ab + size_t(p.K) * ab) ||
      overlaps(a->Y, ybytes, a->W,
               size_t((p.flags & EG_EPI_GATED) ? 2 * p.N - 1 : p.N - 1) * a->ldw * eb + size_t(p.K) * eb) ||
      (res && !debug_out &&
       overlaps(a->Y, ybytes, a->residual, size_t(p.M - 1) * a->ldr * 2 + size_t(p.N) * 2)))
    return fail(EG_ERR_INVALID_ARG, "Y must not alias A, W or the residual");
  return EG_OK;
}

eg_status validate_args(const eg_plan* pl, const eg_args* a, bool debug_out) {
  return validate_args_for(pl->prob, a, debug_out);
}

eg_status ensure_maps(eg_plan* pl, const eg_args* a) {
  const eg_problem& p = pl->prob;
  if (p.K == 0) return EG_OK;
  if (pl->maps_valid && pl->mapA == a->A && pl->mapW == a->W && pl->map_lda == a->lda &&
      pl->map_ldw == a->ldw)
    return EG_OK;
  const int box_k = pl->ke.elems_per_stage;
  const int bn = pl->tune.tile_n;
  CUtensorMap mA, mW;
  eg_status s;
  const bool swap = pl->tune.swap_ab != 0;
  if ((s = encode_map(&mA, a->A, p.dtype, p.M, p.K, a->lda, box_k, swap ? bn : 128)) != EG_OK) return s;
  const int64_t wrows = (p.flags & EG_EPI_GATED) ? 2 * p.N : p.N;  // gated: gate + up halves
  // CTA pairs: each CTA loads half of the weight tile
  const int wbox = swap ? 128 : (pl->tune.cta_pair ? bn / 2 : bn);
  if ((s = encode_map(&mW, a->W, p.dtype, wrows, p.K, a->ldw, box_k, wbox)) != EG_OK) return s;
  pl->tmP = swap ? mW : mA;
  pl->tmQ = swap ? mA : mW;
  pl->mapA = a->A;
  pl->mapW = a->W;
  pl->map_lda = a->lda;
  pl->map_ldw = a->ldw;
  pl->maps_valid = true;
  return EG_OK;
}

// Staged TMA stores for this run's Y: the plan reserved the staging boxes,
// the output is bf16 / fp16 (not the debug accumulators) and Y and its row
// stride are 16-byte aligned.  Encodes (and caches) Y's tensor map.
eg_status ensure_ymap(eg_plan* pl, void* Y, int64_t ldy, uint32_t kflags, bool* use) {
  const eg_problem& p = pl->prob;
  *use = pl->stage_ok && !(kflags & eg::F_DEBUG) && !(p.flags & EG_OUT_E4M3) && aligned16(Y) &&
         (ldy * 2) % 16 == 0;
  if (!*use) return EG_OK;
  if (pl->mapY == Y && pl->map_ldy == ldy) return EG_OK;
  eg_status s = encode_ymap(&pl->tmY, Y, p.M, p.N, ldy, pl->ke.cw);
  if (s != EG_OK) return s;
  pl->mapY = Y;
  pl->map_ldy = ldy;
  return EG_OK;
}

eg::KParams make_params(const eg_plan* pl, const eg_args* a, int act, uint32_t flags, void* Y,
                        int64_t ldy) {
  const eg_problem& p = pl->prob;
  eg::KParams k{};
  k.M = static_cast<int32_t>(p.M);
  k.N = static_cast<int32_t>(p.N);
  k.K = static_cast<int32_t>(p.K);
  k.rows = pl->rows;
  k.cols = pl->cols;
  k.tiles_rows = pl->tiles_rows;
  k.tiles_cols = pl->tiles_cols;
  k.k_tiles = pl->k_tiles;
  k.split_k = pl->tune.split_k;
  k.stream_k = pl->tune.stream_k > 0 ? 1 : 0;
  k.max_contrib = pl->max_contrib;
  k.stages = pl->tune.stages;
  k.act = act;
  k.flags = flags;
  k.kb_count = pl->kb_count;
  k.s_a = a->s_a;
  k.s_w = a->s_w;
  k.bias = static_cast<const __nv_bfloat16*>(a->bias);
  k.R = static_cast<const __nv_bfloat16*>(a->residual);
  k.ldr = a->ldr;
  k.Y = Y;
  k.ldy = ldy;
  k.ws = static_cast<float*>(pl->ws);
  k.counters = pl->counters;
  k.status = pl->status;
  k.wait_limit_ns = pl->wait_limit_ns;
  k.stall_producer = pl->stall;
  const bool res = (flags & (eg::F_RES | eg::F_RES_PRE)) != 0;
  const int yb = (flags & eg::F_DEBUG) ? 4 : out_elt_bytes(p.flags);
  k.vec_ok = aligned16(Y) && (ldy * yb) % 16 == 0 &&
             (!res || (aligned16(a->residual) && (a->ldr * 2) % 16 == 0));
  k.out = (p.flags & EG_OUT_F16) ? eg::OUT_F16 : (p.flags & EG_OUT_E4M3) ? eg::OUT_E4M3 : eg::OUT_BF16;
  k.s_y = a->s_y;
  k.pdl = (p.flags & EG_RUN_PDL) ? 1 : 0;
  k.l2_prefetch = pl->l2_prefetch;
  k.commit_group = pl->commit_group;
  k.acc_release = pl->acc_release;
  k.trace = pl->trace;
  k.trace_ctas = pl->trace_ctas;
  k.cluster_reduce = pl->tune.cluster_reduce;
  k.out_stage_off = pl->out_stage_off;
  // streamed weights: hint L2 to evict them first when the grid reads each
  // weight tile once (one tile column / row over the tokens)
  const bool w_once = pl->tune.swap_ab ? (pl->tiles_cols == 1) : (pl->tiles_rows == 1);
  k.evict_first_p = pl->tune.swap_ab ? w_once : 0;
  k.evict_first_q = pl->tune.swap_ab ? 0 : w_once;
  return k;
}

// Ring stages the UMMA issuer releases with one commit.  A tcgen05.commit
// stalls the tensor pipe for a few hundred cycles unless enough UMMAs are
// queued behind it (measured on GB300 with back-to-back 128 x 256 UMMAs: 4
// per commit run at ~61% of the UMMA rate, 8 at ~81%, 16 at ~97%).
// Releasing stages in pairs halves the commits but hands the producer two
// stages at a time, which exposes the load latency in a 4-stage ring; with
// the 6-stage rings of CTA pairs it pays (bf16 prefill 4096^3: 111 -> 105
// us).  So: pairs of stages for CTA pairs with an even ring of 6 or more,
// else one stage per commit.  Promotion (block scales, INT8) commits its
// accumulator per K block anyway.  EG_COMMIT_GROUP=n overrides (n must
// divide the stages).
int commit_group_for(const eg_problem& p, const eg_tuning& t) {
  const bool promote = p.scale == EG_SCALE_BLOCK || p.dtype == EG_IN_INT8;
  if (promote) return 1;
  int g = (t.cta_pair && t.stages >= 6 && t.stages % 2 == 0) ? 2 : 1;
  if (const char* e = getenv("EG_COMMIT_GROUP")) {
    const int v = atoi(e);
    if (v >= 1 && v <= t.stages && t.stages % v == 0) g = v;
  }
  return g;
}

// Promotion commits each K block's accumulator (4 accumulator buffers); that
// commit also says the block's UMMAs have read their ring stage (block
// scales) or fp16 operand slot (INT8), so the stage / slot needs no commit
// of its own.  A stage is then freed S blocks later, which is safe while S
// <= 4 (the accumulator buffer's next commit cannot have happened yet).
int acc_release_for(const eg_problem& p, const eg_tuning& t) {
  if (const char* e = getenv("EG_ACC_RELEASE"))
    if (atoi(e) == 0) return 0;
  if (p.dtype == EG_IN_INT8) return 1;
  // (a stage may wait for the commit of the K block S blocks back only while
  // S is at most the accumulator buffers: four, or two for 256-wide tiles)
  if (p.scale == EG_SCALE_BLOCK) return t.stages <= (!t.swap_ab && t.tile_n > 128 ? 2 : 4) ? 1 : 0;
  return 0;
}

uint32_t epi_flags(uint32_t f) {
  uint32_t k = 0;
  if (f & EG_EPI_BIAS) k |= eg::F_BIAS;
  if (f & EG_EPI_RESIDUAL) k |= eg::F_RES;
  if (f & EG_EPI_RESIDUAL_PRE_ACT) k |= eg::F_RES_PRE;
  if (f & EG_OUT_DEBUG_ACCUM) k |= eg::F_DEBUG;
  return k;
}

eg_status launch_fused(eg_plan* pl, const eg::KParams& kp, cudaStream_t st) {
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(pl->grid);
  cfg.blockDim = dim3(pl->ke.threads);
  cfg.dynamicSmemBytes = pl->smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  unsigned n = 0;
  if (kp.pdl) {
    attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[n].val.programmaticStreamSerializationAllowed = 1;
    ++n;
  }
  if (kp.cluster_reduce || pl->tune.cta_pair) {
    // the split_k CTAs of a tile, or a CTA pair (consecutive blocks), form
    // one cluster
    attr[n].id = cudaLaunchAttributeClusterDimension;
    attr[n].val.clusterDim.x = pl->tune.cta_pair ? 2u : static_cast<unsigned>(kp.split_k);
    attr[n].val.clusterDim.y = 1;
    attr[n].val.clusterDim.z = 1;
    ++n;
  }
  cfg.attrs = attr;
  cfg.numAttrs = n;
  void* args[4] = {const_cast<CUtensorMap*>(&pl->tmP), const_cast<CUtensorMap*>(&pl->tmQ),
                   const_cast<CUtensorMap*>(&pl->tmY), const_cast<eg::KParams*>(&kp)};
  EG_CUDA(cudaLaunchKernelExC(&cfg, pl->ke.fn, args), "launching the fused kernel");
  return EG_OK;
}

}  // namespace

// --------------------------------------------------------- elementwise ----
// Kernels of the unfused comparison path (8 bf16 per thread, 16-byte access).

namespace eg {

__device__ __forceinline__ float bf(uint16_t b) { return __uint_as_float(uint32_t(b) << 16); }

// T2 = T1 + bias (+ R when the residual comes before the activation)
__global__ void unfused_bias_kernel(const __nv_bfloat16* T1, const __nv_bfloat16* bias,
                                    const __nv_bfloat16* R, int64_t ldr, __nv_bfloat16* T2,
                                    int64_t M, int64_t N, int has_bias, int res_pre) {
  const int64_t nv = N / 8;
  const int64_t total = M * nv;
  for (int64_t v = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; v < total;
       v += int64_t(gridDim.x) * blockDim.x) {
    const int64_t m = v / nv, n = (v % nv) * 8;
    const uint4 t = *reinterpret_cast<const uint4*>(T1 + m * N + n);
    uint4 b = make_uint4(0, 0, 0, 0), r = make_uint4(0, 0, 0, 0);
    if (has_bias) b = *reinterpret_cast<const uint4*>(bias + n);
    if (res_pre) r = *reinterpret_cast<const uint4*>(R + m * ldr + n);
    const uint32_t tw[4] = {t.x, t.y, t.z, t.w}, bw[4] = {b.x, b.y, b.z, b.w},
                   rw[4] = {r.x, r.y, r.z, r.w};
    uint32_t o[4];
#pragma unroll
    for (int h = 0; h < 4; ++h) {
      uint16_t e[2];
#pragma unroll
      for (int q = 0; q < 2; ++q) {
        float x = bf(uint16_t(tw[h] >> (16 * q)));
        if (has_bias) x += bf(uint16_t(bw[h] >> (16 * q)));
        if (res_pre) x += bf(uint16_t(rw[h] >> (16 * q)));
        e[q] = __bfloat16_as_ushort(__float2bfloat16_rn(x));
      }
      o[h] = uint32_t(e[0]) | (uint32_t(e[1]) << 16);
    }
    *reinterpret_cast<uint4*>(T2 + m * N + n) = make_uint4(o[0], o[1], o[2], o[3]);
  }
}

// Y = act(T2) (+ R when the residual comes after the activation)
__global__ void unfused_act_kernel(const __nv_bfloat16* T2, const __nv_bfloat16* R, int64_t ldr,
                                   __nv_bfloat16* Y, int64_t ldy, int64_t M, int64_t N, int act,
                                   int res_post) {
  const int64_t nv = N / 8;
  const int64_t total = M * nv;
  for (int64_t v = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; v < total;
       v += int64_t(gridDim.x) * blockDim.x) {
    const int64_t m = v / nv, n = (v % nv) * 8;
    const uint4 t = *reinterpret_cast<const uint4*>(T2 + m * N + n);
    uint4 r = make_uint4(0, 0, 0, 0);
    if (res_post) r = *reinterpret_cast<const uint4*>(R + m * ldr + n);
    const uint32_t tw[4] = {t.x, t.y, t.z, t.w}, rw[4] = {r.x, r.y, r.z, r.w};
    uint32_t o[4];
#pragma unroll
    for (int h = 0; h < 4; ++h) {
      uint16_t e[2];
#pragma unroll
      for (int q = 0; q < 2; ++q) {
        float x = act_apply(act, bf(uint16_t(tw[h] >> (16 * q))));
        if (res_post) x += bf(uint16_t(rw[h] >> (16 * q)));
        e[q] = __bfloat16_as_ushort(__float2bfloat16_rn(x));
      }
      o[h] = uint32_t(e[0]) | (uint32_t(e[1]) << 16);
    }
    *reinterpret_cast<uint4*>(Y + m * ldy + n) = make_uint4(o[0], o[1], o[2], o[3]);
  }
}

}  // namespace eg

// ------------------------------------------------------------------ ABI ----

extern "C" {

const char* eg_status_string(eg_status s) {
  switch (s) {
    case EG_OK: return "EG_OK";
    case EG_ERR_INVALID_ARG: return "EG_ERR_INVALID_ARG";
    case EG_ERR_UNSUPPORTED: return "EG_ERR_UNSUPPORTED";
    case EG_ERR_NO_MEMORY: return "EG_ERR_NO_MEMORY";
    case EG_ERR_CUDA: return "EG_ERR_CUDA";
    case EG_ERR_DEVICE_TIMEOUT: return "EG_ERR_DEVICE_TIMEOUT";
    case EG_ERR_NOT_TUNED: return "EG_ERR_NOT_TUNED";
  }
  return "EG_ERR_UNKNOWN";
}

const char* eg_last_error_detail(void) { return g_detail.c_str(); }

eg_status eg_quantize_rows(const void* x, int64_t M, int64_t K, int64_t ldx, int32_t dtype,
                           void* q, int64_t ldq, float* s, void* stream) {
  if (M < 0 || K < 0 || M > INT32_MAX || K > INT32_MAX)
    return fail(EG_ERR_INVALID_ARG, "bad sizes M=%lld K=%lld", (long long)M, (long long)K);
  if (dtype != EG_IN_E4M3 && dtype != EG_IN_INT8)
    return fail(EG_ERR_INVALID_ARG, "eg_quantize_rows quantises to E4M3 or INT8 (dtype %d)", dtype);
  if (M == 0) return EG_OK;
  if (!s || (K > 0 && (!x || !q)))
    return fail(EG_ERR_INVALID_ARG, "x, q and s must be non-NULL");
  if (ldx < K || ldq < K) return fail(EG_ERR_INVALID_ARG, "ldx and ldq must be >= K");
  if (reinterpret_cast<uintptr_t>(x) & 1u) return fail(EG_ERR_INVALID_ARG, "x must be 2-byte aligned");
  EG_CUDA(eg::launch_quant_rows(x, M, K, ldx, dtype == EG_IN_E4M3, q, ldq, s,
                                static_cast<cudaStream_t>(stream), false),
          "launching the quantisation kernel");
  return EG_OK;
}

eg_status eg_plan_create(const eg_problem* problem, const eg_tuning* tuning, eg_plan** out) {
  if (!out) return fail(EG_ERR_INVALID_ARG, "out is NULL");
  *out = nullptr;
  eg_status s = validate_problem(problem);
  if (s != EG_OK) return s;
  // INT8 and Block_FP8 gated units: the plan's GEMM is the accumulator
  // output over all 2N weight rows; the combine kernel does the rest
  const bool two_pass = (problem->flags & EG_EPI_GATED) &&
                        (problem->dtype == EG_IN_INT8 || problem->scale == EG_SCALE_BLOCK);
  eg_problem inner = *problem;
  if (two_pass) {
    inner.N = 2 * problem->N;
    inner.act = EG_ACT_NONE;
    inner.flags = (problem->flags & (EG_RUN_PDL | EG_RUN_QUANT_A)) | EG_OUT_DEBUG_ACCUM;
  }
  const eg_problem& p = inner;

  // device checks come after the argument checks, so invalid problems are
  // rejected without touching the GPU
  int dev = -1;
  EG_CUDA(cudaGetDevice(&dev), "cudaGetDevice");
  int major = 0, minor = 0;
  EG_CUDA(cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev), "device query");
  EG_CUDA(cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev), "device query");
  if (major != 10 || minor != 3)
    return fail(EG_ERR_UNSUPPORTED, "the kernels are built for sm_103a; device %d is sm_%d%d", dev,
                major, minor);

  eg_tuning t{};
  // a two-kernel gated unit's GEMM takes the rows of the plain layer of the
  // same K and per-half N (the weight stream per output is twice as long,
  // the shape of the work per tile is the same)
  eg_problem key = p;
  if (two_pass) {
    key = *problem;
    key.flags &= ~static_cast<uint32_t>(EG_EPI_GATED);
  }
  if (tuning) {
    t = *tuning;
  } else if (!eg::tuning_lookup(key, sm_count_of(dev), &t)) {
    return fail(EG_ERR_NOT_TUNED, "no tuning entry or default for this problem");
  }
  eg::KernelEntry ke;
  uint32_t smem = 0;
  int k_tiles = 0;
  if ((s = validate_tuning(p, t, &ke, &smem, &k_tiles)) != EG_OK) return s;

  eg_plan* pl = new eg_plan();
  pl->prob = p;
  pl->tune = t;
  pl->device = dev;
  pl->ke = ke;
  pl->smem = smem;
  pl->k_tiles = k_tiles;
  pl->kb_count = static_cast<int>(p.K / 128);
  const bool swap = t.swap_ab != 0;
  pl->rows = static_cast<int>(swap ? p.N : p.M);
  pl->cols = static_cast<int>(swap ? p.M : p.N);
  pl->tiles_rows = t.cta_pair ? (pl->rows + 255) / 256 : (pl->rows + 127) / 128;
  pl->tiles_cols = (pl->cols + t.tile_n - 1) / t.tile_n;
  pl->wait_limit_ns = default_wait_limit_ns();
  if (const char* e2 = getenv("EG_PDL_L2_PREFETCH")) pl->l2_prefetch = atoi(e2) != 0;
  pl->commit_group = commit_group_for(p, t);
  pl->acc_release = acc_release_for(p, t);
  auto cleanup = [&](eg_status st) {
    eg_plan_destroy(pl);
    return st;
  };
  // The attribute belongs to the kernel function, which plans with other
  // ring depths share: allow the device maximum (each launch still passes
  // its own size), so that a later plan cannot shrink an earlier one's limit.
  cudaError_t e = cudaFuncSetAttribute(ke.fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(kMaxSmem));
  if (e != cudaSuccess) return cleanup(cuda_fail(e, "cudaFuncSetAttribute"));
  // operands arrive through TMA into shared memory: prefer the largest
  // shared-memory carveout so that several CTAs can be resident per SM
  e = cudaFuncSetAttribute(ke.fn, cudaFuncAttributePreferredSharedMemoryCarveout,
                           cudaSharedmemCarveoutMaxShared);
  if (e != cudaSuccess) return cleanup(cuda_fail(e, "setting the shared-memory carveout"));
  plan_staging(pl, dev);
  int per_sm = 0;
  if ((s = residency(pl, dev, &per_sm)) != EG_OK) return cleanup(s);
  plan_grid(pl, sm_count_of(dev), per_sm);
  const size_t tiles = size_t(pl->tiles_rows) * pl->tiles_cols;
  if (pl->max_contrib > 1 && tiles > 0) {
    pl->ws_bytes = size_t(pl->max_contrib) * tiles * size_t(ke.acc_n) * 128 * 4;
    if ((e = cudaMalloc(&pl->ws, pl->ws_bytes)) != cudaSuccess)
      return cleanup(cuda_fail(e, "allocating the split-K workspace"));
    // INT8 accumulates its splits into slot 0 of each tile, which the kernel
    // keeps at zero between calls; it starts at zero here
    if ((e = cudaMemset(pl->ws, 0, pl->ws_bytes)) != cudaSuccess)
      return cleanup(cuda_fail(e, "zeroing the split-K workspace"));
  }
  if ((p.flags & EG_RUN_QUANT_A) && p.M > 0) {
    pl->ldq = (p.K + 15) / 16 * 16;  // 16-byte rows for the TMA loads
    if ((e = cudaMalloc(&pl->qa, size_t(p.M) * size_t(pl->ldq > 0 ? pl->ldq : 16))) != cudaSuccess ||
        (e = cudaMalloc(reinterpret_cast<void**>(&pl->qs), size_t(p.M) * sizeof(float))) != cudaSuccess)
      return cleanup(cuda_fail(e, "allocating the quantised activations"));
  }
  if ((e = cudaMalloc(reinterpret_cast<void**>(&pl->counters), (tiles + 1) * sizeof(int))) !=
          cudaSuccess ||
      (e = cudaMalloc(reinterpret_cast<void**>(&pl->status), sizeof(int))) != cudaSuccess)
    return cleanup(cuda_fail(e, "allocating plan counters"));
  if ((e = cudaMemset(pl->counters, 0, (tiles + 1) * sizeof(int))) != cudaSuccess ||
      (e = cudaMemset(pl->status, 0, sizeof(int))) != cudaSuccess ||
      (e = cudaDeviceSynchronize()) != cudaSuccess)
    return cleanup(cuda_fail(e, "zeroing plan counters"));
  pl->two_pass_gated = two_pass;
  pl->user = *problem;
  if (two_pass && p.M > 0 && p.N > 0 &&
      (e = cudaMalloc(reinterpret_cast<void**>(&pl->gacc), size_t(p.M) * size_t(p.N) * 4u)) != cudaSuccess)
    return cleanup(cuda_fail(e, "allocating the gated unit's accumulators"));
  *out = pl;
  return EG_OK;
}

eg_status eg_plan_workspace_bytes(const eg_plan* plan, size_t* out) {
  if (!plan || !out) return fail(EG_ERR_INVALID_ARG, "NULL argument");
  *out = plan->ws_bytes + (plan->gacc ? size_t(plan->prob.M) * size_t(plan->prob.N) * 4u : 0u);
  return EG_OK;
}

eg_status eg_plan_get_tuning(const eg_plan* plan, eg_tuning* out) {
  if (!plan || !out) return fail(EG_ERR_INVALID_ARG, "NULL argument");
  *out = plan->tune;
  return EG_OK;
}

int32_t eg_plan_last_launch_count(const eg_plan* plan) { return plan ? plan->last_launches : 0; }

eg_status eg_plan_get_launch(const eg_plan* plan, eg_launch_info* out) {
  if (!plan || !out) return fail(EG_ERR_INVALID_ARG, "NULL argument");
  out->grid = plan->grid;
  out->block = plan->ke.threads;
  out->smem_bytes = static_cast<int32_t>(plan->smem);
  out->units = plan->units;
  out->blocks_per_sm = plan->blocks_per_sm;
  out->regs_per_thread = plan->regs;
  return EG_OK;
}

eg_status eg_plan_set_trace(eg_plan* plan, uint64_t* trace, int32_t trace_ctas) {
  if (!plan) return fail(EG_ERR_INVALID_ARG, "plan is NULL");
  if (trace && (trace_ctas < 0 || (reinterpret_cast<uintptr_t>(trace) & 7u)))
    return fail(EG_ERR_INVALID_ARG, "trace must be 8-byte aligned with trace_ctas >= 0");
  plan->trace = trace;
  plan->trace_ctas = trace ? trace_ctas : 0;
  // graphs captured earlier hold the old parameters
  for (auto& g : plan->graphs) cudaGraphExecDestroy(g.exec);
  plan->graphs.clear();
  return EG_OK;
}

eg_status eg_plan_set_test_stall(eg_plan* plan, uint64_t wait_limit_ns, int32_t stall_producer) {
  if (!plan) return fail(EG_ERR_INVALID_ARG, "plan is NULL");
  plan->wait_limit_ns = wait_limit_ns ? wait_limit_ns : default_wait_limit_ns();
  if (stall_producer < 0 || stall_producer > 2)
    return fail(EG_ERR_INVALID_ARG, "stall_producer must be 0, 1 or 2 (got %d)", stall_producer);
  plan->stall = stall_producer;
  return EG_OK;
}

static eg_status run_gemm(eg_plan* pl, const eg_args* a, cudaStream_t st) {
  const eg_problem& p = pl->prob;
  eg_args q;
  if (p.flags & EG_RUN_QUANT_A) {
    // prologue: per-token codes and scales of the bf16 activations, then
    // the GEMM on them (its programmatic dependent)
    EG_CUDA(eg::launch_quant_rows(a->A, p.M, p.K, a->lda, p.dtype == EG_IN_E4M3, pl->qa, pl->ldq,
                                  pl->qs, st, (p.flags & EG_RUN_PDL) != 0),
            "launching the quantisation kernel");
    q = *a;
    q.A = pl->qa;
    q.lda = pl->ldq;
    q.s_a = pl->qs;
    a = &q;
  }
  eg_status s = ensure_maps(pl, a);
  if (s != EG_OK) return s;
  bool ts = false;
  if ((s = ensure_ymap(pl, a->Y, a->ldy, epi_flags(p.flags), &ts)) != EG_OK) return s;
  eg::KParams kp = make_params(pl, a, p.act, epi_flags(p.flags), a->Y, a->ldy);
  kp.tma_store = ts ? 1 : 0;
  if (p.flags & EG_RUN_QUANT_A) kp.pdl = 1;
  return launch_fused(pl, kp, st);
}

// INT8 / Block_FP8 gated unit: the accumulators of the 2N weight rows, then
// the combine kernel (a programmatic dependent of the GEMM with EG_RUN_PDL).
static eg_status run_two_pass_gated(eg_plan* pl, const eg_args* a, cudaStream_t st) {
  const eg_problem& u = pl->user;
  eg_args q = *a;
  q.Y = pl->gacc;
  q.ldy = 2 * u.N;
  q.bias = nullptr;
  q.residual = nullptr;
  q.ldr = 0;
  q.s_y = nullptr;
  eg_status s = run_gemm(pl, &q, st);
  if (s != EG_OK) return s;
  const uint32_t fl = ((u.flags & EG_EPI_BIAS) ? uint32_t(eg::F_BIAS) : 0u) |
                      ((u.flags & EG_EPI_RESIDUAL) ? uint32_t(eg::F_RES) : 0u);
  const int out = (u.flags & EG_OUT_F16) ? eg::OUT_F16 : (u.flags & EG_OUT_E4M3) ? eg::OUT_E4M3 : eg::OUT_BF16;
  const float* s_a = (u.flags & EG_RUN_QUANT_A) ? pl->qs : a->s_a;
  EG_CUDA(eg::launch_gated_combine(pl->gacc, u.M, u.N, u.dtype == EG_IN_INT8, s_a, a->s_w, a->bias,
                                   a->residual, a->ldr, a->Y, a->ldy, u.act, fl, out, a->s_y, st,
                                   (u.flags & EG_RUN_PDL) != 0),
          "launching the gated combine kernel");
  return EG_OK;
}

static eg_status run_direct(eg_plan* pl, const eg_args* a, cudaStream_t st) {
  return pl->two_pass_gated ? run_two_pass_gated(pl, a, st) : run_gemm(pl, a, st);
}

eg_status eg_plan_run(eg_plan* plan, const eg_args* args, void* stream) {
  if (!plan) return fail(EG_ERR_INVALID_ARG, "plan is NULL");
  const eg_problem& p = plan->two_pass_gated ? plan->user : plan->prob;
  eg_status s = validate_args_for(p, args, (p.flags & EG_OUT_DEBUG_ACCUM) != 0);
  if (s != EG_OK) return s;
  plan->last_launches = 0;
  if (p.M == 0 || p.N == 0) return EG_OK;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int launches = ((p.flags & EG_RUN_QUANT_A) ? 2 : 1) + (plan->two_pass_gated ? 1 : 0);
  if (!(p.flags & EG_RUN_GRAPH)) {
    if ((s = run_direct(plan, args, st)) != EG_OK) return s;
    plan->last_launches = launches;
    return EG_OK;
  }
  // graph mode: one captured graph per distinct argument set, the most
  // recently used first; at most kGraphCache of them are kept
  for (size_t i = 0; i < plan->graphs.size(); ++i) {
    if (memcmp(&plan->graphs[i].args, args, sizeof(eg_args)) == 0) {
      if (i > 0) std::rotate(plan->graphs.begin(), plan->graphs.begin() + i, plan->graphs.begin() + i + 1);
      EG_CUDA(cudaGraphLaunch(plan->graphs[0].exec, st), "cudaGraphLaunch");
      plan->last_launches = launches;
      return EG_OK;
    }
  }
  if (!plan->cap_stream)
    EG_CUDA(cudaStreamCreateWithFlags(&plan->cap_stream, cudaStreamNonBlocking), "creating the capture stream");
  EG_CUDA(cudaStreamBeginCapture(plan->cap_stream, cudaStreamCaptureModeThreadLocal), "begin capture");
  s = run_direct(plan, args, plan->cap_stream);
  cudaGraph_t graph = nullptr;
  cudaError_t e = cudaStreamEndCapture(plan->cap_stream, &graph);
  if (s != EG_OK) {
    if (graph) cudaGraphDestroy(graph);
    return s;
  }
  if (e != cudaSuccess) return cuda_fail(e, "end capture");
  cudaGraphExec_t exec = nullptr;
  e = cudaGraphInstantiate(&exec, graph, 0);
  cudaGraphDestroy(graph);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGraphInstantiate");
  if (plan->graphs.size() >= kGraphCache) {
    // the least recently used graph goes; work it queued earlier keeps
    // running (a graph exec may be destroyed while its launches are pending)
    cudaGraphExecDestroy(plan->graphs.back().exec);
    plan->graphs.pop_back();
  }
  plan->graphs.insert(plan->graphs.begin(), GraphEntry{*args, exec});
  EG_CUDA(cudaGraphLaunch(exec, st), "cudaGraphLaunch");
  plan->last_launches = launches;
  return EG_OK;
}

eg_status eg_plan_run_unfused(eg_plan* plan, const eg_args* args, void* T1, void* T2,
                              void* stream) {
  if (!plan) return fail(EG_ERR_INVALID_ARG, "plan is NULL");
  const eg_problem& p = plan->prob;
  if (p.flags & EG_OUT_DEBUG_ACCUM)
    return fail(EG_ERR_INVALID_ARG, "the unfused path has no debug output mode");
  if (p.flags & EG_RUN_QUANT_A)
    return fail(EG_ERR_UNSUPPORTED, "the unfused path takes quantised A (no EG_RUN_QUANT_A)");
  if (p.flags & (EG_OUT_F16 | EG_OUT_E4M3))
    return fail(EG_ERR_UNSUPPORTED, "the unfused path writes bf16 only");
  if ((p.flags & EG_EPI_GATED) || plan->two_pass_gated)
    return fail(EG_ERR_UNSUPPORTED, "the unfused path has no gated unit");
  eg_status s = validate_args(plan, args, false);
  if (s != EG_OK) return s;
  plan->last_launches = 0;
  if (p.M == 0 || p.N == 0) return EG_OK;
  if (!T1 || !T2 || !aligned16(T1) || !aligned16(T2))
    return fail(EG_ERR_INVALID_ARG, "T1 and T2 must be non-NULL and 16-byte aligned");
  if (p.N % 8) return fail(EG_ERR_UNSUPPORTED, "the unfused path needs N %% 8 == 0");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if ((s = ensure_maps(plan, args)) != EG_OK) return s;
  // 1) the same GEMM kernel with no epilogue terms: T1 = bf16(scaled acc)
  bool ts = false;
  if ((s = ensure_ymap(plan, T1, p.N, 0u, &ts)) != EG_OK) return s;
  eg::KParams kp = make_params(plan, args, eg::ACT_NONE, 0u, T1, p.N);
  kp.tma_store = ts ? 1 : 0;
  if ((s = launch_fused(plan, kp, st)) != EG_OK) return s;
  const int64_t nv = p.M * (p.N / 8);
  const int threads = 256;
  const int blocks = static_cast<int>((nv + threads - 1) / threads < 65535 ? (nv + threads - 1) / threads : 65535);
  const bool pre = (p.flags & EG_EPI_RESIDUAL_PRE_ACT) != 0;
  const bool post = (p.flags & EG_EPI_RESIDUAL) != 0;
  // 2) T2 = T1 + bias (+ R before the activation)
  eg::unfused_bias_kernel<<<blocks, threads, 0, st>>>(
      static_cast<const __nv_bfloat16*>(T1), static_cast<const __nv_bfloat16*>(args->bias),
      static_cast<const __nv_bfloat16*>(args->residual), args->ldr, static_cast<__nv_bfloat16*>(T2),
      p.M, p.N, (p.flags & EG_EPI_BIAS) ? 1 : 0, pre ? 1 : 0);
  EG_CUDA(cudaGetLastError(), "launching the unfused bias kernel");
  // 3) Y = act(T2) (+ R after the activation)
  eg::unfused_act_kernel<<<blocks, threads, 0, st>>>(
      static_cast<const __nv_bfloat16*>(T2), static_cast<const __nv_bfloat16*>(args->residual),
      args->ldr, static_cast<__nv_bfloat16*>(args->Y), args->ldy, p.M, p.N, p.act, post ? 1 : 0);
  EG_CUDA(cudaGetLastError(), "launching the unfused activation kernel");
  plan->last_launches = 3;
  return EG_OK;
}

eg_status eg_plan_device_status(eg_plan* plan) {
  if (!plan) return fail(EG_ERR_INVALID_ARG, "plan is NULL");
  EG_CUDA(cudaDeviceSynchronize(), "synchronising");
  int st = 0;
  EG_CUDA(cudaMemcpy(&st, plan->status, sizeof(int), cudaMemcpyDeviceToHost), "reading the status word");
  if (st != 0) {
    // A CTA that gave up on a wait left its split-K tiles unfinished: their
    // arrival counters hold partial counts (the last arriver resets a
    // counter, and it never came) and, for INT8, slot 0 of the workspace
    // holds partial sums (the last arriver re-zeroes it).  Reset both so the
    // plan's next run starts from the state eg_plan_create left.
    const size_t tiles = size_t(plan->tiles_rows) * plan->tiles_cols;
    EG_CUDA(cudaMemset(plan->counters, 0, (tiles + 1) * sizeof(int)), "resetting the tile counters");
    if (plan->ws) EG_CUDA(cudaMemset(plan->ws, 0, plan->ws_bytes), "resetting the split-K workspace");
    EG_CUDA(cudaMemset(plan->status, 0, sizeof(int)), "clearing the status word");
    EG_CUDA(cudaDeviceSynchronize(), "synchronising");
    static const char* where[] = {"", "load warp", "UMMA warp", "epilogue warps", "transform warps",
                                  "teardown"};
    return fail(EG_ERR_DEVICE_TIMEOUT, "a device pipeline wait ran past its limit (%s)",
                (st > 0 && st <= 5) ? where[st] : "unknown");
  }
  return EG_OK;
}

eg_status eg_plan_destroy(eg_plan* plan) {
  if (!plan) return EG_OK;
  if (plan->device >= 0) cudaDeviceSynchronize();
  for (auto& g : plan->graphs) cudaGraphExecDestroy(g.exec);
  if (plan->cap_stream) cudaStreamDestroy(plan->cap_stream);
  if (plan->ws) cudaFree(plan->ws);
  if (plan->qa) cudaFree(plan->qa);
  if (plan->qs) cudaFree(plan->qs);
  if (plan->counters) cudaFree(plan->counters);
  if (plan->status) cudaFree(plan->status);
  if (plan->gacc) cudaFree(plan->gacc);
  delete plan;
  return EG_OK;
}

}  // extern "C"

// --------------------------------------------- no-allocation entry point ---
//
// Some callers cannot allocate device memory on the path where they run the
// layer: code running inside a memory pool or arena that owns every byte of
// the device, allocators that must not be re-entered from within a call, or
// runtimes that forbid cudaMalloc after start-up.  eg_linear_noalloc serves
// them: it runs the same fused kernel, but the kernel's scratch (split-K
// partial sums, per-tile arrival counters and the device status word) lives
// in the fixed array below, which the library's module holds on every device
// that loads it, until the process exits.

namespace {

constexpr size_t kScratchCounterBytes = 64u * 1024u;          // arrival counters + status
constexpr size_t kScratchWorkspaceBytes = 4u * 1024u * 1024u;  // split-K partial sums
constexpr size_t kScratchCounters = kScratchCounterBytes / sizeof(int) - 1;  // last int: status

// Host code may not dereference this name: on the host it is only a stand-in
// for the device array.  The device address comes from cudaGetSymbolAddress.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchCounterBytes +
                                                                 kScratchWorkspaceBytes];

constexpr int kMaxDevices = 64;
std::mutex g_noalloc_mu;
void* g_noalloc_ptr[kMaxDevices] = {};

// Once per device, with that device current: the scratch array's address.
eg_status noalloc_scratch(int dev, void** out) {
  if (dev < 0 || dev >= kMaxDevices) return fail(EG_ERR_UNSUPPORTED, "device index %d out of range", dev);
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  if (!g_noalloc_ptr[dev]) {
    void* p = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress of the scratch array");
    g_noalloc_ptr[dev] = p;
  }
  *out = g_noalloc_ptr[dev];
  return EG_OK;
}

}  // namespace

extern "C" {

eg_status eg_linear_noalloc(const eg_problem* problem, const eg_tuning* tuning,
                            const eg_args* args, void* stream) {
  eg_status s = validate_problem(problem);
  if (s != EG_OK) return s;
  const eg_problem& p = *problem;
  if (p.flags & EG_RUN_GRAPH)
    return fail(EG_ERR_INVALID_ARG, "eg_linear_noalloc keeps no captured graphs (drop EG_RUN_GRAPH)");
  if ((p.flags & EG_EPI_GATED) && (p.dtype == EG_IN_INT8 || p.scale == EG_SCALE_BLOCK))
    return fail(EG_ERR_UNSUPPORTED, "INT8 and Block_FP8 gated units need an accumulator buffer: use a plan");
  if (p.flags & EG_RUN_QUANT_A)
    return fail(EG_ERR_UNSUPPORTED, "eg_linear_noalloc has no buffers for quantised activations "
                                    "(quantise with eg_quantize_rows first)");
  int dev = -1;
  EG_CUDA(cudaGetDevice(&dev), "cudaGetDevice");
  int major = 0, minor = 0;
  EG_CUDA(cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev), "device query");
  EG_CUDA(cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev), "device query");
  if (major != 10 || minor != 3)
    return fail(EG_ERR_UNSUPPORTED, "the kernels are built for sm_103a; device %d is sm_%d%d", dev,
                major, minor);
  eg_tuning t{};
  if (tuning) {
    t = *tuning;
  } else if (!eg::tuning_lookup(p, sm_count_of(dev), &t)) {
    return fail(EG_ERR_NOT_TUNED, "no tuning entry or default for this problem");
  }
  // A plan on the stack: it only carries the launch description to the
  // shared helpers; nothing in it allocates.
  eg_plan pl;
  uint32_t smem = 0;
  int k_tiles = 0;
  if ((s = validate_tuning(p, t, &pl.ke, &smem, &k_tiles)) != EG_OK) return s;
  pl.prob = p;
  pl.tune = t;
  pl.device = -1;  // not a created plan
  pl.smem = smem;
  pl.k_tiles = k_tiles;
  pl.kb_count = static_cast<int>(p.K / 128);
  const bool swap = t.swap_ab != 0;
  pl.rows = static_cast<int>(swap ? p.N : p.M);
  pl.cols = static_cast<int>(swap ? p.M : p.N);
  pl.tiles_rows = t.cta_pair ? (pl.rows + 255) / 256 : (pl.rows + 127) / 128;
  pl.tiles_cols = (pl.cols + t.tile_n - 1) / t.tile_n;
  pl.wait_limit_ns = default_wait_limit_ns();
  pl.commit_group = commit_group_for(p, t);
  pl.acc_release = acc_release_for(p, t);
  if ((s = validate_args(&pl, args, (p.flags & EG_OUT_DEBUG_ACCUM) != 0)) != EG_OK) return s;
  if (p.M == 0 || p.N == 0) return EG_OK;

  // work decomposition and scratch needs
  const size_t tiles = size_t(pl.tiles_rows) * pl.tiles_cols;
  plan_staging(&pl, dev);
  int per_sm = 0;
  if ((s = residency(&pl, dev, &per_sm)) != EG_OK) return s;
  plan_grid(&pl, sm_count_of(dev), per_sm);
  const size_t ws_need =
      pl.max_contrib > 1 ? size_t(pl.max_contrib) * tiles * size_t(pl.ke.acc_n) * 128 * 4 : 0;
  if (tiles > kScratchCounters || ws_need > kScratchWorkspaceBytes)
    return fail(EG_ERR_UNSUPPORTED,
                "problem needs %zu tile counters and %zu bytes of split-K scratch; "
                "eg_linear_noalloc holds %zu counters and %zu bytes",
                tiles, ws_need, kScratchCounters, kScratchWorkspaceBytes);

  void* scratch = nullptr;
  if ((s = noalloc_scratch(dev, &scratch)) != EG_OK) return s;
  int* counters = static_cast<int*>(scratch);
  pl.counters = counters;
  pl.status = counters + kScratchCounters;
  pl.ws = static_cast<unsigned char*>(scratch) + kScratchCounterBytes;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  EG_CUDA(cudaFuncSetAttribute(pl.ke.fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               static_cast<int>(kMaxSmem)),
          "cudaFuncSetAttribute");
  // as eg_plan_create does: the grid above counts on the largest
  // shared-memory carveout
  EG_CUDA(cudaFuncSetAttribute(pl.ke.fn, cudaFuncAttributePreferredSharedMemoryCarveout,
                               cudaSharedmemCarveoutMaxShared),
          "setting the shared-memory carveout");
  // the arrival counters and the status word start every call at zero (the
  // array keeps whatever the previous call left)
  EG_CUDA(cudaMemsetAsync(counters, 0, (tiles + 1) * sizeof(int), st), "clearing tile counters");
  EG_CUDA(cudaMemsetAsync(pl.status, 0, sizeof(int), st), "clearing the status word");
  // INT8 split-K adds every split into one zeroed slot per tile
  if (p.dtype == EG_IN_INT8 && pl.max_contrib > 1)
    EG_CUDA(cudaMemsetAsync(pl.ws, 0, tiles * size_t(pl.ke.acc_n) * 128 * 4, st),
            "clearing the INT8 split-K sums");
  if ((s = ensure_maps(&pl, args)) != EG_OK) return s;
  bool ts = false;
  if ((s = ensure_ymap(&pl, args->Y, args->ldy, epi_flags(p.flags), &ts)) != EG_OK) return s;
  eg::KParams kp = make_params(&pl, args, p.act, epi_flags(p.flags), args->Y, args->ldy);
  kp.tma_store = ts ? 1 : 0;
  return launch_fused(&pl, kp, st);
}

}  // extern "C"
