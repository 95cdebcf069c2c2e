// eg_registry.h -- host-side table of the fused kernel's instantiations.
#pragma once
#include <cstdint>

namespace eg {

struct KernelEntry {
  const void* fn = nullptr;      // __global__ function
  uint32_t stage_bytes = 0;      // shared memory per ring stage
  uint32_t fixed_bytes = 0;      // alignment slack + barriers + op_bytes
  uint32_t op_bytes = 0;         // INT8 fp16 operand slots (follow the ring)
  int threads = 0;
  int elems_per_stage = 0;       // K elements one stage covers
  int tmem_cols = 0;             // TMEM columns one CTA allocates
  int acc_n = 0;                 // accumulator columns per unit (gated: 2 tile_n)
  int regsplit_need = 0;         // registers a setmaxnreg split needs (0: none)
  int cw = 0;                    // epilogue chunk columns (staged store box width)
  int epi_warps = 0;             // epilogue warps (one pair of staging boxes each)
};

// Each returns false when bn has no instantiation for that kind and swap.
#define EG_DECLARE_LOOKUP(name)                      \
  bool name##_noswap(int bn, KernelEntry* out);      \
  bool name##_swap(int bn, KernelEntry* out);        \
  inline bool name(int swap, int bn, KernelEntry* out) { \
    return swap ? name##_swap(bn, out) : name##_noswap(bn, out); \
  }
EG_DECLARE_LOOKUP(lookup_bf16)
EG_DECLARE_LOOKUP(lookup_e4m3_tc)
EG_DECLARE_LOOKUP(lookup_e4m3_block)
EG_DECLARE_LOOKUP(lookup_int8_tc)
EG_DECLARE_LOOKUP(lookup_bf16_gated)
EG_DECLARE_LOOKUP(lookup_e4m3_tc_gated)
#undef EG_DECLARE_LOOKUP
// CTA-pair kernels (no swap-AB): bf16 and FP8 per-token/channel, and FP8
// block scales (256-wide promotion tiles).
bool lookup_bf16_pair(int bn, KernelEntry* out);
bool lookup_e4m3_tc_pair(int bn, KernelEntry* out);
bool lookup_e4m3_block_pair(int bn, KernelEntry* out);

}  // namespace eg

// Instantiation helpers used by the eg_kernels_*.cu files.
#define EG_KERNEL_ENTRY(IN, SC, SWAP, BN) EG_KERNEL_ENTRY_GP(IN, SC, SWAP, BN, false, false)
#define EG_KERNEL_ENTRY_G(IN, SC, SWAP, BN, G) EG_KERNEL_ENTRY_GP(IN, SC, SWAP, BN, G, false)
#define EG_KERNEL_ENTRY_GP(IN, SC, SWAP, BN, G, PR)                                    \
  do {                                                                                 \
    using C_ = ::eg::Cfg<IN, SC, SWAP, BN, G, PR>;                                     \
    out->fn = reinterpret_cast<const void*>(&::eg::fused_linear_kernel<IN, SC, SWAP, BN, G, PR>); \
    out->stage_bytes = C_::kStageBytes;                                                \
    out->fixed_bytes = 1024u + 512u + C_::kOpBytes;                                    \
    out->op_bytes = C_::kOpBytes;                                                      \
    out->threads = C_::kThreads;                                                       \
    out->elems_per_stage = C_::kElemsPerStage;                                         \
    out->tmem_cols = static_cast<int>(C_::kTmemCols);                                  \
    out->acc_n = C_::kAccN;                                                            \
    out->regsplit_need = C_::kRegSplitNeed;                                            \
    out->cw = C_::kCW;                                                                 \
    out->epi_warps = C_::kEpiWarps;                                                    \
    return true;                                                                       \
  } while (0)
