// eg_tuning.h -- per-shape tuning lookup: the offline sweep's table first,
// then a default rule.
#pragma once
#include "../../include/eg.h"

namespace eg {

// Epilogue classes the table keys its rows by: the plain fused layer (any
// bias / residual / activation / output format), the gated unit (two weight
// halves, two accumulators), and the layer behind the per-token
// quantisation prologue (its GEMM runs as the prologue kernel's
// programmatic dependent).
enum : int32_t { EPI_CLASS_PLAIN = 0, EPI_CLASS_GATED = 1, EPI_CLASS_QUANT = 2 };

int32_t epi_class_of(const eg_problem& p);

// One row of the swept table.  m_max is the token bucket the row was tuned
// at (1, 2, 4, 8, 16, 24, 32, 64, ..., 2048); rows with m_max == 0 cover
// every M above the largest bucket.  epi is the epilogue class.
struct TuningRow {
  int32_t dtype, scale;
  int64_t N, K;
  int32_t m_max, epi;
  int32_t tile_n, stages, split_k, swap_ab, stream_k, cluster_reduce, cta_pair;
};

// Fill *out for problem p on a device with `sms` SMs.  Returns false when
// neither the table nor the default rule applies.
bool tuning_lookup(const eg_problem& p, int sms, eg_tuning* out);

// The default rule on its own (used when the table has no row).
bool tuning_default(const eg_problem& p, int sms, eg_tuning* out);

// Shared memory the kernel uses beyond its ring for block scaling: buffers
// of (tile rows + weight block rows) x (K tiles rounded up to 4, + 4)
// floats, two without swap-AB (the current unit's block scales and the next
// unit's, in flight), one with.  A tile has one weight block row, or one
// per 128 columns when it is wider (rows over M).
inline uint64_t block_scale_smem_bytes(const eg_problem& p, int swap_ab, int tile_n,
                                       int elems_per_stage) {
  if (p.scale != EG_SCALE_BLOCK) return 0;
  const int64_t kt = (p.K + elems_per_stage - 1) / elems_per_stage;
  const int wrows = (!swap_ab && tile_n > 128) ? tile_n / 128 : 1;
  return (swap_ab ? 1u : 2u) * static_cast<uint64_t>((swap_ab ? tile_n : 128) + wrows) *
         static_cast<uint64_t>((kt + 3) / 4 * 4 + 4) * 4u;
}

}  // namespace eg
