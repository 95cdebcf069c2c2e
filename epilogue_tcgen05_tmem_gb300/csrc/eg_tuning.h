// eg_tuning.h -- per-shape tuning lookup: the offline sweep's table first,
// then a default rule.
#pragma once
#include "../../include/eg.h"

namespace eg {

// One row of the swept table.  m_max is the token bucket (1,2,4,8,16,24,32)
// the row was tuned at; rows with m_max == 0 cover every M above 32.
struct TuningRow {
  int32_t dtype, scale;
  int64_t N, K;
  int32_t m_max;
  int32_t tile_n, stages, split_k, swap_ab, stream_k;
};

// Fill *out for problem p on a device with `sms` SMs.  Returns false when
// neither the table nor the default rule applies.
bool tuning_lookup(const eg_problem& p, int sms, eg_tuning* out);

// The default rule on its own (used when the table has no row).
bool tuning_default(const eg_problem& p, int sms, eg_tuning* out);

}  // namespace eg
