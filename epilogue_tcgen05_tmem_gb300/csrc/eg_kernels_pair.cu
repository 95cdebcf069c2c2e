// eg_kernels_pair.cu -- fused kernel instantiations for CTA pairs (one
// 256-row tile per 2-CTA cluster, pair UMMAs): bf16 and IN_E4M3 / SC_TC,
// swap_ab = 0, tile_n 128 and 256.
#include "eg_kernel.cuh"
#include "eg_registry.h"

namespace eg {

bool lookup_bf16_pair(int bn, KernelEntry* out) {
  switch (bn) {
    case 128: EG_KERNEL_ENTRY_GP(IN_BF16, SC_NONE, false, 128, false, true);
    case 256: EG_KERNEL_ENTRY_GP(IN_BF16, SC_NONE, false, 256, false, true);
    default: return false;
  }
}

bool lookup_e4m3_tc_pair(int bn, KernelEntry* out) {
  switch (bn) {
    case 128: EG_KERNEL_ENTRY_GP(IN_E4M3, SC_TC, false, 128, false, true);
    case 256: EG_KERNEL_ENTRY_GP(IN_E4M3, SC_TC, false, 256, false, true);
    default: return false;
  }
}

}  // namespace eg
