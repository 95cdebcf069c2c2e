// eg_kernels_block_pair.cu -- fused kernel instantiation for CTA pairs with
// block-scale promotion: IN_E4M3 / SC_BLOCK, swap_ab = 0, 256 x 256 tiles
// (each CTA promotes its 128 rows x 256 columns per 128-K block).
#include "eg_kernel.cuh"
#include "eg_registry.h"

namespace eg {

bool lookup_e4m3_block_pair(int bn, KernelEntry* out) {
  switch (bn) {
    case 256: EG_KERNEL_ENTRY_GP(IN_E4M3, SC_BLOCK, false, 256, false, true);
    default: return false;
  }
}

}  // namespace eg
