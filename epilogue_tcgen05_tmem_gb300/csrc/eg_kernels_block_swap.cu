// eg_kernels_block_swap.cu -- fused kernel instantiations,
// IN_E4M3 / SC_BLOCK, swap_ab = 1.
#include "eg_kernel.cuh"
#include "eg_registry.h"

namespace eg {

bool lookup_e4m3_block_swap(int bn, KernelEntry* out) {
  switch (bn) {
    case 16: EG_KERNEL_ENTRY(IN_E4M3, SC_BLOCK, true, 16);
    case 32: EG_KERNEL_ENTRY(IN_E4M3, SC_BLOCK, true, 32);
    case 64: EG_KERNEL_ENTRY(IN_E4M3, SC_BLOCK, true, 64);
    case 128: EG_KERNEL_ENTRY(IN_E4M3, SC_BLOCK, true, 128);
    default: return false;
  }
}

}  // namespace eg
