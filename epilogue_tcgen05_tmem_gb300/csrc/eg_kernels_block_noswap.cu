// eg_kernels_block_noswap.cu -- fused kernel instantiations,
// IN_E4M3 / SC_BLOCK, swap_ab = 0.
#include "eg_kernel.cuh"
#include "eg_registry.h"

namespace eg {

bool lookup_e4m3_block_noswap(int bn, KernelEntry* out) {
  switch (bn) {
    case 16: EG_KERNEL_ENTRY(IN_E4M3, SC_BLOCK, false, 16);
    case 32: EG_KERNEL_ENTRY(IN_E4M3, SC_BLOCK, false, 32);
    case 64: EG_KERNEL_ENTRY(IN_E4M3, SC_BLOCK, false, 64);
    case 128: EG_KERNEL_ENTRY(IN_E4M3, SC_BLOCK, false, 128);
    case 256: EG_KERNEL_ENTRY(IN_E4M3, SC_BLOCK, false, 256);
    default: return false;
  }
}

}  // namespace eg
