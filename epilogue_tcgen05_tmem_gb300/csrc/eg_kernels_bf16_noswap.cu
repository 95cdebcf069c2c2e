// eg_kernels_bf16_noswap.cu -- fused kernel instantiations,
// IN_BF16 / SC_NONE, swap_ab = 0.
#include "eg_kernel.cuh"
#include "eg_registry.h"

namespace eg {

bool lookup_bf16_noswap(int bn, KernelEntry* out) {
  switch (bn) {
    case 16: EG_KERNEL_ENTRY(IN_BF16, SC_NONE, false, 16);
    case 32: EG_KERNEL_ENTRY(IN_BF16, SC_NONE, false, 32);
    case 64: EG_KERNEL_ENTRY(IN_BF16, SC_NONE, false, 64);
    case 128: EG_KERNEL_ENTRY(IN_BF16, SC_NONE, false, 128);
    case 192: EG_KERNEL_ENTRY(IN_BF16, SC_NONE, false, 192);
    case 224: EG_KERNEL_ENTRY(IN_BF16, SC_NONE, false, 224);
    case 256: EG_KERNEL_ENTRY(IN_BF16, SC_NONE, false, 256);
    default: return false;
  }
}

}  // namespace eg
