// eg_kernels_bf16_swap.cu -- fused kernel instantiations,
// IN_BF16 / SC_NONE, swap_ab = 1.
#include "eg_kernel.cuh"
#include "eg_registry.h"

namespace eg {

bool lookup_bf16_swap(int bn, KernelEntry* out) {
  switch (bn) {
    case 16: EG_KERNEL_ENTRY(IN_BF16, SC_NONE, true, 16);
    case 32: EG_KERNEL_ENTRY(IN_BF16, SC_NONE, true, 32);
    case 64: EG_KERNEL_ENTRY(IN_BF16, SC_NONE, true, 64);
    case 128: EG_KERNEL_ENTRY(IN_BF16, SC_NONE, true, 128);
    case 256: EG_KERNEL_ENTRY(IN_BF16, SC_NONE, true, 256);
    default: return false;
  }
}

}  // namespace eg
