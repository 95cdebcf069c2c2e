// eg_kernels_int8_swap.cu -- fused kernel instantiations,
// IN_INT8 / SC_TC, swap_ab = 1.
#include "eg_kernel.cuh"
#include "eg_registry.h"

namespace eg {

bool lookup_int8_tc_swap(int bn, KernelEntry* out) {
  switch (bn) {
    case 16: EG_KERNEL_ENTRY(IN_INT8, SC_TC, true, 16);
    case 32: EG_KERNEL_ENTRY(IN_INT8, SC_TC, true, 32);
    case 64: EG_KERNEL_ENTRY(IN_INT8, SC_TC, true, 64);
    default: return false;
  }
}

}  // namespace eg
