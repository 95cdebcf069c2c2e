// eg_kernels_fp8_noswap.cu -- fused kernel instantiations,
// IN_E4M3 / SC_TC, swap_ab = 0.
#include "eg_kernel.cuh"
#include "eg_registry.h"

namespace eg {

bool lookup_e4m3_tc_noswap(int bn, KernelEntry* out) {
  switch (bn) {
    case 16: EG_KERNEL_ENTRY(IN_E4M3, SC_TC, false, 16);
    case 32: EG_KERNEL_ENTRY(IN_E4M3, SC_TC, false, 32);
    case 64: EG_KERNEL_ENTRY(IN_E4M3, SC_TC, false, 64);
    case 128: EG_KERNEL_ENTRY(IN_E4M3, SC_TC, false, 128);
    case 192: EG_KERNEL_ENTRY(IN_E4M3, SC_TC, false, 192);
    case 224: EG_KERNEL_ENTRY(IN_E4M3, SC_TC, false, 224);
    case 256: EG_KERNEL_ENTRY(IN_E4M3, SC_TC, false, 256);
    default: return false;
  }
}

}  // namespace eg
