// eg_kernels_bf16_gated.cu -- fused kernel instantiations of the gated
// linear unit (SwiGLU with SiLU), IN_BF16 / SC_NONE: rows over N (decode) with
// tile_n 16..64, rows over M with tile_n 64 or 128.
#include "eg_kernel.cuh"
#include "eg_registry.h"

namespace eg {

bool lookup_bf16_gated_swap(int bn, KernelEntry* out) {
  switch (bn) {
    case 16: EG_KERNEL_ENTRY_G(IN_BF16, SC_NONE, true, 16, true);
    case 32: EG_KERNEL_ENTRY_G(IN_BF16, SC_NONE, true, 32, true);
    case 64: EG_KERNEL_ENTRY_G(IN_BF16, SC_NONE, true, 64, true);
    default: return false;
  }
}

bool lookup_bf16_gated_noswap(int bn, KernelEntry* out) {
  switch (bn) {
    case 64: EG_KERNEL_ENTRY_G(IN_BF16, SC_NONE, false, 64, true);
    case 128: EG_KERNEL_ENTRY_G(IN_BF16, SC_NONE, false, 128, true);
    default: return false;
  }
}

}  // namespace eg
