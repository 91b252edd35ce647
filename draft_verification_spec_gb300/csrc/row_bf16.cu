// bf16 instantiations of the row kernel.
#include "row_kernel.cuh"

namespace sv {

const void* row_kernel_bf16(bool greedy, int nt) {
  if (nt == 256) return greedy ? reinterpret_cast<const void*>(&row_kernel<true, true, 256>)
                               : reinterpret_cast<const void*>(&row_kernel<true, false, 256>);
  return greedy ? reinterpret_cast<const void*>(&row_kernel<true, true, 512>)
                : reinterpret_cast<const void*>(&row_kernel<true, false, 512>);
}

}  // namespace sv
