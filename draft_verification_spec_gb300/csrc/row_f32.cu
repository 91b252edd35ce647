// fp32 instantiations of the row kernel.
#include "row_kernel.cuh"

namespace sv {

const void* row_kernel_f32(bool greedy, int nt) {
  if (nt == 256) return greedy ? reinterpret_cast<const void*>(&row_kernel<false, true, 256>)
                               : reinterpret_cast<const void*>(&row_kernel<false, false, 256>);
  return greedy ? reinterpret_cast<const void*>(&row_kernel<false, true, 512>)
                : reinterpret_cast<const void*>(&row_kernel<false, false, 512>);
}

}  // namespace sv
