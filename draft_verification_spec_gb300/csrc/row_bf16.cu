// bf16 instantiations of the sampling row kernel.
#include "sample_kernel.cuh"

namespace sv {

const void* sample_kernel_bf16(int nt) {
  return nt == 256 ? reinterpret_cast<const void*>(&sample_kernel<true, 256>)
                   : reinterpret_cast<const void*>(&sample_kernel<true, 512>);
}

}  // namespace sv
