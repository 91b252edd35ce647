// fp32 instantiations of the sampling row kernel.
#include "sample_kernel.cuh"

namespace sv {

const void* sample_kernel_f32(int nt) {
  return nt == 256 ? reinterpret_cast<const void*>(&sample_kernel<false, 256>)
                   : reinterpret_cast<const void*>(&sample_kernel<false, 512>);
}

}  // namespace sv
