// bf16 instantiations of the sampling row kernel (16-byte aligned rows, and any rows).
#include "sample_kernel.cuh"

namespace sv {

const void* sample_kernel_bf16(bool aligned) {
  return aligned ? reinterpret_cast<const void*>(&sample_kernel<true, true>)
                 : reinterpret_cast<const void*>(&sample_kernel<true, false>);
}

}  // namespace sv
