// f32 instantiations of the sampling row kernel (16-byte aligned rows, and any rows).
#include "sample_kernel.cuh"

namespace sv {

const void* sample_kernel_f32(bool aligned) {
  return aligned ? reinterpret_cast<const void*>(&sample_kernel<false, true>)
                 : reinterpret_cast<const void*>(&sample_kernel<false, false>);
}

}  // namespace sv
