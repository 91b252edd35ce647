// f32 instantiation of the sampling row kernel.
#include "stream_kernel.cuh"

namespace sv {

const void* sample_kernel_f32(int nt) {
  (void)nt;
  return reinterpret_cast<const void*>(&stream_kernel<false>);
}

}  // namespace sv
