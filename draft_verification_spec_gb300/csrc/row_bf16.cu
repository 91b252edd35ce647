// bf16 instantiation of the sampling row kernel.
#include "stream_kernel.cuh"

namespace sv {

const void* sample_kernel_bf16(int nt) {
  (void)nt;
  return reinterpret_cast<const void*>(&stream_kernel<true>);
}

}  // namespace sv
