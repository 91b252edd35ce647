// bf16 instantiation of the sampling row kernel.
#include "sample_kernel.cuh"

namespace sv {

const void* sample_kernel_bf16() { return reinterpret_cast<const void*>(&sample_kernel<true>); }

}  // namespace sv
