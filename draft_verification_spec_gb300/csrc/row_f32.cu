// fp32 instantiation of the sampling row kernel.
#include "sample_kernel.cuh"

namespace sv {

const void* sample_kernel_f32() { return reinterpret_cast<const void*>(&sample_kernel<false>); }

}  // namespace sv
