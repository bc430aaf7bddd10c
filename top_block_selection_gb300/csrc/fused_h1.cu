// fused_h1.cu - the fused step kernel's instantiations for 1 head (one
// translation unit per head count, so that they compile in parallel).
#include "fused_kernel.cuh"

namespace qsa {
const void* fused_kernel_h1(bool f32q, int form) { return fused_kernel_ptr<1>(f32q, form); }
}  // namespace qsa
