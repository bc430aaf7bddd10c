// fused_h2.cu - the fused step kernel's instantiations for 2 heads (one
// translation unit per head count, so that they compile in parallel).
#include "fused_kernel.cuh"

namespace qsa {
const void* fused_kernel_h2(bool f32q, int form) { return fused_kernel_ptr<2>(f32q, form); }
}  // namespace qsa
