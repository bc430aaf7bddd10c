// fused_h4.cu - the fused step kernel's instantiations for 4 heads (one
// translation unit per head count, so that they compile in parallel).
#include "fused_kernel.cuh"

namespace qsa {
const void* fused_kernel_h4(bool f32q, int form) { return fused_kernel_ptr<4>(f32q, form); }
}  // namespace qsa
