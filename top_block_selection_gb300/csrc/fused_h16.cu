// fused_h16.cu - the fused step kernel's instantiations for 16 heads (one
// translation unit per head count, so that they compile in parallel).
#include "fused_kernel.cuh"

namespace qsa {
const void* fused_kernel_h16(bool f32q, int form) { return fused_kernel_ptr<16>(f32q, form); }
}  // namespace qsa
