// fused_h8.cu - the fused step kernel's instantiations for 8 heads (one
// translation unit per head count, so that they compile in parallel).
#include "fused_kernel.cuh"

namespace qsa {
const void* fused_kernel_h8(bool f32q, int form) { return fused_kernel_ptr<8>(f32q, form); }
}  // namespace qsa
