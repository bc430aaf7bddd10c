// convert.cu - the FP32 -> FP16 operand conversion stage (Strata pull request
// 228, part 1: f32_to_f16_poison_kernel runs beside the scorer, and the fp16
// conversion is part of the qsa select phase).
//
// dst[i] = binary16 round-to-nearest-even of src[i] (cvt.rn.f16.f32). Memory
// bound: each thread moves 8 values per step (two 16-byte loads, one 16-byte
// store) over a grid-stride loop sized to a whole number of waves; unaligned
// buffers take a scalar loop.
#include "qsa_device.cuh"
#include "qsa_internal.h"

namespace qsa {

constexpr int kConvThreads = 256;

__global__ void __launch_bounds__(kConvThreads)
    convert_vec8_kernel(const float4* __restrict__ src, uint4* __restrict__ dst, int64_t n8) {
  pdl_launch_dependents();
  pdl_wait();
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n8;
       i += stride) {
    const float4 a = src[2 * i];
    const float4 b = src[2 * i + 1];
    const __half2 h0 = __floats2half2_rn(a.x, a.y);
    const __half2 h1 = __floats2half2_rn(a.z, a.w);
    const __half2 h2 = __floats2half2_rn(b.x, b.y);
    const __half2 h3 = __floats2half2_rn(b.z, b.w);
    uint4 o;
    o.x = *reinterpret_cast<const uint32_t*>(&h0);
    o.y = *reinterpret_cast<const uint32_t*>(&h1);
    o.z = *reinterpret_cast<const uint32_t*>(&h2);
    o.w = *reinterpret_cast<const uint32_t*>(&h3);
    dst[i] = o;
  }
}

__global__ void __launch_bounds__(kConvThreads)
    convert_scalar_kernel(const float* __restrict__ src, __half* __restrict__ dst, int64_t n) {
  pdl_launch_dependents();
  pdl_wait();
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n;
       i += stride)
    dst[i] = __float2half_rn(src[i]);
}

cudaError_t launch_convert(const float* src, uint16_t* dst, int64_t n, const DeviceInfo& dev,
                           cudaStream_t stream) {
  if (n <= 0) return cudaSuccess;
  const int64_t wave = static_cast<int64_t>(dev.sm_count) * (2048 / kConvThreads);
  const bool vec = (reinterpret_cast<uintptr_t>(src) % 16 == 0) &&
                   (reinterpret_cast<uintptr_t>(dst) % 16 == 0);
  int64_t done = 0;
  if (vec) {
    const int64_t n8 = n / 8;
    if (n8 > 0) {
      int64_t blocks = (n8 + kConvThreads - 1) / kConvThreads;
      if (blocks > wave * 4) blocks = wave * 4;
      plan_add("convert_vec8_kernel");
      cudaError_t e = launch_pdl(convert_vec8_kernel, dim3(static_cast<unsigned>(blocks)),
                                 dim3(kConvThreads), 0, stream,
                                 reinterpret_cast<const float4*>(src), reinterpret_cast<uint4*>(dst),
                                 n8);
      if (e != cudaSuccess) return e;
    }
    done = n8 * 8;
  }
  const int64_t rest = n - done;
  if (rest > 0) {
    int64_t blocks = (rest + kConvThreads - 1) / kConvThreads;
    if (blocks > wave * 4) blocks = wave * 4;
    plan_add("convert_scalar_kernel");
    return launch_pdl(convert_scalar_kernel, dim3(static_cast<unsigned>(blocks)), dim3(kConvThreads),
                      0, stream, src + done, reinterpret_cast<__half*>(dst) + done, rest);
  }
  return cudaSuccess;
}

}  // namespace qsa
