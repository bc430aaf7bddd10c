// qsa_runtime.cu - per-device state: the device status word, device
// attributes, one-time kernel setup, and the driver's tensor-map encoder.
#include <mutex>

#include "qsa_device.cuh"
#include "qsa_internal.h"

namespace qsa {

// One word per device that loads the library; kernels OR a bit into it when a
// bounded wait runs out (bits in qsa_device.cuh).
__device__ uint32_t g_status_word = 0;

namespace {
constexpr int kMaxDevices = 64;
DeviceInfo g_devices[kMaxDevices];
std::mutex g_mutex;
}  // namespace

const DeviceInfo* current_device(cudaError_t* err) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    *err = (e != cudaSuccess) ? e : cudaErrorInvalidDevice;
    return nullptr;
  }
  std::lock_guard<std::mutex> lock(g_mutex);
  DeviceInfo& d = g_devices[dev];
  if (d.ready) return &d;
  d.id = dev;
  if ((e = cudaDeviceGetAttribute(&d.sm_count, cudaDevAttrMultiProcessorCount, dev)) ||
      (e = cudaDeviceGetAttribute(&d.cc_major, cudaDevAttrComputeCapabilityMajor, dev)) ||
      (e = cudaDeviceGetAttribute(&d.cc_minor, cudaDevAttrComputeCapabilityMinor, dev)) ||
      (e = cudaDeviceGetAttribute(&d.max_smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin,
                                  dev))) {
    *err = e;
    return nullptr;
  }
  d.supported = (d.cc_major == 10 && d.cc_minor == 3);
  if (d.supported) {
    void* p = nullptr;
    if ((e = cudaGetSymbolAddress(&p, g_status_word)) != cudaSuccess) {
      *err = e;
      return nullptr;
    }
    d.status_word = static_cast<uint32_t*>(p);
    if ((e = init_score_kernels(d)) != cudaSuccess || (e = init_select_kernels(d)) != cudaSuccess ||
        (e = init_fused_kernels(d)) != cudaSuccess || (e = init_split_reduce_kernel(d)) != cudaSuccess) {
      *err = e;
      return nullptr;
    }
  }
  d.ready = true;
  *err = cudaSuccess;
  return &d;
}

// Waits on an mbarrier that nothing arrives on, for at most timeout_ns, then
// records the expiry in the status word: the bounded-wait path of every
// kernel, exercised on purpose without hanging or faulting the GPU.
__global__ void selftest_wait_kernel(uint32_t* status, uint64_t timeout_ns) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_mbarrier_init();
    if (!mbar_wait_bounded(&bar, 0, timeout_ns)) atomicOr(status, kErrSelftestTimeout);
  }
}

cudaError_t launch_selftest_wait(const DeviceInfo& dev, uint64_t timeout_ns, cudaStream_t stream) {
  selftest_wait_kernel<<<1, 32, 0, stream>>>(dev.status_word, timeout_ns);
  return cudaGetLastError();
}

EncodeTiledFn encode_tiled_fn() {
  static EncodeTiledFn fn = [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      p = nullptr;
    return reinterpret_cast<EncodeTiledFn>(p);
  }();
  return fn;
}

}  // namespace qsa
