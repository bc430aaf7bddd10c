// split_reduce_static.cu - the fixed device scratch behind
// qsa_split_reduce_static: the split reduce's chunk partials and arrival
// counters for callers that cannot allocate device memory when they call
// (a serving loop that must not enter the allocator, whose cudaMalloc /
// cudaFree synchronise the device; a plain C host without a caching
// allocator). No allocation happens here or in the entry point: the array
// is part of the library's device image, one copy per device.
#include <mutex>

#include "qsa.h"
#include "qsa_internal.h"

namespace qsa {

namespace {

static __device__ __align__(256) uint8_t g_split_scratch[QSA_SPLIT_STATIC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_addr[kMaxDevices] = {};

}  // namespace

void* split_static_scratch(cudaError_t* err) {
  int d = 0;
  cudaError_t e = cudaGetDevice(&d);
  if (e != cudaSuccess || d < 0 || d >= kMaxDevices) {
    *err = e != cudaSuccess ? e : cudaErrorInvalidDevice;
    return nullptr;
  }
  std::lock_guard<std::mutex> lock(g_mu);
  if (g_addr[d] == nullptr) {
    // Once per device, with that device current (the caller's).
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_split_scratch);
    if (e != cudaSuccess) {
      *err = e;
      return nullptr;
    }
    g_addr[d] = p;
  }
  return g_addr[d];
}

}  // namespace qsa
