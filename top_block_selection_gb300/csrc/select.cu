// select.cu - exact top-k block selection per query (Strata pull request 228,
// part 1 and pull request 856, "Arithmetic contract and parity": the top-k
// over the block scores, here with a block-index tie-break).
//
// One CTA of kSelThreads threads per query row (see select_row.cuh for the
// algorithm): the row's keys stay in registers (8 or 16 per thread) for rows
// up to 4096 blocks, in shared memory beyond; the first 11-bit radix digit's
// histogram is built while the row is read; a suffix scan finds the boundary
// bin; a small boundary bin is ranked exactly; the winners are rank-sorted.
#include "qsa_internal.h"
#include "select_row.cuh"

namespace qsa {

constexpr int kSelThreads = 256;

__global__ void __launch_bounds__(kSelThreads)
    select_kernel(const float* __restrict__ scores, int32_t nb, int32_t k,
                  int32_t* __restrict__ ids) {
  extern __shared__ __align__(16) uint8_t sm_raw[];
  __shared__ SelectShared sh;
  uint32_t* hist = reinterpret_cast<uint32_t*>(sm_raw);                 // [kSelHistBins]
  uint64_t* cand = reinterpret_cast<uint64_t*>(hist + kSelHistBins);     // [kSelCandMax]
  uint64_t* sel = cand + kSelCandMax;                                    // [k]
  uint32_t* keys = reinterpret_cast<uint32_t*>(sel + k);                 // [nb] (long rows)
  const int64_t row = blockIdx.x;
  const float* s = scores + row * nb;
  int32_t* out = ids + row * k;
  if (nb <= 8 * kSelThreads) {
    uint32_t key[8];
    load_keys_global<kSelThreads, 8>(s, nb, key, hist, threadIdx.x, 1);
    select_row_regs<kSelThreads, 8>(key, nb, k, out, hist, cand, sel, sh, threadIdx.x, 1);
  } else if (nb <= 16 * kSelThreads) {
    uint32_t key[16];
    load_keys_global<kSelThreads, 16>(s, nb, key, hist, threadIdx.x, 1);
    select_row_regs<kSelThreads, 16>(key, nb, k, out, hist, cand, sel, sh, threadIdx.x, 1);
  } else {
    select_row_smem<kSelThreads, true>(s, nb, k, out, keys, hist, cand, sel, sh, threadIdx.x, 1);
  }
}

namespace {
size_t select_smem_bytes(int32_t nb, int32_t k) {
  size_t b = (static_cast<size_t>(kSelCandMax) + k) * sizeof(uint64_t) + kSelHistBins * sizeof(uint32_t);
  if (nb > 16 * kSelThreads) b += static_cast<size_t>(nb) * sizeof(uint32_t);
  return b;
}
}  // namespace

cudaError_t init_select_kernels(const DeviceInfo& dev) {
  cudaFuncAttributes fa;
  cudaError_t e = cudaFuncGetAttributes(&fa, reinterpret_cast<const void*>(&select_kernel));
  if (e != cudaSuccess) return e;
  const size_t most = select_smem_bytes(kMaxSelectNb, kMaxSelectK);
  const size_t room = static_cast<size_t>(dev.max_smem_optin) - fa.sharedSizeBytes;
  return cudaFuncSetAttribute(reinterpret_cast<const void*>(&select_kernel),
                              cudaFuncAttributeMaxDynamicSharedMemorySize,
                              static_cast<int>(most < room ? most : room));
}

cudaError_t launch_select(const float* scores, int32_t nq, int32_t nb, int32_t k, int32_t* ids,
                          const DeviceInfo& dev, cudaStream_t stream) {
  if (nq <= 0) return cudaSuccess;
  const size_t smem = select_smem_bytes(nb, k);
  if (smem + sizeof(SelectShared) > static_cast<size_t>(dev.max_smem_optin))
    return cudaErrorInvalidValue;
  select_kernel<<<static_cast<unsigned>(nq), kSelThreads, smem, stream>>>(scores, nb, k, ids);
  return cudaGetLastError();
}

}  // namespace qsa
