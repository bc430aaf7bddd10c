// select.cu - exact top-k block selection per query (Strata pull request 228,
// part 1 and pull request 856, "Arithmetic contract and parity": the top-k
// over the block scores, here with a block-index tie-break).
//
// Rows of up to 4096 blocks: one CTA of 8 warps per row, the row's keys in
// registers, the selects of the fused kernel (select_row_warp64 by one warp
// on rows of at most 64 blocks; select_row_thr for k <= 128 on rows of up to
// 1024 blocks, then select_row_window, with select_row_regs behind it). Longer rows: a CTA of kSelThreads threads
// selects several rows, kSelG warps per row (select_row_g): the row's keys
// are staged in shared memory, the first 11-bit radix digit finds the
// boundary bin, the boundary bin's keys are compacted and refined, and the
// winners are rank-sorted.
#include <algorithm>
#include <map>
#include <mutex>
#include <tuple>

#include <cuda_fp16.h>

#include "qsa_internal.h"
#include "select_row.cuh"
#include "select_warp.cuh"

namespace qsa {

constexpr int kSelThreads = 256;
constexpr int kSelG = 4;                          // warps per row
constexpr int kSelMaxGroups = kSelThreads / (32 * kSelG);  // rows per CTA at most

// Shared bytes of one row's group: hist, cand, sel (k), keys (nb).
__host__ __device__ inline size_t select_group_bytes(int32_t nb, int32_t k) {
  size_t b = kSelHistBins * sizeof(uint32_t) + (static_cast<size_t>(kSelBinMax) + k) * sizeof(uint64_t) +
             static_cast<size_t>(nb) * sizeof(uint32_t);
  return (b + 15) & ~static_cast<size_t>(15);
}

__global__ void __launch_bounds__(kSelThreads)
    select_kernel(const float* __restrict__ scores, int32_t nq, int32_t nb, int32_t k,
                  int32_t* __restrict__ ids) {
  extern __shared__ __align__(16) uint8_t sm_raw[];
  __shared__ GroupShared sh[kSelMaxGroups];
  constexpr int T = 32 * kSelG;
  const int groups = blockDim.x / T;  // rows per CTA, chosen at launch to fit shared memory
  const int g = threadIdx.x / T;
  const int gtid = threadIdx.x % T;
  const int64_t row = static_cast<int64_t>(blockIdx.x) * groups + g;
  pdl_launch_dependents();
  if (row >= nq) return;  // whole groups leave together; no CTA-wide barrier follows
  pdl_wait();             // the scores may come from the previous kernel on the stream
  uint8_t* base = sm_raw + g * select_group_bytes(nb, k);
  uint32_t* hist = reinterpret_cast<uint32_t*>(base);                 // [kSelHistBins]
  uint64_t* cand = reinterpret_cast<uint64_t*>(hist + kSelHistBins);  // [kSelBinMax]
  uint64_t* sel = cand + kSelBinMax;                                  // [k]
  uint32_t* keys = reinterpret_cast<uint32_t*>(sel + k);              // [nb]
  const float* s = scores + row * nb;
  for (int b0 = 0; b0 < nb; b0 += 8 * T) {
    float v[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int i = b0 + j * T + gtid;
      v[j] = i < nb ? __ldcg(s + i) : 0.0f;
    }
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int i = b0 + j * T + gtid;
      if (i < nb) keys[i] = score_key(v[j]);
    }
  }
  group_sync<T>(1 + g);
  select_row_g<kSelG>(keys, nb, k, ids + row * k, hist, cand, sel, sh[g], gtid, 1 + g);
}

constexpr int kWinThreads = 256;

// Shared bytes of the window select: hist, excl, cand, sel (k), sel_bin (k
// rounded up to 4).
inline size_t select_window_bytes(int32_t k) {
  return 2 * kSelHistBins * sizeof(uint32_t) + (static_cast<size_t>(kSelBinMax) + k) * sizeof(uint64_t) +
         ((static_cast<size_t>(k) + 3) & ~static_cast<size_t>(3)) * sizeof(uint32_t);
}

// Three CTAs per SM (at most 85 registers a thread): the select is bound by
// the latency of its barrier-separated phases, so more rows in flight per SM
// raise the throughput of many-row launches.
template <int R>
__global__ void __launch_bounds__(kWinThreads, 3)
    select_window_kernel(const float* __restrict__ scores, int32_t nb, int32_t k,
                         int32_t* __restrict__ ids) {
  extern __shared__ __align__(16) uint8_t sm_raw[];
  __shared__ SelectShared sh;
  uint32_t* hist = reinterpret_cast<uint32_t*>(sm_raw);
  uint32_t* excl = hist + kSelHistBins;
  uint64_t* cand = reinterpret_cast<uint64_t*>(excl + kSelHistBins);
  uint64_t* sel = cand + kSelBinMax;
  uint32_t* sel_bin = reinterpret_cast<uint32_t*>(sel + k);
  const int tid = threadIdx.x;
  const int64_t row = blockIdx.x;
  pdl_launch_dependents();
  pdl_wait();  // the scores may come from the previous kernel on the stream
  if (nb <= 64) {  // short rows: one warp, no block barrier
    if (tid < 32) {
      const float* s = scores + row * nb;
      const uint32_t k0 = tid < nb ? score_key(__ldcg(s + tid)) : 0u;
      const uint32_t k1 = tid + 32 < nb ? score_key(__ldcg(s + tid + 32)) : 0u;
      select_row_warp64(k0, k1, nb, k, ids + row * k, tid);
    }
    return;
  }
  uint32_t key[R];
  load_keys_regs_global<kWinThreads, R>(scores + row * nb, nb, key, hist, tid);
  int32_t* out = ids + row * k;
  // The threshold select first on rows of up to 1024 blocks (measured: 2,646
  // vs 3,800 cycles per 513-key row); on longer rows the window select alone
  // (4.3 vs 5.1 us for 256 rows of 2048 blocks, three CTAs per SM).
  if (nb <= 1024 && select_row_thr<kWinThreads, R>(key, nb, k, out, cand, sh, tid, 1)) return;
  if (!select_row_window<kWinThreads, R>(key, nb, k, out, hist, excl, cand, sel, sel_bin, sh, tid, 1)) {
    build_first_digit_hist<kWinThreads, R>(key, nb, hist, tid, 1);
    select_row_regs<kWinThreads, R>(key, nb, k, out, hist, cand, sel, sh, tid, 1);
  }
}

constexpr int kWsWarps = 8;
constexpr int kWsMaxNb = 4096;
constexpr int kWsMinRows = 1024;  // fewer rows: one CTA per row has the lower latency

// Shared bytes of the warp select kernel: per warp, kWarpSelCap candidates
// and the staged row (nb + 6 words, rounded up to 4: see the staging).
inline size_t select_warp_bytes(int32_t nb) {
  return static_cast<size_t>(kWsWarps) *
         (kWarpSelCap * sizeof(uint64_t) + ((static_cast<size_t>(nb) + 9) & ~static_cast<size_t>(3)) * 4);
}

__device__ __forceinline__ void cp_async_4(void* smem_dst, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(smem_u32(smem_dst)),
               "l"(reinterpret_cast<uint64_t>(src))
               : "memory");
}

// Many rows: one warp per row, rows grid-strided over the launch's warps.
// The row is staged into the warp's slice of shared memory by 4-byte
// asynchronous copies (all in flight at once; rows need not be 16-byte
// aligned) and selected there (select_row_warp_f32).
// kTail: the row's last column is the tail block (Strata pull request 856,
// "What": the shared tail kernel and the +1e9 dead-tail rule), scored here
// while the copies are in flight: lane h < H sums head h's fp32 products in
// index order, lane 0 sums max(acc_h, 0) in head order and adds 1e9f (the
// pinned order of the tail kernel, every step round-to-nearest-even); the
// score goes to the scores row and into the staged row before the select.
template <bool kTail>
__global__ void __launch_bounds__(kWsWarps * 32)
    select_warp_kernel(const float* scores_in, float* scores_tail,
                       int32_t nq, int32_t nb, int32_t k, int32_t* __restrict__ ids,
                       const __half* __restrict__ q16, const __half* __restrict__ kb_tail0,
                       int32_t H, int32_t D, int64_t kb_batch_stride, int32_t nq_per_batch) {
  extern __shared__ __align__(16) uint8_t sm_raw[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // staged positions [0, nb + shift + 3) with shift < 4, rounded up to whole
  // 16-byte units
  const int row_words = (nb + 9) & ~3;
  uint64_t* cand = reinterpret_cast<uint64_t*>(sm_raw) + warp * kWarpSelCap;
  float* buf = reinterpret_cast<float*>(sm_raw + kWsWarps * kWarpSelCap * sizeof(uint64_t)) +
               warp * row_words;
  pdl_launch_dependents();
  pdl_wait();  // the scores (and q16) may come from earlier kernels on the stream
  for (int64_t row = static_cast<int64_t>(blockIdx.x) * kWsWarps + warp; row < nq;
       row += static_cast<int64_t>(gridDim.x) * kWsWarps) {
    const float* s = scores_in + row * nb;
    // Stage the row from the 16-byte units that hold it: element i lands at
    // buf[i + shift] with shift = (address of s mod 16) / 4, so each unit is
    // one 16-byte copy (an aligned unit holding a row element never crosses
    // an allocation granule, so the words beside the row it brings are
    // readable; they are ignored).
    const int shift = static_cast<int>((reinterpret_cast<uintptr_t>(s) & 15u) >> 2);
    const float* s0 = s - shift;
    const int n_copy = kTail ? nb - 1 : nb;
    for (int p = lane * 4; p < n_copy + shift; p += 128)
      asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(buf + p)),
                   "l"(reinterpret_cast<uint64_t>(s0 + p))
                   : "memory");
    asm volatile("cp.async.commit_group;" ::: "memory");
    float tail = 0.0f;
    if constexpr (kTail) {
      // acc = fl(acc + q_i k_i) for i in order. A product of two fp16 values
      // is exact in fp32, so one fused multiply-add per step rounds exactly as
      // the separate multiply and add do.
      float acc = 0.0f;
      const __half* kb_tail =
          kb_tail0 + (kb_batch_stride != 0
                          ? static_cast<int64_t>(static_cast<int32_t>(row) / nq_per_batch) * kb_batch_stride
                          : 0);
      if (lane < H) {
        const __half2* qr = reinterpret_cast<const __half2*>(q16 + (row * H + lane) * D);
        const __half2* kr = reinterpret_cast<const __half2*>(kb_tail);
#pragma unroll 8
        for (int i = 0; i < D / 2; i += 4) {  // eight 16-byte loads of q in flight
          const uint4 qv = __ldg(reinterpret_cast<const uint4*>(qr + i));
          const uint4 kv = __ldg(reinterpret_cast<const uint4*>(kr + i));
          const __half2* qh = reinterpret_cast<const __half2*>(&qv);
          const __half2* kh = reinterpret_cast<const __half2*>(&kv);
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const float2 qf = __half22float2(qh[j]), kf = __half22float2(kh[j]);
            acc = __fmaf_rn(qf.x, kf.x, acc);
            acc = __fmaf_rn(qf.y, kf.y, acc);
          }
        }
      }
      float t = 0.0f;
      for (int h = 0; h < H; ++h) t = __fadd_rn(t, fmaxf(__shfl_sync(0xFFFFFFFFu, acc, h), 0.0f));
      tail = __fadd_rn(t, 1.0e9f);
      if (lane == 0) scores_tail[row * nb + (nb - 1)] = tail;
    }
    asm volatile("cp.async.wait_group 0;" ::: "memory");
    if (kTail && lane == 0) buf[nb - 1 + shift] = tail;
    __syncwarp();
    select_row_warp_f32(buf, shift, nb, k, ids + row * k, cand, lane);
    __syncwarp();  // the slice is rewritten by the next row
  }
}

bool select_scores_tail(int32_t nq, int32_t nb, int32_t k) {
  return nq >= kWsMinRows && nb >= 2 && nb <= kWsMaxNb && k <= kWarpSelKMax;
}

cudaError_t init_select_kernels(const DeviceInfo& dev) {
  {
    for (const void* fn : {reinterpret_cast<const void*>(&select_warp_kernel<false>),
                           reinterpret_cast<const void*>(&select_warp_kernel<true>)}) {
      cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           static_cast<int>(select_warp_bytes(kWsMaxNb)));
      if (e != cudaSuccess) return e;
    }
  }
  for (const void* fn : {reinterpret_cast<const void*>(&select_window_kernel<8>),
                         reinterpret_cast<const void*>(&select_window_kernel<12>),
                         reinterpret_cast<const void*>(&select_window_kernel<16>)}) {
    cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(select_window_bytes(1024)));
    if (e != cudaSuccess) return e;
  }
  cudaFuncAttributes fa;
  cudaError_t e = cudaFuncGetAttributes(&fa, reinterpret_cast<const void*>(&select_kernel));
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(reinterpret_cast<const void*>(&select_kernel),
                              cudaFuncAttributeMaxDynamicSharedMemorySize,
                              dev.max_smem_optin - static_cast<int>(fa.sharedSizeBytes));
}

cudaError_t launch_select(const float* scores, int32_t nq, int32_t nb, int32_t k, int32_t* ids,
                          const DeviceInfo& dev, cudaStream_t stream, const TailInfo* tail) {
  if (nq <= 0) return cudaSuccess;
  if (tail != nullptr && !select_scores_tail(nq, nb, k)) return cudaErrorInvalidValue;
  if (nq >= kWsMinRows && nb >= 1 && nb <= kWsMaxNb && k <= kWarpSelKMax) {
    const size_t smem = select_warp_bytes(nb);
    auto fn = tail != nullptr ? select_warp_kernel<true> : select_warp_kernel<false>;
    // CTAs per SM for this row length, asked of the runtime once per (device,
    // form, shared bytes): the query is host work that eager callers would
    // otherwise pay on every call.
    int per_sm = 0;
    {
      static std::mutex mu;
      static std::map<std::tuple<int, bool, size_t>, int> cache;
      const auto key = std::make_tuple(dev.id, tail != nullptr, smem);
      std::lock_guard<std::mutex> lock(mu);
      auto it = cache.find(key);
      if (it != cache.end()) {
        per_sm = it->second;
      } else {
        cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, fn, kWsWarps * 32, smem);
        if (e != cudaSuccess) return e;
        cache.emplace(key, per_sm);
      }
    }
    const int64_t want = (static_cast<int64_t>(nq) + kWsWarps - 1) / kWsWarps;
    const int64_t grid = std::min(want, static_cast<int64_t>(std::max(per_sm, 1)) * dev.sm_count);
    plan_add(tail != nullptr ? "select_warp_kernel (tail block scored in)" : "select_warp_kernel");
    // scores is written (the tail column) only in the tail form
    float* scores_w = const_cast<float*>(scores);
    return launch_pdl(fn, dim3(static_cast<unsigned>(grid)), dim3(kWsWarps * 32), smem, stream,
                      scores, scores_w, nq, nb, k, ids,
                      tail ? reinterpret_cast<const __half*>(tail->q16) : nullptr,
                      tail ? reinterpret_cast<const __half*>(tail->kb_tail) : nullptr,
                      tail ? tail->H : 0, tail ? tail->D : 0, tail ? tail->kb_batch_stride : 0,
                      tail ? tail->nq_per_batch : 1);
  }
  if (nb >= 1 && nb <= 16 * kWinThreads && k <= 1024) {
    const size_t smem = select_window_bytes(k);
    const dim3 grid(static_cast<unsigned>(nq)), block(kWinThreads);
    plan_add("select_window_kernel");
    if (nb <= 8 * kWinThreads)
      return launch_pdl(select_window_kernel<8>, grid, block, smem, stream, scores, nb, k, ids);
    if (nb <= 12 * kWinThreads)
      return launch_pdl(select_window_kernel<12>, grid, block, smem, stream, scores, nb, k, ids);
    return launch_pdl(select_window_kernel<16>, grid, block, smem, stream, scores, nb, k, ids);
  }
  const size_t per = select_group_bytes(nb, k);
  const size_t room = static_cast<size_t>(dev.max_smem_optin) - sizeof(GroupShared) * kSelMaxGroups;
  int groups = kSelMaxGroups;
  while (groups > 1 && static_cast<size_t>(groups) * per > room) groups >>= 1;
  if (per > room) return cudaErrorInvalidValue;
  const int64_t grid = (static_cast<int64_t>(nq) + groups - 1) / groups;
  plan_add("select_kernel");
  return launch_pdl(select_kernel, dim3(static_cast<unsigned>(grid)), dim3(groups * 32 * kSelG),
                    groups * per, stream, scores, nq, nb, k, ids);
}

}  // namespace qsa
