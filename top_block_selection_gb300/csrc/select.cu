// select.cu - exact top-k block selection per query (Strata pull request 228,
// part 1 and pull request 856, "Arithmetic contract and parity": the top-k
// over the block scores, here with a block-index tie-break).
//
// One CTA of four warps per query row:
//   1. the row's scores are mapped to order-preserving uint32 keys (-0.0
//      folded onto +0.0) and staged in shared memory, with the row's min and
//      max key reduced by warp redux and a shared-memory step;
//   2. radix select from the first bit where min and max differ, 8 bits per
//      pass: a shared histogram of the candidates' digit, then one warp scans
//      the 256 bins from the top with shuffles and a ballot to find the digit
//      that holds the k-th largest key. It stops early once the keys still
//      needed are exactly one bin;
//   3. the winners (every key above the threshold, plus, when the k-th key is
//      tied, the tied keys with the smallest block indices, taken in index
//      order by ballot-ranked compaction) are gathered as 64-bit keys
//      (key << 32 | ~index), which are all distinct;
//   4. each winner's output slot is its rank among the winners, so ids come
//      out in descending score order with ascending index on ties.
// Rows with nb < k are padded with -1.
#include "qsa_device.cuh"
#include "qsa_internal.h"

namespace qsa {

constexpr int kSelThreads = 128;
constexpr int kSelWarps = kSelThreads / 32;

__device__ __forceinline__ uint32_t lanemask_lt() {
  uint32_t m;
  asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
  return m;
}

__global__ void __launch_bounds__(kSelThreads)
    select_kernel(const float* __restrict__ scores, int32_t nb, int32_t k,
                  int32_t* __restrict__ ids) {
  extern __shared__ uint32_t sm[];
  uint32_t* keys = sm;                                            // [nb]
  uint32_t* hist = keys + ((nb + 3) & ~3);                        // [256]
  uint64_t* sel = reinterpret_cast<uint64_t*>(hist + 256);        // [min(k, nb)]
  __shared__ uint32_t red_min[kSelWarps], red_max[kSelWarps], warp_cnt[kSelWarps];
  __shared__ uint32_t s_digit, s_above, s_cnt, s_count;

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t row = blockIdx.x;
  const float* s = scores + row * nb;
  int32_t* out = ids + row * k;
  const int kk = k < nb ? k : nb;

  uint32_t lmin = 0xFFFFFFFFu, lmax = 0u;
  for (int i = tid; i < nb; i += kSelThreads) {
    const uint32_t key = score_key(s[i]);
    keys[i] = key;
    lmin = min(lmin, key);
    lmax = max(lmax, key);
  }
  lmin = __reduce_min_sync(0xFFFFFFFFu, lmin);
  lmax = __reduce_max_sync(0xFFFFFFFFu, lmax);
  if (lane == 0) {
    red_min[warp] = lmin;
    red_max[warp] = lmax;
  }
  if (tid == 0) s_count = 0;
  __syncthreads();
  uint32_t kmin = red_min[0], kmax = red_max[0];
#pragma unroll
  for (int w = 1; w < kSelWarps; ++w) {
    kmin = min(kmin, red_min[w]);
    kmax = max(kmax, red_max[w]);
  }

  // Selection rule after the search: keys >= thr are taken (take_all), or
  // keys > thr plus the `need` smallest indices whose key == thr.
  uint32_t thr = 0;
  bool take_all = true;
  uint32_t need = static_cast<uint32_t>(kk);
  if (kk > 0 && kk < nb) {
    const uint32_t diff = kmin ^ kmax;
    if (diff == 0) {
      thr = kmax;  // every key equal: k smallest indices
      take_all = false;
    } else {
      int hi = 32 - __clz(diff);  // bits [hi, 32) are common to every key
      uint32_t prefix = (hi >= 32) ? 0u : ((kmax >> hi) << hi);
      bool done = false;
      while (hi > 0 && !done) {
        const int nbits = hi < 8 ? hi : 8;
        const int lo = hi - nbits;
        const uint32_t dmask = (1u << nbits) - 1u;
        for (int i = tid; i < 256; i += kSelThreads) hist[i] = 0;
        __syncthreads();
        for (int i = tid; i < nb; i += kSelThreads) {
          const uint32_t key = keys[i];
          const bool match = (hi >= 32) || (((key ^ prefix) >> hi) == 0);
          if (match) atomicAdd(&hist[(key >> lo) & dmask], 1u);
        }
        __syncthreads();
        if (warp == 0) {
          // lane l holds bins [8*(31-l), 8*(31-l)+8): lane 0 the highest.
          const int bin0 = 8 * (31 - lane);
          uint32_t c[8], local = 0;
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            c[j] = hist[bin0 + j];
            local += c[j];
          }
          uint32_t incl = local;
#pragma unroll
          for (int off = 1; off < 32; off <<= 1) {
            const uint32_t v = __shfl_up_sync(0xFFFFFFFFu, incl, off);
            if (lane >= off) incl += v;
          }
          const uint32_t excl = incl - local;
          const uint32_t hit = __ballot_sync(0xFFFFFFFFu, excl < need && need <= incl);
          if (lane == __ffs(hit) - 1) {
            uint32_t run = excl;
#pragma unroll
            for (int j = 7; j >= 0; --j) {
              if (run + c[j] >= need) {
                s_digit = static_cast<uint32_t>(bin0 + j);
                s_above = run;
                s_cnt = c[j];
                break;
              }
              run += c[j];
            }
          }
        }
        __syncthreads();
        const uint32_t digit = s_digit, above = s_above, cnt = s_cnt;
        need -= above;
        prefix |= digit << lo;
        hi = lo;
        if (cnt == need) {
          thr = prefix;  // every candidate left is a winner: take keys >= prefix
          take_all = true;
          done = true;
        }
        __syncthreads();  // hist is rewritten by the next pass
      }
      if (!done) {
        thr = prefix;
        take_all = false;
      }
    }
  }

  // Gather the winners as distinct 64-bit keys.
  if (kk > 0) {
    for (int i = tid; i < nb; i += kSelThreads) {
      const uint32_t key = keys[i];
      if (take_all ? key >= thr : key > thr) {
        const uint32_t pos = atomicAdd(&s_count, 1u);
        sel[pos] = (static_cast<uint64_t>(key) << 32) | static_cast<uint32_t>(~i);
      }
    }
    if (!take_all) {
      uint32_t taken = 0;  // tied keys taken so far, uniform over the CTA
      for (int base = 0; base < nb && taken < need; base += kSelThreads) {
        const int i = base + tid;
        const bool tie = i < nb && keys[i] == thr;
        const uint32_t m = __ballot_sync(0xFFFFFFFFu, tie);
        if (lane == 0) warp_cnt[warp] = __popc(m);
        __syncthreads();
        uint32_t before = 0, total = 0;
#pragma unroll
        for (int w = 0; w < kSelWarps; ++w) {
          before += (w < warp) ? warp_cnt[w] : 0u;
          total += warp_cnt[w];
        }
        const uint32_t r = taken + before + __popc(m & lanemask_lt());
        if (tie && r < need) {
          const uint32_t pos = atomicAdd(&s_count, 1u);
          sel[pos] = (static_cast<uint64_t>(thr) << 32) | static_cast<uint32_t>(~i);
        }
        taken += total;
        __syncthreads();
      }
    }
  }
  __syncthreads();

  // Rank sort of the winners into their output slots.
  for (int j = tid; j < kk; j += kSelThreads) {
    const uint64_t c = sel[j];
    int rank = 0;
    for (int m = 0; m < kk; ++m) rank += sel[m] > c ? 1 : 0;
    out[rank] = static_cast<int32_t>(~static_cast<uint32_t>(c));
  }
  for (int j = kk + tid; j < k; j += kSelThreads) out[j] = -1;
}

namespace {
size_t select_smem_bytes(int32_t nb, int32_t k) {
  const int kk = k < nb ? k : nb;
  return (static_cast<size_t>((nb + 3) & ~3) + 256) * sizeof(uint32_t) +
         static_cast<size_t>(kk) * sizeof(uint64_t);
}
}  // namespace

cudaError_t init_select_kernels(const DeviceInfo& dev) {
  const size_t most = select_smem_bytes(kMaxSelectNb, kMaxSelectK);
  const int limit = static_cast<int>(most < static_cast<size_t>(dev.max_smem_optin)
                                         ? most
                                         : static_cast<size_t>(dev.max_smem_optin));
  return cudaFuncSetAttribute(reinterpret_cast<const void*>(&select_kernel),
                              cudaFuncAttributeMaxDynamicSharedMemorySize, limit);
}

cudaError_t launch_select(const float* scores, int32_t nq, int32_t nb, int32_t k, int32_t* ids,
                          const DeviceInfo& dev, cudaStream_t stream) {
  if (nq <= 0) return cudaSuccess;
  const size_t smem = select_smem_bytes(nb, k);
  if (smem > static_cast<size_t>(dev.max_smem_optin)) return cudaErrorInvalidValue;
  select_kernel<<<static_cast<unsigned>(nq), kSelThreads, smem, stream>>>(scores, nb, k, ids);
  return cudaGetLastError();
}

}  // namespace qsa
