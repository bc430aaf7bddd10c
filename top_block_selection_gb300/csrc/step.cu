// step.cu - the selection step in one launch, one 128-block tile per CTA:
// fp32 -> fp16 query conversion, tensor-core block scores with the fused
// ReLU / head-sum epilogue, the fp32 tail block with the +1e9 dead-tail rule,
// and the exact top-k select (Strata pull request 228, part 1: the block
// scorer and the "qsa select" phase of scores + selection + fp16 conversion;
// pull request 856, "What": the shared tail kernel and the dead-tail rule).
//
// Work decomposition. Queries are cut into groups of qg queries (bn = qg*H
// TMEM columns, up to 256: one tcgen05.mma covers 128 blocks x bn columns x
// 16 of D). One thread-block cluster of cs CTAs (cs = the number of 128-block
// tiles, at most 16) owns a group: CTA rank r scores tile r, so one chain of
// D/16 MMAs per CTA covers every block of the group, and the cluster shares
// the group's query tile: each CTA rounds 1/cs of the fp32 rows to fp16 and
// stores them into every CTA's operand tile (st.async over DSMEM, counted on
// each CTA's bar_q).
//
// After the MMAs, each CTA's operand tiles are dead: the query tile's bytes
// receive the selection keys of the rows this CTA selects (queries ql with
// ql % cs == r), and the key tile's bytes hold the select's scratch. A
// cluster barrier ("every CTA's MMAs are complete") orders the first key
// store after the last operand read in every CTA.
//
// Roles (288 threads):
//   warp 8      TMA (key tile; fp16 queries), tcgen05.mma issue (one lane),
//               TMEM owner;
//   warps 0-7   the query conversion; on the tail-owner CTA, warps 0-3 score
//               the tail block in the pinned fp32 order while the MMAs run;
//               the epilogue: warp w reads TMEM lane quarter w % 4 (one block
//               per thread) and half w / 4 of the columns, applies ReLU, sums
//               each query's H adjacent columns in fp32 in head order, stores
//               the scores and sends each score's order-preserving key to the
//               selecting CTA (st.async, counted on its bar_keys); then the
//               select, rows_per_cta rows in one or two groups of threads.
// Every mbarrier wait is bounded; a CTA that gives up still reaches both
// cluster barriers, so the cluster never hangs on them.
#include <algorithm>
#include <cstring>
#include <type_traits>

#include "qsa_device.cuh"
#include "qsa_internal.h"
#include "select_row.cuh"

namespace qsa {

namespace {

constexpr int kSWork = 256;  // warps 0..7
constexpr int kSProducerWarp = 8;
constexpr int kSThreads = kSWork + 32;
constexpr int kSTileM = 128;
constexpr int kSRowBytes = 128;
constexpr int kSKAtom = 64;
constexpr int kSMaxCluster = 16;
constexpr int kSMaxBn = 256;
constexpr int kSBarTmem = 9;   // named barrier: TMEM reads done (work warps + producer warp)
constexpr int kSBarTail = 10;  // named barrier: the tail threads (work warps)
constexpr int kSBarKeys = 11;  // named barrier: the rows' keys have arrived (work warps)

struct StepArgs {
  const float* q32;     // fp32 queries [nq,H,D], or nullptr when q arrives as fp16
  __half* q16out;       // optional fp16 copy of the converted queries (fp32 input)
  const __half* kb;     // [nb, D]
  float* scores;        // [nq, nb]
  int32_t* ids;         // [nq, k]
  int32_t nq, D, nb, n_full, has_tail, k;
  int32_t bn, qg, cs, n_chunks, k_steps;
  int32_t rows_per_cta;  // rows this CTA selects at most (ceil(qg / cs))
  int32_t q_multicast;   // fp16 queries: each CTA loads 1/cs of the tile for all
  uint32_t row_bytes;    // bytes of one row's keys (16-byte multiple)
  uint32_t scratch_off;  // offset of the select scratch (the key tile's bytes)
  uint32_t group_bytes;  // scratch bytes of one select group
  uint32_t tmem_cols;
  uint32_t* status;
  uint64_t timeout_ns;
};

__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

__device__ __forceinline__ void cluster_arrive_relaxed() {
  asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}


__device__ __forceinline__ void cluster_wait_acquire() {
  asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

__device__ __forceinline__ uint32_t cluster_map(uint32_t saddr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
  return r;
}

__device__ __forceinline__ void st_async_u32(uint32_t addr, uint32_t v, uint32_t bar) {
  asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.u32 [%0], %1, [%2];" ::"r"(
                   addr),
               "r"(v), "r"(bar)
               : "memory");
}

__device__ __forceinline__ void st_async_v4(uint32_t addr, const uint4& v, uint32_t bar) {
  asm volatile(
      "st.async.shared::cluster.mbarrier::complete_tx::bytes.v4.b32 [%0], {%1, %2, %3, %4}, [%5];" ::"r"(
          addr),
      "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w), "r"(bar)
      : "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// 2-D TMA load multicast to the CTAs of `mask` (same shared offset in each),
// completion counted on each destination CTA's barrier at the same offset.
__device__ __forceinline__ void tma_load_2d_mc(void* smem_dst, const CUtensorMap* tm, int32_t x,
                                               int32_t y, uint64_t* bar, uint16_t mask) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.multicast::cluster"
      " [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(smem_u32(smem_dst)),
      "l"(reinterpret_cast<uint64_t>(tm)), "r"(x), "r"(y), "r"(smem_u32(bar)), "h"(mask)
      : "memory");
}

// Byte offset of fp16 element (row, i) in a K-major tile of `rows` rows stored
// as 64-column chunks of 128-byte rows with the 128-byte swizzle.
__device__ __forceinline__ uint32_t sw128_offset(int rows, int row, int i) {
  const int chunk = i >> 6;
  const int unit = (i & 63) >> 3;
  return static_cast<uint32_t>(chunk * rows * kSRowBytes + row * kSRowBytes +
                               ((unit ^ (row & 7)) << 4) + ((i & 7) << 1));
}

// The selecting CTA of query ql (in the group) is rank ql % cs, row slot
// ql / cs; the key of block b goes to keys[b] of that row.
__device__ __forceinline__ void send_key(uint32_t keys_base, uint32_t row_bytes, uint32_t bar_keys,
                                         int cs, int ql, int b, float score) {
  const uint32_t owner = static_cast<uint32_t>(ql % cs);
  const uint32_t local = keys_base + static_cast<uint32_t>(ql / cs) * row_bytes;
  st_async_u32(cluster_map(local, owner) + static_cast<uint32_t>(b) * 4u, score_key(score),
               cluster_map(bar_keys, owner));
}

template <int H, bool kF32Q>
__global__ void __launch_bounds__(kSThreads, 2)
    select_step_kernel(const __grid_constant__ CUtensorMap tm_kb,
                       const __grid_constant__ CUtensorMap tm_q, const StepArgs a) {
  static_assert(H >= 1 && H <= 32 && 32 % H == 0, "a 32-column TMEM load must hold whole queries");
  extern __shared__ uint8_t smem_raw[];
  __shared__ uint64_t bar_kb, bar_q, bar_acc, bar_keys;
  __shared__ uint32_t tmem_slot;
  __shared__ uint32_t keys_ok;
  __shared__ float tail_acc[kSMaxBn];
  __shared__ NwShared nw_sh[2];
  __shared__ GroupShared g_sh[2];

  const uint32_t raw = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + ((1024u - (raw & 1023u)) & 1023u);
  uint8_t* sQ = smem;                  // n_chunks x bn rows x 128 B; later the rows' keys
  uint8_t* sKB = smem + a.scratch_off; // n_chunks x 128 rows x 128 B; later select scratch
  const uint32_t q_bytes = static_cast<uint32_t>(a.n_chunks * a.bn * kSRowBytes);
  const uint32_t kb_bytes = static_cast<uint32_t>(a.n_chunks * kSTileM * kSRowBytes);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int cs = a.cs;
  const int rank = static_cast<int>(cluster_rank());
  const int group = blockIdx.x / cs;
  const int q0 = group * a.qg;  // first query of the group
  const int col0 = q0 * H;      // first row of the [nq*H, D] query view
  const int qh_rows = min(a.bn, (a.nq - q0) * H);
  const bool tail_owner = a.has_tail && rank == cs - 1;
  const bool producer_warp = warp == kSProducerWarp;
  const uint32_t keys_base = smem_u32(sQ);
  const uint32_t keys_bar = smem_u32(&bar_keys);
  // this CTA's slice of the query tile: rows [r0, r1) (possibly empty)
  const int slice = (a.bn + cs - 1) / cs;
  const int r0 = min(a.bn, rank * slice), r1 = min(a.bn, r0 + slice);

  pdl_launch_dependents();
  if (tid == kSProducerWarp * 32) {
    mbar_init(&bar_kb, 1);
    mbar_init(&bar_q, 1);
    mbar_init(&bar_acc, 1);
    mbar_init(&bar_keys, 1);
    fence_mbarrier_init();
    // Every CTA receives the whole query tile (its own slice included) and
    // the keys of its valid rows (nb keys each), registered before cluster
    // barrier 1 lets any peer store.
    mbar_arrive_expect_tx(&bar_q, q_bytes);
    int rows_valid = 0;
    for (int j = 0; j < a.rows_per_cta; ++j) {
      const int ql = rank + j * cs;
      if (ql < a.qg && q0 + ql < a.nq) ++rows_valid;
    }
    mbar_arrive_expect_tx(&bar_keys, static_cast<uint32_t>(rows_valid) * a.nb * 4u);
    tma_prefetch_desc(&tm_kb);
    if (!kF32Q) tma_prefetch_desc(&tm_q);
    for (int c = 0; c < a.n_chunks; ++c) tma_prefetch_l2_2d(&tm_kb, c * kSKAtom, rank * kSTileM);
    if (kF32Q) {
      const int rows = min(r1, qh_rows) - r0;
      if (rows > 0)
        bulk_prefetch_l2(a.q32 + static_cast<int64_t>(col0 + r0) * a.D,
                         static_cast<uint32_t>(rows) * a.D * 4u);
    }
  }
  // Cluster barrier 1: every CTA has started and initialised its barriers
  // before any peer stores into its shared memory. Arrived before the
  // dependency wait; waited just before the first remote store.
  __syncwarp();
  cluster_arrive_relaxed();
  if (producer_warp) {
    __syncwarp();
    tmem_alloc(&tmem_slot, a.tmem_cols);
    tmem_relinquish();
  }
  pdl_wait();
  if (producer_warp) {
    if (lane == 0) {
      mbar_arrive_expect_tx(&bar_kb, kb_bytes);
      for (int c = 0; c < a.n_chunks; ++c)
        tma_load_2d(sKB + c * kSTileM * kSRowBytes, &tm_kb, c * kSKAtom, rank * kSTileM, &bar_kb);
    }
    __syncwarp();
    cluster_wait_acquire();
    if (!kF32Q && lane == 0) {
      if (a.q_multicast) {
        // this CTA's slice of the fp16 tile, to every CTA of the cluster
        const uint16_t mask = static_cast<uint16_t>((1u << cs) - 1u);
        if (r1 > r0)
          for (int c = 0; c < a.n_chunks; ++c)
            tma_load_2d_mc(sQ + c * a.bn * kSRowBytes + r0 * kSRowBytes, &tm_q, c * kSKAtom,
                           col0 + r0, &bar_q, mask);
      } else {
        for (int c = 0; c < a.n_chunks; ++c)
          tma_load_2d(sQ + c * a.bn * kSRowBytes, &tm_q, c * kSKAtom, col0, &bar_q);
      }
    }
    __syncwarp();
  } else if (kF32Q) {
    // Rows [r0, r1) of the tile, rounded to fp16 (round to nearest even) and
    // stored as 16-byte swizzle units into every CTA of the cluster. Rows
    // past the group's last query and columns past D are zeros, so every CTA
    // receives all q_bytes.
    const int units_per_row = a.n_chunks * (kSKAtom / 8);
    const int n_units = (r1 - r0) * units_per_row;
    const uint32_t sq_local = smem_u32(sQ), bar_local = smem_u32(&bar_q);
    auto load_unit = [&](int u, float4& v0, float4& v1) {
      const int row = r0 + u / units_per_row;
      const int i = (u % units_per_row) * 8;
      v0 = make_float4(0.f, 0.f, 0.f, 0.f);
      v1 = v0;
      if (row < qh_rows && i < a.D) {
        const float4* src =
            reinterpret_cast<const float4*>(a.q32 + static_cast<int64_t>(col0 + row) * a.D + i);
        v0 = __ldg(src);
        v1 = __ldg(src + 1);
      }
    };
    float4 v0, v1;
    if (tid < n_units) load_unit(tid, v0, v1);
    cluster_wait_acquire();
    for (int u = tid; u < n_units; u += kSWork) {
      if (u != tid) load_unit(u, v0, v1);
      const int row = r0 + u / units_per_row;
      const int i = (u % units_per_row) * 8;
      const __half2 h01 = __floats2half2_rn(v0.x, v0.y), h23 = __floats2half2_rn(v0.z, v0.w);
      const __half2 h45 = __floats2half2_rn(v1.x, v1.y), h67 = __floats2half2_rn(v1.z, v1.w);
      uint4 pk;
      pk.x = *reinterpret_cast<const uint32_t*>(&h01);
      pk.y = *reinterpret_cast<const uint32_t*>(&h23);
      pk.z = *reinterpret_cast<const uint32_t*>(&h45);
      pk.w = *reinterpret_cast<const uint32_t*>(&h67);
      if (a.q16out != nullptr && row < qh_rows && i < a.D)
        *reinterpret_cast<uint4*>(a.q16out + static_cast<int64_t>(col0 + row) * a.D + i) = pk;
      const uint32_t off = sw128_offset(a.bn, row, i);
      for (int dst = 0; dst < cs; ++dst)
        st_async_v4(cluster_map(sq_local + off, static_cast<uint32_t>(dst)), pk,
                    cluster_map(bar_local, static_cast<uint32_t>(dst)));
    }
  } else {
    cluster_wait_acquire();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem_base = tmem_slot;

  if (producer_warp) {
    // ------------------------------------------------- MMA issue (one lane)
    if (lane == 0) {
      const bool ok = mbar_wait_bounded(&bar_q, 0, a.timeout_ns) &&
                      mbar_wait_bounded(&bar_kb, 0, a.timeout_ns);
      if (ok) {
        // peers' st.async writes of the query tile, then the tensor core's reads
        fence_proxy_async_smem();
        tc_fence_after_sync();
        const uint32_t idesc = idesc_f16_f32(kSTileM, a.bn);
        const uint32_t a_base = smem_u32(sKB), b_base = smem_u32(sQ);
        for (int step = 0; step < a.k_steps; ++step) {
          const int c = step >> 2, kk = step & 3;
          mma_f16_ss(tmem_base, smem_desc_k_sw128(a_base + c * kSTileM * kSRowBytes + kk * 32),
                     smem_desc_k_sw128(b_base + c * a.bn * kSRowBytes + kk * 32), idesc,
                     step > 0 ? 1u : 0u);
        }
      } else {
        atomicOr(a.status, kErrScoreLoadTimeout);
        // drain the loads still in flight before the bytes are reused
        mbar_wait_bounded(&bar_q, 0, a.timeout_ns);
        mbar_wait_bounded(&bar_kb, 0, a.timeout_ns);
      }
      // arrives once the MMAs (if any) have completed: the operands are dead
      mma_commit(&bar_acc);
      if (!mbar_wait_bounded(&bar_acc, 0, a.timeout_ns)) atomicOr(a.status, kErrScoreMmaTimeout);
    }
    __syncwarp();
    // Cluster barrier 2: this CTA's operand tiles are dead.
    cluster_arrive_relaxed();
    // TMEM is freed once the epilogue has read it.
    asm volatile("bar.sync %0, %1;" ::"n"(kSBarTmem), "n"(kSThreads) : "memory");
    tc_fence_after_sync();
    tmem_dealloc(tmem_base, a.tmem_cols);
    return;
  }

  // ---------------------------- tail block (the owner CTA's 256 threads)
  // Pinned fp32 order: per head a sequential sum over i of the exact
  // products, then a sequential sum over h of max(acc_h, 0), then + 1e9f.
  // The dot products read the query tile before cluster barrier 2; the head
  // sums, stores and keys come after it.
  if (tail_owner) {
    if (!mbar_wait_bounded(&bar_q, 0, a.timeout_ns) && tid == 0)
      atomicOr(a.status, kErrScoreLoadTimeout);
    const __half* krow = a.kb + static_cast<int64_t>(a.nb - 1) * a.D;
    for (int p = tid; p < qh_rows; p += kSWork) {
      float acc = 0.0f;
      for (int i = 0; i < a.D; i += 8) {
        const uint4 kv = __ldg(reinterpret_cast<const uint4*>(krow + i));
        const uint4 qv = *reinterpret_cast<const uint4*>(sQ + sw128_offset(a.bn, p, i));
        const __half* kh = reinterpret_cast<const __half*>(&kv);
        const __half* qh = reinterpret_cast<const __half*>(&qv);
#pragma unroll
        for (int j = 0; j < 8; ++j)
          acc = __fadd_rn(acc, __fmul_rn(__half2float(qh[j]), __half2float(kh[j])));
      }
      tail_acc[p] = acc;
    }
    asm volatile("bar.sync %0, %1;" ::"n"(kSBarTail), "n"(kSWork) : "memory");
  }

  // ------------------------------------------------ epilogue (warps 0..7)
  // bn >= 64: warp w reads TMEM lane quarter w % 4 (one block per thread)
  // and the half w / 4 of the columns; bn == 32: warps 0-3, every column.
  constexpr int kQPerLoad = 32 / H;
  constexpr int kMaxLoads = kSMaxBn / 2 / 32;
  constexpr bool kKeep = kMaxLoads * kQPerLoad <= 16;  // keys held in registers
  float keep[kKeep ? kMaxLoads * kQPerLoad : 1];
  const int quarter = warp & 3;
  const int ncolw = a.bn >= 64 ? a.bn / 2 : a.bn;
  const bool epi_warp = a.bn >= 64 || warp < 4;
  const int c_begin = a.bn >= 64 ? (warp >> 2) * ncolw : 0;
  const int b = rank * kSTileM + quarter * 32 + lane;
  const bool b_ok = b < a.n_full;
  const bool my_acc = mbar_wait_bounded(&bar_acc, 0, a.timeout_ns);
  const bool acc_ok = __all_sync(0xFFFFFFFFu, my_acc);
  if (!acc_ok && lane == 0) atomicOr(a.status, kErrScoreMmaTimeout);
  tc_fence_after_sync();
  // Cluster barrier 2: this thread has read its last operand byte.
  cluster_arrive_relaxed();
  const uint32_t taddr = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16);
  // One 32-column load: the scores of kQPerLoad queries of block b.
  auto scores_of = [&](int ld, float (&sc)[kQPerLoad]) {
    uint32_t r[32];
    tmem_ld_32cols(taddr + c_begin + ld * 32, r);
    tmem_ld_wait();
#pragma unroll
    for (int j = 0; j < kQPerLoad; ++j) {
      float s = 0.0f;
#pragma unroll
      for (int h = 0; h < H; ++h) s = __fadd_rn(s, fmaxf(__uint_as_float(r[j * H + h]), 0.0f));
      sc[j] = s;
    }
  };
  if (acc_ok && epi_warp) {
    float* out = a.scores + b;
#pragma unroll
    for (int ld = 0; ld < kMaxLoads; ++ld) {
      if (ld * 32 < ncolw) {
        float sc[kQPerLoad];
        scores_of(ld, sc);
#pragma unroll
        for (int j = 0; j < kQPerLoad; ++j) {
          const int ql = (c_begin + ld * 32) / H + j;
          if (kKeep) keep[ld * kQPerLoad + j] = sc[j];
          if (b_ok && q0 + ql < a.nq) out[static_cast<int64_t>(q0 + ql) * a.nb] = sc[j];
        }
      }
    }
  }
  if (kKeep) {
    tc_fence_before_sync();
    asm volatile("bar.arrive %0, %1;" ::"n"(kSBarTmem), "n"(kSThreads) : "memory");
  }
  cluster_wait_acquire();
  // Keys to the selecting CTAs: every peer's operand tiles are dead now.
  if (acc_ok && epi_warp) {
#pragma unroll
    for (int ld = 0; ld < kMaxLoads; ++ld) {
      if (ld * 32 < ncolw) {
        float sc[kQPerLoad];
        if (kKeep) {
#pragma unroll
          for (int j = 0; j < kQPerLoad; ++j) sc[j] = keep[ld * kQPerLoad + j];
        } else {
          scores_of(ld, sc);  // recomputed from TMEM: the same bits
        }
#pragma unroll
        for (int j = 0; j < kQPerLoad; ++j) {
          const int ql = (c_begin + ld * 32) / H + j;
          if (b_ok && q0 + ql < a.nq) send_key(keys_base, a.row_bytes, keys_bar, cs, ql, b, sc[j]);
        }
      }
    }
  }
  if (!kKeep) {
    tc_fence_before_sync();
    asm volatile("bar.arrive %0, %1;" ::"n"(kSBarTmem), "n"(kSThreads) : "memory");
  }
  if (tail_owner) {
    for (int ql = tid; ql * H < qh_rows; ql += kSWork) {
      float s = 0.0f;
#pragma unroll
      for (int h = 0; h < H; ++h) s = __fadd_rn(s, fmaxf(tail_acc[ql * H + h], 0.0f));
      const float score = __fadd_rn(s, 1.0e9f);
      a.scores[static_cast<int64_t>(q0 + ql) * a.nb + (a.nb - 1)] = score;
      send_key(keys_base, a.row_bytes, keys_bar, cs, ql, a.nb - 1, score);
    }
  }

  // ---------------------------------------------------------- select
  // Every key of this CTA's rows has arrived once bar_keys completes; one
  // thread waits (bounded) and tells the others.
  if (tid == 0) {
    keys_ok = mbar_wait_bounded(&bar_keys, 0, a.timeout_ns) ? 1u : 0u;
    if (!keys_ok) atomicOr(a.status, kErrFusedWaitTimeout);
  }
  asm volatile("bar.sync %0, %1;" ::"n"(kSBarKeys), "n"(kSWork) : "memory");
  if (!keys_ok) return;
  const int skip = a.has_tail ? a.nb - 1 : -1;
  auto run_rows = [&](auto tag) {
    constexpr int T = decltype(tag)::value;
    const int g = tid / T, gtid = tid % T;
    uint8_t* scr = sKB + g * a.group_bytes;
    uint32_t* hist = reinterpret_cast<uint32_t*>(scr);                  // kSelHistBins
    uint64_t* cand = reinterpret_cast<uint64_t*>(hist + kSelHistBins);  // kSelBinMax
    uint64_t* sel = cand + kSelBinMax;                                  // k
    uint32_t* sel_bin = reinterpret_cast<uint32_t*>(sel + a.k);         // k
    for (int j = g; j < a.rows_per_cta; j += kSWork / T) {
      const int ql = rank + j * cs;
      if (ql >= a.qg || q0 + ql >= a.nq) break;
      const uint32_t* keys = reinterpret_cast<const uint32_t*>(sQ + j * a.row_bytes);
      int32_t* out = a.ids + static_cast<int64_t>(q0 + ql) * a.k;
      if (!select_row_narrow<T>(keys, a.nb, a.k, skip, out, hist, cand, sel, sel_bin, nw_sh[g],
                                gtid, 1 + g)) {
        group_sync<T>(1 + g);
        select_row_g<T / 32>(keys, a.nb, a.k, out, hist, cand, sel, g_sh[g], gtid, 1 + g);
      }
      group_sync<T>(1 + g);
    }
  };
  if (a.rows_per_cta >= 2) run_rows(std::integral_constant<int, 128>{});
  else run_rows(std::integral_constant<int, 256>{});
}

template <int H, bool F>
const void* step_ptr() {
  return reinterpret_cast<const void*>(&select_step_kernel<H, F>);
}

const void* step_kernel_for(int H, bool f32q) {
  switch (H) {
    case 1: return f32q ? step_ptr<1, true>() : step_ptr<1, false>();
    case 2: return f32q ? step_ptr<2, true>() : step_ptr<2, false>();
    case 4: return f32q ? step_ptr<4, true>() : step_ptr<4, false>();
    case 8: return f32q ? step_ptr<8, true>() : step_ptr<8, false>();
    case 16: return f32q ? step_ptr<16, true>() : step_ptr<16, false>();
    case 32: return f32q ? step_ptr<32, true>() : step_ptr<32, false>();
    default: return nullptr;
  }
}

bool encode_2d(CUtensorMap* tm, const void* base, uint64_t cols, uint64_t rows, uint32_t box_cols,
               uint32_t box_rows) {
  EncodeTiledFn enc = encode_tiled_fn();
  if (!enc) return false;
  const cuuint64_t dims[2] = {cols, rows};
  const cuuint64_t strides[1] = {cols * 2};
  const cuuint32_t box[2] = {box_cols, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  return enc(tm, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<void*>(base), dims, strides, box,
             estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int g_step_static_smem = 0;

// The step's launch shape for a problem, or false when this kernel does not
// take it (the caller then uses the 8-CTA fused kernel).
struct StepPlan {
  int bn, qg, cs, n_chunks, rows_per_cta;
  bool q_multicast;
  size_t smem, q_bytes, kb_bytes, row_bytes, group_bytes, scratch_off;
  int64_t groups;
};

bool plan_step(int32_t nq, int32_t H, int32_t D, int64_t nb, int64_t n_full, int32_t k,
               const DeviceInfo& dev, StepPlan* p) {
  if (nq <= 0 || n_full <= 0 || D > 128) return false;
  const int64_t m_tiles = (n_full + kSTileM - 1) / kSTileM;
  if (m_tiles > kSMaxCluster) return false;
  // columns: the queries of a group times H, a multiple of 16, at most 256;
  // whole queries per 32-column TMEM load
  int bn = kSMaxBn;
  const int64_t need = static_cast<int64_t>(nq) * H;
  while (bn > 32 && bn / 2 >= need) bn /= 2;
  if (bn < H || bn % 32 != 0) bn = std::max(32, H);
  if (bn > kSMaxBn) return false;
  p->bn = bn;
  p->qg = bn / H;
  p->cs = static_cast<int>(m_tiles);
  // fp16 queries are multicast one slice per CTA when the slices are whole
  // 8-row swizzle atoms; otherwise every CTA loads the whole tile
  p->q_multicast = bn % p->cs == 0 && (bn / p->cs) % 8 == 0;
  p->n_chunks = (D + kSKAtom - 1) / kSKAtom;
  p->rows_per_cta = (p->qg + p->cs - 1) / p->cs;
  p->q_bytes = static_cast<size_t>(p->n_chunks) * bn * kSRowBytes;
  p->kb_bytes = static_cast<size_t>(p->n_chunks) * kSTileM * kSRowBytes;
  p->row_bytes = (static_cast<size_t>(nb) * 4 + 15) & ~static_cast<size_t>(15);
  if (static_cast<size_t>(p->rows_per_cta) * p->row_bytes > p->q_bytes) return false;
  const size_t k4 = (static_cast<size_t>(k) + 3) & ~static_cast<size_t>(3);
  p->group_bytes = kSelHistBins * 4 + static_cast<size_t>(kSelBinMax) * 8 + static_cast<size_t>(k) * 8 + k4 * 4;
  p->group_bytes = (p->group_bytes + 15) & ~static_cast<size_t>(15);
  const int n_groups = p->rows_per_cta >= 2 ? 2 : 1;
  p->scratch_off = p->q_bytes;  // 1024-byte multiple
  const size_t tail = std::max(p->kb_bytes, n_groups * p->group_bytes);
  p->smem = p->scratch_off + tail + 1024;  // + alignment slack
  // two CTAs per SM, so that 16-CTA clusters of a step fit on the GPU at once
  if (p->smem + g_step_static_smem > 113 * 1024) return false;
  if (p->smem + g_step_static_smem > static_cast<size_t>(dev.max_smem_optin)) return false;
  p->groups = (nq + p->qg - 1) / p->qg;
  return true;
}

}  // namespace

cudaError_t init_step_kernels(const DeviceInfo& dev) {
  for (int H : {1, 2, 4, 8, 16, 32})
    for (bool f : {false, true}) {
      const void* fn = step_kernel_for(H, f);
      cudaFuncAttributes fa;
      cudaError_t e = cudaFuncGetAttributes(&fa, fn);
      if (e != cudaSuccess) return e;
      g_step_static_smem = std::max(g_step_static_smem, static_cast<int>(fa.sharedSizeBytes));
      e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               dev.max_smem_optin - static_cast<int>(fa.sharedSizeBytes));
      if (e != cudaSuccess) return e;
      e = cudaFuncSetAttribute(fn, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
      if (e != cudaSuccess) return e;
      e = cudaFuncSetAttribute(fn, cudaFuncAttributePreferredSharedMemoryCarveout,
                               cudaSharedmemCarveoutMaxShared);
      if (e != cudaSuccess) return e;
    }
  return cudaSuccess;
}

bool step_supported(int32_t nq, int32_t H, int32_t D, int64_t nb, int64_t n_full, int32_t k,
                    const DeviceInfo& dev) {
  StepPlan p;
  return plan_step(nq, H, D, nb, n_full, k, dev, &p);
}

cudaError_t launch_step(const FusedProblem& fp, const DeviceInfo& dev, cudaStream_t stream) {
  StepPlan p;
  if (fp.n_batches != 1 || !plan_step(fp.nq, fp.H, fp.D, fp.nb, fp.n_full, fp.k, dev, &p))
    return cudaErrorInvalidValue;
  StepArgs a;
  a.q32 = fp.q32;
  a.q16out = reinterpret_cast<__half*>(fp.q16out);
  a.kb = reinterpret_cast<const __half*>(fp.kb);
  a.scores = fp.scores;
  a.ids = fp.ids;
  a.nq = fp.nq;
  a.D = fp.D;
  a.nb = static_cast<int32_t>(fp.nb);
  a.n_full = static_cast<int32_t>(fp.n_full);
  a.has_tail = fp.has_tail ? 1 : 0;
  a.k = fp.k;
  a.bn = p.bn;
  a.qg = p.qg;
  a.cs = p.cs;
  a.n_chunks = p.n_chunks;
  a.k_steps = fp.D / 16;
  a.rows_per_cta = p.rows_per_cta;
  a.q_multicast = p.q_multicast ? 1 : 0;
  a.row_bytes = static_cast<uint32_t>(p.row_bytes);
  a.scratch_off = static_cast<uint32_t>(p.scratch_off);
  a.group_bytes = static_cast<uint32_t>(p.group_bytes);
  a.tmem_cols = static_cast<uint32_t>(std::max(32, p.bn));
  a.status = dev.status_word;
  a.timeout_ns = kWaitTimeoutNs;

  CUtensorMap tm_kb, tm_q;
  memset(&tm_kb, 0, sizeof(tm_kb));
  memset(&tm_q, 0, sizeof(tm_q));
  if (!encode_2d(&tm_kb, fp.kb, fp.D, fp.n_full, kSKAtom, kSTileM)) return cudaErrorInvalidValue;
  if (fp.q32 == nullptr &&
      !encode_2d(&tm_q, fp.q16, fp.D, static_cast<uint64_t>(fp.nq) * fp.H, kSKAtom,
                 p.q_multicast ? p.bn / p.cs : p.bn))
    return cudaErrorInvalidValue;
  const void* fn = step_kernel_for(fp.H, fp.q32 != nullptr);
  if (fn == nullptr) return cudaErrorInvalidValue;
  plan_add("select_step_kernel (one 128-block tile per CTA, clusters of up to 16)");
  const int64_t blocks = p.groups * p.cs;
  if (blocks > 0x7FFFFFFFLL) return cudaErrorInvalidValue;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(blocks));
  cfg.blockDim = dim3(kSThreads);
  cfg.dynamicSmemBytes = p.smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = static_cast<unsigned>(p.cs);
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  void* args[] = {&tm_kb, &tm_q, &a};
  cudaError_t e = cudaLaunchKernelExC(&cfg, fn, args);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace qsa
