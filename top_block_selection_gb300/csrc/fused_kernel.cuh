// fused_kernel.cuh - the whole selection step in one launch: (fp32 -> fp16 query
// conversion,) tensor-core block scores with the fused ReLU / head-sum
// epilogue, the fp32 tail block with the +1e9 dead-tail rule, and the exact
// top-k select (Strata pull request 228, part 1: the block scorer and the
// "qsa select" phase of scores + selection + fp16 conversion; pull request
// 856, "What": the shared tail kernel and the dead-tail rule).
//
// Work decomposition. Queries are cut into groups of Qg queries (bn = Qg*H
// TMEM columns). One thread-block cluster of C CTAs (8; 16 in the wide form)
// owns a group: CTA rank r scores the 128-block tiles r, r+C, r+2C, ... of
// that group, so the cluster covers every KV block once while the group's
// query tile is shared by all its CTAs; CTA r selects the group's rows r,
// r+C, ....
//
// Roles inside a CTA (288 threads):
//   warp 8      TMA producer and tcgen05.mma issuer (one lane), TMEM owner;
//               two shared-memory stages for Kb tiles and two TMEM
//               accumulators, so tile t+1 is multiplied while tile t drains;
//   warps 0-7   the fp32 -> fp16 query conversion; then (warps 0-3 of the
//               tail-owner CTA) the tail block while the tiles load; then the
//               epilogue: warp w reads TMEM lane quarter w % 4 (one KV block
//               per thread) and half w / 4 of the columns, applies ReLU, sums
//               the H adjacent columns of each query in registers and stores
//               the scores (a warp writes 32 consecutive blocks); after the
//               cluster barrier, the select, one row at a time.
// When the rows a CTA selects fit in its shared memory next to the operand
// tiles ("DSMEM mode"), every producer of a score (epilogue or tail thread,
// on any CTA of the cluster) also stores the score's order-preserving key
// into the selecting CTA's key array over distributed shared memory
// (st.shared::cluster), so the select does not read the row back from
// global memory; otherwise it reads the row after the barrier.
// fp32 queries are rounded to fp16 (cvt.rn) straight into the 128-byte-
// swizzled operand layout. In DSMEM mode each CTA of the cluster rounds one
// eighth of the group's rows and stores them (st.async) into all eight CTAs'
// operand tiles, counted on each CTA's bar_q, so the cluster reads the fp32
// tile from L2 once; otherwise every CTA converts the whole tile. fp16
// queries arrive by TMA. Every wait is bounded; a CTA that gives up still reaches the
// cluster barriers, so the cluster never hangs on them.
#pragma once

#include <algorithm>
#include <cstring>

#include "qsa_device.cuh"
#include "qsa_internal.h"
#include "select_row.cuh"

namespace qsa {

constexpr int kWork = 256;         // warps 0..7: query conversion, tail, epilogue, select
constexpr int kProducerWarp = 8;   // warp 8: TMA + tcgen05.mma issue, TMEM owner
constexpr int kFThreads = kWork + 32;
constexpr int kFTileM = 128;
constexpr int kFRowBytes = 128;
constexpr int kFKAtom = 64;

struct FusedArgs {
  const float* q32;     // fp32 queries [nq,H,D], or nullptr when q arrives as fp16
  const __half* q16in;  // fp16 queries [nq,H,D] (fp16 input only)
  __half* q16out;       // optional fp16 copy of the converted queries (fp32 input only)
  const __half* kb;     // [nb, D]
  float* scores;        // [nq, nb]
  int32_t* ids;         // [nq, k]
  int32_t nq, D, nb, n_full, has_tail, k;
  int32_t groups_per_batch;  // query groups of one batch; blocks are (batch, group, rank)
  int64_t q_batch_elems;     // nq * H * D: q32 / q16 / q16out elements per batch
  int64_t kb_batch_stride;   // kb elements between batches; 0 = one kb shared by all
  int32_t bn, qg, m_tiles, n_chunks, k_steps;
  int32_t kb_stages;    // shared-memory stages for Kb tiles (2; 1 in the lean form)
  uint32_t tmem_cols;
  uint32_t sel_bytes;   // shared bytes of one select group (cand + sel, plus keys +
                        // hist in global mode)
  int32_t dsmem;        // 1: keys and first-digit histograms arrive over DSMEM
  int32_t q_share;      // 1: each CTA converts 1/8 of the fp32 query tile and
                        //    stores it into all eight CTAs' operand tiles (DSMEM)
  uint32_t row_bytes;   // DSMEM mode: bytes of one row's keys + histogram
  uint32_t rows_off;    // DSMEM mode: offset of the row regions in dynamic smem
  uint32_t* status;
  uint64_t timeout_ns;
};

__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

__device__ __forceinline__ void cluster_sync_release_acquire() {
  asm volatile(
      "barrier.cluster.arrive.release.aligned;\n\t"
      "barrier.cluster.wait.acquire.aligned;" ::
          : "memory");
}

// Arrive without release semantics: orders nothing but the CTA's start and
// the mbarrier initialisation made visible by fence.mbarrier_init (a release
// arrive waited about a microsecond here).
__device__ __forceinline__ void cluster_arrive_relaxed() {
  asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}

__device__ __forceinline__ void cluster_wait_acquire() {
  asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Address of the same shared-memory offset in CTA `rank` of this cluster.
__device__ __forceinline__ uint32_t cluster_map(uint32_t saddr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
  return r;
}

// Remote store that signals its 4 bytes on the destination CTA's mbarrier
// (both addresses in the same peer CTA).
__device__ __forceinline__ void st_async_u32(uint32_t addr, uint32_t v, uint32_t bar) {
  asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.u32 [%0], %1, [%2];" ::"r"(
                   addr),
               "r"(v), "r"(bar)
               : "memory");
}

// 16-byte remote store, signalled on the destination CTA's mbarrier.
__device__ __forceinline__ void st_async_v4(uint32_t addr, const uint4& v, uint32_t bar) {
  asm volatile(
      "st.async.shared::cluster.mbarrier::complete_tx::bytes.v4.b32 [%0], {%1, %2, %3, %4}, [%5];" ::"r"(
          addr),
      "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w), "r"(bar)
      : "memory");
}

// Sends one score's key to keys[b] of the row's region in the CTA that
// selects the row (rank ql % kCluster, row slot ql / kCluster), counted on that CTA's
// bar_keys. A remote store, not a remote atomic (those are slow): the owner
// builds the row's histogram itself. The owner waits on its own barrier for
// the bytes of all its rows, so no cluster-wide release (which would also
// wait for this thread's global score stores) is needed.
template <int kCluster>
__device__ __forceinline__ void send_key(uint32_t rows_base, uint32_t row_bytes, uint32_t bar_keys,
                                         int ql, int b, float score) {
  const uint32_t owner = static_cast<uint32_t>(ql % kCluster);
  const uint32_t local = rows_base + static_cast<uint32_t>(ql / kCluster) * row_bytes;
  st_async_u32(cluster_map(local, owner) + static_cast<uint32_t>(b) * 4u, score_key(score),
               cluster_map(bar_keys, owner));
}

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

// Byte offset of fp16 element (row, i) in a K-major tile of `rows` rows stored
// as 64-column chunks of 128-byte rows with the 128-byte swizzle (16-byte
// unit u of row r lives at unit u ^ (r & 7)).
__device__ __forceinline__ uint32_t sw128_offset(int rows, int row, int i) {
  const int chunk = i >> 6;
  const int unit = (i & 63) >> 3;
  return static_cast<uint32_t>(chunk * rows * kFRowBytes + row * kFRowBytes +
                               ((unit ^ (row & 7)) << 4) + ((i & 7) << 1));
}

// Forms of the kernel (the cluster size is set at launch):
//   kFormRegular  8-CTA clusters, two Kb stages, at most 96 registers;
//   kFormLean     8-CTA clusters, at most 72 registers (with one Kb stage,
//                 three CTAs fit an SM), for launches of many waves where
//                 CTAs overlap one another;
//   kFormWide     16-CTA clusters (one 128-block tile per CTA for 2048
//                 blocks), for launches of one or two clusters (decode-shaped
//                 steps), where the SMs are idle anyway and each CTA's load
//                 and MMA chain halve.
constexpr int kFormRegular = 0, kFormLean = 1, kFormWide = 2;

template <int H, bool kF32Q, int kForm>
__global__ void __maxnreg__(kForm == kFormLean ? 72 : 96)
    fused_step_kernel(const __grid_constant__ CUtensorMap tm_kb,
                      const __grid_constant__ CUtensorMap tm_q, const FusedArgs a) {
  constexpr int kCluster = kForm == kFormWide ? 16 : 8;
  static_assert(32 % H == 0, "a 32-column TMEM load must hold whole queries");
  extern __shared__ uint8_t smem_raw[];
  __shared__ uint64_t bar_full[2], bar_empty[2], bar_acc_full[2], bar_acc_empty[2], bar_q, bar_keys;
  __shared__ uint32_t tmem_slot;
  __shared__ int failed;
  __shared__ float tail_acc[256];
  __shared__ SelectShared sel_sh;
  __shared__ GroupShared sel_gsh;

  const uint32_t raw = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + ((1024u - (raw & 1023u)) & 1023u);
  uint8_t* sQ = smem;                                             // n_chunks x bn rows x 128 B
  uint8_t* sKB = sQ + a.n_chunks * a.bn * kFRowBytes;              // kb_stages stages
  const int stage_bytes = a.n_chunks * kFTileM * kFRowBytes;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int rank = static_cast<int>(cluster_rank());
  const int cluster_id = blockIdx.x / kCluster;
  const int batch = cluster_id / a.groups_per_batch;
  const int group = cluster_id - batch * a.groups_per_batch;
  const int q0 = group * a.qg;                 // first query of the group (in its batch)
  // this block's batch: its slices of every tensor
  const float* q32b = kF32Q ? a.q32 + batch * a.q_batch_elems : nullptr;
  __half* q16outb = a.q16out != nullptr ? a.q16out + batch * a.q_batch_elems : nullptr;
  const __half* kbb = a.kb + batch * a.kb_batch_stride;
  float* scoresb = a.scores + static_cast<int64_t>(batch) * a.nq * a.nb;
  int32_t* idsb = a.ids + static_cast<int64_t>(batch) * a.nq * a.k;
  const int kb_z = a.kb_batch_stride != 0 ? batch : 0;  // kb tensor map: 3rd coordinate
  const int q_row0 = batch * a.nq * H;                  // fp16 q tensor map: batch row offset
  const int col0 = q0 * H;                     // first row of the [nq*H, D] query view
  const int qh_rows = min(a.bn, (a.nq - q0) * H);
  const int n_local = a.m_tiles > rank ? (a.m_tiles - rank + kCluster - 1) / kCluster : 0;
  const bool tail_owner = a.has_tail && rank == kCluster - 1;
  const bool need_q = n_local > 0 || tail_owner || (kF32Q && q16outb != nullptr && rank == 0);
  const int rows_here = a.qg > rank ? (a.qg - rank + kCluster - 1) / kCluster : 0;
  const uint32_t rows_base = smem_u32(smem + a.rows_off);
  const uint32_t keys_bar = smem_u32(&bar_keys);
  const bool producer_warp = warp == kProducerWarp;

  // Programmatic dependent launch: the next kernel on the stream may start its
  // own set-up now; this kernel reads nothing produced by earlier work on the
  // stream before pdl_wait() below.
  pdl_launch_dependents();
  if (tid == kProducerWarp * 32) {
    for (int s = 0; s < 2; ++s) {
      mbar_init(&bar_full[s], 1);
      mbar_init(&bar_empty[s], 1);
      mbar_init(&bar_acc_full[s], 1);
      mbar_init(&bar_acc_empty[s], kWork);
    }
    mbar_init(&bar_q, 1);
    mbar_init(&bar_keys, 1);
    failed = 0;
    fence_mbarrier_init();
    // DSMEM mode: this CTA expects the keys of its valid rows (nb keys each),
    // registered before the cluster barrier that lets peers send.
    if (a.dsmem) {
      int rows_valid = 0;
      for (int r = 0; r < rows_here && q0 + rank + r * kCluster < a.nq; ++r) ++rows_valid;
      mbar_arrive_expect_tx(&bar_keys, static_cast<uint32_t>(rows_valid * a.nb) * 4u);
    }
    // Shared query tile: the eight CTAs' slices arrive on bar_q.
    if (a.q_share)
      mbar_arrive_expect_tx(&bar_q, static_cast<uint32_t>(a.n_chunks * a.bn * kFRowBytes));
    if (n_local > 0) tma_prefetch_desc(&tm_kb);
    if (!kF32Q && need_q) tma_prefetch_desc(&tm_q);
    // Start this CTA's first operand tiles on their way from HBM to L2 while
    // the previous kernel finishes; the loads proper come after the wait.
    for (int t = 0; t < 2 && t < n_local; ++t)
      for (int c = 0; c < a.n_chunks; ++c)
        tma_prefetch_l2_3d(&tm_kb, c * kFKAtom, (rank + t * kCluster) * kFTileM, kb_z);
    if (a.q_share) {
      const int rows_per = a.bn / kCluster, r0 = rank * rows_per;
      const int rows = min(rows_per, qh_rows - r0);
      if (rows > 0) {
        const char* qp = reinterpret_cast<const char*>(q32b + static_cast<int64_t>(col0 + r0) * a.D);
        bulk_prefetch_l2(qp, static_cast<uint32_t>(rows) * a.D * 4u);
      }
    } else if (need_q) {
      if (kF32Q) {
        const char* qp = reinterpret_cast<const char*>(q32b + static_cast<int64_t>(col0) * a.D);
        const uint32_t q_bytes = static_cast<uint32_t>(qh_rows) * a.D * 4u;
        for (uint32_t off = 0; off < q_bytes; off += 16384u)
          bulk_prefetch_l2(qp + off, min(16384u, q_bytes - off));
      } else {
        for (int c = 0; c < a.n_chunks; ++c)
          tma_prefetch_l2_2d(&tm_q, c * kFKAtom, q_row0 + col0);
      }
    }
  }
  // DSMEM mode: peers store into this CTA's shared memory (keys, counted on
  // bar_keys) only after every CTA of the cluster has started and initialised
  // its barriers: this arrive, and the wait before a thread's first remote
  // store. Arriving before the dependency wait lets the barrier complete
  // while the previous kernel finishes.
  __syncwarp();
  if (a.dsmem) cluster_arrive_relaxed();
  // The TMEM allocation comes before the wait too, and every CTA then gives
  // up its allocation permit, also one that allocates nothing: a CTA holding
  // the permit keeps the SM from taking another CTA (measured: ranks without
  // tiles that kept it halved the resident clusters, and early-launched CTAs
  // that kept it across the wait held back half the next step's clusters
  // until the previous step had completed).
  if (producer_warp) {
    __syncwarp();
    if (n_local > 0) tmem_alloc(&tmem_slot, a.tmem_cols);
    tmem_relinquish();
  }
  pdl_wait();
  if (tid == kProducerWarp * 32) {
    if (!kF32Q && need_q) {
      mbar_arrive_expect_tx(&bar_q, static_cast<uint32_t>(a.n_chunks * a.bn * kFRowBytes));
      for (int c = 0; c < a.n_chunks; ++c)
        tma_load_2d(sQ + c * a.bn * kFRowBytes, &tm_q, c * kFKAtom, q_row0 + col0, &bar_q);
    }
    for (int t = 0; t < a.kb_stages && t < n_local; ++t) {
      const int m = rank + t * kCluster;
      mbar_arrive_expect_tx(&bar_full[t], static_cast<uint32_t>(stage_bytes));
      for (int c = 0; c < a.n_chunks; ++c)
        tma_load_3d(sKB + t * stage_bytes + c * kFTileM * kFRowBytes, &tm_kb, c * kFKAtom,
                    m * kFTileM, kb_z, &bar_full[t]);
    }
  }
  __syncwarp();
  // Work warps that already waited on the cluster start barrier (share mode).
  bool cl_waited = false;
  if (!producer_warp && kF32Q && a.q_share) {
    // This CTA's slice of the query tile: rows [rank*bn/8, (rank+1)*bn/8),
    // rounded to fp16 and stored as 16-byte swizzle units into every CTA of
    // the cluster (its own included), counted on each CTA's bar_q. Rows past
    // the last query and columns past D are sent as zeros, so every CTA
    // receives the whole tile.
    const int rows_per = a.bn / kCluster;
    const int units_per_row = a.n_chunks * (kFKAtom / 8);
    const int n_units = rows_per * units_per_row;
    const uint32_t sq_local = smem_u32(sQ), bar_local = smem_u32(&bar_q);
    auto load_unit = [&](int u, float4& v0, float4& v1) {
      const int row = rank * rows_per + u / units_per_row;
      const int i = (u % units_per_row) * 8;
      v0 = make_float4(0.f, 0.f, 0.f, 0.f);
      v1 = v0;
      if (row < qh_rows && i < a.D) {
        const float4* src =
            reinterpret_cast<const float4*>(q32b + static_cast<int64_t>(col0 + row) * a.D + i);
        v0 = __ldg(src);
        v1 = __ldg(src + 1);
      }
    };
    // The first unit's loads are in flight during the cluster wait.
    float4 v0, v1;
    if (tid < n_units) load_unit(tid, v0, v1);
    cluster_wait_acquire();
    cl_waited = true;
    for (int u = tid; u < n_units; u += kWork) {
      if (u != tid) load_unit(u, v0, v1);
      const int row = rank * rows_per + u / units_per_row;
      const int i = (u % units_per_row) * 8;
      const __half2 h01 = __floats2half2_rn(v0.x, v0.y), h23 = __floats2half2_rn(v0.z, v0.w);
      const __half2 h45 = __floats2half2_rn(v1.x, v1.y), h67 = __floats2half2_rn(v1.z, v1.w);
      uint4 pk;
      pk.x = *reinterpret_cast<const uint32_t*>(&h01);
      pk.y = *reinterpret_cast<const uint32_t*>(&h23);
      pk.z = *reinterpret_cast<const uint32_t*>(&h45);
      pk.w = *reinterpret_cast<const uint32_t*>(&h67);
      if (q16outb != nullptr && row < qh_rows && i < a.D)
        *reinterpret_cast<uint4*>(q16outb + static_cast<int64_t>(col0 + row) * a.D + i) = pk;
      const uint32_t off = sw128_offset(a.bn, row, i);
#pragma unroll
      for (int dst = 0; dst < kCluster; ++dst)
        st_async_v4(cluster_map(sq_local + off, static_cast<uint32_t>(dst)), pk,
                    cluster_map(bar_local, static_cast<uint32_t>(dst)));
    }
  } else if (!producer_warp && kF32Q && need_q) {
    // fp32 queries -> fp16 (round to nearest even) -> swizzled operand tile,
    // by the kWork threads. Rows past the last query and columns past D are 0.
    const int f4_per_row = a.n_chunks * (kFKAtom / 4);
    if (kWork % f4_per_row == 0) {
      // Each thread keeps one 4-column group and steps down the rows.
      const int rstep = kWork / f4_per_row;
      const int i = (tid % f4_per_row) * 4;
      const int r0 = tid / f4_per_row;
      const bool col_ok = i < a.D;
      const int64_t src_step = static_cast<int64_t>(rstep) * a.D;
      const float* src = q32b + static_cast<int64_t>(col0 + r0) * a.D + i;
      for (int base = r0; base < a.bn; base += 8 * rstep, src += 8 * src_step) {
        float4 v[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          v[j] = make_float4(0.f, 0.f, 0.f, 0.f);
          if (base + j * rstep < qh_rows && col_ok)
            v[j] = __ldg(reinterpret_cast<const float4*>(src + j * src_step));
        }
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const int row = base + j * rstep;
          if (row < a.bn) {
            const __half2 h01 = __floats2half2_rn(v[j].x, v[j].y);
            const __half2 h23 = __floats2half2_rn(v[j].z, v[j].w);
            uint2 pk;
            pk.x = *reinterpret_cast<const uint32_t*>(&h01);
            pk.y = *reinterpret_cast<const uint32_t*>(&h23);
            *reinterpret_cast<uint2*>(sQ + sw128_offset(a.bn, row, i)) = pk;
            if (q16outb != nullptr && rank == 0 && row < qh_rows && col_ok)
              *reinterpret_cast<uint2*>(q16outb + static_cast<int64_t>(col0 + row) * a.D + i) = pk;
          }
        }
      }
    } else {
      const int total = a.bn * f4_per_row;
      for (int base = 0; base < total; base += 8 * kWork) {
        float4 v[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const int f = base + j * kWork + tid;
          const int row = f / f4_per_row;
          const int i = (f - row * f4_per_row) * 4;
          v[j] = make_float4(0.f, 0.f, 0.f, 0.f);
          if (f < total && row < qh_rows && i < a.D)
            v[j] = __ldg(reinterpret_cast<const float4*>(q32b + static_cast<int64_t>(col0 + row) * a.D + i));
        }
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const int f = base + j * kWork + tid;
          if (f < total) {
            const int row = f / f4_per_row;
            const int i = (f - row * f4_per_row) * 4;
            const __half2 h01 = __floats2half2_rn(v[j].x, v[j].y);
            const __half2 h23 = __floats2half2_rn(v[j].z, v[j].w);
            uint2 pk;
            pk.x = *reinterpret_cast<const uint32_t*>(&h01);
            pk.y = *reinterpret_cast<const uint32_t*>(&h23);
            *reinterpret_cast<uint2*>(sQ + sw128_offset(a.bn, row, i)) = pk;
            if (q16outb != nullptr && rank == 0 && row < qh_rows && i < a.D)
              *reinterpret_cast<uint2*>(q16outb + static_cast<int64_t>(col0 + row) * a.D + i) = pk;
          }
        }
      }
    }
    fence_proxy_async_smem();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem_base = tmem_slot;

  if (producer_warp) {
    // ---------------------------------------------------- producer / MMA
    if (lane == 0 && n_local > 0) {
      const uint32_t idesc = idesc_f16_f32(kFTileM, a.bn);
      bool ok = (kF32Q && !a.q_share) ? true : mbar_wait_bounded(&bar_q, 0, a.timeout_ns);
      // Peers' st.async writes of the query tile, then the tensor core's reads.
      if (a.q_share) fence_proxy_async_smem();
      for (int t = 0; t < n_local && ok; ++t) {
        const int s = t & 1;  // accumulator
        const uint32_t use = static_cast<uint32_t>(t >> 1);
        const int ks = t % a.kb_stages;  // Kb stage
        const uint32_t kuse = static_cast<uint32_t>(t / a.kb_stages);
        if (!mbar_wait_bounded(&bar_full[ks], kuse & 1u, a.timeout_ns)) { ok = false; break; }
        if (t >= 2 && !mbar_wait_bounded(&bar_acc_empty[s], (use - 1) & 1u, a.timeout_ns)) {
          ok = false;
          break;
        }
        tc_fence_after_sync();
        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(s * a.bn);
        const uint32_t a_base = smem_u32(sKB + ks * stage_bytes);
        const uint32_t b_base = smem_u32(sQ);
        for (int step = 0; step < a.k_steps; ++step) {
          const int c = step >> 2, kk = step & 3;
          mma_f16_ss(d_tmem, smem_desc_k_sw128(a_base + c * kFTileM * kFRowBytes + kk * 32),
                     smem_desc_k_sw128(b_base + c * a.bn * kFRowBytes + kk * 32), idesc,
                     step > 0 ? 1u : 0u);
        }
        mma_commit(&bar_acc_full[s]);
        mma_commit(&bar_empty[ks]);
        if (t + a.kb_stages < n_local) {
          if (!mbar_wait_bounded(&bar_empty[ks], kuse & 1u, a.timeout_ns)) { ok = false; break; }
          const int m = rank + (t + a.kb_stages) * kCluster;
          mbar_arrive_expect_tx(&bar_full[ks], static_cast<uint32_t>(stage_bytes));
          for (int c = 0; c < a.n_chunks; ++c)
            tma_load_3d(sKB + ks * stage_bytes + c * kFTileM * kFRowBytes, &tm_kb, c * kFKAtom,
                        m * kFTileM, kb_z, &bar_full[ks]);
        }
      }
      if (!ok) {
        failed = 1;
        atomicOr(a.status, kErrScoreLoadTimeout);
        // Complete both accumulators' "full" barriers so the epilogue does not
        // wait out its own bound, then drain loads still in flight.
        mma_commit(&bar_acc_full[0]);
        mma_commit(&bar_acc_full[1]);
        for (int s = 0; s < a.kb_stages && s < n_local; ++s) mbar_wait_bounded(&bar_full[s], 0, a.timeout_ns);
      }
    }
    __syncwarp();
    if (a.dsmem) cluster_wait_acquire();  // pairs with the early arrive
  } else {
    // Peers' shared memory is written below (keys over DSMEM): every CTA of
    // the cluster must have started, which the early arrive and one wait per
    // thread guarantee. Each warp waits just before its first remote store
    // (warp-uniform flag), which keeps the cluster's start skew off the
    // loads, the MMAs and the tail's dot products.
    bool waited = !a.dsmem || cl_waited;
    // ------------------------------ tail block (warps 0..3 of the owner)
    if (tail_owner && warp < 4) {
      if ((!kF32Q || a.q_share) && !mbar_wait_bounded(&bar_q, 0, a.timeout_ns)) {
        failed = 1;
        atomicOr(a.status, kErrScoreLoadTimeout);
      }
      const int pairs = qh_rows;
      const __half* krow = kbb + static_cast<int64_t>(a.nb - 1) * a.D;
      for (int p = tid; p < pairs; p += 128) {
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
      asm volatile("bar.sync 3, 128;" ::: "memory");
      if (!waited) {
        cluster_wait_acquire();
        waited = true;
      }
      for (int ql = tid; ql * H < pairs; ql += 128) {
        float s = 0.0f;
#pragma unroll
        for (int h = 0; h < H; ++h) s = __fadd_rn(s, fmaxf(tail_acc[ql * H + h], 0.0f));
        const float score = __fadd_rn(s, 1.0e9f);
        scoresb[static_cast<int64_t>(q0 + ql) * a.nb + (a.nb - 1)] = score;
        if (a.dsmem) send_key<kCluster>(rows_base, a.row_bytes, keys_bar, ql, a.nb - 1, score);
      }
    }
    // ---------------------------------------- epilogue (warps 0..7)
    // Warp w reads TMEM lane quarter w % 4 (one KV block per thread) and the
    // half w / 4 of the tile's columns.
    const int quarter = warp & 3;
    const int half_cols = a.bn >> 1;
    const int c_begin = (warp >> 2) * half_cols;
    for (int t = 0; t < n_local; ++t) {
      const int s = t & 1;
      const uint32_t use = static_cast<uint32_t>(t >> 1);
      if (!mbar_wait_bounded(&bar_acc_full[s], use & 1u, a.timeout_ns)) {
        failed = 1;
        if (lane == 0) atomicOr(a.status, kErrScoreMmaTimeout);
        break;
      }
      tc_fence_after_sync();
      if (!waited) {
        cluster_wait_acquire();
        waited = true;
      }
      if (failed) break;
      const int b = (rank + t * kCluster) * kFTileM + quarter * 32 + lane;
      const bool b_ok = b < a.n_full;
      float* out = scoresb + b;
      const uint32_t taddr =
          tmem_base + static_cast<uint32_t>(s * a.bn) + (static_cast<uint32_t>(quarter * 32) << 16);
      constexpr int kQPerLoad = 32 / H;
      for (int c0 = c_begin; c0 < c_begin + half_cols; c0 += 32) {
        uint32_t r[32];
        tmem_ld_32cols(taddr + c0, r);
        tmem_ld_wait();
#pragma unroll
        for (int j = 0; j < kQPerLoad; ++j) {
          float sc = 0.0f;
#pragma unroll
          for (int h = 0; h < H; ++h) sc = __fadd_rn(sc, fmaxf(__uint_as_float(r[j * H + h]), 0.0f));
          const int ql = c0 / H + j;
          if (b_ok && q0 + ql < a.nq) {
            out[static_cast<int64_t>(q0 + ql) * a.nb] = sc;
            if (a.dsmem) send_key<kCluster>(rows_base, a.row_bytes, keys_bar, ql, b, sc);
          }
        }
      }
      tc_fence_before_sync();
      mbar_arrive(&bar_acc_empty[s]);
    }
    if (!waited) cluster_wait_acquire();
  }

  // Share mode: every slice of the query tile has landed here before this
  // CTA's shared memory is reused (select scratch) or released.
  if (a.q_share && tid == 0 && !mbar_wait_bounded(&bar_q, 0, a.timeout_ns))
    atomicOr(a.status, kErrScoreLoadTimeout);
  tc_fence_before_sync();
  __syncthreads();
  if (n_local > 0 && producer_warp) tmem_dealloc(tmem_base, a.tmem_cols);

  if (a.dsmem) {
    // Every key of this CTA's rows has arrived once bar_keys completes.
    if (producer_warp) return;  // the select runs on the kWork threads
    if (!mbar_wait_bounded(&bar_keys, 0, a.timeout_ns)) {
      if (tid == 0) atomicOr(a.status, kErrFusedWaitTimeout);
    }
  } else {
    // Every score of the group is written and visible after this barrier.
    cluster_sync_release_acquire();
    if (producer_warp) return;  // the select runs on the kWork threads
  }

  // ---------------------------------------------------------- select
  // One row at a time with the kWork threads (the lowest latency per row).
  // Keys come from the row regions (DSMEM mode) or from global memory;
  // hist / cand / sel reuse the dead operand tiles.
  uint32_t* hist = reinterpret_cast<uint32_t*>(smem);
  uint32_t* excl = hist + kSelHistBins;
  uint64_t* cand = reinterpret_cast<uint64_t*>(excl + kSelHistBins);
  uint64_t* sel = cand + kSelBinMax;
  uint32_t* sel_bin = reinterpret_cast<uint32_t*>(sel + a.k);
  uint32_t* staged = sel_bin + ((a.k + 3) & ~3);
  for (int r = 0; r < rows_here; ++r) {
    const int qi = q0 + rank + r * kCluster;
    if (qi >= a.nq) break;
    int32_t* out = idsb + static_cast<int64_t>(qi) * a.k;
    const float* row = scoresb + static_cast<int64_t>(qi) * a.nb;
    const uint32_t* rk = reinterpret_cast<const uint32_t*>(smem + a.rows_off + r * a.row_bytes);
    if (a.nb <= 64) {
      // Short rows: one warp, no block barrier (the other warps go on to the
      // loop's barrier).
      if (warp == 0) {
        uint32_t k0 = 0, k1 = 0;
        if (a.dsmem) {
          if (lane < a.nb) k0 = rk[lane];
          if (lane + 32 < a.nb) k1 = rk[lane + 32];
        } else {
          if (lane < a.nb) k0 = score_key(__ldcg(row + lane));
          if (lane + 32 < a.nb) k1 = score_key(__ldcg(row + lane + 32));
        }
        select_row_warp64(k0, k1, a.nb, a.k, out, lane);
      }
    } else if (a.nb <= 8 * kWork) {
      uint32_t key[8];
      if (a.dsmem) load_keys_regs<kWork, 8>(rk, a.nb, key, hist, tid);
      else load_keys_regs_global<kWork, 8>(row, a.nb, key, hist, tid);
      if (!select_row_thr<kWork, 8>(key, a.nb, a.k, out, cand, sel_sh, tid, 1) &&
          !select_row_window<kWork, 8>(key, a.nb, a.k, out, hist, excl, cand, sel, sel_bin, sel_sh,
                                        tid, 1)) {
        build_first_digit_hist<kWork, 8>(key, a.nb, hist, tid, 1);
        select_row_regs<kWork, 8>(key, a.nb, a.k, out, hist, cand, sel, sel_sh, tid, 1);
      }
    } else if (a.nb <= 16 * kWork) {
      uint32_t key[16];
      if (a.dsmem) load_keys_regs<kWork, 16>(rk, a.nb, key, hist, tid);
      else load_keys_regs_global<kWork, 16>(row, a.nb, key, hist, tid);
      if (!select_row_thr<kWork, 16>(key, a.nb, a.k, out, cand, sel_sh, tid, 1) &&
          !select_row_window<kWork, 16>(key, a.nb, a.k, out, hist, excl, cand, sel, sel_bin, sel_sh,
                                        tid, 1)) {
        build_first_digit_hist<kWork, 16>(key, a.nb, hist, tid, 1);
        select_row_regs<kWork, 16>(key, a.nb, a.k, out, hist, cand, sel, sel_sh, tid, 1);
      }
    } else {
      const uint32_t* keys = rk;
      if (!a.dsmem) {
        for (int b0 = 0; b0 < a.nb; b0 += 8 * kWork) {
          float v[8];
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            const int i = b0 + j * kWork + tid;
            v[j] = i < a.nb ? __ldcg(row + i) : 0.0f;
          }
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            const int i = b0 + j * kWork + tid;
            if (i < a.nb) staged[i] = score_key(v[j]);
          }
        }
        group_sync<kWork>(1);
        keys = staged;
      }
      select_row_g<kWork / 32>(keys, a.nb, a.k, out, hist, cand, sel, sel_gsh, tid, 1);
    }
    group_sync<kWork>(1);
  }
}

// The kernel of (f32 queries?, form) for H heads; taking the addresses
// instantiates the kernels in the calling translation unit.
template <int H>
const void* fused_kernel_ptr(bool f32q, int form) {
  if (f32q) {
    return form == kFormLean   ? reinterpret_cast<const void*>(&fused_step_kernel<H, true, kFormLean>)
           : form == kFormWide ? reinterpret_cast<const void*>(&fused_step_kernel<H, true, kFormWide>)
                               : reinterpret_cast<const void*>(&fused_step_kernel<H, true, kFormRegular>);
  }
  return form == kFormLean   ? reinterpret_cast<const void*>(&fused_step_kernel<H, false, kFormLean>)
         : form == kFormWide ? reinterpret_cast<const void*>(&fused_step_kernel<H, false, kFormWide>)
                             : reinterpret_cast<const void*>(&fused_step_kernel<H, false, kFormRegular>);
}

// One per H, each in its own translation unit (compiled in parallel).
const void* fused_kernel_h1(bool f32q, int form);
const void* fused_kernel_h2(bool f32q, int form);
const void* fused_kernel_h4(bool f32q, int form);
const void* fused_kernel_h8(bool f32q, int form);
const void* fused_kernel_h16(bool f32q, int form);
const void* fused_kernel_h32(bool f32q, int form);

}  // namespace qsa
