// score_tc.cu - QSA block scores on the sm_103a tensor cores, and the tail
// block kernel.
//
// score(qi, b) = sum_h relu(sum_i kb[b, i] * q[qi, h, i])   (Strata pull request
// 228, part 1, "qsa_block_scores_wmma": the multi-query block scorer).
//
// Full blocks: the contraction is the GEMM  Kb[n_full, D] x Q2[nq*H, D]^T  with
// Q2 the [nq*H, D] view of q, computed swap-AB so that the 128 KV blocks of a
// tile sit on the 128 TMEM lanes and the (query, head) pairs of the tile, head
// fastest, sit on the TMEM columns. One CTA per (128-block, bn-column) tile:
//   - thread 0 issues TMA loads of the tile's Kb rows and Q2 rows, one
//     mbarrier per 64-wide K chunk (128-byte swizzled rows), then the
//     tcgen05.mma kind::f16 steps (M=128, N=bn, K=16 each; fp16 in, fp32
//     accumulate in TMEM) as each chunk lands, and one tcgen05.commit;
//   - all four warps then read their 32 TMEM lanes (one KV block per thread),
//     apply ReLU per head and sum the H adjacent columns of each query in
//     registers, and store scores[qi, b] (a warp writes 32 consecutive b).
// The [nq*H, n_full] pre-activation matrix never leaves TMEM and registers.
//
// Tail block (Strata pull request 856, "What": the shared tail kernel and the
// +1e9 dead-tail rule): the rows of q staged in shared memory, one thread per
// (query, head) sums the fp32 products over i in order; one thread per query then sums max(acc_h, 0) over h in
// order and adds 1e9f. Every step is a round-to-nearest-even fp32 operation
// (no contraction, no reassociation), so the result is reproducible bit for
// bit.
#include <algorithm>

#include "qsa_device.cuh"
#include "qsa_internal.h"

namespace qsa {

constexpr int kTileM = 128;        // KV blocks per tile = MMA M = TMEM lanes
constexpr int kKAtom = 64;         // fp16 elements per 128-byte swizzled row
constexpr int kRowBytes = 128;
constexpr int kScoreThreads = 128; // 4 warps = the 4 TMEM lane quarters
constexpr int kTailThreads = 256;

struct ScoreArgs {
  float* scores;
  int32_t nq, nb, n_full;
  int32_t bn;          // TMEM columns (query-head pairs) per tile, multiple of 32
  int32_t q_per_tile;  // bn / H
  int32_t n_chunks;    // ceil(D / 64)
  int32_t k_steps;     // D / 16
  uint32_t tmem_cols;  // power of two >= bn
  uint32_t* status;
  uint64_t timeout_ns;
  int32_t kb_z;        // persistent kernel: 1 when each batch has its own kb (3rd map coordinate)
};

template <int H>
__global__ void __launch_bounds__(kScoreThreads, 1)
    score_tc_kernel(const __grid_constant__ CUtensorMap tm_kb,
                    const __grid_constant__ CUtensorMap tm_q, const ScoreArgs a) {
  static_assert(32 % H == 0, "a 32-column TMEM load must hold whole queries");
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + ((1024u - (raw & 1023u)) & 1023u);
  uint8_t* sA = smem;                                           // n_chunks x [128 rows x 128 B]
  uint8_t* sB = sA + a.n_chunks * kTileM * kRowBytes;           // n_chunks x [bn rows x 128 B]
  uint64_t* bars = reinterpret_cast<uint64_t*>(sB + a.n_chunks * a.bn * kRowBytes);
  uint64_t* mma_bar = bars + a.n_chunks;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(mma_bar + 1);
  volatile int* failed = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int m0 = blockIdx.x * kTileM;
  const int col0 = blockIdx.y * a.bn;

  pdl_launch_dependents();
  if (threadIdx.x == 0) {
    for (int c = 0; c < a.n_chunks; ++c) mbar_init(&bars[c], 1);
    mbar_init(mma_bar, 1);
    *failed = 0;
    fence_mbarrier_init();
    tma_prefetch_desc(&tm_kb);
    tma_prefetch_desc(&tm_q);
  }
  if (warp == 0) {
    tmem_alloc(tmem_slot, a.tmem_cols);
    tmem_relinquish();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem_d = *tmem_slot;
  pdl_wait();  // q and kb may come from the previous kernel on the stream

  if (threadIdx.x == 0) {
    const uint32_t chunk_bytes = static_cast<uint32_t>((kTileM + a.bn) * kRowBytes);
    for (int c = 0; c < a.n_chunks; ++c) {
      mbar_arrive_expect_tx(&bars[c], chunk_bytes);
      tma_load_2d(sA + c * kTileM * kRowBytes, &tm_kb, c * kKAtom, m0, &bars[c]);
      tma_load_2d(sB + c * a.bn * kRowBytes, &tm_q, c * kKAtom, col0, &bars[c]);
    }
    const uint32_t idesc = idesc_f16_f32(kTileM, a.bn);
    bool ok = true;
    for (int c = 0; c < a.n_chunks; ++c) {
      if (!mbar_wait_bounded(&bars[c], 0, a.timeout_ns)) {
        ok = false;
        break;
      }
      tc_fence_after_sync();
      const uint32_t a_base = smem_u32(sA + c * kTileM * kRowBytes);
      const uint32_t b_base = smem_u32(sB + c * a.bn * kRowBytes);
#pragma unroll
      for (int s = 0; s < kKAtom / 16; ++s) {
        const int step = c * (kKAtom / 16) + s;
        if (step < a.k_steps)
          mma_f16_ss(tmem_d, smem_desc_k_sw128(a_base + s * 32), smem_desc_k_sw128(b_base + s * 32),
                     idesc, step > 0 ? 1u : 0u);
      }
    }
    mma_commit(mma_bar);  // arrives once every MMA issued above has completed
    if (!ok) {
      *failed = 1;
      atomicOr(a.status, kErrScoreLoadTimeout);
      // Loads may still be in flight into this CTA's shared memory: wait for
      // them (bounded) before the CTA may finish.
      for (int c = 0; c < a.n_chunks; ++c) mbar_wait_bounded(&bars[c], 0, a.timeout_ns);
    }
  }
  __syncwarp();

  if (!mbar_wait_bounded(mma_bar, 0, a.timeout_ns)) {
    *failed = 1;
    if (lane == 0) atomicOr(a.status, kErrScoreMmaTimeout);
  }
  __syncthreads();
  if (*failed == 0) {
    tc_fence_after_sync();
    const int lane_base = (warp & 3) * 32;
    const int b = m0 + lane_base + lane;
    const bool b_ok = b < a.n_full;
    float* out = a.scores + b;
    const int q0 = blockIdx.y * a.q_per_tile;
    constexpr int kQPerLoad = 32 / H;
    for (int c0 = 0; c0 < a.bn; c0 += 32) {
      uint32_t r[32];
      tmem_ld_32cols(tmem_d + (static_cast<uint32_t>(lane_base) << 16) + c0, r);
      tmem_ld_wait();
#pragma unroll
      for (int j = 0; j < kQPerLoad; ++j) {
        float s = 0.0f;
#pragma unroll
        for (int h = 0; h < H; ++h) s = __fadd_rn(s, fmaxf(__uint_as_float(r[j * H + h]), 0.0f));
        const int qidx = q0 + c0 / H + j;
        if (b_ok && qidx < a.nq) out[static_cast<size_t>(qidx) * a.nb] = s;
      }
    }
  }
  tc_fence_before_sync();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem_d, a.tmem_cols);
}

// ------------------------------------------------- persistent variant
// For problems of many tiles: one CTA per SM walks a contiguous run of tiles
// in m-fastest order (so the query tile changes rarely), with warp roles:
// warp 8 lane 0 issues the TMA loads (kb tiles into a 3-stage ring, the query
// tile when the run moves to the next column tile), warp 9 lane 0 issues the
// MMAs into two TMEM accumulators, and warps 0-7 (two per TMEM lane quarter,
// one column half each, four 32-column TMEM loads in flight) drain an
// accumulator with the same ReLU / head-sum epilogue, in the same order,
// while the next tile's MMAs run. Each score is computed exactly as by
// score_tc_kernel.
constexpr int kPStages = 3;
constexpr int kPEpiWarps = 8;                   // two per TMEM lane quarter
constexpr int kPThreads = 32 * (kPEpiWarps + 2);  // + TMA producer + MMA issuer
constexpr int kPProducerWarp = kPEpiWarps, kPMmaWarp = kPEpiWarps + 1;

__device__ __forceinline__ void mbar_arrive_local(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

struct PersistArgs {
  int64_t m_tiles, tiles;  // tiles = n_batches * n_tiles_b * m_tiles
  int64_t n_tiles_b;       // column tiles of one batch (batches never share a column tile)
  int64_t rows_per_batch;  // nq * H: q rows of one batch
  int64_t scores_per_batch;  // nq * nb
};

template <int H>
__global__ void __launch_bounds__(kPThreads, 1)
    score_tc_persistent_kernel(const __grid_constant__ CUtensorMap tm_kb,
                               const __grid_constant__ CUtensorMap tm_q, const ScoreArgs a,
                               const PersistArgs pa) {
  static_assert(32 % H == 0, "a 32-column TMEM load must hold whole queries");
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + ((1024u - (raw & 1023u)) & 1023u);
  const int a_bytes = a.n_chunks * kTileM * kRowBytes;  // one kb stage
  const int q_tile_bytes = a.n_chunks * a.bn * kRowBytes;
  uint8_t* sQbase = smem;                                // 2 x n_chunks x [bn rows x 128 B]
  uint8_t* sA = sQbase + 2 * q_tile_bytes;               // kPStages kb stages
  // Two query-tile buffers: the j-th query tile of the run goes to buffer
  // j % 2, loaded as soon as the MMAs on tile j - 2 are done, so a change of
  // query tile does not wait for its load.
  __shared__ uint64_t full[kPStages], empty[kPStages], acc_full[2], acc_empty[2], q_full[2], q_free[2];
  __shared__ uint32_t tmem_slot;
  __shared__ volatile int failed;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // This CTA's contiguous run of tiles [t0, t1).
  const int64_t per = pa.tiles / gridDim.x, extra = pa.tiles % gridDim.x;
  const int64_t bx = blockIdx.x;
  const int64_t t0 = bx * per + (bx < extra ? bx : extra);
  const int64_t count = per + (blockIdx.x < extra ? 1 : 0);
  const int32_t count32 = static_cast<int32_t>(count);
  const int32_t m_tiles32 = static_cast<int32_t>(pa.m_tiles);
  const int32_t n_tiles_b32 = static_cast<int32_t>(pa.n_tiles_b);

  pdl_launch_dependents();
  if (threadIdx.x == 0) {
    for (int s = 0; s < kPStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&acc_full[s], 1);
      mbar_init(&acc_empty[s], 32 * kPEpiWarps);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&q_full[s], 1);
      mbar_init(&q_free[s], 1);
    }
    failed = 0;
    fence_mbarrier_init();
    tma_prefetch_desc(&tm_kb);
    tma_prefetch_desc(&tm_q);
  }
  if (warp == kPProducerWarp) {
    tmem_alloc(&tmem_slot, 2u * a.tmem_cols);
    tmem_relinquish();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem_base = tmem_slot;
  pdl_wait();  // q and kb may come from the previous kernel on the stream

  if (warp == kPProducerWarp) {
    // ------------------------------------------------ TMA producer
    if (lane == 0) {
      int64_t cur_n = -1;
      int32_t issued = 0;
      int32_t jq = -1;  // query tiles of the run loaded so far, minus one
      const uint32_t q_bytes = static_cast<uint32_t>(q_tile_bytes);
      for (int32_t i = 0; i < count32 && !failed; ++i) {
        // tile t: column tile g (batch g / n_tiles_b), block tile m
        // 32-bit index arithmetic: the host keeps tiles below 2^31
        const int32_t t = static_cast<int32_t>(t0 + i), n = t / m_tiles32, m = t - n * m_tiles32;
        const int32_t bt = n / n_tiles_b32, nb_ = n - bt * n_tiles_b32;
        if (n != cur_n) {
          ++jq;
          const int qb = jq & 1;
          // buffer qb is free once every MMA on query tile jq - 2 has completed
          if (jq >= 2 && !mbar_wait_bounded(&q_free[qb], static_cast<uint32_t>(((jq >> 1) - 1) & 1),
                                            a.timeout_ns)) {
            failed = 1;
            break;
          }
          mbar_arrive_expect_tx(&q_full[qb], q_bytes);
          for (int c = 0; c < a.n_chunks; ++c)
            tma_load_2d(sQbase + qb * q_tile_bytes + c * a.bn * kRowBytes, &tm_q, c * kKAtom,
                        static_cast<int32_t>(static_cast<int64_t>(bt) * pa.rows_per_batch + nb_ * a.bn),
                        &q_full[qb]);
          cur_n = n;
        }
        const int s = static_cast<int>(i % kPStages);
        const int32_t use = i / kPStages;
        if (use > 0 && !mbar_wait_bounded(&empty[s], static_cast<uint32_t>((use - 1) & 1), a.timeout_ns)) {
          failed = 1;
          break;
        }
        mbar_arrive_expect_tx(&full[s], static_cast<uint32_t>(a_bytes));
        for (int c = 0; c < a.n_chunks; ++c)
          tma_load_3d(sA + s * a_bytes + c * kTileM * kRowBytes, &tm_kb, c * kKAtom,
                      static_cast<int32_t>(m * kTileM), a.kb_z ? static_cast<int32_t>(bt) : 0, &full[s]);
        issued = i + 1;
      }
      if (failed) {
        // Loads may still be in flight into shared memory: wait for the last
        // ones issued (bounded) before the CTA may finish.
        atomicOr(a.status, kErrScoreLoadTimeout);
        for (int32_t j = issued > kPStages ? issued - kPStages : 0; j < issued; ++j)
          mbar_wait_bounded(&full[j % kPStages], static_cast<uint32_t>((j / kPStages) & 1), a.timeout_ns);
        for (int32_t j = jq > 1 ? jq - 1 : 0; j <= jq; ++j)  // the (up to) two query loads in flight
          mbar_wait_bounded(&q_full[j & 1], static_cast<uint32_t>((j >> 1) & 1), a.timeout_ns);
      }
    }
  } else if (warp == kPMmaWarp) {
    // ------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t idesc = idesc_f16_f32(kTileM, a.bn);
      int64_t cur_n = -1;
      int32_t jq = -1;  // the run's query tile in use
      for (int32_t i = 0; i < count32 && !failed; ++i) {
        const int32_t t = static_cast<int32_t>(t0 + i), n = t / m_tiles32;
        if (n != cur_n) {
          if (jq >= 0) mma_commit(&q_free[jq & 1]);  // fires when the old tile's MMAs are done
          ++jq;
          if (!mbar_wait_bounded(&q_full[jq & 1], static_cast<uint32_t>((jq >> 1) & 1), a.timeout_ns)) {
            failed = 1;
            break;
          }
          cur_n = n;
        }
        uint8_t* sQ = sQbase + (jq & 1) * q_tile_bytes;
        const int s = static_cast<int>(i % kPStages);
        const int acc = static_cast<int>(i & 1);
        if (!mbar_wait_bounded(&full[s], static_cast<uint32_t>((i / kPStages) & 1), a.timeout_ns)) {
          failed = 1;
          break;
        }
        if (i >= 2 && !mbar_wait_bounded(&acc_empty[acc], static_cast<uint32_t>(((i >> 1) - 1) & 1),
                                         a.timeout_ns)) {
          failed = 1;
          break;
        }
        tc_fence_after_sync();
        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc) * a.tmem_cols;
        for (int c = 0; c < a.n_chunks; ++c) {
          const uint32_t a_base = smem_u32(sA + s * a_bytes + c * kTileM * kRowBytes);
          const uint32_t b_base = smem_u32(sQ + c * a.bn * kRowBytes);
#pragma unroll
          for (int ks = 0; ks < kKAtom / 16; ++ks) {
            const int step = c * (kKAtom / 16) + ks;
            if (step < a.k_steps)
              mma_f16_ss(d_tmem, smem_desc_k_sw128(a_base + ks * 32),
                         smem_desc_k_sw128(b_base + ks * 32), idesc, step > 0 ? 1u : 0u);
          }
        }
        mma_commit(&empty[s]);
        mma_commit(&acc_full[acc]);
      }
      if (failed) atomicOr(a.status, kErrScoreMmaTimeout);
    }
  } else {
    // ------------------------------------------------ epilogue (warps 0-7)
    const int lane_base = (warp & 3) * 32;
    const int half_cols = a.bn >> 1;
    const int c_begin = (warp >> 2) * half_cols;
    constexpr int kQPerLoad = 32 / H;
    for (int32_t i = 0; i < count32; ++i) {
      const int acc = static_cast<int>(i & 1);
      if (failed || !mbar_wait_bounded(&acc_full[acc], static_cast<uint32_t>((i >> 1) & 1), a.timeout_ns)) {
        failed = 1;
        break;
      }
      tc_fence_after_sync();
      const int32_t t = static_cast<int32_t>(t0 + i), n = t / m_tiles32, m = t - n * m_tiles32;
      const int32_t bt = n / n_tiles_b32, nb_ = n - bt * n_tiles_b32;
      const int b = static_cast<int>(m) * kTileM + lane_base + lane;
      const bool b_ok = b < a.n_full;
      float* out = a.scores + static_cast<int64_t>(bt) * pa.scores_per_batch + b;
      const int q0 = static_cast<int>(nb_) * a.q_per_tile;
      const uint32_t taddr = tmem_base + static_cast<uint32_t>(acc) * a.tmem_cols +
                             (static_cast<uint32_t>(lane_base) << 16);
      for (int cb = c_begin; cb < c_begin + half_cols; cb += 128) {
        // up to four 32-column loads in flight, then one wait
        const int nld = min(4, (c_begin + half_cols - cb) / 32);
        uint32_t r[4][32];
#pragma unroll
        for (int u = 0; u < 4; ++u)
          if (u < nld) tmem_ld_32cols(taddr + cb + u * 32, r[u]);
        tmem_ld_wait();
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          if (u >= nld) continue;
          const int c0 = cb + u * 32;
#pragma unroll
          for (int j = 0; j < kQPerLoad; ++j) {
            float sc = 0.0f;
#pragma unroll
            for (int h = 0; h < H; ++h) sc = __fadd_rn(sc, fmaxf(__uint_as_float(r[u][j * H + h]), 0.0f));
            const int qidx = q0 + c0 / H + j;
            if (b_ok && qidx < a.nq) out[static_cast<size_t>(qidx) * a.nb] = sc;
          }
        }
      }
      tc_fence_before_sync();
      mbar_arrive_local(&acc_empty[acc]);
    }
  }
  tc_fence_before_sync();
  __syncthreads();
  if (warp == kPProducerWarp) tmem_dealloc(tmem_base, 2u * a.tmem_cols);
}

// Tail block: one CTA per kTailThreads (query, head) rows (whole queries),
// the rows staged in shared memory by coalesced 16-byte copies (row stride
// 2 D + 16 bytes, so each thread's 16-byte reads of its own row are free of
// bank conflicts); thread r then sums row r's products in index order, and
// one thread per query sums its heads' max(acc, 0) in head order and adds
// 1e9f.
__global__ void __launch_bounds__(kTailThreads)
    tail_kernel(const __half* __restrict__ q, const __half* __restrict__ kb_tail,
                float* __restrict__ scores, int32_t nq, int32_t H, int32_t D, int64_t nb) {
  extern __shared__ __align__(16) uint8_t tail_rows[];
  __shared__ float acc_s[kTailThreads];
  pdl_launch_dependents();
  pdl_wait();
  const int q_per_block = kTailThreads / H;
  const int64_t q0 = static_cast<int64_t>(blockIdx.x) * q_per_block;
  const int64_t row0 = q0 * H;
  const int rows = static_cast<int>(min(static_cast<int64_t>(q_per_block), static_cast<int64_t>(nq) - q0)) * H;
  const int stride = 2 * D + 16;
  const int units = D / 8;  // 16-byte units per row
  // 16-byte asynchronous copies, all in flight at once (q and its rows are
  // 16-byte aligned: D % 16 == 0).
  for (int u = threadIdx.x; u < rows * units; u += kTailThreads) {
    const int r = u / units, c = u - r * units;
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(tail_rows + r * stride + c * 16)),
                 "l"(reinterpret_cast<uint64_t>(q + (row0 + r) * D + c * 8))
                 : "memory");
  }
  asm volatile("cp.async.commit_group;\n\tcp.async.wait_group 0;" ::: "memory");
  __syncthreads();
  float acc = 0.0f;
  if (static_cast<int>(threadIdx.x) < rows) {
    const uint8_t* rp = tail_rows + threadIdx.x * stride;
    for (int i = 0; i < D; i += 8) {
      const uint4 qv = *reinterpret_cast<const uint4*>(rp + i * 2);
      const uint4 kv = __ldg(reinterpret_cast<const uint4*>(kb_tail + i));
      const __half* qh = reinterpret_cast<const __half*>(&qv);
      const __half* kh = reinterpret_cast<const __half*>(&kv);
#pragma unroll
      for (int j = 0; j < 8; ++j)
        acc = __fadd_rn(acc, __fmul_rn(__half2float(qh[j]), __half2float(kh[j])));
    }
  }
  acc_s[threadIdx.x] = acc;
  __syncthreads();
  const int ql = threadIdx.x;
  if (ql * H < rows) {
    float t = 0.0f;
    for (int hh = 0; hh < H; ++hh) t = __fadd_rn(t, fmaxf(acc_s[ql * H + hh], 0.0f));
    scores[(q0 + ql) * nb + (nb - 1)] = __fadd_rn(t, 1.0e9f);
  }
}

inline size_t tail_smem_bytes(int32_t D) {
  return static_cast<size_t>(kTailThreads) * (2 * static_cast<size_t>(D) + 16);
}

// ------------------------------------------------------------------ host
namespace {

uint32_t tmem_cols_for(int bn) {
  uint32_t c = 32;
  while (c < static_cast<uint32_t>(bn)) c <<= 1;
  return c;
}

// Dynamic shared memory for one CTA: operand tiles, barriers, slack for the
// 1024-byte alignment; then padded so that no more CTAs fit on an SM than its
// 512 TMEM columns can serve at once.
size_t score_smem_bytes(int bn, int n_chunks, uint32_t tmem_cols) {
  size_t need = static_cast<size_t>(n_chunks) * (kTileM + bn) * kRowBytes +
                (n_chunks + 1) * sizeof(uint64_t) + 16 + 1024;
  const size_t max_ctas = 512 / tmem_cols;
  const size_t per_sm = 233472;  // 228 KB of shared memory per SM
  const size_t floor_bytes = per_sm / (max_ctas + 1) + 1;
  return std::max(need, floor_bytes);
}

template <int H>
const void* score_kernel_ptr() {
  return reinterpret_cast<const void*>(&score_tc_kernel<H>);
}

template <int H>
const void* persistent_kernel_ptr() {
  return reinterpret_cast<const void*>(&score_tc_persistent_kernel<H>);
}

const void* persistent_kernel_for(int H) {
  switch (H) {
    case 1: return persistent_kernel_ptr<1>();
    case 2: return persistent_kernel_ptr<2>();
    case 4: return persistent_kernel_ptr<4>();
    case 8: return persistent_kernel_ptr<8>();
    case 16: return persistent_kernel_ptr<16>();
    case 32: return persistent_kernel_ptr<32>();
    default: return nullptr;
  }
}

const void* score_kernel_for(int H) {
  switch (H) {
    case 1: return score_kernel_ptr<1>();
    case 2: return score_kernel_ptr<2>();
    case 4: return score_kernel_ptr<4>();
    case 8: return score_kernel_ptr<8>();
    case 16: return score_kernel_ptr<16>();
    case 32: return score_kernel_ptr<32>();
    default: return nullptr;
  }
}

bool encode_2d_f16(CUtensorMap* tm, const void* base, uint64_t cols, uint64_t rows,
                   uint32_t box_cols, uint32_t box_rows) {
  EncodeTiledFn enc = encode_tiled_fn();
  if (!enc) return false;
  const cuuint64_t dims[2] = {cols, rows};
  const cuuint64_t strides[1] = {cols * 2};
  const cuuint32_t box[2] = {box_cols, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  return enc(tm, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<void*>(base), dims, strides, box,
             estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 3-D fp16 map [z][rows][cols] with a z stride in elements (a multiple of 8).
bool encode_3d_f16(CUtensorMap* tm, const void* base, uint64_t cols, uint64_t rows, uint64_t zs,
                   uint64_t z_stride, uint32_t box_cols, uint32_t box_rows) {
  EncodeTiledFn enc = encode_tiled_fn();
  if (!enc) return false;
  const cuuint64_t dims[3] = {cols, rows, zs};
  const cuuint64_t strides[2] = {cols * 2, z_stride * 2};
  const cuuint32_t box[3] = {box_cols, box_rows, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  return enc(tm, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, const_cast<void*>(base), dims, strides, box,
             estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Columns per tile: the widest of 256/128/64/32 that still gives at least one
// CTA per SM; narrower tiles spread small problems over more SMs.
int choose_bn(int64_t m_tiles, int64_t cols, int sm_count) {
  for (int bn : {256, 128, 64}) {
    const int64_t n_tiles = (cols + bn - 1) / bn;
    if (m_tiles * n_tiles >= sm_count) return bn;
  }
  return 32;
}

}  // namespace

cudaError_t init_score_kernels(const DeviceInfo& dev) {
  {
    cudaError_t e = cudaFuncSetAttribute(reinterpret_cast<const void*>(&tail_kernel),
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(tail_smem_bytes(256)));
    if (e != cudaSuccess) return e;
  }
  for (int H : {1, 2, 4, 8, 16, 32}) {
    for (const void* fn : {score_kernel_for(H), persistent_kernel_for(H)}) {
      cudaFuncAttributes fa;
      cudaError_t e = cudaFuncGetAttributes(&fa, fn);
      if (e != cudaSuccess) return e;
      e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               dev.max_smem_optin - static_cast<int>(fa.sharedSizeBytes));
      if (e != cudaSuccess) return e;
    }
  }
  return cudaSuccess;
}

namespace {
// The persistent kernel's plan for p (batches included): full-width tiles
// (256 columns), at least four per SM, and its shared memory within bounds.
struct PersistPlan {
  bool ok;
  int bn;
  int64_t m_tiles, n_tiles_b, tiles;
};
PersistPlan persistent_plan(const ScoreProblem& p, const DeviceInfo& dev) {
  PersistPlan pp{false, 0, 0, 0, 0};
  if (p.nq <= 0 || p.n_full <= 0) return pp;
  const int64_t nbat = p.n_batches > 1 ? p.n_batches : 1;
  const int64_t cols_b = static_cast<int64_t>(p.nq) * p.H;
  pp.m_tiles = (p.n_full + kTileM - 1) / kTileM;
  pp.bn = choose_bn(pp.m_tiles, nbat * cols_b, dev.sm_count);
  pp.n_tiles_b = (cols_b + pp.bn - 1) / pp.bn;
  pp.tiles = nbat * pp.n_tiles_b * pp.m_tiles;
  if (pp.tiles > 0x7FFFFFFFLL) return pp;  // the kernel indexes tiles in 32 bits
  const int n_chunks = (p.D + kKAtom - 1) / kKAtom;
  const size_t psmem = static_cast<size_t>(n_chunks) * (2 * pp.bn + kPStages * kTileM) * kRowBytes + 1024;
  pp.ok = pp.bn == 256 && pp.tiles >= 4LL * dev.sm_count &&
          psmem <= static_cast<size_t>(dev.max_smem_optin) - 1024;
  return pp;
}
}  // namespace

bool scores_persistent(const ScoreProblem& p, const DeviceInfo& dev) { return persistent_plan(p, dev).ok; }

cudaError_t launch_scores(const ScoreProblem& p, const DeviceInfo& dev, cudaStream_t stream) {
  const PersistPlan pp = persistent_plan(p, dev);
  // Several batches (each with its own kb, or one shared) run only on the
  // persistent kernel, with the tail left to the select.
  if (p.n_batches > 1 && (!pp.ok || (p.has_tail && !p.skip_tail))) return cudaErrorInvalidValue;
  if (p.nq > 0 && p.n_full > 0) {
    const int64_t nbat = p.n_batches > 1 ? p.n_batches : 1;
    const int64_t cols = static_cast<int64_t>(p.nq) * p.H;
    const int64_t m_tiles = (p.n_full + kTileM - 1) / kTileM;
    const int bn = pp.ok ? pp.bn : choose_bn(m_tiles, cols, dev.sm_count);
    const int64_t n_tiles = (cols + bn - 1) / bn;
    if (m_tiles > 0x7FFFFFFF || n_tiles > 65535) return cudaErrorInvalidValue;
    CUtensorMap tm_kb, tm_q;
    if (!encode_2d_f16(&tm_q, p.q, p.D, nbat * cols, kKAtom, bn)) return cudaErrorInvalidValue;
    ScoreArgs a;
    a.scores = p.scores;
    a.nq = p.nq;
    a.nb = static_cast<int32_t>(p.nb);
    a.n_full = static_cast<int32_t>(p.n_full);
    a.bn = bn;
    a.q_per_tile = bn / p.H;
    a.n_chunks = (p.D + kKAtom - 1) / kKAtom;
    a.k_steps = p.D / 16;
    a.tmem_cols = tmem_cols_for(bn);
    a.status = dev.status_word;
    a.timeout_ns = kWaitTimeoutNs;
    a.kb_z = p.kb_batch_stride != 0 ? 1 : 0;
    // Many full-width tiles: the persistent kernel (one CTA per SM, pipelined
    // loads, MMAs and epilogue); the same arithmetic per score.
    const size_t psmem = static_cast<size_t>(a.n_chunks) * (2 * bn + kPStages * kTileM) * kRowBytes + 1024;
    if (pp.ok) {
      const uint64_t zs = p.kb_batch_stride != 0 ? static_cast<uint64_t>(nbat) : 1u;
      const uint64_t zst = p.kb_batch_stride != 0 ? static_cast<uint64_t>(p.kb_batch_stride)
                                                  : static_cast<uint64_t>(p.n_full) * p.D;
      if (!encode_3d_f16(&tm_kb, p.kb, p.D, p.n_full, zs, zst, kKAtom, kTileM)) return cudaErrorInvalidValue;
      PersistArgs pa{pp.m_tiles, pp.tiles, pp.n_tiles_b, cols, static_cast<int64_t>(p.nq) * p.nb};
      const dim3 pgrid(static_cast<unsigned>(std::min<int64_t>(dev.sm_count, pa.tiles)));
      const dim3 pblock(kPThreads);
      plan_add("score_tc_persistent_kernel");
      cudaError_t e = cudaErrorInvalidValue;
      switch (p.H) {
        case 1: e = launch_pdl(score_tc_persistent_kernel<1>, pgrid, pblock, psmem, stream, tm_kb, tm_q, a, pa); break;
        case 2: e = launch_pdl(score_tc_persistent_kernel<2>, pgrid, pblock, psmem, stream, tm_kb, tm_q, a, pa); break;
        case 4: e = launch_pdl(score_tc_persistent_kernel<4>, pgrid, pblock, psmem, stream, tm_kb, tm_q, a, pa); break;
        case 8: e = launch_pdl(score_tc_persistent_kernel<8>, pgrid, pblock, psmem, stream, tm_kb, tm_q, a, pa); break;
        case 16: e = launch_pdl(score_tc_persistent_kernel<16>, pgrid, pblock, psmem, stream, tm_kb, tm_q, a, pa); break;
        case 32: e = launch_pdl(score_tc_persistent_kernel<32>, pgrid, pblock, psmem, stream, tm_kb, tm_q, a, pa); break;
        default: break;
      }
      if (e != cudaSuccess) return e;
      if (p.nq > 0 && p.has_tail && !p.skip_tail) {
        const int q_per_block = kTailThreads / p.H;
        const int64_t grid = (p.nq + q_per_block - 1) / q_per_block;
        plan_add("tail_kernel");
        return launch_pdl(tail_kernel, dim3(static_cast<unsigned>(grid)), dim3(kTailThreads),
                          tail_smem_bytes(p.D), stream, reinterpret_cast<const __half*>(p.q),
                          reinterpret_cast<const __half*>(p.kb) + (p.nb - 1) * p.D, p.scores,
                          p.nq, p.H, p.D, p.nb);
      }
      return cudaSuccess;
    }
    if (!encode_2d_f16(&tm_kb, p.kb, p.D, p.n_full, kKAtom, kTileM)) return cudaErrorInvalidValue;
    const size_t smem = score_smem_bytes(bn, a.n_chunks, a.tmem_cols);
    if (smem > static_cast<size_t>(dev.max_smem_optin)) return cudaErrorInvalidValue;
    const dim3 grid(static_cast<unsigned>(m_tiles), static_cast<unsigned>(n_tiles));
    const dim3 block(kScoreThreads);
    plan_add("score_tc_kernel");
    cudaError_t e;
    switch (p.H) {
      case 1: e = launch_pdl(score_tc_kernel<1>, grid, block, smem, stream, tm_kb, tm_q, a); break;
      case 2: e = launch_pdl(score_tc_kernel<2>, grid, block, smem, stream, tm_kb, tm_q, a); break;
      case 4: e = launch_pdl(score_tc_kernel<4>, grid, block, smem, stream, tm_kb, tm_q, a); break;
      case 8: e = launch_pdl(score_tc_kernel<8>, grid, block, smem, stream, tm_kb, tm_q, a); break;
      case 16: e = launch_pdl(score_tc_kernel<16>, grid, block, smem, stream, tm_kb, tm_q, a); break;
      case 32: e = launch_pdl(score_tc_kernel<32>, grid, block, smem, stream, tm_kb, tm_q, a); break;
      default: return cudaErrorInvalidValue;
    }
    if (e != cudaSuccess) return e;
  }
  if (p.nq > 0 && p.has_tail && !p.skip_tail) {
    const int q_per_block = kTailThreads / p.H;
    const int64_t grid = (p.nq + q_per_block - 1) / q_per_block;
    plan_add("tail_kernel");
    return launch_pdl(tail_kernel, dim3(static_cast<unsigned>(grid)), dim3(kTailThreads),
                      tail_smem_bytes(p.D), stream,
                      reinterpret_cast<const __half*>(p.q),
                      reinterpret_cast<const __half*>(p.kb) + (p.nb - 1) * p.D, p.scores, p.nq,
                      p.H, p.D, p.nb);
  }
  return cudaSuccess;
}

}  // namespace qsa
