// split_reduce.cu - the flash-attention decode split reduce (1bit-MONSTER
// llama.cpp pull request 30, "What" and "Changes"; its review asks for a
// bounded scale stage).
//
// Per group g and row r: maximum = max_b partial_max; scale_b =
// exp(partial_max_b - maximum), once per (row, block); sum = sum_b scale_b *
// partial_sum_b; out[c] = (sum_b scale_b * partial_out_b[c]) / sum.
//
// GB300 layout of the work: the blocks are cut into chunks of kSrChunk
// (128) and a group's rows into splits of Rs rows; CTA (chunk, split, group)
// bulk-copies its rows' fp16 partial outputs for the chunk into shared
// memory (when the rows are 16-byte aligned), finds the rows' maxima over all
// blocks meanwhile (partial_max is small and L2-resident), stages the
// chunk's scales and partial sums (bounded whatever the context length), and
// runs the all-rows output pass: a work item is a quad of 4 channels of one
// row over one run of kSrRun blocks (four runs per chunk keep all warps
// busy). Chunk partials go to the caller's workspace; the last CTA of a
// (group, split) to finish (an arrival counter) bulk-copies them back and
// adds them in chunk order, then divides. With one chunk the CTA writes the
// output directly.
//
// Arithmetic, fixed operation for operation (the CPU oracle's pinned fp32
// procedure follows the same steps): scale = exp_pinned(fl(pm - maximum));
// inside a run, acc = fl(acc + fl(scale * x)) block by block from 0 (no
// fused multiply-add); a chunk's runs added in order from 0; chunk partials
// added in chunk order from 0; out = fl(O / sum).
#include <cuda_fp16.h>

#include <algorithm>
#include <cstring>

#include "qsa_device.cuh"
#include "qsa_internal.h"

namespace qsa {

namespace {

constexpr int kSrThreads = 256;

// exp(x) for x <= 0 in fp32: Cody and Waite's reduction x = n ln2 + t
// (ln 2 split so that n * kLn2Hi is exact for |n| <= 128), the degree-7
// Taylor polynomial of exp(t) in Horner form with separately rounded
// multiplies and adds, and an exact scaling by 2^n. Below -86 the result is
// 0. Constants: log2(e), the split of ln 2 and 1/k!, rounded to fp32.
__device__ __forceinline__ float exp_pinned(float x) {
  const float xc = fmaxf(x, -87.0f);
  const float n = rintf(__fmul_rn(xc, 0x1.715476p+0f));
  const float t = __fsub_rn(__fsub_rn(xc, __fmul_rn(n, 0x1.62e4p-1f)), __fmul_rn(n, 0x1.7f7d1cp-20f));
  float p = 0x1.a01a02p-13f;                         // 1/7!
  p = __fadd_rn(__fmul_rn(p, t), 0x1.6c16c2p-10f);  // 1/6!
  p = __fadd_rn(__fmul_rn(p, t), 0x1.111112p-7f);   // 1/5!
  p = __fadd_rn(__fmul_rn(p, t), 0x1.555556p-5f);   // 1/4!
  p = __fadd_rn(__fmul_rn(p, t), 0x1.555556p-3f);   // 1/3!
  p = __fadd_rn(__fmul_rn(p, t), 0.5f);             // 1/2!
  p = __fadd_rn(__fmul_rn(p, t), 1.0f);             // 1/1!
  p = __fadd_rn(__fmul_rn(p, t), 1.0f);             // 1/0!
  const int ni = max(static_cast<int>(n), -126);
  const float two_n = __int_as_float((ni + 127) << 23);
  return x < -86.0f ? 0.0f : __fmul_rn(p, two_n);
}

struct SrArgs {
  const float* pm;      // [G][R][B]
  const float* ps;      // [G][R][B]
  const __half* po;     // [G][R][B][C]
  float* out;           // [G][R][C]
  uint32_t* count;      // [G][R] arrival counters, one per (group, row split); zero between calls
  float* part_sum;      // [G][S][R]
  float* part_out;      // [G][S][R][C]
  uint32_t* status;     // device status word (bounded-wait failures)
  uint64_t timeout_ns;
  int R, B, C, S;
  int RS, Rs;           // row splits per group, rows per split
  int staged;           // 1: the chunk's partial outputs are staged by bulk copies
  int pm_vec;           // 1: partial_max and partial_sum rows are 16-byte aligned
  int stage_bytes;      // dynamic shared memory before the run partials
};

__global__ void __launch_bounds__(kSrThreads) split_reduce_kernel(const SrArgs a) {
  // [Rs][kSrChunk][C] fp16 when staged (stage_bytes), then the run partials
  extern __shared__ __align__(128) uint8_t sr_stage[];
  __shared__ float s_max[kSrMaxRows];
  __shared__ float s_part[kSrMaxRows];
  __shared__ float s_rowsum[kSrMaxRows];

  __shared__ __align__(8) uint64_t bar_stage;
  __shared__ int s_last, s_ok;
  const int j = blockIdx.x, rs = blockIdx.y, g = blockIdx.z;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int R = a.R, B = a.B, C = a.C;
  const int r0 = rs * a.Rs;
  const int nr = min(a.Rs, R - r0);  // rows of this CTA
  const int64_t grb = static_cast<int64_t>(g) * R * B;
  const int b0 = j * kSrChunk;
  const int nbk = min(kSrChunk, B - b0);
  const uint32_t row_bytes = static_cast<uint32_t>(nbk) * C * 2u;
  // Dynamic shared memory: [stage_bytes of staged partial outputs]
  // [run partials kSrRuns x quads float4][run sums kSrRuns x Rs]
  // [scales Rs x kSrChunk][partial sums Rs x kSrChunk].
  const int nquads_max = a.Rs * (C / 4);
  float4* run_out = reinterpret_cast<float4*>(sr_stage + a.stage_bytes);
  float* run_sum = reinterpret_cast<float*>(run_out + kSrRuns * nquads_max);
  float* s_scale = run_sum + kSrRuns * a.Rs;
  float* s_psum = s_scale + a.Rs * kSrChunk;

  pdl_launch_dependents();
  if (tid == 0) {
    if (a.staged) {
      mbar_init(&bar_stage, 1);
      fence_mbarrier_init();
      // The chunk's partial outputs on their way to L2 while the previous
      // kernel finishes (a hint; the copies proper come after the wait).
      for (int r = 0; r < nr; ++r)
        bulk_prefetch_l2(a.po + (grb + static_cast<int64_t>(r0 + r) * B + b0) * C, row_bytes);
    }
    if (a.pm_vec) {
      // the rows' maxima inputs and this chunk's partial sums (whole 16-byte
      // pieces; a hint only)
      for (int r = 0; r < nr; ++r) {
        const int64_t row = grb + static_cast<int64_t>(r0 + r) * B;
        bulk_prefetch_l2(a.pm + row, static_cast<uint32_t>(B) * 4u);
        const uint32_t ps_bytes = (static_cast<uint32_t>(nbk) * 4u) & ~15u;
        if (ps_bytes) bulk_prefetch_l2(a.ps + row + b0, ps_bytes);
      }
    }
  }
  pdl_wait();
  if (a.staged && tid == 0) {
    mbar_arrive_expect_tx(&bar_stage, row_bytes * static_cast<uint32_t>(nr));
    for (int r = 0; r < nr; ++r)
      bulk_load(sr_stage + static_cast<size_t>(r) * kSrChunk * C * 2,
                a.po + (grb + static_cast<int64_t>(r0 + r) * B + b0) * C, row_bytes, &bar_stage);
  }

  // Row maxima over every block, while the copies fly: the CTA's warps
  // split its rows (several warps per row when there are fewer than 8),
  // 16-byte loads when the rows allow, many loads in flight per lane.
  {
    constexpr int kWarps = kSrThreads / 32;
    const int wpr = nr < kWarps ? kWarps / nr : 1;
    const float ninf = __int_as_float(0xff800000u);
    for (int task = warp; task < nr * wpr; task += kWarps) {
      const int r = task / wpr, part = task - r * wpr;
      const float* row = a.pm + grb + static_cast<int64_t>(r0 + r) * B;
      float m = ninf;
      if (a.pm_vec) {
        const int n4 = B / 4, len = (n4 + wpr - 1) / wpr;
        const float4* row4 = reinterpret_cast<const float4*>(row);
        const int hi = min(n4, (part + 1) * len);
#pragma unroll 8
        for (int i = part * len + lane; i < hi; i += 32) {
          const float4 v = __ldg(row4 + i);
          m = fmaxf(m, fmaxf(fmaxf(v.x, v.y), fmaxf(v.z, v.w)));
        }
      } else {
        const int len = (B + wpr - 1) / wpr;
        const int hi = min(B, (part + 1) * len);
#pragma unroll 8
        for (int b = part * len + lane; b < hi; b += 32) m = fmaxf(m, __ldg(row + b));
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
      if (lane == 0) s_part[task] = m;
    }
    __syncthreads();
    if (tid < nr) {
      float m = ninf;
      for (int p = 0; p < wpr; ++p) m = fmaxf(m, s_part[tid * wpr + p]);
      s_max[tid] = m;
    }
    __syncthreads();
  }

  // This chunk's scales and partial sums, staged per row.
  for (int i = tid; i < nr * nbk; i += kSrThreads) {
    const int r = i / nbk, bl = i - r * nbk;
    const int64_t at = grb + static_cast<int64_t>(r0 + r) * B + b0 + bl;
    const float pmv = __ldg(a.pm + at);
    s_psum[r * kSrChunk + bl] = __ldg(a.ps + at);
    s_scale[r * kSrChunk + bl] = exp_pinned(__fsub_rn(pmv, s_max[r]));
  }
  if (tid == 0) s_ok = a.staged ? mbar_wait_bounded(&bar_stage, 0, a.timeout_ns) : 1;
  __syncthreads();
  if (!s_ok) {
    // The copies never completed: record it, give them one more bounded
    // wait so none lands after the CTA has gone, and leave (no output; the
    // workspace counters must be zeroed again before the next call).
    if (tid == 0) {
      atomicOr(a.status, kErrSplitLoadTimeout);
      mbar_wait_bounded(&bar_stage, 0, a.timeout_ns);
    }
    return;
  }

  // Output pass. Work item = (run of kSrRun blocks, quad of 4 channels of a
  // row); consecutive threads take consecutive quads (256 contiguous bytes
  // per warp and block). A run accumulates from 0 block by block; the quad
  // at channel 0 also accumulates the row's sum. Run partials go to shared
  // memory and are then added in run order.
  const int qpr = C / 4;
  const int nquads = nr * qpr;
  const int nruns = (nbk + kSrRun - 1) / kSrRun;
  const int stride = C / 4;  // uint2 (4 halves) per block
  for (int item = tid; item < nruns * nquads; item += kSrThreads) {
    const int run = item / nquads, q = item - run * nquads;
    const int r = q / qpr, c = (q - r * qpr) * 4;
    const int bl_lo = run * kSrRun, bl_hi = min(nbk, bl_lo + kSrRun);
    const float* srow = s_scale + r * kSrChunk;
    const float* psrow = s_psum + r * kSrChunk;
    float o0 = 0.0f, o1 = 0.0f, o2 = 0.0f, o3 = 0.0f, acc_s = 0.0f;
    if (a.staged) {
      const uint2* src = reinterpret_cast<const uint2*>(sr_stage) +
                         static_cast<size_t>(r) * kSrChunk * stride + c / 4;
#pragma unroll 8
      for (int bl = bl_lo; bl < bl_hi; ++bl) {
        const uint2 v = src[bl * stride];
        const float sc = srow[bl];
        const __half2 h01 = *reinterpret_cast<const __half2*>(&v.x);
        const __half2 h23 = *reinterpret_cast<const __half2*>(&v.y);
        o0 = __fadd_rn(o0, __fmul_rn(sc, __low2float(h01)));
        o1 = __fadd_rn(o1, __fmul_rn(sc, __high2float(h01)));
        o2 = __fadd_rn(o2, __fmul_rn(sc, __low2float(h23)));
        o3 = __fadd_rn(o3, __fmul_rn(sc, __high2float(h23)));
        if (c == 0) acc_s = __fadd_rn(acc_s, __fmul_rn(sc, psrow[bl]));
      }
    } else {
      const uint2* src = reinterpret_cast<const uint2*>(
          a.po + ((grb + static_cast<int64_t>(r0 + r) * B + b0) * C + c));
#pragma unroll 8
      for (int bl = bl_lo; bl < bl_hi; ++bl) {
        const uint2 v = __ldg(src + bl * stride);
        const float sc = srow[bl];
        const __half2 h01 = *reinterpret_cast<const __half2*>(&v.x);
        const __half2 h23 = *reinterpret_cast<const __half2*>(&v.y);
        o0 = __fadd_rn(o0, __fmul_rn(sc, __low2float(h01)));
        o1 = __fadd_rn(o1, __fmul_rn(sc, __high2float(h01)));
        o2 = __fadd_rn(o2, __fmul_rn(sc, __low2float(h23)));
        o3 = __fadd_rn(o3, __fmul_rn(sc, __high2float(h23)));
        if (c == 0) acc_s = __fadd_rn(acc_s, __fmul_rn(sc, psrow[bl]));
      }
    }
    run_out[run * nquads + q] = make_float4(o0, o1, o2, o3);
    if (c == 0) run_sum[run * nr + r] = acc_s;
  }
  __syncthreads();
  float acc_q[kSrMaxQuadsPerThread][4];
  float acc_sq[kSrMaxQuadsPerThread];
#pragma unroll
  for (int u = 0; u < kSrMaxQuadsPerThread; ++u) {
    acc_q[u][0] = acc_q[u][1] = acc_q[u][2] = acc_q[u][3] = 0.0f;
    acc_sq[u] = 0.0f;
    const int q = tid + u * kSrThreads;
    if (q >= nquads) continue;
    const int r = q / qpr, c = q - r * qpr;
    for (int run = 0; run < nruns; ++run) {
      const float4 v = run_out[run * nquads + q];
      acc_q[u][0] = __fadd_rn(acc_q[u][0], v.x);
      acc_q[u][1] = __fadd_rn(acc_q[u][1], v.y);
      acc_q[u][2] = __fadd_rn(acc_q[u][2], v.z);
      acc_q[u][3] = __fadd_rn(acc_q[u][3], v.w);
      acc_sq[u] = __fadd_rn(acc_sq[u], run_sum[run * nr + r]);
    }
    if (c == 0) s_rowsum[r] = acc_sq[u];
  }

  const int64_t grc = (static_cast<int64_t>(g) * R + r0) * C;
  if (a.S == 1) {
    // One chunk: its partials are the totals (0 + x is exact).
    __syncthreads();
#pragma unroll
    for (int u = 0; u < kSrMaxQuadsPerThread; ++u) {
      const int q = tid + u * kSrThreads;
      if (q >= nquads) continue;
      const int r = q / qpr, c = (q - r * qpr) * 4;
      const float L = s_rowsum[r];
      *reinterpret_cast<float4*>(a.out + grc + static_cast<int64_t>(r) * C + c) =
          make_float4(__fdiv_rn(acc_q[u][0], L), __fdiv_rn(acc_q[u][1], L),
                      __fdiv_rn(acc_q[u][2], L), __fdiv_rn(acc_q[u][3], L));
    }
    return;
  }

  // Several chunks: publish this chunk's partials, then the last CTA of the
  // (group, row split) adds them in chunk order.
  const int64_t gs = static_cast<int64_t>(g) * a.S;
#pragma unroll
  for (int u = 0; u < kSrMaxQuadsPerThread; ++u) {
    const int q = tid + u * kSrThreads;
    if (q >= nquads) continue;
    const int r = q / qpr, c = (q - r * qpr) * 4;
    *reinterpret_cast<float4*>(a.part_out + ((gs + j) * R + r0 + r) * C + c) =
        make_float4(acc_q[u][0], acc_q[u][1], acc_q[u][2], acc_q[u][3]);
    if (c == 0) a.part_sum[(gs + j) * R + r0 + r] = acc_sq[u];
  }
  __threadfence();
  __syncthreads();
  uint32_t* counter = a.count + static_cast<int64_t>(g) * R + rs;
  if (tid == 0) s_last = atomicAdd(counter, 1u) == static_cast<uint32_t>(a.S - 1);
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  if (tid == 0) *counter = 0;  // ready for the next call
#pragma unroll
  for (int u = 0; u < kSrMaxQuadsPerThread; ++u) {
    acc_q[u][0] = acc_q[u][1] = acc_q[u][2] = acc_q[u][3] = 0.0f;
    acc_sq[u] = 0.0f;
  }
  const int64_t jstride = static_cast<int64_t>(R) * C;  // floats between chunks
  if (a.staged) {
    // The chunk partials of this CTA's rows, staged by bulk copies in rounds
    // that fill the staging buffer, added in chunk order.
    fence_proxy_async_global();  // peers' partials, acquired above, seen by the copies
    const uint32_t slice = static_cast<uint32_t>(nr) * C * 4u;  // one chunk's rows
    const int per_round = static_cast<int>(static_cast<uint32_t>(a.stage_bytes) / slice);
    float* stage = reinterpret_cast<float*>(sr_stage);
    for (int j0 = 0, round = 1; j0 < a.S; j0 += per_round, ++round) {
      const int nj = min(per_round, a.S - j0);
      if (tid == 0) {
        // the stage was last read through the generic proxy
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        mbar_arrive_expect_tx(&bar_stage, slice * static_cast<uint32_t>(nj));
        for (int jj = 0; jj < nj; ++jj)
          bulk_load(stage + static_cast<size_t>(jj) * nr * C,
                    a.part_out + ((gs + j0 + jj) * R + r0) * C, slice, &bar_stage);
      }
      for (int i = tid; i < nj * nr; i += kSrThreads) {
        const int jj = i / nr, r = i - jj * nr;
        s_psum[i] = __ldcg(a.part_sum + (gs + j0 + jj) * R + r0 + r);  // nj * nr <= 64 * Rs
      }
      if (tid == 0) s_ok = mbar_wait_bounded(&bar_stage, round & 1, a.timeout_ns);
      __syncthreads();
      if (!s_ok) {
        if (tid == 0) {
          atomicOr(a.status, kErrSplitLoadTimeout);
          mbar_wait_bounded(&bar_stage, round & 1, a.timeout_ns);
        }
        return;
      }
#pragma unroll
      for (int u = 0; u < kSrMaxQuadsPerThread; ++u) {
        const int q = tid + u * kSrThreads;
        if (q >= nquads) continue;
        const int r = q / qpr, c = (q - r * qpr) * 4;
        for (int jj = 0; jj < nj; ++jj) {
          const float4 v = *reinterpret_cast<const float4*>(stage + (static_cast<size_t>(jj) * nr + r) * C + c);
          acc_sq[u] = __fadd_rn(acc_sq[u], s_psum[jj * nr + r]);
          acc_q[u][0] = __fadd_rn(acc_q[u][0], v.x);
          acc_q[u][1] = __fadd_rn(acc_q[u][1], v.y);
          acc_q[u][2] = __fadd_rn(acc_q[u][2], v.z);
          acc_q[u][3] = __fadd_rn(acc_q[u][3], v.w);
        }
      }
      __syncthreads();  // the stage is refilled by the next round
    }
  } else {
#pragma unroll
    for (int u = 0; u < kSrMaxQuadsPerThread; ++u) {
      const int q = tid + u * kSrThreads;
      if (q >= nquads) continue;
      const int r = q / qpr, c = (q - r * qpr) * 4;
      const float4* po4 = reinterpret_cast<const float4*>(a.part_out + (gs * R + r0 + r) * C + c);
      const float* psum = a.part_sum + gs * R + r0 + r;
#pragma unroll 16
      for (int jj = 0; jj < a.S; ++jj) {
        const float4 v = __ldcg(po4 + jj * (jstride / 4));
        acc_sq[u] = __fadd_rn(acc_sq[u], __ldcg(psum + static_cast<int64_t>(jj) * R));
        acc_q[u][0] = __fadd_rn(acc_q[u][0], v.x);
        acc_q[u][1] = __fadd_rn(acc_q[u][1], v.y);
        acc_q[u][2] = __fadd_rn(acc_q[u][2], v.z);
        acc_q[u][3] = __fadd_rn(acc_q[u][3], v.w);
      }
    }
  }
#pragma unroll
  for (int u = 0; u < kSrMaxQuadsPerThread; ++u) {
    const int q = tid + u * kSrThreads;
    if (q >= nquads) continue;
    const int r = q / qpr, c = (q - r * qpr) * 4;
    const float L = acc_sq[u];
    *reinterpret_cast<float4*>(a.out + grc + static_cast<int64_t>(r) * C + c) =
        make_float4(__fdiv_rn(acc_q[u][0], L), __fdiv_rn(acc_q[u][1], L),
                    __fdiv_rn(acc_q[u][2], L), __fdiv_rn(acc_q[u][3], L));
  }
}

// ------------------------------------ cluster form: one cluster per row
// One thread-block cluster of cs CTAs per (group, row); CTA rank q reduces the
// chunks [q*cpc, (q+1)*cpc) of 128 blocks: it bulk-copies each chunk's fp16
// partial outputs (whole rows of C channels, one contiguous copy per chunk)
// into shared memory and finds the maximum of its blocks' partial_max; each
// CTA stores its maximum into every CTA's shared memory (distributed shared
// memory), so once they have arrived every CTA has the row's maximum. It
// then forms its chunks' partials in the fixed order (runs of 32 blocks
// accumulated block by block, a chunk's runs added in order) and stores them
// into CTA rank 0's shared memory; once they have all arrived rank 0 adds
// them in chunk order and divides. Every exchange is a remote store counted
// on the reader's mbarrier (st.async), so no CTA waits on a remote load or on
// a cluster-wide release. The arithmetic is the row-split kernel's,
// operation for operation: the same bits, with no workspace, no arrival
// counter and no global round trip. Only a few bytes per chunk cross between
// CTAs (distributed shared memory moves bulk data slowly).
constexpr int kScThreads = 256;
constexpr int kScMaxCpc = 4;    // chunks per CTA at most
constexpr int kScMaxCs = 8;     // CTAs per cluster at most (portable)

struct ScArgs {
  const float* pm;     // [G][R][B]
  const float* ps;     // [G][R][B]
  const __half* po;    // [G][R][B][C]
  float* out;          // [G][R][C]
  uint32_t* status;
  uint64_t timeout_ns;
  int R, B, C, cs, cpc;
};

__device__ __forceinline__ uint32_t sc_cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
// Stores v at the same shared-memory offset as `local` in CTA `rank` of the
// cluster (another CTA than the caller's), its 4 bytes counted on that CTA's
// mbarrier at the offset of `bar`.
__device__ __forceinline__ void sc_st_peer(float* local, uint32_t rank, float v, uint64_t* bar) {
  uint32_t addr, baddr;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(addr) : "r"(smem_u32(local)), "r"(rank));
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(baddr) : "r"(smem_u32(bar)), "r"(rank));
  asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.u32 [%0], %1, [%2];" ::"r"(addr),
               "r"(__float_as_uint(v)), "r"(baddr)
               : "memory");
}

__global__ void __launch_bounds__(kScThreads)
    split_cluster_kernel(const ScArgs a) {
  extern __shared__ __align__(128) uint8_t sc_stage[];  // [cpc][128][C] fp16, then floats
  __shared__ __align__(8) uint64_t bar_chunk[kScMaxCpc];
  __shared__ __align__(8) uint64_t bar_max, bar_gather;
  __shared__ float s_red[kScThreads / 32];
  __shared__ float s_lmax[kScMaxCs];  // every CTA's maximum, pushed by its owner
  __shared__ int s_ok;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int R = a.R, B = a.B, C = a.C, cpc = a.cpc, cs = a.cs;
  const int q = static_cast<int>(sc_cluster_rank());
  const int row_id = blockIdx.x / cs;  // (group, row)
  const int64_t row = row_id;
  const int n_chunks = (B + kSrChunk - 1) / kSrChunk;
  const int j0 = q * cpc, j1 = min(n_chunks, j0 + cpc);  // this CTA's chunks
  const int b_lo = j0 * kSrChunk, b_hi = min(B, j1 * kSrChunk);
  const size_t chunk_halves = static_cast<size_t>(kSrChunk) * C;
  float* s_scale = reinterpret_cast<float*>(sc_stage + static_cast<size_t>(cpc) * chunk_halves * 2);
  float* s_psum = s_scale + cpc * kSrChunk;
  float* run_out = s_psum + cpc * kSrChunk;                       // [cpc][kSrRuns][C]
  float* run_sum = run_out + static_cast<size_t>(cpc) * kSrRuns * C;  // [cpc][kSrRuns]
  float* gather = run_sum + cpc * kSrRuns;  // rank 0: [n_chunks][C + 1], pushed by the owners
  const __half* stage = reinterpret_cast<const __half*>(sc_stage);
  (void)R;

  pdl_launch_dependents();
  if (tid == 0) {
    for (int i = 0; i < kScMaxCpc; ++i) mbar_init(&bar_chunk[i], 1);
    mbar_init(&bar_max, 1);
    mbar_init(&bar_gather, 1);
    fence_mbarrier_init();
    // Registered before the cluster's start barrier lets any peer store:
    // the other CTAs' maxima here, and (rank 0) the other CTAs' chunk
    // partials and sums. A CTA's own values go in with plain stores.
    mbar_arrive_expect_tx(&bar_max, static_cast<uint32_t>(cs - 1) * 4u);
    if (q == 0)
      mbar_arrive_expect_tx(&bar_gather, static_cast<uint32_t>(n_chunks - (j1 - j0)) * (C + 1) * 4u);
    s_ok = 1;
    // this CTA's inputs on their way to L2 while the previous kernel
    // finishes (hints: they change no value a later load observes)
    bulk_prefetch_l2(a.po + (row * B + b_lo) * C, static_cast<uint32_t>(b_hi - b_lo) * C * 2u);
    const uint32_t pbytes = (static_cast<uint32_t>(b_hi - b_lo) * 4u) & ~15u;
    if (((row * B + b_lo) & 3) == 0 && pbytes) {
      bulk_prefetch_l2(a.pm + row * B + b_lo, pbytes);
      bulk_prefetch_l2(a.ps + row * B + b_lo, pbytes);
    }
  }
  __syncthreads();
  // Cluster start barrier: every CTA has started and initialised its
  // barriers; arrived before the dependency wait, waited before the first
  // remote store.
  asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
  pdl_wait();
  if (tid == 0) {
    for (int j = j0; j < j1; ++j) {
      const int nbk = min(kSrChunk, B - j * kSrChunk);
      const uint32_t bytes = static_cast<uint32_t>(nbk) * C * 2u;
      mbar_arrive_expect_tx(&bar_chunk[j - j0], bytes);
      bulk_load(sc_stage + static_cast<size_t>(j - j0) * chunk_halves * 2,
                a.po + (row * B + static_cast<int64_t>(j) * kSrChunk) * C, bytes, &bar_chunk[j - j0]);
    }
  }
  // This CTA's blocks' partial_max and partial_sum in registers (both loads
  // in flight together), its maximum, then the row's over the cluster.
  const float* pmr = a.pm + row * B;
  const float* psr = a.ps + row * B;
  constexpr int kScPer = kScMaxCpc * kSrChunk / kScThreads;  // blocks per thread at most
  float pmv[kScPer], psv[kScPer];
#pragma unroll
  for (int i = 0; i < kScPer; ++i) {
    const int b = b_lo + tid + i * kScThreads;
    pmv[i] = b < b_hi ? __ldg(pmr + b) : __int_as_float(0xff800000u);
    psv[i] = b < b_hi ? __ldg(psr + b) : 0.0f;
  }
  float m = pmv[0];
#pragma unroll
  for (int i = 1; i < kScPer; ++i) m = fmaxf(m, pmv[i]);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
  if (lane == 0) s_red[warp] = m;
  __syncthreads();
  asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
  if (tid < cs) {
    float mm = s_red[0];
    for (int w = 1; w < kScThreads / 32; ++w) mm = fmaxf(mm, s_red[w]);
    if (tid == q)
      s_lmax[q] = mm;
    else
      sc_st_peer(&s_lmax[q], static_cast<uint32_t>(tid), mm, &bar_max);  // to CTA tid
  }
  if (tid == 0 && !mbar_wait_bounded(&bar_max, 0, a.timeout_ns)) {
    s_ok = 0;
    atomicOr(a.status, kErrSplitLoadTimeout);
  }
  __syncthreads();  // every CTA's maximum has arrived here
  float M = s_lmax[0];
  for (int p = 1; p < cs; ++p) M = fmaxf(M, s_lmax[p]);
#pragma unroll
  for (int i = 0; i < kScPer; ++i) {
    const int b = b_lo + tid + i * kScThreads;
    if (b < b_hi) {
      s_scale[b - b_lo] = exp_pinned(__fsub_rn(pmv[i], M));
      s_psum[b - b_lo] = psv[i];
    }
  }
  if (tid == 0) {
    for (int j = j0; j < j1; ++j)
      if (!mbar_wait_bounded(&bar_chunk[j - j0], 0, a.timeout_ns)) {
        s_ok = 0;
        atomicOr(a.status, kErrSplitLoadTimeout);
      }
    if (!s_ok)
      for (int j = j0; j < j1; ++j) mbar_wait_bounded(&bar_chunk[j - j0], 0, a.timeout_ns);
  }
  __syncthreads();  // chunks landed, scales staged
  // Runs: work item = (chunk, run, quad of 4 channels); the quad at channel 0
  // also accumulates the run's sum.
  const int qpr = C / 4;
  const int items = (j1 - j0) * kSrRuns * qpr;
  if (s_ok) {
    for (int it = tid; it < items; it += kScThreads) {
      const int jr = it / qpr, qq = it - jr * qpr;   // jr = local chunk * kSrRuns + run
      const int jl = jr / kSrRuns, u = jr - jl * kSrRuns;
      const int c = qq * 4;
      const int bc = (j0 + jl) * kSrChunk;           // first block of the chunk
      const int bl_lo = bc + u * kSrRun, bl_hi = min(B, bl_lo + kSrRun);
      float o0 = 0.0f, o1 = 0.0f, o2 = 0.0f, o3 = 0.0f, acc_s = 0.0f;
      const uint2* src = reinterpret_cast<const uint2*>(stage + static_cast<size_t>(jl) * chunk_halves + c) +
                         static_cast<size_t>(bl_lo - bc) * (C / 4);
      const float* scl = s_scale + (bl_lo - b_lo);
      const float* psl = s_psum + (bl_lo - b_lo);
      auto step = [&](int i) {
        const uint2 v = src[static_cast<size_t>(i) * (C / 4)];
        const float sc = scl[i];
        const float2 f01 = __half22float2(*reinterpret_cast<const __half2*>(&v.x));
        const float2 f23 = __half22float2(*reinterpret_cast<const __half2*>(&v.y));
        o0 = __fadd_rn(o0, __fmul_rn(sc, f01.x));
        o1 = __fadd_rn(o1, __fmul_rn(sc, f01.y));
        o2 = __fadd_rn(o2, __fmul_rn(sc, f23.x));
        o3 = __fadd_rn(o3, __fmul_rn(sc, f23.y));
        if (qq == 0) acc_s = __fadd_rn(acc_s, __fmul_rn(sc, psl[i]));
      };
      const int len = bl_hi - bl_lo;
      if (len == kSrRun) {
#pragma unroll
        for (int i = 0; i < kSrRun; ++i) step(i);  // a whole run: no loop control
      } else {
        for (int i = 0; i < len; ++i) step(i);
      }
      *reinterpret_cast<float4*>(run_out + static_cast<size_t>(jr) * C + c) = make_float4(o0, o1, o2, o3);
      if (qq == 0) run_sum[jr] = acc_s;
    }
  }
  __syncthreads();
  // Chunk partials: a chunk's runs added in order from 0.
  for (int x = tid; x < (j1 - j0) * (C + 1); x += kScThreads) {
    const int jl = x / (C + 1), c = x - jl * (C + 1);
    const int nbk = min(kSrChunk, B - (j0 + jl) * kSrChunk);
    const int nr = (nbk + kSrRun - 1) / kSrRun;
    float part = 0.0f;
    for (int u = 0; u < nr; ++u)
      part = __fadd_rn(part, c < C ? run_out[(static_cast<size_t>(jl) * kSrRuns + u) * C + c]
                                   : run_sum[jl * kSrRuns + u]);
    float* dst = gather + static_cast<size_t>(j0 + jl) * (C + 1) + c;
    if (q == 0)
      *dst = part;
    else
      sc_st_peer(dst, 0u, part, &bar_gather);  // to rank 0
  }
  if (q != 0) return;  // its stores are on their way; rank 0 waits for them
  if (tid == 0 && !mbar_wait_bounded(&bar_gather, 0, a.timeout_ns)) {
    s_ok = 0;
    atomicOr(a.status, kErrSplitLoadTimeout);
  }
  __syncthreads();  // every chunk partial has arrived here
  if (s_ok) {
    // chunk partials in chunk order, then the division
    for (int c = tid; c < C; c += kScThreads) {
      float tot = 0.0f, tot_s = 0.0f;
      for (int j = 0; j < n_chunks; ++j) {
        tot = __fadd_rn(tot, gather[static_cast<size_t>(j) * (C + 1) + c]);
        tot_s = __fadd_rn(tot_s, gather[static_cast<size_t>(j) * (C + 1) + C]);
      }
      a.out[row * C + c] = __fdiv_rn(tot, tot_s);
    }
  }
}

size_t split_cluster_smem(int C, int cpc, int n_chunks) {
  return static_cast<size_t>(cpc) * kSrChunk * C * 2 + 2 * static_cast<size_t>(cpc) * kSrChunk * 4 +
         static_cast<size_t>(cpc) * kSrRuns * C * 4 + static_cast<size_t>(cpc) * kSrRuns * 4 +
         static_cast<size_t>(n_chunks) * (C + 1) * 4 + 16;
}

// Rows per CTA: the whole chunk of a CTA's rows must fit one staging buffer,
// and the grid should cover the GPU about twice.
void split_rows(int32_t G, int32_t R, int32_t B, int32_t C, int sm_count, int* RS, int* Rs) {
  const int64_t S = (static_cast<int64_t>(B) + kSrChunk - 1) / kSrChunk;
  const int64_t row_chunk = static_cast<int64_t>(kSrChunk) * C * 2;
  int rows = static_cast<int>(std::max<int64_t>(1, kSrStageBytes / row_chunk));
  rows = std::min(rows, static_cast<int>(R));
  const int64_t want = 2LL * sm_count;
  while (rows > 1 && static_cast<int64_t>(G) * S * ((R + rows - 1) / rows) < want) rows = (rows + 1) / 2;
  *Rs = rows;
  *RS = (R + rows - 1) / rows;
}

}  // namespace

size_t split_reduce_workspace_bytes(int32_t G, int32_t R, int32_t B, int32_t C) {
  const int64_t S = (static_cast<int64_t>(B) + kSrChunk - 1) / kSrChunk;
  if (G <= 0 || S <= 1) return 0;
  const size_t counters = (static_cast<size_t>(G) * R * sizeof(uint32_t) + 15) & ~static_cast<size_t>(15);
  const size_t sums = (static_cast<size_t>(G) * S * R * sizeof(float) + 15) & ~static_cast<size_t>(15);
  return counters + sums + static_cast<size_t>(G) * S * R * C * sizeof(float);
}

cudaError_t init_split_reduce_kernel(const DeviceInfo& dev) {
  cudaError_t e = cudaFuncSetAttribute(split_reduce_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, kSrSmemMax);
  if (e != cudaSuccess) return e;
  cudaFuncAttributes fa;
  if ((e = cudaFuncGetAttributes(&fa, reinterpret_cast<const void*>(&split_cluster_kernel))) !=
      cudaSuccess)
    return e;
  return cudaFuncSetAttribute(split_cluster_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              dev.max_smem_optin - static_cast<int>(fa.sharedSizeBytes));
}

cudaError_t launch_split_reduce(const SplitReduceProblem& p, const DeviceInfo& dev,
                                cudaStream_t stream) {
  if (p.G <= 0) return cudaSuccess;
  // The cluster form when a chunk's rows are whole 16-byte units, the CTAs
  // of a row fit one portable cluster and their staging fits one CTA: as
  // many CTAs per row (up to 8) as leave each at most kScMaxCpc chunks.
  {
    const int n_chunks = (p.B + kSrChunk - 1) / kSrChunk;
    int cpc = std::max(1, (n_chunks + kScMaxCs - 1) / kScMaxCs);
    const int cs = (n_chunks + cpc - 1) / cpc;
    const size_t smem = split_cluster_smem(p.C, cpc, n_chunks);
    const int64_t rows = static_cast<int64_t>(p.G) * p.R;
    if (p.C % 8 == 0 && reinterpret_cast<uintptr_t>(p.partial_out) % 16 == 0 && cpc <= kScMaxCpc &&
        cs <= kScMaxCs && smem + 1024 <= static_cast<size_t>(dev.max_smem_optin) &&
        rows * cs <= 0x7FFFFFFFLL) {
      ScArgs s;
      s.pm = p.partial_max;
      s.ps = p.partial_sum;
      s.po = reinterpret_cast<const __half*>(p.partial_out);
      s.out = p.out;
      s.status = dev.status_word;
      s.timeout_ns = kWaitTimeoutNs;
      s.R = p.R;
      s.B = p.B;
      s.C = p.C;
      s.cs = cs;
      s.cpc = cpc;
      cudaLaunchConfig_t cfg = {};
      cfg.gridDim = dim3(static_cast<unsigned>(rows * cs));
      cfg.blockDim = dim3(kScThreads);
      cfg.dynamicSmemBytes = smem;
      cfg.stream = stream;
      cudaLaunchAttribute attr[2];
      attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
      attr[0].val.programmaticStreamSerializationAllowed = 1;
      attr[1].id = cudaLaunchAttributeClusterDimension;
      attr[1].val.clusterDim.x = static_cast<unsigned>(cs);
      attr[1].val.clusterDim.y = 1;
      attr[1].val.clusterDim.z = 1;
      cfg.attrs = attr;
      cfg.numAttrs = 2;
      plan_add("split_cluster_kernel");
      return cudaLaunchKernelEx(&cfg, split_cluster_kernel, s);
    }
  }
  SrArgs a;
  a.pm = p.partial_max;
  a.ps = p.partial_sum;
  a.po = reinterpret_cast<const __half*>(p.partial_out);
  a.out = p.out;
  a.R = p.R;
  a.B = p.B;
  a.C = p.C;
  a.S = (p.B + kSrChunk - 1) / kSrChunk;
  a.status = dev.status_word;
  a.timeout_ns = kWaitTimeoutNs;
  split_rows(p.G, p.R, p.B, p.C, dev.sm_count, &a.RS, &a.Rs);
  // Bulk copies need 16-byte aligned rows (C a multiple of 8 and an aligned
  // base), and one row's chunk must fit the staging buffer (C <= 768).
  a.staged = (p.C % 8 == 0 && reinterpret_cast<uintptr_t>(p.partial_out) % 16 == 0 &&
              static_cast<int64_t>(kSrChunk) * p.C * 2 <= kSrStageBytes)
                 ? 1 : 0;
  a.pm_vec = (p.B % 4 == 0 && reinterpret_cast<uintptr_t>(p.partial_max) % 16 == 0 &&
              reinterpret_cast<uintptr_t>(p.partial_sum) % 16 == 0)
                 ? 1 : 0;
  a.stage_bytes = a.staged ? a.Rs * kSrChunk * p.C * 2 : 0;
  const size_t smem = static_cast<size_t>(a.stage_bytes) +
                      static_cast<size_t>(kSrRuns) * (a.Rs * p.C / 4) * 16 +
                      static_cast<size_t>(kSrRuns) * a.Rs * 4 +
                      2 * static_cast<size_t>(a.Rs) * kSrChunk * 4;
  uint8_t* ws = static_cast<uint8_t*>(p.workspace);
  const size_t counters = (static_cast<size_t>(p.G) * p.R * sizeof(uint32_t) + 15) & ~static_cast<size_t>(15);
  const size_t sums = (static_cast<size_t>(p.G) * a.S * p.R * sizeof(float) + 15) & ~static_cast<size_t>(15);
  a.count = a.S > 1 ? reinterpret_cast<uint32_t*>(ws) : nullptr;
  a.part_sum = a.S > 1 ? reinterpret_cast<float*>(ws + counters) : nullptr;
  a.part_out = a.S > 1 ? reinterpret_cast<float*>(ws + counters + sums) : nullptr;
  plan_add("split_reduce_kernel");
  return launch_pdl(split_reduce_kernel,
                    dim3(static_cast<unsigned>(a.S), static_cast<unsigned>(a.RS),
                         static_cast<unsigned>(p.G)),
                    dim3(kSrThreads), smem, stream, a);
}

}  // namespace qsa
