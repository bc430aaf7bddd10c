// split_reduce.cu - the flash-attention decode split reduce (1bit-MONSTER
// llama.cpp pull request 30, "What" and "Changes"; its review asks for a
// bounded scale stage).
//
// Per group g and row r: maximum = max_b partial_max; scale_b =
// exp(partial_max_b - maximum), once per (row, block); sum = sum_b scale_b *
// partial_sum_b; out[c] = (sum_b scale_b * partial_out_b[c]) / sum.
//
// GB300 layout of the work: the blocks are cut into chunks of kSrChunk
// (64); CTA (j, g) reduces chunk j of group g. Each CTA finds the rows'
// maxima over all blocks (partial_max is small and L2-resident), stages its
// chunk's scales in shared memory (R x 64 floats: bounded whatever the
// context length), and runs the all-rows output pass: a thread owns a quad
// of 4 channels of one row and accumulates fp32 over the chunk's blocks from
// 8-byte fp16 loads (a warp reads 256 contiguous bytes per block). Chunk
// partials go to the caller's workspace; the last CTA of a group to finish
// (an arrival counter) adds them in chunk order and divides. With one chunk
// the CTA writes the output directly.
//
// Arithmetic, fixed operation for operation (the CPU oracle's pinned fp32
// procedure follows the same steps): scale = exp_pinned(fl(pm - maximum));
// inside a chunk, acc = fl(acc + fl(scale * x)) block by block (no fused
// multiply-add); chunk partials added in chunk order; out = fl(O / sum).
#include <cuda_fp16.h>

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
  uint32_t* count;      // [G] arrival counters (zero between calls)
  float* part_sum;      // [G][S][R]
  float* part_out;      // [G][S][R][C]
  int R, B, C, S;
};

__global__ void __launch_bounds__(kSrThreads) split_reduce_kernel(const SrArgs a) {
  __shared__ float s_max[kSrMaxRows];
  __shared__ float s_rowsum[kSrMaxRows];
  __shared__ float s_scale[kSrMaxRows * kSrChunk];
  __shared__ int s_last;
  const int j = blockIdx.x, g = blockIdx.y;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int R = a.R, B = a.B, C = a.C;
  const int64_t grb = static_cast<int64_t>(g) * R * B;

  pdl_launch_dependents();
  pdl_wait();

  // Row maxima over every block (one warp per row).
  for (int r = warp; r < R; r += kSrThreads / 32) {
    const float* row = a.pm + grb + static_cast<int64_t>(r) * B;
    float m = __int_as_float(0xff800000u);  // -inf
    for (int b = lane; b < B; b += 32) m = fmaxf(m, __ldg(row + b));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
    if (lane == 0) s_max[r] = m;
  }
  __syncthreads();

  // This chunk's scales, staged per row.
  const int b0 = j * kSrChunk;
  const int nbk = min(kSrChunk, B - b0);
  for (int i = tid; i < R * nbk; i += kSrThreads) {
    const int r = i / nbk, bl = i - r * nbk;
    const float d = __fsub_rn(__ldg(a.pm + grb + static_cast<int64_t>(r) * B + b0 + bl), s_max[r]);
    s_scale[r * kSrChunk + bl] = exp_pinned(d);
  }
  __syncthreads();

  // Output pass: thread -> quads (row, 4 channels); the quad at channel 0
  // also accumulates the row's sum.
  const int qpr = C / 4;
  const int nquads = R * qpr;
  float acc_q[kSrMaxQuadsPerThread][4];
  float acc_sq[kSrMaxQuadsPerThread];
#pragma unroll
  for (int u = 0; u < kSrMaxQuadsPerThread; ++u) {
    acc_q[u][0] = acc_q[u][1] = acc_q[u][2] = acc_q[u][3] = 0.0f;
    acc_sq[u] = 0.0f;
    const int q = tid + u * kSrThreads;
    if (q >= nquads) continue;
    const int r = q / qpr, c = (q - r * qpr) * 4;
    const uint2* src = reinterpret_cast<const uint2*>(
        a.po + ((grb + static_cast<int64_t>(r) * B + b0) * C + c));
    const float* srow = s_scale + r * kSrChunk;
    const float* psrow = a.ps + grb + static_cast<int64_t>(r) * B + b0;
    const int64_t stride = C / 4;  // uint2 (4 halves) per block
    float o0 = 0.0f, o1 = 0.0f, o2 = 0.0f, o3 = 0.0f, acc_s = 0.0f;
    for (int bl0 = 0; bl0 < nbk; bl0 += 8) {
      uint2 v[8];
      float pv[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        if (bl0 + e < nbk) {
          v[e] = __ldg(src + (bl0 + e) * stride);
          pv[e] = c == 0 ? __ldg(psrow + bl0 + e) : 0.0f;
        }
      }
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        if (bl0 + e < nbk) {
          const float s = srow[bl0 + e];
          const __half2 h01 = *reinterpret_cast<const __half2*>(&v[e].x);
          const __half2 h23 = *reinterpret_cast<const __half2*>(&v[e].y);
          o0 = __fadd_rn(o0, __fmul_rn(s, __low2float(h01)));
          o1 = __fadd_rn(o1, __fmul_rn(s, __high2float(h01)));
          o2 = __fadd_rn(o2, __fmul_rn(s, __low2float(h23)));
          o3 = __fadd_rn(o3, __fmul_rn(s, __high2float(h23)));
          if (c == 0) acc_s = __fadd_rn(acc_s, __fmul_rn(s, pv[e]));
        }
      }
    }
    acc_q[u][0] = o0;
    acc_q[u][1] = o1;
    acc_q[u][2] = o2;
    acc_q[u][3] = o3;
    acc_sq[u] = acc_s;
    if (c == 0) s_rowsum[r] = acc_s;
  }

  const int64_t grc = static_cast<int64_t>(g) * R * C;
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
  // group adds them in chunk order.
  const int64_t gs = static_cast<int64_t>(g) * a.S;
#pragma unroll
  for (int u = 0; u < kSrMaxQuadsPerThread; ++u) {
    const int q = tid + u * kSrThreads;
    if (q >= nquads) continue;
    const int r = q / qpr, c = (q - r * qpr) * 4;
    *reinterpret_cast<float4*>(a.part_out + ((gs + j) * R + r) * C + c) =
        make_float4(acc_q[u][0], acc_q[u][1], acc_q[u][2], acc_q[u][3]);
    if (c == 0) a.part_sum[(gs + j) * R + r] = acc_sq[u];
  }
  __threadfence();
  __syncthreads();
  if (tid == 0) s_last = atomicAdd(a.count + g, 1u) == static_cast<uint32_t>(a.S - 1);
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  if (tid == 0) a.count[g] = 0;  // ready for the next call
#pragma unroll
  for (int u = 0; u < kSrMaxQuadsPerThread; ++u) {
    const int q = tid + u * kSrThreads;
    if (q >= nquads) continue;
    const int r = q / qpr, c = (q - r * qpr) * 4;
    float L = 0.0f, o0 = 0.0f, o1 = 0.0f, o2 = 0.0f, o3 = 0.0f;
    for (int jj = 0; jj < a.S; ++jj) {
      const float4 v = __ldcg(reinterpret_cast<const float4*>(a.part_out + ((gs + jj) * R + r) * C + c));
      L = __fadd_rn(L, __ldcg(a.part_sum + (gs + jj) * R + r));
      o0 = __fadd_rn(o0, v.x);
      o1 = __fadd_rn(o1, v.y);
      o2 = __fadd_rn(o2, v.z);
      o3 = __fadd_rn(o3, v.w);
    }
    *reinterpret_cast<float4*>(a.out + grc + static_cast<int64_t>(r) * C + c) =
        make_float4(__fdiv_rn(o0, L), __fdiv_rn(o1, L), __fdiv_rn(o2, L), __fdiv_rn(o3, L));
  }
}

}  // namespace

size_t split_reduce_workspace_bytes(int32_t G, int32_t R, int32_t B, int32_t C) {
  const int64_t S = (static_cast<int64_t>(B) + kSrChunk - 1) / kSrChunk;
  if (G <= 0 || S <= 1) return 0;
  const size_t counters = (static_cast<size_t>(G) * sizeof(uint32_t) + 15) & ~static_cast<size_t>(15);
  const size_t sums = (static_cast<size_t>(G) * S * R * sizeof(float) + 15) & ~static_cast<size_t>(15);
  return counters + sums + static_cast<size_t>(G) * S * R * C * sizeof(float);
}

cudaError_t launch_split_reduce(const SplitReduceProblem& p, const DeviceInfo& dev,
                                cudaStream_t stream) {
  (void)dev;
  if (p.G <= 0) return cudaSuccess;
  SrArgs a;
  a.pm = p.partial_max;
  a.ps = p.partial_sum;
  a.po = reinterpret_cast<const __half*>(p.partial_out);
  a.out = p.out;
  a.R = p.R;
  a.B = p.B;
  a.C = p.C;
  a.S = (p.B + kSrChunk - 1) / kSrChunk;
  uint8_t* ws = static_cast<uint8_t*>(p.workspace);
  const size_t counters = (static_cast<size_t>(p.G) * sizeof(uint32_t) + 15) & ~static_cast<size_t>(15);
  const size_t sums = (static_cast<size_t>(p.G) * a.S * p.R * sizeof(float) + 15) & ~static_cast<size_t>(15);
  a.count = a.S > 1 ? reinterpret_cast<uint32_t*>(ws) : nullptr;
  a.part_sum = a.S > 1 ? reinterpret_cast<float*>(ws + counters) : nullptr;
  a.part_out = a.S > 1 ? reinterpret_cast<float*>(ws + counters + sums) : nullptr;
  return launch_pdl(split_reduce_kernel, dim3(static_cast<unsigned>(a.S), static_cast<unsigned>(p.G)),
                    dim3(kSrThreads), 0, stream, a);
}

}  // namespace qsa
