// fused.cu - host side of the fused step kernel (fused_kernel.cuh): the
// choice of form and cluster size, shared-memory layout, tensor maps and the
// launch. The kernels themselves are instantiated in fused_h{1,...,32}.cu.
#include <map>
#include <mutex>
#include <tuple>

#include "fused_kernel.cuh"

namespace qsa {

// ------------------------------------------------------------------ host
namespace {

constexpr int kCluster = 8;  // CTAs per cluster in the regular and lean forms
constexpr int kClusterWide = 16;

const void* fused_kernel_for(int H, bool f32q, int form) {
  switch (H) {
    case 1: return fused_kernel_h1(f32q, form);
    case 2: return fused_kernel_h2(f32q, form);
    case 4: return fused_kernel_h4(f32q, form);
    case 8: return fused_kernel_h8(f32q, form);
    case 16: return fused_kernel_h16(f32q, form);
    case 32: return fused_kernel_h32(f32q, form);
    default: return nullptr;
  }
}

// 3-D fp16 map: [z][rows][cols] with a z stride in elements (a multiple of 8).
bool encode_f16_3d(CUtensorMap* tm, const void* base, uint64_t cols, uint64_t rows, uint64_t zs,
                   uint64_t z_stride, uint32_t box_cols, uint32_t box_rows) {
  EncodeTiledFn enc = encode_tiled_fn();
  if (!enc) return false;
  const cuuint64_t dims[3] = {cols, rows, zs};
  const cuuint64_t strides[2] = {cols * 2, z_stride * 2};
  const cuuint32_t box[3] = {box_cols, box_rows, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  return enc(tm, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, const_cast<void*>(base), dims, strides, box,
             estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool encode_f16_2d(CUtensorMap* tm, const void* base, uint64_t cols, uint64_t rows,
                   uint32_t box_cols, uint32_t box_rows) {
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

}  // namespace

int g_fused_static_smem = 0;

cudaError_t init_fused_kernels(const DeviceInfo& dev) {
  for (int H : {1, 2, 4, 8, 16, 32})
    for (bool f : {false, true})
      for (int form : {kFormRegular, kFormLean, kFormWide}) {
        const void* fn = fused_kernel_for(H, f, form);
        cudaFuncAttributes fa;
        cudaError_t e = cudaFuncGetAttributes(&fa, fn);
        if (e != cudaSuccess) return e;
        g_fused_static_smem = std::max(g_fused_static_smem, static_cast<int>(fa.sharedSizeBytes));
        e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 dev.max_smem_optin - static_cast<int>(fa.sharedSizeBytes));
        if (e != cudaSuccess) return e;
        // Always the largest shared-memory carveout: two CTAs of a cluster per
        // SM need it, and a smaller carveout chosen from one launch's request
        // left room for one cluster CTA per SM (half the clusters resident).
        e = cudaFuncSetAttribute(fn, cudaFuncAttributePreferredSharedMemoryCarveout,
                                 cudaSharedmemCarveoutMaxShared);
        if (e != cudaSuccess) return e;
        if (form == kFormWide) {  // 16-CTA clusters are beyond the portable size of 8
          e = cudaFuncSetAttribute(fn, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
          if (e != cudaSuccess) return e;
        }
      }
  return cudaSuccess;
}

namespace {
// Columns per query group: 64 unless that would need more than about two
// waves of 8-CTA clusters, then 128.
int fused_bn(int32_t nq, int32_t H, const DeviceInfo& dev) {
  const int64_t groups64 = (nq + (64 / std::min(64, H)) - 1) / (64 / std::min(64, H));
  return groups64 * kCluster > 4LL * dev.sm_count ? 128 : std::max(64, static_cast<int>(H));
}
}  // namespace

int64_t fused_blocks(int32_t nq, int32_t H, const DeviceInfo& dev) {
  const int qg = fused_bn(nq, H, dev) / H;
  return ((static_cast<int64_t>(nq) + qg - 1) / qg) * kCluster;
}

namespace {
// Whether a cluster of the wide form fits the device with this launch's
// shared memory (asked of the runtime once per kernel and size): if not, the
// launch takes the 8-CTA form instead of failing.
bool wide_fits(const void* fn, const cudaLaunchConfig_t& cfg, const DeviceInfo& dev) {
  static std::mutex mu;
  static std::map<std::tuple<int, const void*, size_t>, bool> cache;
  const auto key = std::make_tuple(dev.id, fn, cfg.dynamicSmemBytes);
  std::lock_guard<std::mutex> lock(mu);
  auto it = cache.find(key);
  if (it != cache.end()) return it->second;
  int n = 0;
  const bool ok = cudaOccupancyMaxActiveClusters(&n, fn, &cfg) == cudaSuccess && n >= 1;
  cudaGetLastError();  // a refused query leaves no sticky error behind
  cache.emplace(key, ok);
  return ok;
}

cudaError_t launch_fused_impl(const FusedProblem& p, const DeviceInfo& dev, cudaStream_t stream,
                              bool allow_wide) {
  if (p.nq <= 0) return cudaSuccess;
  const int bn = fused_bn(p.nq, p.H, dev);
  const int qg = bn / p.H;
  const int64_t groups = (p.nq + qg - 1) / qg;
  const int32_t m_tiles = static_cast<int32_t>((p.n_full + kFTileM - 1) / kFTileM);
  // Wide form (16-CTA clusters) for one or two clusters with at least one
  // block tile per CTA: decode-shaped steps, where most SMs are idle and each
  // CTA's kb load and MMA chain halve.
  const bool wide = allow_wide && static_cast<int64_t>(p.n_batches) * groups <= 2 &&
                    m_tiles >= kClusterWide && bn % kClusterWide == 0;
  const int cluster = wide ? kClusterWide : kCluster;
  const int64_t blocks = static_cast<int64_t>(p.n_batches) * groups * cluster;
  if (blocks > 0x7FFFFFFFLL || groups > 0x7FFFFFFFLL) return cudaErrorInvalidValue;
  FusedArgs a;
  a.q32 = p.q32;
  a.q16in = reinterpret_cast<const __half*>(p.q16);
  a.q16out = reinterpret_cast<__half*>(p.q16out);
  a.kb = reinterpret_cast<const __half*>(p.kb);
  a.scores = p.scores;
  a.ids = p.ids;
  a.nq = p.nq;
  a.groups_per_batch = static_cast<int32_t>(groups);
  a.q_batch_elems = static_cast<int64_t>(p.nq) * p.H * p.D;
  a.kb_batch_stride = p.kb_batch_stride;
  a.D = p.D;
  a.nb = static_cast<int32_t>(p.nb);
  a.n_full = static_cast<int32_t>(p.n_full);
  a.has_tail = p.has_tail ? 1 : 0;
  a.k = p.k;
  a.bn = bn;
  a.qg = qg;
  a.m_tiles = m_tiles;
  a.n_chunks = (p.D + kFKAtom - 1) / kFKAtom;
  a.k_steps = p.D / 16;
  a.tmem_cols = 2u * static_cast<uint32_t>(bn) <= 32u ? 32u : 2u * static_cast<uint32_t>(bn);
  a.status = dev.status_word;
  a.timeout_ns = kWaitTimeoutNs;
  const int rows_per_cta = (qg + cluster - 1) / cluster;
  // Lean form for launches of several waves (CTAs overlap one another's
  // phases): one Kb stage and at most 72 registers, so three CTAs fit an SM;
  // only while three CTAs' TMEM columns fit the SM's 512.
  const bool lean = !wide && blocks > 2LL * dev.sm_count && 3u * (2u * static_cast<uint32_t>(bn)) <= 512u;
  a.kb_stages = lean ? 1 : 2;
  const size_t operand_bytes =
      static_cast<size_t>(a.n_chunks) * (bn + a.kb_stages * kFTileM) * kFRowBytes;
  const size_t budget = static_cast<size_t>(dev.max_smem_optin) - g_fused_static_smem - 1024;
  // Select scratch in the operand region after the epilogue: hist, excl,
  // cand, sel, sel_bin, and (global mode, long rows) the row's staged keys
  // (16-byte aligned: k is rounded up to a multiple of 4).
  const size_t k4 = (static_cast<size_t>(p.k) + 3) & ~static_cast<size_t>(3);
  const size_t core = 2 * kSelHistBins * sizeof(uint32_t) +
                      (static_cast<size_t>(kSelBinMax) + p.k) * sizeof(uint64_t) +
                      k4 * sizeof(uint32_t);
  // DSMEM mode when the keys of the rows this CTA selects fit beside the
  // operand tiles.
  const size_t row_bytes = (static_cast<size_t>(a.nb) * sizeof(uint32_t) + 15) & ~static_cast<size_t>(15);
  const size_t rows_off = (std::max(operand_bytes, core) + 1023) & ~static_cast<size_t>(1023);
  a.dsmem = (rows_off + rows_per_cta * row_bytes <= budget) ? 1 : 0;
  a.q_share = (p.q32 != nullptr && a.dsmem && bn % cluster == 0) ? 1 : 0;
  const size_t sel_bytes = a.dsmem ? core : core + static_cast<size_t>(a.nb) * sizeof(uint32_t);
  a.sel_bytes = static_cast<uint32_t>(sel_bytes);
  a.row_bytes = static_cast<uint32_t>(row_bytes);
  a.rows_off = static_cast<uint32_t>(rows_off);
  size_t smem = a.dsmem ? rows_off + rows_per_cta * row_bytes : std::max(operand_bytes, sel_bytes);
  smem += 1024;  // alignment slack
  if (smem + g_fused_static_smem > static_cast<size_t>(dev.max_smem_optin)) return cudaErrorInvalidValue;

  CUtensorMap tm_kb, tm_q;
  memset(&tm_kb, 0, sizeof(tm_kb));
  memset(&tm_q, 0, sizeof(tm_q));
  if (p.n_full > 0) {
    const uint64_t zs = p.kb_batch_stride != 0 ? static_cast<uint64_t>(p.n_batches) : 1u;
    const uint64_t zst = p.kb_batch_stride != 0 ? static_cast<uint64_t>(p.kb_batch_stride)
                                                : static_cast<uint64_t>(p.n_full) * p.D;
    if (!encode_f16_3d(&tm_kb, p.kb, p.D, p.n_full, zs, zst, kFKAtom, kFTileM))
      return cudaErrorInvalidValue;
  }
  if (p.q32 == nullptr &&
      !encode_f16_2d(&tm_q, p.q16, p.D, static_cast<uint64_t>(p.n_batches) * p.nq * p.H, kFKAtom, bn))
    return cudaErrorInvalidValue;
  const bool f32q = p.q32 != nullptr;
  const void* fn = fused_kernel_for(p.H, f32q, wide ? kFormWide : lean ? kFormLean : kFormRegular);
  if (fn == nullptr) return cudaErrorInvalidValue;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(blocks));
  cfg.blockDim = dim3(kFThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = static_cast<unsigned>(cluster);
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  if (wide && !wide_fits(fn, cfg, dev)) return launch_fused_impl(p, dev, stream, false);
  plan_add(wide   ? "fused_step_kernel (16-CTA clusters)"
           : lean ? "fused_step_kernel (8-CTA clusters, lean form)"
                  : "fused_step_kernel (8-CTA clusters)");
  void* args[] = {&tm_kb, &tm_q, &a};
  cudaError_t e = cudaLaunchKernelExC(&cfg, fn, args);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_fused(const FusedProblem& p, const DeviceInfo& dev, cudaStream_t stream) {
  return launch_fused_impl(p, dev, stream, true);
}

}  // namespace qsa
