// qsa_internal.h - host-side declarations shared by the C-ABI layer and the
// kernel translation units. Not installed; not part of the ABI.
#pragma once

#include <cstdint>
#include <utility>
#include <cuda.h>
#include <cuda_runtime.h>

namespace qsa {

// Launches `kernel` with programmatic stream serialization: it may start
// while the previous kernel on the stream finishes; the kernel itself must
// call pdl_wait() before reading what earlier work produced.
template <typename... Params, typename... Args>
cudaError_t launch_pdl(void (*kernel)(Params...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t stream, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

struct DeviceInfo {
  int id = -1;
  int sm_count = 0;
  int cc_major = 0, cc_minor = 0;
  int max_smem_optin = 0;
  uint32_t* status_word = nullptr;  // device address of this device's status word
  bool supported = false;           // compute capability 10.3
  bool ready = false;               // kernel attributes set
};

// Info for the current device, initialised once per device (attributes of the
// kernels are set then). Returns nullptr and sets *err on a CUDA failure.
const DeviceInfo* current_device(cudaError_t* err);

// cuTensorMapEncodeTiled from the driver, looked up once.
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn encode_tiled_fn();

// The launch plan of the last library call on this thread, which qsa_arm()
// reports: each entry point clears it (plan_begin) and every launcher
// appends the kernel it launched (plan_add, a static string), so a chain of
// separate kernels or a different form of a kernel cannot pass for another.
void plan_begin();
void plan_add(const char* kernel);

// Per-TU one-time kernel attribute setup, called from current_device().
cudaError_t init_score_kernels(const DeviceInfo& dev);
cudaError_t init_select_kernels(const DeviceInfo& dev);

// Launchers. Each returns cudaSuccess or the first CUDA error; arguments are
// already validated by the caller.
cudaError_t launch_convert(const float* src, uint16_t* dst, int64_t n, const DeviceInfo& dev,
                           cudaStream_t stream);

struct ScoreProblem {
  const uint16_t* q;
  const uint16_t* kb;
  float* scores;
  int32_t nq, H, D;
  int64_t nb, n_full;
  bool has_tail;
  bool skip_tail;  // the tail column is left to the select (select_scores_tail)
  // n_batches > 1: that many batches of nq queries, q, scores contiguous per
  // batch; kb per batch at kb_batch_stride elements (0: one kb shared). Only
  // the persistent kernel takes batches (scores_persistent), with skip_tail
  // or no tail.
  int32_t n_batches = 1;
  int64_t kb_batch_stride = 0;
};
// True when launch_scores runs the persistent score kernel for p (many
// full-width tiles; the only form that takes batches).
bool scores_persistent(const ScoreProblem& p, const DeviceInfo& dev);
// Returns cudaErrorInvalidValue if a tensor map cannot be encoded, or for
// batches the persistent kernel cannot take.
cudaError_t launch_scores(const ScoreProblem& p, const DeviceInfo& dev, cudaStream_t stream);

// The fused step: optional fp32->fp16 conversion of q, block scores (full
// blocks and tail) and the top-k select in one cluster launch. Exactly one of
// q32 / q16 is non-null; q16out (fp32 input only) may be null.
struct FusedProblem {
  const float* q32;
  const uint16_t* q16;
  uint16_t* q16out;
  const uint16_t* kb;
  float* scores;
  int32_t* ids;
  int32_t nq, H, D;
  int64_t nb, n_full;
  bool has_tail;
  int32_t k;
  int32_t n_batches;        // independent query batches in this launch (>= 1)
  int64_t kb_batch_stride;  // kb elements between batches; 0 = kb shared by all batches
};
cudaError_t init_fused_kernels(const DeviceInfo& dev);
// CTAs the fused kernel would launch for one batch of nq queries of H heads.
int64_t fused_blocks(int32_t nq, int32_t H, const DeviceInfo& dev);
cudaError_t launch_fused(const FusedProblem& p, const DeviceInfo& dev, cudaStream_t stream);

// The tail block of a chained step, scored by the select kernel itself (fp16
// queries [nq, H, D] and the tail's key row); see select_scores_tail.
struct TailInfo {
  const uint16_t* q16;
  const uint16_t* kb_tail;  // the tail's key row (of batch 0)
  int32_t H, D;
  int64_t kb_batch_stride = 0;  // elements between batches' kb; 0: one kb
  int32_t nq_per_batch = 1;     // rows of one batch (used when kb_batch_stride != 0)
};
// True when launch_select with a TailInfo scores the tail column (column nb-1)
// itself before selecting: many rows, k <= 128, nb <= 4096.
bool select_scores_tail(int32_t nq, int32_t nb, int32_t k);
cudaError_t launch_select(const float* scores, int32_t nq, int32_t nb, int32_t k, int32_t* ids,
                          const DeviceInfo& dev, cudaStream_t stream,
                          const TailInfo* tail = nullptr);

// Launches the bounded-wait self-test (see qsa_selftest_bounded_wait).
cudaError_t launch_selftest_wait(const DeviceInfo& dev, uint64_t timeout_ns, cudaStream_t stream);

// Flash-attention decode split reduce (split_reduce.cu).
constexpr int kSrChunk = 128;             // blocks per CTA (the bounded scale stage)
constexpr int kSrRun = 32;                // blocks per run inside a chunk
constexpr int kSrRuns = kSrChunk / kSrRun;
constexpr int kSrMaxRows = 32;            // rows (query heads per KV head)
constexpr int kSrMaxQuadsPerThread = 4;   // R * C / 4 <= 4 * 256
constexpr int kSrStageBytes = 96 * 1024;  // staged fp16 partial outputs per CTA
constexpr int kSrSmemMax =
    kSrStageBytes + kSrRuns * 1024 * 16 + kSrRuns * kSrMaxRows * 4 + 2 * kSrMaxRows * kSrChunk * 4;
struct SplitReduceProblem {
  const float* partial_max;
  const float* partial_sum;
  const uint16_t* partial_out;
  float* out;
  void* workspace;  // split_reduce_workspace_bytes(G, R, B, C) bytes; counters zero
  int32_t G, R, B, C;
};
size_t split_reduce_workspace_bytes(int32_t G, int32_t R, int32_t B, int32_t C);
cudaError_t init_split_reduce_kernel(const DeviceInfo& dev);
// Address of the current device's fixed split-reduce scratch
// (QSA_SPLIT_STATIC_SCRATCH_BYTES), looked up once per device; null and *err
// set on failure.
void* split_static_scratch(cudaError_t* err);
cudaError_t launch_split_reduce(const SplitReduceProblem& p, const DeviceInfo& dev,
                                cudaStream_t stream);

constexpr int kMaxSelectK = 1024;
constexpr int kMaxSelectNb = 32768;
constexpr uint64_t kWaitTimeoutNs = 2000000000ull;  // 2 s bound on any device-side wait

}  // namespace qsa
