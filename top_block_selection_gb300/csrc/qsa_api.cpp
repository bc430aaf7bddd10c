// qsa_api.cpp - the C ABI (include/qsa.h): host-side validation, block
// partition, and stream-ordered launches. Arguments are checked before any
// CUDA call, so a bad call returns a status without touching the device.
#include "qsa.h"

#include <cstdint>
#include <cstdio>
#include <cuda_runtime.h>

#include "qsa_internal.h"

namespace qsa {
void plan_begin();
void plan_add(const char* kernel);
}  // namespace qsa

namespace {

using qsa::DeviceInfo;

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

bool supported_heads(int32_t H) {
  return H == 1 || H == 2 || H == 4 || H == 8 || H == 16 || H == 32;
}

cudaStream_t as_cuda(qsa_stream_t s) { return reinterpret_cast<cudaStream_t>(s); }

thread_local const char* t_last_cuda_error = "no error";

// The kernels the last call on this thread launched, in order (static names).
constexpr int kPlanMax = 8;
thread_local const char* t_plan[kPlanMax];
thread_local int t_plan_n = 0;
thread_local bool t_plan_any = false;

qsa_status cuda_fail(cudaError_t e) {
  t_last_cuda_error = cudaGetErrorString(e);
  return QSA_ERR_CUDA;
}

qsa_status from_cuda(cudaError_t e) { return e == cudaSuccess ? QSA_OK : cuda_fail(e); }

// Returns the current device's info, or an error status. Entry points that
// launch pass launching = true, which starts this thread's plan record.
qsa_status device_or_error(const DeviceInfo** out, bool launching = true) {
  cudaError_t e = cudaSuccess;
  const DeviceInfo* d = qsa::current_device(&e);
  if (!d) return cuda_fail(e);
  if (!d->supported) return QSA_ERR_UNSUPPORTED_ARCH;
  *out = d;
  if (launching) qsa::plan_begin();
  return QSA_OK;
}

struct Geometry {
  int64_t nb = 0, n_full = 0;
  bool has_tail = false;
};

// Checks shared by every scoring entry point; fills g on success.
qsa_status check_scores(const uint16_t* q, const uint16_t* kb, int32_t nq, int32_t H, int32_t D,
                        int64_t n_kv, int32_t block, const float* scores, Geometry* g) {
  if (nq < 0 || n_kv < 0 || block < 1 || H < 1 || D < 1) return QSA_ERR_INVALID_ARG;
  if (!supported_heads(H) || D % 16 != 0 || D < 16 || D > 256) return QSA_ERR_UNSUPPORTED_GEOMETRY;
  g->nb = n_kv / block + (n_kv % block != 0 ? 1 : 0);
  g->n_full = n_kv / block;
  g->has_tail = (n_kv % block) != 0;
  if (g->nb > 0x7FFFFFFFLL || static_cast<int64_t>(nq) * H > 0x7FFFFFFFLL)
    return QSA_ERR_UNSUPPORTED_GEOMETRY;
  if (nq == 0 || g->nb == 0) return QSA_OK;
  if (!q || !kb || !scores) return QSA_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(kb, 16) || !aligned(scores, 16)) return QSA_ERR_MISALIGNED;
  return QSA_OK;
}

qsa_status check_select(const float* scores, int32_t nq, int64_t nb, int32_t k,
                        const int32_t* ids) {
  if (nq < 0 || nb < 0 || k < 1) return QSA_ERR_INVALID_ARG;
  if (k > qsa::kMaxSelectK || nb > qsa::kMaxSelectNb) return QSA_ERR_UNSUPPORTED_GEOMETRY;
  if (nq == 0) return QSA_OK;
  if (!ids || (nb > 0 && !scores)) return QSA_ERR_INVALID_ARG;
  if (!aligned(ids, 4) || !aligned(scores, 4)) return QSA_ERR_MISALIGNED;
  return QSA_OK;
}

qsa_status run_scores(const uint16_t* q, const uint16_t* kb, int32_t nq, int32_t H, int32_t D,
                      const Geometry& g, float* scores, const DeviceInfo& dev,
                      cudaStream_t stream, bool skip_tail = false) {
  if (nq == 0 || g.nb == 0) return QSA_OK;
  qsa::ScoreProblem p{q, kb, scores, nq, H, D, g.nb, g.n_full, g.has_tail, skip_tail};
  return from_cuda(qsa::launch_scores(p, dev, stream));
}

// The single-batch steps run either the one fused cluster kernel or the
// separate stages (convert, score + tail, select) chained by programmatic
// dependent launch. Fused wins while its CTAs fit in a few waves (it saves the
// scores round trip and the launch gaps); past that the separate score kernel,
// which tiles 128 key blocks per MMA against many queries, does less work per
// score. Both write identical scores and ids.
bool use_separate(int32_t nq, int32_t H, const DeviceInfo& dev) {
  return qsa::fused_blocks(nq, H, dev) > 4LL * dev.sm_count;
}

// With many rows the select kernel scores the tail column itself (one launch
// fewer; the same pinned fp32 order, so the same bits).
qsa_status run_separate(const uint16_t* q, const uint16_t* kb, int32_t nq, int32_t H, int32_t D,
                        const Geometry& g, int32_t k, float* scores, int32_t* ids,
                        const DeviceInfo& dev, cudaStream_t stream) {
  const int32_t nb = static_cast<int32_t>(g.nb);
  const bool tail_in_select = g.has_tail && qsa::select_scores_tail(nq, nb, k);
  qsa_status st = run_scores(q, kb, nq, H, D, g, scores, dev, stream, tail_in_select);
  if (st != QSA_OK) return st;
  if (!tail_in_select) return from_cuda(qsa::launch_select(scores, nq, nb, k, ids, dev, stream));
  const qsa::TailInfo t{q, kb + (g.nb - 1) * D, H, D};
  return from_cuda(qsa::launch_select(scores, nq, nb, k, ids, dev, stream, &t));
}

// Batches with their own kb: past a few waves of the fused kernel the chain
// (persistent scores over every batch's tiles, then one select over every
// batch's rows, the tail block scored there) does the same work with less
// per score, when the persistent kernel and the row select can take it.
bool batched_chain_ok(int32_t n_batches, int32_t nq, int32_t H, int32_t D, const Geometry& g, int32_t k,
                      int64_t kb_batch_stride, const DeviceInfo& dev) {
  if (n_batches < 2 || g.nb == 0 || g.n_full == 0) return false;
  const int64_t rows = static_cast<int64_t>(n_batches) * nq;
  if (rows > 0x7FFFFFFFLL) return false;
  if (static_cast<int64_t>(n_batches) * qsa::fused_blocks(nq, H, dev) <= 4LL * dev.sm_count) return false;
  qsa::ScoreProblem sp{nullptr, nullptr, nullptr, nq, H, D, g.nb, g.n_full, g.has_tail, g.has_tail};
  sp.n_batches = n_batches;
  sp.kb_batch_stride = kb_batch_stride;
  if (!qsa::scores_persistent(sp, dev)) return false;
  return !g.has_tail || qsa::select_scores_tail(static_cast<int32_t>(rows), static_cast<int32_t>(g.nb), k);
}

qsa_status run_batched_chain(const uint16_t* q, const uint16_t* kb, int64_t kb_batch_stride,
                             int32_t n_batches, int32_t nq, int32_t H, int32_t D, const Geometry& g,
                             int32_t k, float* scores, int32_t* ids, const DeviceInfo& dev,
                             cudaStream_t stream) {
  qsa::ScoreProblem sp{q, kb, scores, nq, H, D, g.nb, g.n_full, g.has_tail, g.has_tail};
  sp.n_batches = n_batches;
  sp.kb_batch_stride = kb_batch_stride;
  qsa_status st = from_cuda(qsa::launch_scores(sp, dev, stream));
  if (st != QSA_OK) return st;
  const int32_t rows = n_batches * nq, nb = static_cast<int32_t>(g.nb);
  if (!g.has_tail) return from_cuda(qsa::launch_select(scores, rows, nb, k, ids, dev, stream));
  qsa::TailInfo t{q, kb + (g.nb - 1) * D, H, D};
  t.kb_batch_stride = kb_batch_stride;
  t.nq_per_batch = nq;
  return from_cuda(qsa::launch_select(scores, rows, nb, k, ids, dev, stream, &t));
}

}  // namespace

namespace qsa {
void plan_begin() {
  t_plan_n = 0;
  t_plan_any = true;
}
void plan_add(const char* kernel) {
  if (t_plan_n < kPlanMax) t_plan[t_plan_n++] = kernel;
}
}  // namespace qsa

extern "C" {

int qsa_abi_version(void) { return QSA_ABI_VERSION; }

const char* qsa_last_cuda_error(void) { return t_last_cuda_error; }

const char* qsa_status_str(qsa_status s) {
  switch (s) {
    case QSA_OK: return "QSA_OK";
    case QSA_ERR_INVALID_ARG: return "QSA_ERR_INVALID_ARG";
    case QSA_ERR_UNSUPPORTED_GEOMETRY: return "QSA_ERR_UNSUPPORTED_GEOMETRY";
    case QSA_ERR_UNSUPPORTED_ARCH: return "QSA_ERR_UNSUPPORTED_ARCH";
    case QSA_ERR_MISALIGNED: return "QSA_ERR_MISALIGNED";
    case QSA_ERR_CUDA: return "QSA_ERR_CUDA";
    case QSA_ERR_TIMEOUT: return "QSA_ERR_TIMEOUT";
  }
  return "QSA_ERR_UNKNOWN";
}

const char* qsa_arm(void) {
  thread_local char buf[1024];
  int n = snprintf(buf, sizeof buf,
                   "sm_103a: TMA + tcgen05.mma kind::f16 (M128, fp32 in TMEM) scorer with fused "
                   "ReLU/head-sum epilogue; fp32 pinned-order tail (+1e9); exact top-k select "
                   "(one warp for rows of <= 64 blocks, threshold + rank for k <= 128, radix "
                   "select otherwise; "
                   "block-index tie-break); cvt.rn fp32->fp16 stage | last call on this thread: ");
  if (!t_plan_any) {
    snprintf(buf + n, sizeof buf - n, "none");
  } else if (t_plan_n == 0) {
    snprintf(buf + n, sizeof buf - n, "no launch");
  } else {
    n += snprintf(buf + n, sizeof buf - n, "%d launch%s: ", t_plan_n, t_plan_n == 1 ? "" : "es");
    for (int i = 0; i < t_plan_n && n < static_cast<int>(sizeof buf); ++i)
      n += snprintf(buf + n, sizeof buf - n, "%s%s", i ? " -> " : "", t_plan[i]);
  }
  return buf;
}

int64_t qsa_num_blocks(int64_t n_kv, int32_t block) {
  if (n_kv < 0 || block < 1) return -1;
  return n_kv / block + (n_kv % block != 0 ? 1 : 0);
}

qsa_status qsa_f32_to_f16(const float* src, uint16_t* dst, int64_t n, qsa_stream_t stream) {
  if (n < 0) return QSA_ERR_INVALID_ARG;
  if (n == 0) return QSA_OK;
  if (!src || !dst) return QSA_ERR_INVALID_ARG;
  if (!aligned(src, 4) || !aligned(dst, 2)) return QSA_ERR_MISALIGNED;
  const DeviceInfo* dev = nullptr;
  qsa_status st = device_or_error(&dev);
  if (st != QSA_OK) return st;
  return from_cuda(qsa::launch_convert(src, dst, n, *dev, as_cuda(stream)));
}

qsa_status qsa_block_scores(const uint16_t* q, const uint16_t* kb, int32_t nq, int32_t H,
                            int32_t D, int64_t n_kv, int32_t block, float* scores,
                            qsa_stream_t stream) {
  Geometry g;
  qsa_status st = check_scores(q, kb, nq, H, D, n_kv, block, scores, &g);
  if (st != QSA_OK || nq == 0 || g.nb == 0) return st;
  const DeviceInfo* dev = nullptr;
  if ((st = device_or_error(&dev)) != QSA_OK) return st;
  return run_scores(q, kb, nq, H, D, g, scores, *dev, as_cuda(stream));
}

qsa_status qsa_select(const float* scores, int32_t nq, int32_t nb, int32_t k, int32_t* ids,
                      qsa_stream_t stream) {
  qsa_status st = check_select(scores, nq, nb, k, ids);
  if (st != QSA_OK || nq == 0) return st;
  const DeviceInfo* dev = nullptr;
  if ((st = device_or_error(&dev)) != QSA_OK) return st;
  return from_cuda(qsa::launch_select(scores, nq, nb, k, ids, *dev, as_cuda(stream)));
}

qsa_status qsa_score_select(const uint16_t* q, const uint16_t* kb, int32_t nq, int32_t H,
                            int32_t D, int64_t n_kv, int32_t block, int32_t k, float* scores,
                            int32_t* ids, qsa_stream_t stream) {
  Geometry g;
  qsa_status st = check_scores(q, kb, nq, H, D, n_kv, block, scores, &g);
  if (st != QSA_OK) return st;
  if ((st = check_select(scores, nq, g.nb, k, ids)) != QSA_OK) return st;
  if (nq == 0) return QSA_OK;
  if (g.nb > 0 && (!q || !kb)) return QSA_ERR_INVALID_ARG;
  const DeviceInfo* dev = nullptr;
  if ((st = device_or_error(&dev)) != QSA_OK) return st;
  if (g.nb > 0 && use_separate(nq, H, *dev))
    return run_separate(q, kb, nq, H, D, g, k, scores, ids, *dev, as_cuda(stream));
  qsa::FusedProblem p{nullptr, q,       nullptr,  kb, scores, ids, nq, H, D, g.nb, g.n_full,
                      g.has_tail, k, 1, 0};
  return from_cuda(qsa::launch_fused(p, *dev, as_cuda(stream)));
}

qsa_status qsa_select_step(const float* q32, uint16_t* q16, const uint16_t* kb, int32_t nq,
                           int32_t H, int32_t D, int64_t n_kv, int32_t block, int32_t k,
                           float* scores, int32_t* ids, qsa_stream_t stream) {
  Geometry g;
  // q16 is optional here; the scoring checks see the (aligned) q32 in its place.
  qsa_status st = check_scores(reinterpret_cast<const uint16_t*>(q32), kb, nq, H, D, n_kv, block,
                               scores, &g);
  if (st != QSA_OK) return st;
  if ((st = check_select(scores, nq, g.nb, k, ids)) != QSA_OK) return st;
  if (nq == 0) return QSA_OK;
  if (!q32) return QSA_ERR_INVALID_ARG;
  if (!aligned(q32, 16) || !aligned(q16, 16)) return QSA_ERR_MISALIGNED;
  const DeviceInfo* dev = nullptr;
  if ((st = device_or_error(&dev)) != QSA_OK) return st;
  if (q16 && g.nb > 0 && use_separate(nq, H, *dev)) {
    cudaStream_t s = as_cuda(stream);
    const int64_t n = static_cast<int64_t>(nq) * H * D;
    if ((st = from_cuda(qsa::launch_convert(q32, q16, n, *dev, s))) != QSA_OK) return st;
    return run_separate(q16, kb, nq, H, D, g, k, scores, ids, *dev, s);
  }
  qsa::FusedProblem p{q32, nullptr, q16, kb, scores, ids, nq, H, D, g.nb, g.n_full,
                      g.has_tail, k, 1, 0};
  return from_cuda(qsa::launch_fused(p, *dev, as_cuda(stream)));
}

int32_t qsa_select_step_launches(int32_t nq, int32_t H, int32_t D, int64_t n_kv, int32_t block,
                                 int32_t k, int32_t with_q16) {
  if (nq < 0 || n_kv < 0 || block < 1 || H < 1 || D < 1 || k < 1) return -1;
  if (!supported_heads(H) || D % 16 != 0 || D < 16 || D > 256 || k > qsa::kMaxSelectK) return -1;
  const int64_t nb = n_kv / block + (n_kv % block != 0 ? 1 : 0);
  if (nb > qsa::kMaxSelectNb || static_cast<int64_t>(nq) * H > 0x7FFFFFFFLL) return -1;
  if (nq == 0 || nb == 0) return 0;
  const DeviceInfo* dev = nullptr;
  if (device_or_error(&dev, false) != QSA_OK) return -1;
  if (!with_q16 || !use_separate(nq, H, *dev)) return 1;
  // convert (nq * H * D is a multiple of 8: one vector launch), the score
  // kernel when there are full blocks, the tail kernel when there is a tail
  // that the select does not score itself, and the select.
  const bool tail_kernel = n_kv % block != 0 && !qsa::select_scores_tail(nq, static_cast<int32_t>(nb), k);
  return 1 + (n_kv / block > 0 ? 1 : 0) + (tail_kernel ? 1 : 0) + 1;
}

// Shared by the two batched entry points: batch count and kb stride rules.
static qsa_status check_batches(int32_t n_batches, int64_t kb_batch_stride, int64_t nb, int32_t D) {
  if (n_batches < 0 || kb_batch_stride < 0) return QSA_ERR_INVALID_ARG;
  if (kb_batch_stride != 0 && kb_batch_stride < nb * D) return QSA_ERR_INVALID_ARG;
  if (kb_batch_stride % 8 != 0) return QSA_ERR_MISALIGNED;
  return QSA_OK;
}

qsa_status qsa_score_select_batched(const uint16_t* q, const uint16_t* kb, int64_t kb_batch_stride,
                                    int32_t n_batches, int32_t nq, int32_t H, int32_t D,
                                    int64_t n_kv, int32_t block, int32_t k, float* scores,
                                    int32_t* ids, qsa_stream_t stream) {
  Geometry g;
  qsa_status st = check_scores(q, kb, nq, H, D, n_kv, block, scores, &g);
  if (st != QSA_OK) return st;
  if ((st = check_select(scores, nq, g.nb, k, ids)) != QSA_OK) return st;
  if ((st = check_batches(n_batches, kb_batch_stride, g.nb, D)) != QSA_OK) return st;
  if (nq == 0 || n_batches == 0) return QSA_OK;
  if (static_cast<int64_t>(n_batches) * nq * H > 0x7FFFFFFFLL) return QSA_ERR_UNSUPPORTED_GEOMETRY;
  if (g.nb > 0 && (!q || !kb)) return QSA_ERR_INVALID_ARG;
  // Batches sharing one kb: one step over n_batches * nq queries.
  if (kb_batch_stride == 0)
    return qsa_score_select(q, kb, n_batches * nq, H, D, n_kv, block, k, scores, ids, stream);
  const DeviceInfo* dev = nullptr;
  if ((st = device_or_error(&dev)) != QSA_OK) return st;
  if (batched_chain_ok(n_batches, nq, H, D, g, k, kb_batch_stride, *dev))
    return run_batched_chain(q, kb, kb_batch_stride, n_batches, nq, H, D, g, k, scores, ids, *dev,
                             as_cuda(stream));
  qsa::FusedProblem p{nullptr, q,       nullptr,  kb, scores, ids, nq, H, D, g.nb, g.n_full,
                      g.has_tail, k, n_batches, kb_batch_stride};
  return from_cuda(qsa::launch_fused(p, *dev, as_cuda(stream)));
}

qsa_status qsa_select_step_batched(const float* q32, uint16_t* q16, const uint16_t* kb,
                                   int64_t kb_batch_stride, int32_t n_batches, int32_t nq,
                                   int32_t H, int32_t D, int64_t n_kv, int32_t block, int32_t k,
                                   float* scores, int32_t* ids, qsa_stream_t stream) {
  Geometry g;
  qsa_status st = check_scores(reinterpret_cast<const uint16_t*>(q32), kb, nq, H, D, n_kv, block,
                               scores, &g);
  if (st != QSA_OK) return st;
  if ((st = check_select(scores, nq, g.nb, k, ids)) != QSA_OK) return st;
  if ((st = check_batches(n_batches, kb_batch_stride, g.nb, D)) != QSA_OK) return st;
  if (nq == 0 || n_batches == 0) return QSA_OK;
  if (static_cast<int64_t>(n_batches) * nq * H > 0x7FFFFFFFLL) return QSA_ERR_UNSUPPORTED_GEOMETRY;
  if (!q32) return QSA_ERR_INVALID_ARG;
  if (!aligned(q32, 16) || !aligned(q16, 16)) return QSA_ERR_MISALIGNED;
  // Batches sharing one kb are one step over n_batches * nq queries (the
  // buffers are laid out as such): it takes the single-step plan, the chain
  // of separate kernels when it is large and q16 is given.
  if (kb_batch_stride == 0)
    return qsa_select_step(q32, q16, kb, n_batches * nq, H, D, n_kv, block, k, scores, ids, stream);
  const DeviceInfo* dev = nullptr;
  if ((st = device_or_error(&dev)) != QSA_OK) return st;
  if (q16 && batched_chain_ok(n_batches, nq, H, D, g, k, kb_batch_stride, *dev)) {
    cudaStream_t s = as_cuda(stream);
    const int64_t n = static_cast<int64_t>(n_batches) * nq * H * D;
    if ((st = from_cuda(qsa::launch_convert(q32, q16, n, *dev, s))) != QSA_OK) return st;
    return run_batched_chain(q16, kb, kb_batch_stride, n_batches, nq, H, D, g, k, scores, ids, *dev, s);
  }
  qsa::FusedProblem p{q32, nullptr, q16, kb, scores, ids, nq, H, D, g.nb, g.n_full,
                      g.has_tail, k, n_batches, kb_batch_stride};
  return from_cuda(qsa::launch_fused(p, *dev, as_cuda(stream)));
}

qsa_status qsa_select_step_host(const float* q32_host, const uint16_t* kb_host, int32_t nq,
                                int32_t H, int32_t D, int64_t n_kv, int32_t block, int32_t k,
                                float* scores_host, int32_t* ids_host, float* q32_dev,
                                uint16_t* q16_dev, uint16_t* kb_dev, float* scores_dev,
                                int32_t* ids_dev, qsa_stream_t stream) {
  Geometry g;
  qsa_status st = check_scores(reinterpret_cast<const uint16_t*>(q32_dev), kb_dev, nq, H, D, n_kv,
                               block, scores_dev, &g);
  if (st != QSA_OK) return st;
  if ((st = check_select(scores_dev, nq, g.nb, k, ids_dev)) != QSA_OK) return st;
  if (nq == 0) return QSA_OK;
  if (!q32_host || !ids_host || !q32_dev || !ids_dev) return QSA_ERR_INVALID_ARG;
  if (g.nb > 0 && !kb_host) return QSA_ERR_INVALID_ARG;
  const DeviceInfo* dev = nullptr;
  if ((st = device_or_error(&dev)) != QSA_OK) return st;
  cudaStream_t s = as_cuda(stream);
  const size_t q_bytes = static_cast<size_t>(nq) * H * D * sizeof(float);
  const size_t kb_bytes = static_cast<size_t>(g.nb) * D * sizeof(uint16_t);
  const size_t s_bytes = static_cast<size_t>(nq) * g.nb * sizeof(float);
  const size_t id_bytes = static_cast<size_t>(nq) * k * sizeof(int32_t);
  if (cudaMemcpyAsync(q32_dev, q32_host, q_bytes, cudaMemcpyHostToDevice, s) != cudaSuccess)
    return cuda_fail(cudaGetLastError());
  if (kb_bytes &&
      cudaMemcpyAsync(kb_dev, kb_host, kb_bytes, cudaMemcpyHostToDevice, s) != cudaSuccess)
    return cuda_fail(cudaGetLastError());
  st = qsa_select_step(q32_dev, q16_dev, kb_dev, nq, H, D, n_kv, block, k, scores_dev, ids_dev,
                       stream);
  if (st != QSA_OK) return st;
  if (s_bytes && scores_host &&
      cudaMemcpyAsync(scores_host, scores_dev, s_bytes, cudaMemcpyDeviceToHost, s) != cudaSuccess)
    return cuda_fail(cudaGetLastError());
  if (cudaMemcpyAsync(ids_host, ids_dev, id_bytes, cudaMemcpyDeviceToHost, s) != cudaSuccess)
    return cuda_fail(cudaGetLastError());
  return QSA_OK;
}

qsa_status qsa_select_step_host_packed(const void* in_host, int32_t nq, int32_t H, int32_t D,
                                       int64_t n_kv, int32_t block, int32_t k, void* out_host,
                                       int32_t with_scores, void* in_dev, uint16_t* q16_dev,
                                       void* out_dev, qsa_stream_t stream) {
  if (nq < 0 || H < 1 || D < 1) return QSA_ERR_INVALID_ARG;
  const int64_t nb = qsa_num_blocks(n_kv, block);
  if (nb < 0) return QSA_ERR_INVALID_ARG;
  const size_t q_bytes = static_cast<size_t>(nq) * H * D * sizeof(float);
  const size_t kb_bytes = static_cast<size_t>(nb) * D * sizeof(uint16_t);
  const size_t s_bytes = static_cast<size_t>(nq) * nb * sizeof(float);
  const size_t id_bytes = static_cast<size_t>(nq) * (k > 0 ? k : 0) * sizeof(int32_t);
  char* in_d = static_cast<char*>(in_dev);
  char* out_d = static_cast<char*>(out_dev);
  float* q32_dev = reinterpret_cast<float*>(in_d);
  uint16_t* kb_dev = in_d ? reinterpret_cast<uint16_t*>(in_d + q_bytes) : nullptr;
  float* scores_dev = reinterpret_cast<float*>(out_d);
  int32_t* ids_dev = out_d ? reinterpret_cast<int32_t*>(out_d + s_bytes) : nullptr;
  Geometry g;
  qsa_status st = check_scores(reinterpret_cast<const uint16_t*>(q32_dev), kb_dev, nq, H, D, n_kv,
                               block, scores_dev, &g);
  if (st != QSA_OK) return st;
  if ((st = check_select(scores_dev, nq, g.nb, k, ids_dev)) != QSA_OK) return st;
  if (nq == 0) return QSA_OK;
  if (!in_host || !out_host || !in_dev || !out_dev) return QSA_ERR_INVALID_ARG;
  const DeviceInfo* dev = nullptr;
  if ((st = device_or_error(&dev)) != QSA_OK) return st;
  cudaStream_t s = as_cuda(stream);
  // One copy in (queries then keys), one copy out (scores then ids, or ids).
  if (cudaMemcpyAsync(in_dev, in_host, q_bytes + kb_bytes, cudaMemcpyHostToDevice, s) != cudaSuccess)
    return cuda_fail(cudaGetLastError());
  st = qsa_select_step(q32_dev, q16_dev, kb_dev, nq, H, D, n_kv, block, k, scores_dev, ids_dev,
                       stream);
  if (st != QSA_OK) return st;
  const void* src = with_scores ? static_cast<const void*>(scores_dev) : static_cast<const void*>(ids_dev);
  const size_t out_bytes = with_scores ? s_bytes + id_bytes : id_bytes;
  if (cudaMemcpyAsync(out_host, src, out_bytes, cudaMemcpyDeviceToHost, s) != cudaSuccess)
    return cuda_fail(cudaGetLastError());
  return QSA_OK;
}

// Shape rules of the split reduce; fills *ws with the workspace it needs.
static qsa_status check_split(int32_t G, int32_t R, int32_t B, int32_t C, size_t* ws) {
  if (G < 0 || R < 1 || B < 1 || C < 1) return QSA_ERR_INVALID_ARG;
  if (R > qsa::kSrMaxRows || C % 4 != 0 || C < 4 || G > 65535 ||
      static_cast<int64_t>(R) * C > 4LL * qsa::kSrMaxQuadsPerThread * 256)
    return QSA_ERR_UNSUPPORTED_GEOMETRY;
  *ws = qsa::split_reduce_workspace_bytes(G, R, B, C);
  return QSA_OK;
}

size_t qsa_split_reduce_workspace_bytes(int32_t G, int32_t R, int32_t B, int32_t C) {
  size_t ws = 0;
  return check_split(G, R, B, C, &ws) == QSA_OK ? ws : 0;
}

qsa_status qsa_split_reduce(const float* partial_max, const float* partial_sum,
                            const uint16_t* partial_out, int32_t G, int32_t R, int32_t B,
                            int32_t C, float* out, void* workspace, size_t workspace_bytes,
                            qsa_stream_t stream) {
  size_t need = 0;
  qsa_status st = check_split(G, R, B, C, &need);
  if (st != QSA_OK) return st;
  if (G == 0) return QSA_OK;
  if (!partial_max || !partial_sum || !partial_out || !out) return QSA_ERR_INVALID_ARG;
  if (need > 0 && (!workspace || workspace_bytes < need)) return QSA_ERR_INVALID_ARG;
  if (!aligned(partial_max, 4) || !aligned(partial_sum, 4) || !aligned(partial_out, 8) ||
      !aligned(out, 16) || (need > 0 && !aligned(workspace, 16)))
    return QSA_ERR_MISALIGNED;
  const DeviceInfo* dev = nullptr;
  if ((st = device_or_error(&dev)) != QSA_OK) return st;
  qsa::SplitReduceProblem p{partial_max, partial_sum, partial_out, out, workspace, G, R, B, C};
  return from_cuda(qsa::launch_split_reduce(p, *dev, as_cuda(stream)));
}

qsa_status qsa_split_reduce_static(const float* partial_max, const float* partial_sum,
                                   const uint16_t* partial_out, int32_t G, int32_t R, int32_t B,
                                   int32_t C, float* out, qsa_stream_t stream) {
  size_t need = 0;
  qsa_status st = check_split(G, R, B, C, &need);
  if (st != QSA_OK) return st;
  if (need > QSA_SPLIT_STATIC_SCRATCH_BYTES) return QSA_ERR_UNSUPPORTED_GEOMETRY;
  if (G == 0) return QSA_OK;
  if (!partial_max || !partial_sum || !partial_out || !out) return QSA_ERR_INVALID_ARG;
  if (!aligned(partial_max, 4) || !aligned(partial_sum, 4) || !aligned(partial_out, 8) ||
      !aligned(out, 16))
    return QSA_ERR_MISALIGNED;
  const DeviceInfo* dev = nullptr;
  if ((st = device_or_error(&dev)) != QSA_OK) return st;
  cudaError_t e = cudaSuccess;
  void* scratch = qsa::split_static_scratch(&e);
  if (!scratch) return cuda_fail(e);
  cudaStream_t s = as_cuda(stream);
  if (need > 0) {
    // The counters lead the workspace layout and must be zero; an earlier
    // call of another shape may have left partials where they now sit.
    const size_t counters = (static_cast<size_t>(G) * R * sizeof(uint32_t) + 15) & ~static_cast<size_t>(15);
    if ((e = cudaMemsetAsync(scratch, 0, counters, s)) != cudaSuccess) return cuda_fail(e);
  }
  qsa::SplitReduceProblem p{partial_max, partial_sum, partial_out, out, scratch, G, R, B, C};
  return from_cuda(qsa::launch_split_reduce(p, *dev, s));
}

qsa_status qsa_selftest_bounded_wait(uint64_t timeout_ns, qsa_stream_t stream) {
  if (timeout_ns == 0 || timeout_ns > 1000000000ull) return QSA_ERR_INVALID_ARG;
  const DeviceInfo* dev = nullptr;
  qsa_status st = device_or_error(&dev);
  if (st != QSA_OK) return st;
  return from_cuda(qsa::launch_selftest_wait(*dev, timeout_ns, as_cuda(stream)));
}

qsa_status qsa_device_status(int clear, uint32_t* bits, qsa_stream_t stream) {
  const DeviceInfo* dev = nullptr;
  qsa_status st = device_or_error(&dev, false);
  if (st != QSA_OK) return st;
  cudaError_t e = cudaStreamSynchronize(as_cuda(stream));
  if (e != cudaSuccess) return cuda_fail(e);
  uint32_t v = 0;
  if ((e = cudaMemcpy(&v, dev->status_word, sizeof(v), cudaMemcpyDeviceToHost)) != cudaSuccess)
    return cuda_fail(e);
  if (bits) *bits = v;
  if (v != 0 && clear) {
    if ((e = cudaMemset(dev->status_word, 0, sizeof(uint32_t))) != cudaSuccess ||
        (e = cudaDeviceSynchronize()) != cudaSuccess)
      return cuda_fail(e);
  }
  return v == 0 ? QSA_OK : QSA_ERR_TIMEOUT;
}

}  // extern "C"
