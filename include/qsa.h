/*
 * qsa.h - C ABI of libqsa, a GB300 (sm_103a) library for QSA block scoring and
 * top-k block selection.
 *
 * The operation (Strata pull request 228, part 1, "qsa_block_scores_wmma: the
 * prompt scorer arm on tensor cores"): for every query qi and KV block b,
 *
 *     score(qi, b) = sum_{h < H} relu( sum_{i < D} kb[b, i] * q[qi, h, i] )
 *
 * with fp16 operands and fp32 accumulation, followed by the selection of the k
 * highest-scoring blocks per query. A context of n_kv tokens is cut into
 * nb = ceil(n_kv / block) blocks; when n_kv % block != 0 the last block is a
 * partial "tail" that a separate kernel scores in one fixed fp32 order and
 * forces into the selection by adding 1e9 to its score (Strata pull request
 * 856, section "What": the shared tail-block kernel and the +1e9 dead-tail
 * rule).
 *
 * Conventions for every entry point:
 *   - Buffers are device pointers owned by the caller unless stated otherwise.
 *     The library allocates no device memory and keeps no pointer after a
 *     call returns.
 *   - Work is enqueued on `stream` (a cudaStream_t; NULL is the legacy default
 *     stream) and runs asynchronously; no entry point synchronizes except
 *     qsa_device_status().
 *   - Arguments are validated on the host before anything is launched. A
 *     failed check returns an error status and launches nothing. There is no
 *     CPU fallback: every result is computed by the library's CUDA kernels.
 *   - Empty work (nq == 0, nb == 0, n == 0) returns QSA_OK without a launch.
 *   - The device must be compute capability 10.3 (sm_103a); other devices get
 *     QSA_ERR_UNSUPPORTED_ARCH.
 *   - Kernels bound every wait; a wait that runs out records a timeout in a
 *     device status word that qsa_device_status() reports.
 *   - Not thread-safe per stream in the sense of CUDA streams only: calls from
 *     several host threads are safe; work on one stream runs in order.
 */
#ifndef QSA_H_
#define QSA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* A cudaStream_t, declared without CUDA headers. */
typedef struct CUstream_st* qsa_stream_t;

typedef enum {
  QSA_OK = 0,
  QSA_ERR_INVALID_ARG = 1,          /* null pointer, negative size, k < 1, block < 1 ... */
  QSA_ERR_UNSUPPORTED_GEOMETRY = 2, /* H, D, k or nb outside the supported ranges below */
  QSA_ERR_UNSUPPORTED_ARCH = 3,     /* current device is not sm_103 */
  QSA_ERR_MISALIGNED = 4,           /* a pointer breaks the alignment rule stated below */
  QSA_ERR_CUDA = 5,                 /* a CUDA runtime/driver call or launch failed */
  QSA_ERR_TIMEOUT = 6               /* a kernel gave up a bounded wait (qsa_device_status) */
} qsa_status;

/* ABI version of this header; bumps when a signature changes. */
#define QSA_ABI_VERSION 1
int qsa_abi_version(void);

/* Static, NUL-terminated name of a status code. */
const char* qsa_status_str(qsa_status status);

/* NUL-terminated description of the arm (the kernels this library runs),
 * followed by the plan the last launching call on this thread ran: the
 * number of launches and each kernel by name, in order (for example one
 * fused_step_kernel launch, or a chain of convert, score and select
 * kernels), or "none" before any such call. So a fallback cannot pass for
 * the fast path (after Strata pull request 228, part 1, which prints the arm
 * that ran). The text lives in thread-local storage: valid until the next
 * qsa_arm() call on the same thread. */
const char* qsa_arm(void);

/* Static text of the last CUDA error that made a call of this thread return
 * QSA_ERR_CUDA ("no error" if none has). */
const char* qsa_last_cuda_error(void);

/* nb = ceil(n_kv / block): the number of KV blocks, the tail included.
 * Returns -1 if n_kv < 0 or block < 1. */
int64_t qsa_num_blocks(int64_t n_kv, int32_t block);

/*
 * qsa_f32_to_f16 - the FP32 -> FP16 operand conversion stage (Strata pull
 * request 228, part 1: f32_to_f16_poison_kernel runs beside the scorer; the
 * "fp16 conversion" is part of the qsa select phase).
 *
 *   src  f32[n], dst f16[n] (raw binary16 bits, uint16_t), device memory.
 *   dst[i] = binary16 round-to-nearest-even of src[i]; overflow gives +-inf;
 *   NaN gives a NaN (its payload is not kept).
 *   src and dst must not overlap. Any alignment of 4 (src) / 2 (dst) bytes
 *   works; 16-byte aligned buffers take the vectorised path.
 *   Errors: QSA_ERR_INVALID_ARG for n < 0 or a null pointer with n > 0;
 *   QSA_ERR_MISALIGNED for a src not 4-byte or dst not 2-byte aligned.
 */
qsa_status qsa_f32_to_f16(const float* src, uint16_t* dst, int64_t n, qsa_stream_t stream);

/*
 * qsa_block_scores - every block score, tail included (Strata pull request
 * 228, part 1, the score definition; pull request 856, "What", the tail).
 *
 *   q       f16 [nq, H, D] row-major (D contiguous), device, 16-byte aligned.
 *   kb      f16 [nb, D] row-major, one key vector per block, device, 16-byte
 *           aligned; must hold nb = ceil(n_kv / block) rows (the C ABI cannot
 *           check this, the Python binding does).
 *   scores  f32 [nq, nb] row-major, device, 16-byte aligned; written exactly
 *           once per entry and nowhere else.
 *   Full blocks b < n_kv / block: fp16 x fp16 products accumulated in fp32 by
 *   the tensor cores (tcgen05), then per-head ReLU and the head sum in fp32.
 *   Each such score lies within B = 2^-9.5 * S + 8 * 2^-24 * |score| of the
 *   exact score, S = sum over h and i of |q * kb|.
 *   Tail block (n_kv % block != 0, column nb-1): acc_h = sequential fp32 sum
 *   over i of q[qi,h,i]*kb[nb-1,i]; t = sequential fp32 sum over h of
 *   max(acc_h, 0); score = t + 1e9f, each step rounded to nearest even.
 *   Supported: nq >= 0; H in {1, 2, 4, 8, 16, 32}; D a multiple of 16 with
 *   16 <= D <= 256; block >= 1; n_kv >= 0; nq * H < 2^31; nb < 2^31.
 *   Inputs must be finite.
 */
qsa_status qsa_block_scores(const uint16_t* q, const uint16_t* kb, int32_t nq, int32_t H,
                            int32_t D, int64_t n_kv, int32_t block, float* scores,
                            qsa_stream_t stream);

/*
 * qsa_select - top-k block selection per query (Strata pull request 228,
 * part 1; pull request 856, "Arithmetic contract and parity": top-k over the
 * block scores).
 *
 *   scores  f32 [nq, nb] row-major, device, 4-byte aligned, finite (NaN is
 *           not supported).
 *   ids     int32 [nq, k] row-major, device, 4-byte aligned.
 *   ids[qi, :] lists the min(k, nb) blocks with the largest scores, in
 *   descending score order; equal scores are ordered by ascending block index
 *   (the smaller index wins a tie at the k-th place); -0.0 and +0.0 are
 *   equal; entries past nb (when nb < k) are -1. Exact: no tolerance.
 *   Supported: 1 <= k <= 1024; 0 <= nb <= 32768.
 */
qsa_status qsa_select(const float* scores, int32_t nq, int32_t nb, int32_t k, int32_t* ids,
                      qsa_stream_t stream);

/*
 * qsa_score_select - the metric path: the results of qsa_block_scores and
 * then qsa_select, with the same arguments and rules as those two (and
 * bit-identical results). Both outputs are written: scores [nq, nb] and ids
 * [nq, k]. Up to a few waves of work this is one fused launch; a larger
 * problem (more than four fused CTAs per SM, e.g. 2048 queries of 8 heads)
 * runs the score and select kernels in turn instead, chained by
 * programmatic dependent launch; the tail block is scored by the select
 * kernel when it selects one row per warp (at least 1024 rows, k <= 128,
 * nb <= 4096), else by a tail kernel between the two. The results are the
 * same bits either way.
 */
qsa_status qsa_score_select(const uint16_t* q, const uint16_t* kb, int32_t nq, int32_t H,
                            int32_t D, int64_t n_kv, int32_t block, int32_t k, float* scores,
                            int32_t* ids, qsa_stream_t stream);

/*
 * qsa_select_step - one whole pass of the selection phase for one query
 * batch, in one launch: q arrives as f32 and is rounded to fp16 (as by
 * qsa_f32_to_f16) on its way into the tensor cores, then every block is
 * scored and the top-k selected (as by qsa_score_select).
 *
 *   q32  f32 [nq, H, D] device, 16-byte aligned.
 *   q16  optional: NULL, or f16 [nq, H, D] device, 16-byte aligned, which
 *        then receives the converted queries.
 *   The other arguments as for qsa_score_select.
 * A problem too large for the fused launch (as for qsa_score_select) runs
 * the conversion into q16 and then the separate kernels when q16 is given,
 * and the fused launch when it is NULL (no buffer for the fp16 operand).
 */
qsa_status qsa_select_step(const float* q32, uint16_t* q16, const uint16_t* kb, int32_t nq,
                           int32_t H, int32_t D, int64_t n_kv, int32_t block, int32_t k,
                           float* scores, int32_t* ids, qsa_stream_t stream);

/*
 * qsa_select_step_launches - the number of kernel launches one call of
 * qsa_select_step with these sizes makes on the current device: 1 for the
 * fused launch, more for the separate kernels, 0 when there is nothing to
 * compute (nq == 0 or nb == 0). with_q16 says whether the call passes a q16
 * buffer. Returns -1 for sizes qsa_select_step would reject or when the
 * current device cannot run the library. Launches nothing.
 */
int32_t qsa_select_step_launches(int32_t nq, int32_t H, int32_t D, int64_t n_kv, int32_t block,
                                 int32_t k, int32_t with_q16);

/*
 * qsa_select_step_batched / qsa_score_select_batched - n_batches independent
 * query batches in one launch (the selection phase's batch loop over query
 * batches, made one launch). Batch b is exactly qsa_select_step /
 * qsa_score_select on batch b's slices (bit-identical results). With
 * per-batch keys (kb_batch_stride != 0) the call is one fused launch while
 * that is at most about four CTAs per SM; past that (and, for
 * qsa_select_step_batched, given a q16 buffer) it runs the chain: one
 * conversion of every batch's queries, one persistent score launch over
 * every batch's tiles and one select launch over every batch's rows (which
 * scores each batch's tail block), when those kernels can take the sizes
 * (at least four 128 x 256 tiles per SM; with a tail, at least 1024 rows in
 * all, k <= 128, nb <= 4096), else the fused launch. Batches that share one
 * kb (kb_batch_stride == 0) are one step over n_batches * nq queries and
 * take the single-step plan (one fused launch, or for a large step given a
 * q16 buffer the chain of separate kernels, as qsa_select_step /
 * qsa_score_select):
 *   q32 / q     f32 / f16 [n_batches, nq, H, D]; q16 (optional) likewise.
 *   kb          f16: one [nb, D] shared by every batch when kb_batch_stride
 *               is 0 (the block keys of one context, shared by its query
 *               batches); otherwise batch b's [nb, D] keys start at
 *               kb + b * kb_batch_stride (elements; a multiple of 8 and at
 *               least nb * D).
 *   scores      f32 [n_batches, nq, nb]; ids int32 [n_batches, nq, k].
 * n_batches == 0 returns QSA_OK without a launch; n_batches * nq * H < 2^31.
 * Errors as for the single-batch calls; QSA_ERR_INVALID_ARG for a negative
 * count or stride or a stride below nb * D; QSA_ERR_MISALIGNED for a stride
 * that is not a multiple of 8.
 */
qsa_status qsa_select_step_batched(const float* q32, uint16_t* q16, const uint16_t* kb,
                                   int64_t kb_batch_stride, int32_t n_batches, int32_t nq,
                                   int32_t H, int32_t D, int64_t n_kv, int32_t block, int32_t k,
                                   float* scores, int32_t* ids, qsa_stream_t stream);
qsa_status qsa_score_select_batched(const uint16_t* q, const uint16_t* kb, int64_t kb_batch_stride,
                                    int32_t n_batches, int32_t nq, int32_t H, int32_t D,
                                    int64_t n_kv, int32_t block, int32_t k, float* scores,
                                    int32_t* ids, qsa_stream_t stream);

/*
 * qsa_select_step_host - qsa_select_step from HOST buffers: enqueues on
 * `stream` the copies q32_host -> q32_dev and kb_host -> kb_dev, the step,
 * and the copies scores_dev -> scores_host (unless scores_host is NULL: the
 * scores then stay in scores_dev) and ids_dev -> ids_host. Host buffers
 * should be page-locked for the copies to be asynchronous; they must stay
 * valid until the stream has finished the call's work (synchronize the
 * stream before reading scores_host / ids_host). Device buffers are the
 * caller's, sized as for qsa_select_step (kb_dev: nb rows).
 * Each host <-> device copy has a fixed cost of about 2 us on top of its
 * bytes, and copies in one direction do not overlap one another:
 * qsa_select_step_host_packed below makes one copy each way.
 */
qsa_status qsa_select_step_host(const float* q32_host, const uint16_t* kb_host, int32_t nq,
                                int32_t H, int32_t D, int64_t n_kv, int32_t block, int32_t k,
                                float* scores_host, int32_t* ids_host, float* q32_dev,
                                uint16_t* q16_dev, uint16_t* kb_dev, float* scores_dev,
                                int32_t* ids_dev, qsa_stream_t stream);

/*
 * qsa_select_step_host_packed - qsa_select_step_host with each direction's
 * buffers packed into one allocation, so that each direction is one copy
 * (the pages' selection step fed from and read back to the host):
 *   in_host / in_dev   q32 [nq,H,D] f32 at byte 0, then kb [nb,D] f16 at byte
 *                      nq*H*D*4 (in_dev 16-byte aligned); in_host should be
 *                      page-locked; in_dev is overwritten by the copy.
 *   out_dev            scores [nq,nb] f32 at byte 0, then ids [nq,k] int32 at
 *                      byte nq*nb*4.
 *   out_host           with_scores != 0: scores then ids, as out_dev;
 *                      with_scores == 0: ids [nq,k] only (the scores stay in
 *                      out_dev).
 *   q16_dev            optional fp16 copy of the converted queries, as for
 *                      qsa_select_step.
 * Enqueued on `stream`; host buffers must stay valid until the stream has
 * finished the call's work. Errors as for qsa_select_step_host.
 */
qsa_status qsa_select_step_host_packed(const void* in_host, int32_t nq, int32_t H, int32_t D,
                                       int64_t n_kv, int32_t block, int32_t k, void* out_host,
                                       int32_t with_scores, void* in_dev, uint16_t* q16_dev,
                                       void* out_dev, qsa_stream_t stream);

/*
 * qsa_split_reduce - the flash-attention decode split reduce (a second
 * workload: 1bit-MONSTER llama.cpp pull request 30, "What" and "Changes",
 * the multipass reduce's output pass; its review's bounded scale stage).
 * For each of G groups (a sequence and KV head) and R rows (the query heads
 * sharing that KV head), B KV blocks have left partials; the call computes
 *
 *   maximum[r] = max_b partial_max[r,b]
 *   scale[r,b] = exp(partial_max[r,b] - maximum[r])      once per (row, block)
 *   sum[r]     = sum_b scale[r,b] * partial_sum[r,b]
 *   out[r,c]   = (sum_b scale[r,b] * partial_out[r,b,c]) / sum[r]
 *
 *   partial_max, partial_sum  f32 [G, R, B] device, 4-byte aligned, finite.
 *   partial_out               f16 [G, R, B, C] device, 8-byte aligned.
 *   out                       f32 [G, R, C] device, 16-byte aligned.
 *   workspace                 device, 16-byte aligned, at least
 *                             qsa_split_reduce_workspace_bytes(G, R, B, C)
 *                             bytes (0 when B <= 128: NULL allowed). Its first
 *                             bytes hold arrival counters that must be zero
 *                             before the first call (zero-fill it once); every
 *                             call that completes leaves them zero again. A
 *                             call whose staging wait ran out (bit 3 of the
 *                             status word, QSA_ERR_TIMEOUT from
 *                             qsa_device_status) returns early and may leave
 *                             them nonzero: zero-fill the workspace again
 *                             before its next use. Calls that may run at the
 *                             same time need separate workspaces. Shapes the
 *                             one-cluster-per-row form takes (C % 8 == 0,
 *                             partial_out 16-byte aligned, B <= 4096, a CTA's
 *                             chunks fitting in its shared memory) leave the
 *                             workspace untouched.
 * Arithmetic (fixed, so results are reproducible bit for bit on any GB300):
 * the blocks are reduced in chunks of 128 (the scales of a chunk staged on
 * chip), each chunk in runs of 32 blocks; in a run, sum and out accumulate
 * block by block from 0 in fp32, each term fl(scale * x) then one rounded
 * add (no fused multiply-add); a chunk's runs are added in order, then the
 * chunk partials in chunk order; out = fl(O / sum).
 * exp is a fixed fp32 routine (Cody-Waite reduction, degree-7 Taylor
 * polynomial; within 3 ulp of exp; arguments below -86 give 0).
 * Supported: G >= 0 (0: nothing to do), 1 <= R <= 32, B >= 1, 4 <= C,
 * C % 4 == 0, R * C <= 4096, G <= 65535.
 * Errors: QSA_ERR_INVALID_ARG (a NULL buffer, B < 1, R < 1, G < 0, a
 * workspace smaller than required), QSA_ERR_UNSUPPORTED_GEOMETRY, QSA_ERR_MISALIGNED.
 * Order of the checks: the sizes first (INVALID_ARG for negative or zero
 * sizes, then UNSUPPORTED_GEOMETRY), then G == 0 returns QSA_OK without
 * looking at any pointer, then the pointers (INVALID_ARG for a NULL buffer
 * or a short workspace), then their alignment (MISALIGNED).
 */
size_t qsa_split_reduce_workspace_bytes(int32_t G, int32_t R, int32_t B, int32_t C);
qsa_status qsa_split_reduce(const float* partial_max, const float* partial_sum,
                            const uint16_t* partial_out, int32_t G, int32_t R, int32_t B,
                            int32_t C, float* out, void* workspace, size_t workspace_bytes,
                            qsa_stream_t stream);

/*
 * qsa_split_reduce_static - qsa_split_reduce without a caller workspace, for
 * callers that cannot allocate device memory at call time (a serving loop
 * that must stay out of the allocator, whose cudaMalloc / cudaFree
 * synchronise the device; a plain C host without a caching allocator). The
 * pages have no counterpart of this entry point: it is library plumbing, not
 * part of the method.
 *
 * Same arguments (less the workspace) and bit-identical results. The chunk
 * partials and arrival counters live in one fixed array of
 * QSA_SPLIT_STATIC_SCRATCH_BYTES per device inside the library; nothing is
 * allocated. Shapes whose qsa_split_reduce_workspace_bytes exceeds it
 * return QSA_ERR_UNSUPPORTED_GEOMETRY without a launch.
 * Every call first clears the array's counter area on `stream` (an
 * asynchronous memset, no allocation), then launches the reduce.
 * Calls that may run at the same time on one device (other streams or other
 * host threads) share the array and race: serialise them.
 * The first call on each device looks up the array's address
 * (cudaGetSymbolAddress, with that device current) and keeps it for the
 * life of the process; make that first call before any stream capture on
 * the device. The kept address assumes that the device's primary context
 * lives as long as the process: after cudaDeviceReset (or a release and
 * re-creation of the primary context) the array may move, so do not call
 * this entry point on that device again in the same process.
 * Order of the checks: the sizes as for qsa_split_reduce, then a workspace
 * need above QSA_SPLIT_STATIC_SCRATCH_BYTES (UNSUPPORTED_GEOMETRY), then
 * G == 0 returns QSA_OK without looking at any pointer, then the pointers
 * (INVALID_ARG) and their alignment (MISALIGNED).
 */
#define QSA_SPLIT_STATIC_SCRATCH_BYTES (4u << 20)
qsa_status qsa_split_reduce_static(const float* partial_max, const float* partial_sum,
                                   const uint16_t* partial_out, int32_t G, int32_t R, int32_t B,
                                   int32_t C, float* out, qsa_stream_t stream);

/*
 * qsa_device_status - synchronizes `stream`, then reads the current device's
 * status word, where kernels record a bounded wait that ran out. Returns
 * QSA_OK if it is clear, QSA_ERR_TIMEOUT if not (and clears it when `clear`
 * is nonzero), or QSA_ERR_CUDA if the synchronization itself failed. The
 * word's raw bits are stored in *bits when bits is not NULL.
 */
qsa_status qsa_device_status(int clear, uint32_t* bits, qsa_stream_t stream);

/*
 * qsa_selftest_bounded_wait - failure-detection self-test. Launches one
 * kernel that waits on a barrier nothing completes, for at most timeout_ns
 * (1 ns .. 1 s), then gives up and sets bit 31 of the device status word,
 * exactly as a real kernel does when one of its bounded waits runs out. The
 * GPU context stays usable. A following qsa_device_status() returns
 * QSA_ERR_TIMEOUT with that bit set (and clears it when asked).
 * Errors: QSA_ERR_INVALID_ARG for a timeout outside the range.
 */
qsa_status qsa_selftest_bounded_wait(uint64_t timeout_ns, qsa_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* QSA_H_ */
