/*
 * qsa.h - C ABI of the GB300 (sm_103a) QSA-indexer library: paged MQA-logits
 * scoring and per-row top-k selection.
 *
 * The compute calls - scoring (qsa_paged_mqa_logits and its _ragged / _ex
 * forms), selection (qsa_select_topk, qsa_select_topk_bounded) and both in
 * one call (qsa_paged_mqa_topk, qsa_paged_mqa_topk_noalloc) - follow the
 * problem statement of the pages:
 *   - vLLM #62589 "Tile QSA indexer scoring and skip invisible columns",
 *     Dispatch and Details: qsa_mqa_paged(...) scores request-major query rows
 *     against a paged compressed-key cache; top_k_per_row_decode reads
 *     [0, visible_blocks[row]).
 *   - SGLang #48649 test body: torch_qsa_mqa_decode(q, compressed_cache,
 *     page_table, context_lens, max_model_len) then
 *     qsa_fast_topk(logits, row_starts, context_lens, topk).
 *   - aiter #4221, commit extending fp8_paged_mqa_logits to KVBlockSize>=1:
 *     the fp8 block-flat cache (KVB e4m3 key rows, then KVB fp32 scales),
 *     column c of request b at block table[b][c / KVB], slot c % KVB.
 *
 * Conventions for every call:
 *   - Pointers marked "device" are CUDA device (or managed) memory owned by the
 *     caller; the library never frees or retains them.  `desc` is host memory,
 *     read during the call only.
 *   - `stream` is a cudaStream_t (NULL = legacy default stream).  Work is
 *     enqueued asynchronously; no compute call synchronises the host with the
 *     device, so they can be captured in a CUDA graph (the first call of
 *     qsa_paged_mqa_topk_noalloc on a device excepted, see there).
 *   - The library allocates no device memory per call.
 *   - Kernels are launched with programmatic stream serialisation: a call's
 *     kernel may start while the kernel before it in the stream is still
 *     running, and it waits for that kernel before it reads q, weights, keys,
 *     scales or logits and before it writes anything.  The row metadata -
 *     visible_cols, next_n_lens and block_table - may be read before that
 *     wait, so the kernel just before a compute call in its stream must not
 *     write them (copies, and kernels further back in the stream, may).  The
 *     library's own kernels never write them, and each of them waits for its
 *     own predecessor before it lets the next kernel start.
 *   - Argument errors are detected on the host, before anything is enqueued,
 *     and returned synchronously (QSA_ERR_INVALID_ARG / QSA_ERR_UNSUPPORTED);
 *     a failed launch returns QSA_ERR_CUDA.  qsa_last_error() describes the
 *     most recent failure of the calling thread.
 *   - Device-resident values (page ids, visible counts) are not read by the
 *     host.  They are clamped on the device (visible to [0, capacity], page ids
 *     to [0, num_pages)), so bad values give wrong numbers, never a fault.
 *   - Not thread-safe with respect to qsa_force_variant().
 */
#ifndef QSA_H_
#define QSA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define QSA_ABI_VERSION 1

typedef enum qsa_status {
  QSA_OK = 0,
  QSA_ERR_INVALID_ARG = 1, /* null / misaligned pointer, bad size or stride */
  QSA_ERR_UNSUPPORTED = 2, /* valid request this library cannot serve (e.g. head_dim != 128) */
  QSA_ERR_CUDA = 3         /* a CUDA runtime call or kernel launch failed */
} qsa_status;

typedef enum qsa_kv_dtype {
  QSA_KV_BF16 = 0,     /* keys are bf16 [page_cols][head_dim] per page; no scales */
  QSA_KV_FP8_E4M3 = 1  /* keys are OCP e4m3fn bytes [page_cols][head_dim] per page,
                          each key dequantised by one fp32 scale (k = e4m3 * scale) */
} qsa_kv_dtype;

/* Kernel variants the host dispatch chooses between (qsa_plan_variant). */
typedef enum qsa_variant {
  QSA_VARIANT_AUTO = -1,
  QSA_VARIANT_ROWCORE = 0, /* CUDA-core scorer, one row at a time; any shape */
  QSA_VARIANT_UMMA = 1,    /* tcgen05 scorer: 128 keys in M, a request's rows x heads in N */
  QSA_VARIANT_UMMA_TOPK = 2, /* tcgen05 scorer with the selection in the same kernel
                               (qsa_paged_mqa_topk; reported by qsa_last_variant only) */
  QSA_VARIANT_UMMA_LEAN = 3 /* tcgen05 scorer in its lean form: 8 warps and half an SM's
                               shared memory, so that a call's CTAs share the SMs with the
                               kernel before it; groups of at most 64 rows x heads, at most
                               256 rows, bf16 keys or fp8 keys with fp8 q */
} qsa_variant;

/* Shape of one qsa_paged_mqa_logits call.  All sizes are host values. */
typedef struct qsa_paged_desc {
  int32_t num_requests;     /* B >= 0                                                  */
  int32_t rows_per_req;     /* query rows per request, >= 1; rows are request-major:
                               row r belongs to request r / rows_per_req              */
  int32_t num_heads;        /* H, 1..64 index heads                                    */
  int32_t head_dim;         /* D; must be 128 (else QSA_ERR_UNSUPPORTED)               */
  int32_t page_cols;        /* compressed keys (columns) per page / KV block, >= 1     */
  int32_t max_pages;        /* entries per block-table row (row stride), >= 1          */
  int32_t num_pages;        /* pages in the pool; page ids are clamped below this      */
  int32_t kv_dtype;         /* qsa_kv_dtype                                            */
  int64_t out_cols;         /* logits row width and row stride (floats), >= 0          */
  int64_t key_page_stride;  /* bytes between consecutive pages' keys; multiple of 16,
                               >= page_cols * head_dim * (2 for bf16, 1 for fp8)       */
  int64_t scale_page_stride;/* fp8: bytes between consecutive pages' scale vectors,
                               multiple of 4 (block-flat: == key_page_stride); bf16: 0 */
} qsa_paged_desc;

/*
 * qsa_paged_mqa_logits - index logits of every query row against its
 * request's paged keys.
 *
 * Defines (ROCm/ATOM #2651 "Changes": per-head ReLU before the heads are
 * summed; aiter #4221 "Technical details": ReLU then weight; vLLM #62589
 * first commit: fp32 accumulation), for row r, request b = r / rows_per_req
 * and column c < out_cols:
 *
 *   c >= visible_cols[r]:  out_logits[r*out_cols + c] = -inf
 *   otherwise:             p = block_table[b*max_pages + c / page_cols],
 *                          j = c % page_cols,
 *                          key = K[p][j][:] (bf16), or e4m3(K8[p][j][:]) * scale(p, j),
 *                          out = sum_h weights[r*H+h] * max(0, dot(q[r][h][:], key))
 *                          accumulated in fp32 (order unspecified); +0.0 for zero.
 *
 * Arguments (device pointers unless stated):
 *   desc         host; shape as above.
 *   q            bf16 [R][H][D], R = num_requests * rows_per_req; 16-byte aligned.
 *   weights      fp32 [R][H] per-row per-head weights (any finite sign).
 *   kv_cache     key of (page p, slot j) at (char*)kv_cache + p*key_page_stride
 *                + j*D*esize (esize 2 bf16, 1 fp8); 16-byte aligned.
 *   scales       fp8: scale of (p, j) at (char*)scales + p*scale_page_stride + 4*j;
 *                block-flat: scales = (char*)kv_cache + page_cols*D.  bf16: NULL
 *                (a non-NULL scales with bf16 keys, or NULL with fp8 keys, is
 *                rejected as mixed operand types, as SGLang #48649's
 *                rejects_mixed_operand_dtypes test does).
 *   block_table  int32 [num_requests][max_pages] physical page ids; only the
 *                entries covering a request's visible columns are read.  Read
 *                early (see the conventions above), as is visible_cols.
 *   visible_cols int32 [R] visible column count of each row.
 *   out_logits   fp32 [R][out_cols]; every element is written.
 *   stream       cudaStream_t.
 * Returns QSA_OK once the work is enqueued.
 */
qsa_status qsa_paged_mqa_logits(const qsa_paged_desc* desc, const void* q, const float* weights,
                                const void* kv_cache, const float* scales,
                                const int32_t* block_table, const int32_t* visible_cols,
                                float* out_logits, void* stream);

/*
 * qsa_paged_mqa_logits_ragged - qsa_paged_mqa_logits with a live-row count per
 * request (aiter #4221 "Ragged next_n for confidence-scheduled verification":
 * a request's leading next_n_lens[b] rows are live, the rest stay -inf).
 *
 * Row i of request b (r = b*rows_per_req + i) is live when
 * i < clamp(next_n_lens[b], 0, rows_per_req); a live row is scored exactly as
 * qsa_paged_mqa_logits scores it, and every logit of a dead row is -inf,
 * whatever its q, weights and visible count (its keys are not read).
 *
 *   next_n_lens  int32 [num_requests] (device), 4-byte aligned, or NULL: every
 *                row live (the call is then qsa_paged_mqa_logits).
 * Other arguments, errors and ownership as qsa_paged_mqa_logits.
 */
qsa_status qsa_paged_mqa_logits_ragged(const qsa_paged_desc* desc, const void* q, const float* weights,
                                       const void* kv_cache, const float* scales,
                                       const int32_t* block_table, const int32_t* visible_cols,
                                       const int32_t* next_n_lens, float* out_logits, void* stream);

/* q element types of qsa_paged_mqa_logits_ex. */
typedef enum { QSA_Q_BF16 = 0, QSA_Q_FP8_E4M3 = 1 } qsa_q_dtype;

/*
 * qsa_paged_mqa_logits_ex - qsa_paged_mqa_logits_ragged with the q element type
 * given.  With QSA_Q_FP8_E4M3 (aiter #4221 "Motivation": q and keys are e4m3
 * codes, weights, key scales and logits fp32; q has no scale of its own, the
 * weights carry it) q is OCP e4m3fn codes [R][H][D], 16-byte aligned, and the keys
 * must be fp8 too (QSA_KV_FP8_E4M3; bf16 keys with fp8 q are rejected as mixed
 * operand types); the definition is qsa_paged_mqa_logits's with
 * q[r][h][d] = e4m3(Q8[r][h][d]).  The tcgen05 scorer multiplies the raw fp8
 * q and keys (products exact, fp32 accumulation); the tolerance of fp8 keys
 * applies.  QSA_Q_BF16 is qsa_paged_mqa_logits_ragged.
 */
qsa_status qsa_paged_mqa_logits_ex(const qsa_paged_desc* desc, int32_t q_dtype, const void* q,
                                   const float* weights, const void* kv_cache, const float* scales,
                                   const int32_t* block_table, const int32_t* visible_cols,
                                   const int32_t* next_n_lens, float* out_logits, void* stream);

/*
 * qsa_select_topk - per-row top-k column indices of a logits matrix.
 *
 * For each row r (vLLM #62589 "Details": top-k reads only [0, visible)):
 *   n = visible_cols[r] clamped to [0, row_stride];
 *   n <= k: out_idx[r] = 0, 1, ..., n-1, then -1 in the remaining k - n slots
 *           (SGLang #48649: rows that fit in top-k select every column);
 *   n >  k: the k columns that come first in the order (logit descending,
 *           column ascending); -0.0 and +0.0 compare equal.
 * The selected columns are written in ascending column order.  NaN logits
 * inside [0, n) give an unspecified (but in-bounds) selection.
 *
 * Arguments (device pointers): logits fp32 rows of row_stride floats;
 * visible_cols int32 [num_rows]; out_idx int32 [num_rows][k].
 * num_rows >= 0, row_stride >= 1, 1 <= k <= 2048.
 * visible_cols is read before the kernel waits for the kernel before it in
 * the stream, the logits after (see the conventions above).
 */
qsa_status qsa_select_topk(const float* logits, int64_t num_rows, int64_t row_stride,
                           const int32_t* visible_cols, int32_t k, int32_t* out_idx,
                           void* stream);

/*
 * qsa_select_topk_bounded - qsa_select_topk with the caller's host bound on
 * the visible counts.
 *
 * A serving host knows the longest context of its batch (SGLang #48649's
 * test body hands max_model_len to the scorer beside context_lens; vLLM
 * #62589 "Dispatch" picks its decode path from host metadata).  The results
 * are exactly qsa_select_topk's; max_visible, the caller's bound on the
 * clamped counts (0 or less: none), only chooses the launch.  With a bound
 * of at most 8192 columns, and at most two rows an SM, every row is
 * selected by one CTA of 1024 threads holding the row's keys in registers
 * (faster for decode rows than the general form, which must allow rows of
 * any length).  A wrong bound costs speed only: a row longer than it is
 * still selected exactly, from global memory.
 *
 * Arguments as qsa_select_topk, plus max_visible (host value).  Errors as
 * qsa_select_topk.
 */
qsa_status qsa_select_topk_bounded(const float* logits, int64_t num_rows, int64_t row_stride,
                                   const int32_t* visible_cols, int64_t max_visible, int32_t k,
                                   int32_t* out_idx, void* stream);

/*
 * qsa_paged_mqa_topk - qsa_paged_mqa_logits_ex and then the top-k of every row,
 * in one call.
 *
 * The pages score and then select in two steps, and vLLM #62589 "Details"
 * notes that the only consumer of the logits, the decode top-k, reads each
 * row's [0, visible) alone.  The call runs the scoring launch and the top-k
 * launch, which measure faster on GB300 than selecting inside the scoring
 * kernel; with QSA_VARIANT_UMMA_TOPK forced (qsa_force_variant), a row's
 * selection starts in the scoring kernel as soon as every tile of the row is
 * stored, with the logits still in L2.
 *
 * Results: out_logits exactly as qsa_paged_mqa_logits_ex writes them; out_idx
 * exactly as qsa_select_topk(out_logits, R, out_cols, n, k, out_idx) writes
 * it, where n[r] is the row's scored visible count: visible_cols[r] clamped
 * to [0, min(out_cols, max_pages * page_cols)], and 0 for a dead row of the
 * ragged call (so a dead row selects nothing: k slots of -1).
 *
 * Arguments: as qsa_paged_mqa_logits_ex, plus
 *   k            1..2048 selected columns per row.
 *   max_visible  host value: the caller's bound on the visible counts, or 0
 *                (unknown; out_cols and the page capacity bound them).  Like
 *                vLLM #62589's single_row_decode flag it only steers the
 *                dispatch: the top-k launch's form, as in
 *                qsa_select_topk_bounded, and with the fused kernel forced,
 *                the selection runs in the scoring kernel for at most 256 rows
 *                whose bound is at most 16384 columns, and as a separate top-k
 *                launch (which splits long rows over a thread-block cluster)
 *                otherwise.  A wrong bound costs speed only.
 *   out_idx      int32 [R][k] (device), 4-byte aligned.
 *   workspace    device memory of at least qsa_paged_mqa_topk_workspace(desc)
 *                bytes, 4-byte aligned (NULL when that size is 0).  It must
 *                hold zeros before the first call; every completed call leaves
 *                it zero again (a call that set qsa_device_status bit 0 may
 *                not: zero it before the next call).  Calls that may run at the
 *                same time (other streams) need their own workspaces.
 * Errors as qsa_paged_mqa_logits_ex; k out of range, a NULL or misaligned
 * out_idx, or a missing or short workspace: QSA_ERR_INVALID_ARG.
 */
qsa_status qsa_paged_mqa_topk(const qsa_paged_desc* desc, int32_t q_dtype, const void* q, const float* weights,
                              const void* kv_cache, const float* scales, const int32_t* block_table,
                              const int32_t* visible_cols, const int32_t* next_n_lens, int32_t k,
                              int64_t max_visible, float* out_logits, int32_t* out_idx, void* workspace,
                              size_t workspace_bytes, void* stream);

/* Workspace bytes qsa_paged_mqa_topk needs for `desc` (host only; 0 when the
 * call never selects inside the scoring kernel - every shape unless
 * QSA_VARIANT_UMMA_TOPK is forced): 4 * (2 * G + 1) for the G <= 256 row
 * groups of the tcgen05 scorer. */
qsa_status qsa_paged_mqa_topk_workspace(const qsa_paged_desc* desc, size_t* bytes);

/*
 * qsa_paged_mqa_topk_noalloc - qsa_paged_mqa_topk with the library's own fixed
 * counter array in place of the caller's workspace.  The pages have no
 * counterpart: it exists for callers that want the fused call without owning
 * device memory for it.  It allocates nothing: the counters are a static
 * device array of 257 words, enough for 128 row groups.  A call that would
 * select inside the scoring kernel over more groups is rejected with
 * QSA_ERR_UNSUPPORTED before anything is enqueued; calls that take the
 * scoring and top-k launches instead (every call unless QSA_VARIANT_UMMA_TOPK
 * is forced, and then more than 256 rows, rows longer than 16384 columns, the
 * CUDA-core scorer's shapes) never touch the array and take any number of
 * groups.  The array must read zero when a call starts: it
 * is zero when the library is loaded, and every call that completes leaves it
 * zero.  A call that set qsa_device_status bit 0 may not:
 * qsa_device_status(flags, 1) then zeroes the array as well as the fault word,
 * or the caller zeroes it in stream order (a cudaMemsetAsync of the address
 * and size qsa_paged_mqa_topk_noalloc_counters gives).  The first call on each
 * device looks the array's address up (with that device current) and must
 * come before any stream capture on that device; the address is kept for the
 * life of the process, so cudaDeviceReset while the library is loaded is not
 * supported.  Calls that may overlap (other streams or host threads) share the
 * one array and race: give each of them qsa_paged_mqa_topk with its own
 * workspace instead.  Arguments, results and the other errors as
 * qsa_paged_mqa_topk.
 */
qsa_status qsa_paged_mqa_topk_noalloc(const qsa_paged_desc* desc, int32_t q_dtype, const void* q,
                                      const float* weights, const void* kv_cache, const float* scales,
                                      const int32_t* block_table, const int32_t* visible_cols,
                                      const int32_t* next_n_lens, int32_t k, int64_t max_visible,
                                      float* out_logits, int32_t* out_idx, void* stream);

/* Device address (*device_ptr) and size in bytes (*bytes) of the counter array
 * of qsa_paged_mqa_topk_noalloc on the current device, looked up as that
 * call's first use on the device does (so not during a stream capture).  For
 * callers that zero the array in stream order after a call that set
 * qsa_device_status bit 0; nothing else may write it. */
qsa_status qsa_paged_mqa_topk_noalloc_counters(void** device_ptr, size_t* bytes);

/*
 * qsa_plan_variant - host-only dispatch decision for `desc` (no CUDA call).
 * Writes the qsa_variant qsa_paged_mqa_logits would launch (honouring
 * qsa_force_variant) to *variant.  The choice uses host metadata only, with no
 * device sync, as vLLM #62589 "Dispatch" does for its one-row kernel.  On
 * GB300 the tcgen05 scorer measures faster than the CUDA-core one-row scorer
 * at every row count (single-row decode included), so shapes it supports go
 * to it - its lean form for decode-sized calls (at most 256 rows, groups of
 * at most 64 rows x heads, three 32 KB key stages in its shared memory), its
 * full form otherwise; everything else (head counts other than 1, 2, 4, ...,
 * 64, page sizes that are not a multiple of 8 dividing 128 or a multiple of
 * 128, misaligned fp8 scales) goes to the CUDA-core scorer.
 */
qsa_status qsa_plan_variant(const qsa_paged_desc* desc, int32_t* variant);

/* qsa_plan_variant for q of element type q_dtype (qsa_q_dtype), as
 * qsa_paged_mqa_logits_ex with that q_dtype would choose: fp8 keys with fp8 q
 * may take the lean tcgen05 form, fp8 keys with bf16 q never do (their keys
 * are widened by the converter warps of the full form). */
qsa_status qsa_plan_variant_ex(const qsa_paged_desc* desc, int32_t q_dtype, int32_t* variant);

/* Force a variant for later calls (QSA_VARIANT_AUTO restores the dispatch).
 * A forced scorer (ROWCORE, UMMA, UMMA_LEAN) that cannot serve a shape makes
 * the call return QSA_ERR_UNSUPPORTED, and qsa_paged_mqa_topk then runs it
 * and the top-k launch.  QSA_VARIANT_UMMA_TOPK makes qsa_paged_mqa_topk select
 * inside the scoring kernel for every shape the tcgen05 scorer serves (the
 * dispatch never does) and leaves the scoring calls' dispatch as it is.  Meant for tests and A/B measurements. */
void qsa_force_variant(int32_t variant);

/* Variant launched by this thread's last successful scoring call
 * (qsa_paged_mqa_logits and its _ragged / _ex forms, qsa_paged_mqa_topk). */
int32_t qsa_last_variant(void);

/* Static description of a status code, and of this thread's last failure. */
const char* qsa_status_string(int32_t status);
const char* qsa_last_error(void);

/*
 * qsa_device_status - the library's device fault word.  Bit 0 is set after a
 * scoring kernel gave up waiting on one of its internal barriers (about one
 * second): that launch left its output incomplete and returned early instead
 * of hanging the GPU.  Bit 1: a top-k launch gave up waiting for its row copy
 * (its selection for that row is unspecified).  Bit 2: a qsa_page_stream
 * launch gave up waiting for a page (its checksum is unspecified).  Synchronises the current
 * device, then writes the word to *flags (host pointer).  When `clear` is
 * non-zero it then clears the word and zeroes the counter array of
 * qsa_paged_mqa_topk_noalloc on the current device (synchronously), so the
 * next no-alloc call starts clean after a failed one.
 */
qsa_status qsa_device_status(uint32_t* flags, int32_t clear);

/*
 * qsa_page_stream - measurement, not part of the scoring path: streams the
 * listed pages from device memory into shared memory the way the scorers
 * fetch a request's key pages (one copy per page, in list order, one CTA per
 * SM taking a contiguous share), with no arithmetic on them, so the time of
 * a launch is the rate HBM delivers that gather - the achievable side of the
 * roofline of the key-cache reads that the paged scoring of vLLM #62589
 * "Overview" (keys gathered through a per-request block table) makes.
 *
 *   base        device pointer to pool_pages pages, page p at base + p * page_stride
 *               (16-byte aligned); read only.
 *   page_stride bytes from one page to the next (a multiple of 16).
 *   page_bytes  bytes copied from the start of each listed page: a multiple of
 *               16 in 16 .. 65536, at most page_stride.
 *   pages       device int32 [num_listed]: page indices; one outside
 *               [0, pool_pages) is clamped into it (no fault).
 *   checksum    device uint32, XORed with the XOR of every 32-bit word of every
 *               listed page copy (a page listed twice cancels): zero it first
 *               to read the checksum of one launch.  Written only by this call.
 *   stream      cudaStream_t (NULL: the legacy default stream); asynchronous.
 *
 * Returns QSA_ERR_INVALID_ARG for a null pointer with num_listed > 0, a
 * misaligned base or stride, page_bytes or pool_pages out of range;
 * QSA_ERR_CUDA when the launch fails.  num_listed == 0 launches nothing.
 */
qsa_status qsa_page_stream(const void* base, int64_t page_stride, int32_t page_bytes, const int32_t* pages,
                           int64_t num_listed, int64_t pool_pages, uint32_t* checksum, void* stream);

/* QSA_ABI_VERSION of the loaded library. */
int32_t qsa_abi_version(void);

#ifdef __cplusplus
}
#endif

#endif /* QSA_H_ */
