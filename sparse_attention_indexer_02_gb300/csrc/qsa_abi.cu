// C ABI entry points: host-side validation, variant dispatch and launches.
// Declarations, argument meaning and error behaviour are in include/qsa.h.
#include <stdarg.h>
#include <stdio.h>
#include <string.h>

#include <atomic>
#include <mutex>

#include "qsa_internal.h"

namespace {

thread_local char g_last_error[512] = "";
thread_local int32_t g_last_variant = -1;
std::atomic<int32_t> g_forced_variant{QSA_VARIANT_AUTO};

qsa_status fail(qsa_status st, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_last_error, sizeof g_last_error, fmt, ap);
  va_end(ap);
  return st;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

qsa_status validate_desc(const qsa_paged_desc* d) {
  if (!d) return fail(QSA_ERR_INVALID_ARG, "desc is NULL");
  if (d->num_requests < 0) return fail(QSA_ERR_INVALID_ARG, "num_requests < 0");
  if (d->rows_per_req < 1) return fail(QSA_ERR_INVALID_ARG, "rows_per_req < 1");
  if (d->num_heads < 1) return fail(QSA_ERR_INVALID_ARG, "num_heads < 1");
  if (d->num_heads > 64) return fail(QSA_ERR_UNSUPPORTED, "num_heads > 64");
  if (d->head_dim != 128) return fail(QSA_ERR_UNSUPPORTED, "head_dim must be 128 (got %d)", d->head_dim);
  if (d->page_cols < 1) return fail(QSA_ERR_INVALID_ARG, "page_cols < 1");
  if (d->max_pages < 1) return fail(QSA_ERR_INVALID_ARG, "max_pages < 1");
  if (d->num_pages < 1) return fail(QSA_ERR_INVALID_ARG, "num_pages < 1");
  if (d->out_cols < 0) return fail(QSA_ERR_INVALID_ARG, "out_cols < 0");
  if (d->kv_dtype != QSA_KV_BF16 && d->kv_dtype != QSA_KV_FP8_E4M3)
    return fail(QSA_ERR_INVALID_ARG, "unknown kv_dtype %d", d->kv_dtype);
  const int64_t rows = (int64_t)d->num_requests * d->rows_per_req;
  if (rows > 0x7FFFFFFFLL) return fail(QSA_ERR_INVALID_ARG, "num_requests * rows_per_req overflows int32");
  const int64_t esize = d->kv_dtype == QSA_KV_BF16 ? 2 : 1;
  const int64_t key_bytes = (int64_t)d->page_cols * d->head_dim * esize;
  if (d->key_page_stride % 16 != 0 || d->key_page_stride < key_bytes)
    return fail(QSA_ERR_INVALID_ARG, "key_page_stride must be a multiple of 16 and >= %lld",
                (long long)key_bytes);
  if (d->kv_dtype == QSA_KV_FP8_E4M3 &&
      (d->scale_page_stride % 4 != 0 || d->scale_page_stride < 4LL * d->page_cols))
    return fail(QSA_ERR_INVALID_ARG, "scale_page_stride must be a multiple of 4 and >= 4 * page_cols");
  return QSA_OK;
}

}  // namespace

namespace qsa {

cudaError_t device_info(DeviceInfo* info) {
  static std::mutex mu;
  static DeviceInfo cache[64];
  static bool have[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lock(mu);
  if (dev >= 0 && dev < 64 && have[dev]) {
    *info = cache[dev];
    return cudaSuccess;
  }
  DeviceInfo d{dev, 0, 0};
  e = cudaDeviceGetAttribute(&d.num_sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  e = cudaDeviceGetAttribute(&d.max_smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
  if (e != cudaSuccess) return e;
  if (dev >= 0 && dev < 64) {
    cache[dev] = d;
    have[dev] = true;
  }
  *info = d;
  return cudaSuccess;
}

}  // namespace qsa

extern "C" {

int32_t qsa_abi_version(void) { return QSA_ABI_VERSION; }

const char* qsa_status_string(int32_t s) {
  switch (s) {
    case QSA_OK: return "QSA_OK";
    case QSA_ERR_INVALID_ARG: return "QSA_ERR_INVALID_ARG";
    case QSA_ERR_UNSUPPORTED: return "QSA_ERR_UNSUPPORTED";
    case QSA_ERR_CUDA: return "QSA_ERR_CUDA";
    default: return "unknown qsa_status";
  }
}

const char* qsa_last_error(void) { return g_last_error; }

void qsa_force_variant(int32_t v) { g_forced_variant.store(v); }

int32_t qsa_last_variant(void) { return g_last_variant; }

}  // extern "C"

namespace {

// Variant for `d` with q of type q8 (fp8) or bf16; see qsa_plan_variant.
qsa_status plan(const qsa_paged_desc* d, bool q8, int32_t* variant) {
  qsa_status st = validate_desc(d);
  if (st != QSA_OK) return st;
  if (!variant) return fail(QSA_ERR_INVALID_ARG, "variant is NULL");
  const int32_t forced = g_forced_variant.load();
  const char* why = nullptr;
  if (forced == QSA_VARIANT_ROWCORE) {
    *variant = QSA_VARIANT_ROWCORE;
  } else if (forced == QSA_VARIANT_UMMA) {
    if (!qsa::umma_supports(*d, &why))
      return fail(QSA_ERR_UNSUPPORTED, "forced tcgen05 variant cannot serve this shape: %s", why);
    *variant = QSA_VARIANT_UMMA;
  } else if (forced == QSA_VARIANT_UMMA_LEAN) {
    if (!qsa::umma_lean_supports(*d, q8, &why))
      return fail(QSA_ERR_UNSUPPORTED, "forced lean tcgen05 variant cannot serve this shape: %s", why);
    *variant = QSA_VARIANT_UMMA_LEAN;
  } else if (qsa::umma_lean_supports(*d, q8, &why)) {
    // decode-sized calls: the lean form, whose CTAs share the SMs with the
    // kernel before it and stream their first keys while it finishes
    *variant = QSA_VARIANT_UMMA_LEAN;
  } else if (qsa::umma_supports(*d, &why)) {
    // Measured on GB300: the tcgen05 scorer is faster than the CUDA-core
    // one-row scorer at every row count, single-row decode included (its
    // padded N = 16 costs nothing against HBM), so it takes every shape it
    // serves; the one-row scorer serves the rest.
    *variant = QSA_VARIANT_UMMA;
  } else {
    *variant = QSA_VARIANT_ROWCORE;
  }
  return QSA_OK;
}

}  // namespace

extern "C" {

qsa_status qsa_plan_variant(const qsa_paged_desc* d, int32_t* variant) { return plan(d, false, variant); }

qsa_status qsa_plan_variant_ex(const qsa_paged_desc* d, int32_t q_dtype, int32_t* variant) {
  if (q_dtype != QSA_Q_BF16 && q_dtype != QSA_Q_FP8_E4M3)
    return fail(QSA_ERR_INVALID_ARG, "q_dtype must be QSA_Q_BF16 or QSA_Q_FP8_E4M3 (got %d)", q_dtype);
  if (d && q_dtype == QSA_Q_FP8_E4M3 && d->kv_dtype != QSA_KV_FP8_E4M3)
    return fail(QSA_ERR_INVALID_ARG, "fp8 q needs fp8 keys (mixed operand types)");
  return plan(d, q_dtype == QSA_Q_FP8_E4M3, variant);
}

qsa_status qsa_paged_mqa_logits(const qsa_paged_desc* d, const void* q, const float* weights,
                                const void* kv_cache, const float* scales,
                                const int32_t* block_table, const int32_t* visible_cols,
                                float* out_logits, void* stream) {
  return qsa_paged_mqa_logits_ragged(d, q, weights, kv_cache, scales, block_table, visible_cols, nullptr,
                                     out_logits, stream);
}

qsa_status qsa_paged_mqa_logits_ragged(const qsa_paged_desc* d, const void* q, const float* weights,
                                       const void* kv_cache, const float* scales,
                                       const int32_t* block_table, const int32_t* visible_cols,
                                       const int32_t* next_n_lens, float* out_logits, void* stream) {
  return qsa_paged_mqa_logits_ex(d, QSA_Q_BF16, q, weights, kv_cache, scales, block_table, visible_cols,
                                 next_n_lens, out_logits, stream);
}

}  // extern "C"

namespace {

// Validation, variant choice and launch parameters shared by the scoring
// calls.  Returns QSA_OK with *empty set when there is nothing to compute.
qsa_status prepare_scoring(const qsa_paged_desc* d, int32_t q_dtype, const void* q, const float* weights,
                           const void* kv_cache, const float* scales, const int32_t* block_table,
                           const int32_t* visible_cols, const int32_t* next_n_lens, float* out_logits,
                           qsa::ScoreParams* p, int32_t* variant, bool* empty) {
  qsa_status st = validate_desc(d);
  if (st != QSA_OK) return st;
  const int64_t rows = (int64_t)d->num_requests * d->rows_per_req;
  const bool fp8 = d->kv_dtype == QSA_KV_FP8_E4M3;
  if (q_dtype != QSA_Q_BF16 && q_dtype != QSA_Q_FP8_E4M3)
    return fail(QSA_ERR_INVALID_ARG, "q_dtype must be QSA_Q_BF16 or QSA_Q_FP8_E4M3 (got %d)", q_dtype);
  const bool q8 = q_dtype == QSA_Q_FP8_E4M3;
  if (q8 && !fp8) return fail(QSA_ERR_INVALID_ARG, "fp8 q needs fp8 keys (mixed operand types)");
  if (fp8 && !scales) return fail(QSA_ERR_INVALID_ARG, "fp8 keys need a scales pointer");
  if (!fp8 && scales) return fail(QSA_ERR_INVALID_ARG, "bf16 keys take no scales (mixed operand types)");
  *empty = rows == 0 || d->out_cols == 0;
  if (*empty) return QSA_OK;
  if (!q || !weights || !kv_cache || !block_table || !visible_cols || !out_logits)
    return fail(QSA_ERR_INVALID_ARG, "a required pointer is NULL");
  if (!aligned(q, 16) || !aligned(kv_cache, 16))
    return fail(QSA_ERR_INVALID_ARG, "q and kv_cache must be 16-byte aligned");
  if (!aligned(weights, 4) || !aligned(block_table, 4) || !aligned(visible_cols, 4) ||
      !aligned(out_logits, 4) || (fp8 && !aligned(scales, 4)) || !aligned(next_n_lens, 4))
    return fail(QSA_ERR_INVALID_ARG,
                "weights, block_table, visible_cols, next_n_lens, out_logits, scales must be 4-byte aligned");
  st = plan(d, q8, variant);
  if (st != QSA_OK) return st;
  // the tcgen05 scorer bulk-copies fp8 scales, which needs a 16-byte aligned base
  if ((*variant == QSA_VARIANT_UMMA || *variant == QSA_VARIANT_UMMA_LEAN) && fp8 && !aligned(scales, 16)) {
    if (g_forced_variant.load() != QSA_VARIANT_AUTO)
      return fail(QSA_ERR_UNSUPPORTED, "forced tcgen05 variant needs 16-byte aligned fp8 scales");
    *variant = QSA_VARIANT_ROWCORE;
  }
  p->q = static_cast<const uint16_t*>(q);
  p->weights = weights;
  p->kv = static_cast<const uint8_t*>(kv_cache);
  p->scales = reinterpret_cast<const uint8_t*>(scales);
  p->block_table = block_table;
  p->visible = visible_cols;
  p->next_n_lens = next_n_lens;
  p->out = out_logits;
  p->out_cols = d->out_cols;
  p->key_page_stride = d->key_page_stride;
  p->scale_page_stride = fp8 ? d->scale_page_stride : 0;
  const int64_t cap = (int64_t)d->max_pages * d->page_cols;
  p->capacity = cap < d->out_cols ? cap : d->out_cols;
  p->num_requests = d->num_requests;
  p->rows_per_req = d->rows_per_req;
  p->num_rows = (int32_t)rows;
  p->num_heads = d->num_heads;
  p->page_cols = d->page_cols;
  p->max_pages = d->max_pages;
  p->num_pages = d->num_pages;
  p->fp8 = fp8 ? 1 : 0;
  p->q8 = q8 ? 1 : 0;
  return QSA_OK;
}

qsa_status launch_scoring(const qsa::ScoreParams& p, int32_t variant, cudaStream_t s,
                          const qsa::FuseArgs* fuse) {
  const char* msg = "launch failed";
  cudaError_t e = variant == QSA_VARIANT_ROWCORE
                      ? qsa::launch_rowcore(p, s, &msg)
                      : qsa::launch_umma(p, s, &msg, fuse, variant == QSA_VARIANT_UMMA_LEAN);
  if (e == cudaErrorInvalidValue && msg && strcmp(msg, "launch failed") != 0)
    return fail(QSA_ERR_UNSUPPORTED, "%s", msg);
  if (e != cudaSuccess)
    return fail(QSA_ERR_CUDA, "scoring launch (variant %d): %s", variant, cudaGetErrorString(e));
  g_last_variant = variant;
  return QSA_OK;
}

// The fused selection is used for decode-sized calls: at most kFuseMaxRows
// rows, none longer than kFuseMaxVisible columns (up to there one CTA a row is
// as fast as any split of the row, the top-k kernel's own rule; longer rows go
// to the cluster split of the separate top-k launch).
constexpr int64_t kFuseMaxRows = 256;
constexpr int64_t kFuseMaxVisible = 16384;

// Whether qsa_paged_mqa_topk may select inside the scoring kernel for `d`
// (the row count and the caller's bound are checked at the call).  Measured on
// GB300, the lean scorer followed by the top-k launch is faster than the fused
// kernel at every decode shape (single-row decode 17.9 vs 18.4 us a step,
// tiny_mtp 9.1 vs 12.1 us), so the dispatch does not fuse; forcing
// QSA_VARIANT_UMMA_TOPK fuses every shape the tcgen05 scorer serves.
bool fusable(const qsa_paged_desc* d) {
  const char* why = nullptr;
  if (!qsa::umma_supports(*d, &why)) return false;
  return g_forced_variant.load() == QSA_VARIANT_UMMA_TOPK;
}

// Workspace words of the fused selection for `d` (0: the shape is never fused).
int64_t fused_words(const qsa_paged_desc* d) {
  if (!fusable(d)) return 0;
  const int64_t G = qsa::umma_num_groups(*d);
  return G >= 1 && G <= qsa::kFuseMaxGroups ? 2 * G + 1 : 0;
}

// Counters of qsa_paged_mqa_topk_noalloc: a fixed array in the library's
// own device memory instead of a caller workspace (zero when the library is
// loaded; every completed call leaves it zero).
constexpr int kNoAllocGroups = 128;
constexpr int kNoAllocWords = 2 * kNoAllocGroups + 1;
static __device__ __align__(256) uint32_t g_noalloc_counters[kNoAllocWords];

// Device address of g_noalloc_counters on the current device, looked up once
// per device (with that device current).
cudaError_t noalloc_counters(uint32_t** out) {
  static std::mutex mu;
  static uint32_t* addr[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(mu);
  if (!addr[dev]) {
    void* a = nullptr;
    e = cudaGetSymbolAddress(&a, g_noalloc_counters);
    if (e != cudaSuccess) return e;
    addr[dev] = static_cast<uint32_t*>(a);
  }
  *out = addr[dev];
  return cudaSuccess;
}

// qsa_paged_mqa_topk (workspace given) and qsa_paged_mqa_topk_noalloc (the
// library's counter array, looked up only when the fused selection runs).
qsa_status topk_call(const qsa_paged_desc* d, int32_t q_dtype, const void* q, const float* weights,
                     const void* kv_cache, const float* scales, const int32_t* block_table,
                     const int32_t* visible_cols, const int32_t* next_n_lens, int32_t k, int64_t max_visible,
                     float* out_logits, int32_t* out_idx, void* workspace, size_t workspace_bytes, bool noalloc,
                     void* stream) {
  qsa::ScoreParams p;
  int32_t variant = 0;
  bool empty = false;
  qsa_status st = prepare_scoring(d, q_dtype, q, weights, kv_cache, scales, block_table, visible_cols,
                                  next_n_lens, out_logits, &p, &variant, &empty);
  if (st != QSA_OK) return st;
  if (k < 1 || k > 2048) return fail(QSA_ERR_INVALID_ARG, "k must be in 1..2048 (got %d)", k);
  if (empty) {
    g_last_variant = -1;
    if ((int64_t)d->num_requests * d->rows_per_req == 0) return QSA_OK;
    // rows but no column: every row selects nothing
    if (!out_idx || !aligned(out_idx, 4)) return fail(QSA_ERR_INVALID_ARG, "out_idx must be 4-byte aligned");
    const size_t n = (size_t)d->num_requests * d->rows_per_req * k * sizeof(int32_t);
    cudaError_t e = cudaMemsetAsync(out_idx, 0xFF, n, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return fail(QSA_ERR_CUDA, "filling out_idx: %s", cudaGetErrorString(e));
    return QSA_OK;
  }
  if (!out_idx || !aligned(out_idx, 4)) return fail(QSA_ERR_INVALID_ARG, "out_idx must be non-NULL, 4-byte aligned");
  const int64_t words = fused_words(d);
  if (!noalloc && words > 0 && (!workspace || !aligned(workspace, 4) || workspace_bytes < (size_t)words * 4))
    return fail(QSA_ERR_INVALID_ARG, "workspace must be 4-byte aligned and hold %lld bytes", (long long)words * 4);
  const int64_t bound = max_visible > 0 && max_visible < p.capacity ? max_visible : p.capacity;
  // the fused selection runs in the full form of the tcgen05 scorer
  const bool fused =
      words > 0 && variant != QSA_VARIANT_ROWCORE && p.num_rows <= kFuseMaxRows && bound <= kFuseMaxVisible;
  if (fused && noalloc) {
    if (words > kNoAllocWords)
      return fail(QSA_ERR_UNSUPPORTED,
                  "qsa_paged_mqa_topk_noalloc holds counters for %d row groups and this call selects in the "
                  "scoring kernel over %lld: call qsa_paged_mqa_topk with a workspace of %lld bytes",
                  kNoAllocGroups, (long long)(words - 1) / 2, (long long)words * 4);
    uint32_t* counters = nullptr;
    cudaError_t e = noalloc_counters(&counters);
    if (e != cudaSuccess) return fail(QSA_ERR_CUDA, "counter address: %s", cudaGetErrorString(e));
    workspace = counters;
  }
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (fused) {
    const qsa::FuseArgs fa{out_idx, static_cast<uint32_t*>(workspace), k};
    st = launch_scoring(p, QSA_VARIANT_UMMA, s, &fa);
    if (st == QSA_OK) g_last_variant = QSA_VARIANT_UMMA_TOPK;
    return st;
  }
  st = launch_scoring(p, variant, s, nullptr);
  if (st != QSA_OK) return st;
  cudaError_t e = qsa::launch_topk(out_logits, p.num_rows, p.out_cols, visible_cols, next_n_lens, p.rows_per_req,
                                   p.capacity, max_visible, k, out_idx, s);
  if (e != cudaSuccess) return fail(QSA_ERR_CUDA, "top-k launch: %s", cudaGetErrorString(e));
  return QSA_OK;
}

}  // namespace

extern "C" {

qsa_status qsa_paged_mqa_logits_ex(const qsa_paged_desc* d, int32_t q_dtype, const void* q,
                                   const float* weights, const void* kv_cache, const float* scales,
                                   const int32_t* block_table, const int32_t* visible_cols,
                                   const int32_t* next_n_lens, float* out_logits, void* stream) {
  qsa::ScoreParams p;
  int32_t variant = 0;
  bool empty = false;
  qsa_status st = prepare_scoring(d, q_dtype, q, weights, kv_cache, scales, block_table, visible_cols,
                                  next_n_lens, out_logits, &p, &variant, &empty);
  if (st != QSA_OK) return st;
  if (empty) {
    g_last_variant = -1;
    return QSA_OK;
  }
  return launch_scoring(p, variant, static_cast<cudaStream_t>(stream), nullptr);
}

qsa_status qsa_paged_mqa_topk_workspace(const qsa_paged_desc* d, size_t* bytes) {
  qsa_status st = validate_desc(d);
  if (st != QSA_OK) return st;
  if (!bytes) return fail(QSA_ERR_INVALID_ARG, "bytes is NULL");
  *bytes = (size_t)fused_words(d) * 4;
  return QSA_OK;
}

qsa_status qsa_paged_mqa_topk(const qsa_paged_desc* d, int32_t q_dtype, const void* q, const float* weights,
                              const void* kv_cache, const float* scales, const int32_t* block_table,
                              const int32_t* visible_cols, const int32_t* next_n_lens, int32_t k,
                              int64_t max_visible, float* out_logits, int32_t* out_idx, void* workspace,
                              size_t workspace_bytes, void* stream) {
  return topk_call(d, q_dtype, q, weights, kv_cache, scales, block_table, visible_cols, next_n_lens, k, max_visible,
                   out_logits, out_idx, workspace, workspace_bytes, false, stream);
}

qsa_status qsa_paged_mqa_topk_noalloc(const qsa_paged_desc* d, int32_t q_dtype, const void* q,
                                      const float* weights, const void* kv_cache, const float* scales,
                                      const int32_t* block_table, const int32_t* visible_cols,
                                      const int32_t* next_n_lens, int32_t k, int64_t max_visible,
                                      float* out_logits, int32_t* out_idx, void* stream) {
  return topk_call(d, q_dtype, q, weights, kv_cache, scales, block_table, visible_cols, next_n_lens, k, max_visible,
                   out_logits, out_idx, nullptr, 0, true, stream);
}

qsa_status qsa_paged_mqa_topk_noalloc_counters(void** device_ptr, size_t* bytes) {
  if (!device_ptr || !bytes) return fail(QSA_ERR_INVALID_ARG, "device_ptr and bytes must be non-NULL");
  uint32_t* counters = nullptr;
  cudaError_t e = noalloc_counters(&counters);
  if (e != cudaSuccess) return fail(QSA_ERR_CUDA, "counter address: %s", cudaGetErrorString(e));
  *device_ptr = counters;
  *bytes = sizeof(g_noalloc_counters);
  return QSA_OK;
}

qsa_status qsa_page_stream(const void* base, int64_t page_stride, int32_t page_bytes, const int32_t* pages,
                           int64_t num_listed, int64_t pool_pages, uint32_t* checksum, void* stream) {
  if (num_listed < 0) return fail(QSA_ERR_INVALID_ARG, "num_listed < 0");
  if (num_listed == 0) return QSA_OK;
  if (!base || !pages || !checksum) return fail(QSA_ERR_INVALID_ARG, "a required pointer is NULL");
  if (reinterpret_cast<uintptr_t>(base) % 16 != 0 || page_stride % 16 != 0 || page_stride < 16)
    return fail(QSA_ERR_INVALID_ARG, "base and page_stride must be multiples of 16 bytes");
  if (page_bytes < 16 || page_bytes > 65536 || page_bytes % 16 != 0 || page_bytes > page_stride)
    return fail(QSA_ERR_INVALID_ARG, "page_bytes must be a multiple of 16 in 16..65536 and at most page_stride");
  if (pool_pages < 1) return fail(QSA_ERR_INVALID_ARG, "pool_pages < 1");
  if (reinterpret_cast<uintptr_t>(pages) % 4 != 0 || reinterpret_cast<uintptr_t>(checksum) % 4 != 0)
    return fail(QSA_ERR_INVALID_ARG, "pages and checksum must be 4-byte aligned");
  cudaError_t e = qsa::launch_page_stream(static_cast<const uint8_t*>(base), page_stride, page_bytes, pages,
                                          num_listed, pool_pages, checksum, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return fail(QSA_ERR_CUDA, "page stream launch: %s", cudaGetErrorString(e));
  return QSA_OK;
}

qsa_status qsa_device_status(uint32_t* flags, int32_t clear) {
  if (!flags) return fail(QSA_ERR_INVALID_ARG, "flags is NULL");
  cudaError_t e = qsa::read_fault_word(flags, clear != 0);
  if (e != cudaSuccess) return fail(QSA_ERR_CUDA, "reading the device fault word: %s", cudaGetErrorString(e));
  if (clear) {
    // the device is idle (read_fault_word synchronised it): put the no-alloc
    // call's counters back to zero too, whatever a failed call left there
    uint32_t* counters = nullptr;
    e = noalloc_counters(&counters);
    if (e == cudaSuccess) e = cudaMemset(counters, 0, sizeof(g_noalloc_counters));
    if (e == cudaSuccess) e = cudaDeviceSynchronize();
    if (e != cudaSuccess) return fail(QSA_ERR_CUDA, "clearing the no-alloc counters: %s", cudaGetErrorString(e));
  }
  return QSA_OK;
}

qsa_status qsa_select_topk(const float* logits, int64_t num_rows, int64_t row_stride,
                           const int32_t* visible_cols, int32_t k, int32_t* out_idx, void* stream) {
  return qsa_select_topk_bounded(logits, num_rows, row_stride, visible_cols, 0, k, out_idx, stream);
}

qsa_status qsa_select_topk_bounded(const float* logits, int64_t num_rows, int64_t row_stride,
                                   const int32_t* visible_cols, int64_t max_visible, int32_t k, int32_t* out_idx,
                                   void* stream) {
  if (num_rows < 0) return fail(QSA_ERR_INVALID_ARG, "num_rows < 0");
  if (row_stride < 1) return fail(QSA_ERR_INVALID_ARG, "row_stride < 1");
  if (k < 1 || k > 2048) return fail(QSA_ERR_INVALID_ARG, "k must be in 1..2048 (got %d)", k);
  if (num_rows > 0x7FFFFFFFLL) return fail(QSA_ERR_INVALID_ARG, "num_rows exceeds 2^31 - 1");
  if (num_rows == 0) return QSA_OK;
  if (!logits || !visible_cols || !out_idx) return fail(QSA_ERR_INVALID_ARG, "a required pointer is NULL");
  if (!aligned(logits, 4) || !aligned(visible_cols, 4) || !aligned(out_idx, 4))
    return fail(QSA_ERR_INVALID_ARG, "pointers must be 4-byte aligned");
  cudaError_t e = qsa::launch_topk(logits, num_rows, row_stride, visible_cols, nullptr, 1, row_stride, max_visible, k,
                                   out_idx, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return fail(QSA_ERR_CUDA, "top-k launch: %s", cudaGetErrorString(e));
  return QSA_OK;
}

}  // extern "C"
