/*
 * CPU oracle for paged MQA-logits scoring and per-row top-k selection.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path links, loads or calls
 * this file: only tests/, __graft_entry__.smoke() and bench.py's CPU baseline
 * (and its `--impl reference` arm) use it.  It shares no code, header, table
 * or constant with the CUDA library.
 *
 * It is the plain definition, written out element by element in double
 * precision, with no blocking, fusion or reordering:
 *
 *   for row r of request b = r / rows_per_req and column c < out_cols:
 *     c >= visible[r]         ->  logit[r][c] = -inf
 *     otherwise  p = block_table[b][c / page_cols],  j = c % page_cols
 *                key[d]  = bf16(K[p][j][d])                   (bf16 cache)
 *                        | e4m3(K8[p][j][d]) * scale[p][j]    (fp8 cache)
 *                logit   = sum_h w[r][h] * max(0, sum_d q[r][h][d] * key[d])
 *                q[r][h][d] = bf16(Q[r][h][d]), or e4m3(Q8[r][h][d]) with fp8 q
 *                (aiter #4221 "Motivation": both q and the keys are e4m3 codes while
 *                the weights, key scales and logits stay fp32; q has no scale of its own)
 *                (max(0, NaN) is NaN, as torch.relu: poisoned keys stay visible)
 *                rounded once to fp32; a zero result is stored as +0.0
 *
 * Sources, by page and section:
 *  - per-head ReLU before the head sum: ROCm/ATOM #2651 "Changes" (stacked
 *    scorer applies the per-head ReLU before summing heads back out of M);
 *    aiter #4221 "Technical details" (ReLU then weight, "ReLU*w").
 *  - fp32 accumulation of the dot is the kernels' precision; the oracle uses
 *    double and rounds once (vLLM #62589, first commit: "fp32 accumulation").
 *  - column -> page gather: aiter #4221 commit "extend fp8_paged_mqa_logits to
 *    KVBlockSize>=1" (block = table[b][col / KVB], token = col % KVB).
 *  - fp8 block-flat layout: same commit (KVB fp8 key rows, then KVB fp32
 *    scales); the scale dequantises the key (k = e4m3 * scale).
 *  - -inf past the visible count: aiter #4221 test gate ("exact -inf mask").
 *  - top-k over [0, visible): vLLM #62589 "Details"; rows with at most k
 *    visible columns select all of them (SGLang #48649 test list,
 *    "decode_skips_rows_that_fit_topk"); unused slots are -1 (SGLang #48649
 *    test body filters idx >= 0).
 *  - tie rule (value descending, then column ascending) is this library's
 *    reading: the pages leave ties to the implementation (vLLM #62589,
 *    MI300X comment: "so tie-break decides").
 *
 * bf16 and e4m3 are decoded from their format definitions:
 *  - bfloat16: 1 sign bit, 8 exponent bits (bias 127), 7 fraction bits,
 *    subnormals when the exponent field is 0, inf/NaN when it is 255.
 *  - OCP OFP8 E4M3 ("fn"): 1 sign bit, 4 exponent bits (bias 7), 3 fraction
 *    bits, subnormals when the exponent field is 0, no infinities, NaN only
 *    for S.1111.111; largest finite magnitude 448.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_OK 0
#define ORACLE_BAD_ARG 1
#define ORACLE_BAD_DATA 2

double qsa_oracle_bf16_value(uint16_t bits) {
  int sign = (bits >> 15) & 1;
  int expo = (bits >> 7) & 0xFF;
  int frac = bits & 0x7F;
  double mag;
  if (expo == 0xFF) {
    mag = frac ? NAN : INFINITY;
  } else if (expo == 0) {
    mag = ldexp((double)frac / 128.0, -126);
  } else {
    mag = ldexp(1.0 + (double)frac / 128.0, expo - 127);
  }
  return sign ? -mag : mag;
}

double qsa_oracle_e4m3_value(uint8_t code) {
  int sign = (code >> 7) & 1;
  int expo = (code >> 3) & 0xF;
  int frac = code & 0x7;
  double mag;
  if (expo == 0xF && frac == 0x7) {
    mag = NAN;
  } else if (expo == 0) {
    mag = ldexp((double)frac / 8.0, -6);
  } else {
    mag = ldexp(1.0 + (double)frac / 8.0, expo - 7);
  }
  return sign ? -mag : mag;
}

static double f32_bits_to_double(const uint8_t* p) {
  float f;
  memcpy(&f, p, sizeof f);
  return (double)f;
}

typedef struct {
  int32_t num_requests, rows_per_req, num_heads, head_dim, page_cols, max_pages, num_pages,
      kv_dtype;
  int64_t out_cols, key_page_stride, scale_page_stride;
  int32_t q_dtype; /* 0: bf16 q, 1: e4m3 q */
  const void* q;
  const float* weights;
  const uint8_t* kv;
  const uint8_t* scales;
  const int32_t* block_table;
  const int32_t* visible;
  const int64_t* rows;
  int64_t num_sel;
  float* out;
  int32_t num_threads, thread_id;
  int status;
} logits_job;

/* One output row: the definition above, column by column. */
static int oracle_row(const logits_job* J, int64_t r, float* out_row) {
  const int64_t D = J->head_dim, H = J->num_heads;
  const int64_t b = r / J->rows_per_req;
  const int64_t vis = J->visible[r];
  double* key = (double*)malloc(sizeof(double) * (size_t)D);
  if (!key) return ORACLE_BAD_ARG;
  for (int64_t c = 0; c < J->out_cols; ++c) {
    if (c >= vis) {
      out_row[c] = -INFINITY;
      continue;
    }
    const int64_t p = J->block_table[b * J->max_pages + c / J->page_cols];
    const int64_t j = c % J->page_cols;
    if (p < 0 || p >= J->num_pages) {
      free(key);
      return ORACLE_BAD_DATA;
    }
    if (J->kv_dtype == 0) {
      const uint8_t* src = J->kv + p * J->key_page_stride + j * D * 2;
      for (int64_t d = 0; d < D; ++d) {
        uint16_t bits = (uint16_t)(src[2 * d] | (src[2 * d + 1] << 8));
        key[d] = qsa_oracle_bf16_value(bits);
      }
    } else {
      const uint8_t* src = J->kv + p * J->key_page_stride + j * D;
      const double scale = f32_bits_to_double(J->scales + p * J->scale_page_stride + 4 * j);
      for (int64_t d = 0; d < D; ++d) key[d] = qsa_oracle_e4m3_value(src[d]) * scale;
    }
    double acc = 0.0;
    for (int64_t h = 0; h < H; ++h) {
      double dot = 0.0;
      if (J->q_dtype == 0) {
        const uint16_t* qh = (const uint16_t*)J->q + (r * H + h) * D;
        for (int64_t d = 0; d < D; ++d) dot += qsa_oracle_bf16_value(qh[d]) * key[d];
      } else {
        const uint8_t* qh = (const uint8_t*)J->q + (r * H + h) * D;
        for (int64_t d = 0; d < D; ++d) dot += qsa_oracle_e4m3_value(qh[d]) * key[d];
      }
      /* ReLU that lets NaN through, as torch.relu does: a poisoned key shows. */
      const double relu = dot < 0.0 ? 0.0 : dot;
      acc += (double)J->weights[r * H + h] * relu;
    }
    float v = (float)acc;
    if (v == 0.0f) v = 0.0f; /* a zero logit is +0.0 */
    out_row[c] = v;
  }
  free(key);
  return ORACLE_OK;
}

static void* logits_worker(void* arg) {
  logits_job* J = (logits_job*)arg;
  for (int64_t i = J->thread_id; i < J->num_sel; i += J->num_threads) {
    const int64_t r = J->rows ? J->rows[i] : i;
    int st = oracle_row(J, r, J->out + i * J->out_cols);
    if (st != ORACLE_OK) {
      J->status = st;
      break;
    }
  }
  return NULL;
}

/* Logits of the selected rows (rows == NULL: every row, in order) into
 * out[num_sel][out_cols], q bf16 (q_dtype 0) or e4m3 (q_dtype 1).  Returns 0,
 * or non-zero on bad arguments / page ids. */
int qsa_oracle_paged_mqa_logits_ex(int32_t num_requests, int32_t rows_per_req, int32_t num_heads,
                                   int32_t head_dim, int32_t page_cols, int32_t max_pages,
                                   int32_t num_pages, int32_t kv_dtype, int64_t out_cols,
                                   int64_t key_page_stride, int64_t scale_page_stride, int32_t q_dtype,
                                   const void* q, const float* weights, const uint8_t* kv,
                                   const uint8_t* scales, const int32_t* block_table,
                                   const int32_t* visible, const int64_t* rows, int64_t num_sel,
                                   float* out, int32_t num_threads) {
  if (num_requests < 0 || rows_per_req < 1 || num_heads < 1 || head_dim < 1 || page_cols < 1 ||
      max_pages < 1 || num_pages < 1 || out_cols < 0 || (kv_dtype != 0 && kv_dtype != 1) ||
      (q_dtype != 0 && q_dtype != 1))
    return ORACLE_BAD_ARG;
  if (!q || !weights || !kv || !block_table || !visible || !out) return ORACLE_BAD_ARG;
  if (kv_dtype == 1 && !scales) return ORACLE_BAD_ARG;
  const int64_t R = (int64_t)num_requests * rows_per_req;
  const int64_t cap = (int64_t)max_pages * page_cols;
  if (!rows) num_sel = R;
  for (int64_t i = 0; i < num_sel; ++i) {
    const int64_t r = rows ? rows[i] : i;
    if (r < 0 || r >= R) return ORACLE_BAD_ARG;
    if (visible[r] < 0 || visible[r] > out_cols || visible[r] > cap) return ORACLE_BAD_DATA;
  }
  if (num_threads < 1) num_threads = 1;
  if (num_threads > 256) num_threads = 256;
  logits_job jobs[256];
  pthread_t tids[256];
  for (int t = 0; t < num_threads; ++t) {
    logits_job J = {num_requests, rows_per_req, num_heads, head_dim, page_cols, max_pages,
                    num_pages, kv_dtype, out_cols, key_page_stride, scale_page_stride, q_dtype, q,
                    weights, kv, scales, block_table, visible, rows, num_sel, out,
                    num_threads, t, ORACLE_OK};
    jobs[t] = J;
  }
  if (num_threads == 1) {
    logits_worker(&jobs[0]);
    return jobs[0].status;
  }
  for (int t = 0; t < num_threads; ++t) pthread_create(&tids[t], NULL, logits_worker, &jobs[t]);
  int status = ORACLE_OK;
  for (int t = 0; t < num_threads; ++t) {
    pthread_join(tids[t], NULL);
    if (jobs[t].status != ORACLE_OK) status = jobs[t].status;
  }
  return status;
}

/* The same with bf16 q. */
int qsa_oracle_paged_mqa_logits(int32_t num_requests, int32_t rows_per_req, int32_t num_heads,
                                int32_t head_dim, int32_t page_cols, int32_t max_pages,
                                int32_t num_pages, int32_t kv_dtype, int64_t out_cols,
                                int64_t key_page_stride, int64_t scale_page_stride,
                                const uint16_t* q, const float* weights, const uint8_t* kv,
                                const uint8_t* scales, const int32_t* block_table,
                                const int32_t* visible, const int64_t* rows, int64_t num_sel,
                                float* out, int32_t num_threads) {
  return qsa_oracle_paged_mqa_logits_ex(num_requests, rows_per_req, num_heads, head_dim, page_cols,
                                        max_pages, num_pages, kv_dtype, out_cols, key_page_stride,
                                        scale_page_stride, 0, q, weights, kv, scales, block_table,
                                        visible, rows, num_sel, out, num_threads);
}

/* ------------------------------------------------------------------------- */
/* Top-k: sort the visible columns by (value descending, column ascending),   */
/* keep the first k, emit them in ascending column order, pad with -1.        */
/* ------------------------------------------------------------------------- */

typedef struct {
  float v;
  int32_t c;
} cand;

static int cand_cmp(const void* a, const void* b) {
  const cand* x = (const cand*)a;
  const cand* y = (const cand*)b;
  if (x->v > y->v) return -1;
  if (x->v < y->v) return 1;
  return (x->c > y->c) - (x->c < y->c);
}

static int int_cmp(const void* a, const void* b) {
  int32_t x = *(const int32_t*)a, y = *(const int32_t*)b;
  return (x > y) - (x < y);
}

typedef struct {
  const float* logits;
  int64_t num_rows, row_stride;
  const int32_t* visible;
  int32_t k;
  int32_t* out;
  int32_t num_threads, thread_id;
  int status;
} topk_job;

static void* topk_worker(void* arg) {
  topk_job* J = (topk_job*)arg;
  cand* buf = (cand*)malloc(sizeof(cand) * (size_t)(J->row_stride > 0 ? J->row_stride : 1));
  if (!buf) {
    J->status = ORACLE_BAD_ARG;
    return NULL;
  }
  for (int64_t r = J->thread_id; r < J->num_rows; r += J->num_threads) {
    const int64_t n = J->visible[r];
    int32_t* o = J->out + r * J->k;
    const float* row = J->logits + r * J->row_stride;
    if (n <= J->k) {
      for (int64_t i = 0; i < J->k; ++i) o[i] = i < n ? (int32_t)i : -1;
      continue;
    }
    for (int64_t c = 0; c < n; ++c) {
      buf[c].v = row[c];
      buf[c].c = (int32_t)c;
    }
    qsort(buf, (size_t)n, sizeof(cand), cand_cmp);
    for (int32_t i = 0; i < J->k; ++i) o[i] = buf[i].c;
    qsort(o, (size_t)J->k, sizeof(int32_t), int_cmp);
  }
  free(buf);
  return NULL;
}

int qsa_oracle_select_topk(const float* logits, int64_t num_rows, int64_t row_stride,
                           const int32_t* visible, int32_t k, int32_t* out_idx,
                           int32_t num_threads) {
  if (!logits || !visible || !out_idx || num_rows < 0 || row_stride < 1 || k < 1)
    return ORACLE_BAD_ARG;
  for (int64_t r = 0; r < num_rows; ++r)
    if (visible[r] < 0 || visible[r] > row_stride) return ORACLE_BAD_DATA;
  if (num_threads < 1) num_threads = 1;
  if (num_threads > 256) num_threads = 256;
  topk_job jobs[256];
  pthread_t tids[256];
  for (int t = 0; t < num_threads; ++t) {
    topk_job J = {logits, num_rows, row_stride, visible, k, out_idx, num_threads, t, ORACLE_OK};
    jobs[t] = J;
  }
  if (num_threads == 1) {
    topk_worker(&jobs[0]);
    return jobs[0].status;
  }
  for (int t = 0; t < num_threads; ++t) pthread_create(&tids[t], NULL, topk_worker, &jobs[t]);
  int status = ORACLE_OK;
  for (int t = 0; t < num_threads; ++t) {
    pthread_join(tids[t], NULL);
    if (jobs[t].status != ORACLE_OK) status = jobs[t].status;
  }
  return status;
}
