/*
 * Reference oracle for the paged-KV attention step — TEST INFRASTRUCTURE ONLY.
 *
 * Plain, slow, float64 CPU code that states what the step computes, written
 * from the pages' descriptions and nothing else.  Only the test suite, the
 * package smoke check and the benchmark's CPU-baseline leg may load it; the
 * product path never calls into this file, and this file shares no code,
 * header or constant with the CUDA library.
 *
 * Sources (page title, then the section on it):
 *  - "vLLM 推理全流程深度解析" (vLLM inference deep dive), the
 *    reshape_and_cache section: a token whose slot is negative is skipped;
 *    otherwise block = slot / block_size, offset = slot % block_size, and the
 *    token's [num_kv_heads, head_size] K and V rows land in
 *    cache[block, offset, :, :] of the global pool
 *    [num_blocks, block_size, num_kv_heads, head_size].
 *  - same page, the paged_attention_v1 section: the kernel looks up the
 *    request's physical blocks through block_tables, forms q.k scores,
 *    softmax-normalises them and takes the weighted sum of V.
 *  - "Tour: One forward pass", stop 3: seq_len = num_computed + query_len;
 *    stop 10: causal attention, R1 reads 541 keys, R2 130, R3 298; only the
 *    first num_actual_tokens output rows are written.
 *  - "vLLM MHA Code Path: From QKV to Paged KV Cache", section "One Path
 *    Covers MHA, GQA, and MQA": Hq divisible by Hkv, several query heads
 *    share one K/V head; "Worked Trace: One Decode Token", after step 10:
 *    the current token attends to itself, future positions are excluded.
 *
 * Readings taken where the pages are silent:
 *  - query heads are grouped contiguously: head h uses KV head h / (Hq/Hkv);
 *  - query row i of a request sits at absolute position ctx + i with
 *    ctx = seq_len - query_len, and sees keys 0 .. ctx + i (bottom-right
 *    causal alignment);
 *  - a negative slot is a pad; a slot >= num_blocks * block_size, a block id
 *    outside [0, num_blocks), seq_len < query_len, a decreasing
 *    query_start_loc or a block-table row shorter than ceil(seq_len /
 *    block_size) make the item invalid: it is skipped and reported in the
 *    returned error bits, nothing is written for it.
 *
 * Numbers: bf16 inputs are widened exactly to double; every sum, the max,
 * exp and the division run in double, in the order of the definition.
 *
 * int8 KV cache ("vLLM 推理全流程深度解析", the closing note of the
 * paged_attention section names KV-cache int8 quantisation as a decode
 * speed-up and gives no format).  Reading: one fp32 scale per cache (per
 * layer) and symmetric codes, code = clamp(rne(x / scale), -127, 127) with x
 * the bf16 value widened to fp32 and the division done in fp32 (a NaN input
 * gives code 0); the cached value is code * scale.  Attention over an int8
 * cache is the definition above with those values as K and V.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* error bits, OR-ed into the return value */
#define ORC_ERR_SLOT_RANGE 1   /* slot >= num_blocks * block_size          */
#define ORC_ERR_QSL 2          /* query_start_loc decreasing / out of rows */
#define ORC_ERR_SEQ_LEN 4      /* seq_len < query_len or negative          */
#define ORC_ERR_BT_WIDTH 8     /* block-table row too short for seq_len    */
#define ORC_ERR_BLOCK_ID 16    /* block id outside [0, num_blocks)         */

static double bf16_to_double(uint16_t bits) {
  uint32_t w = ((uint32_t)bits) << 16;
  float f;
  memcpy(&f, &w, sizeof f);
  return (double)f;
}

int oracle_num_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

void oracle_set_num_threads(int n) {
#ifdef _OPENMP
  if (n > 0) omp_set_num_threads(n);
#else
  (void)n;
#endif
}

/* Cache write.  k, v: [n_tokens, hkv, d] bf16 with a row stride (elements)
 * between tokens; caches: [num_blocks, block_size, hkv, d] bf16, contiguous.
 * Returns the OR of error bits (0 when every non-negative slot was in range). */
int oracle_write(const uint16_t *k, int64_t k_row_stride, const uint16_t *v,
                 int64_t v_row_stride, uint16_t *key_cache,
                 uint16_t *value_cache, int64_t num_blocks, int block_size,
                 int hkv, int d, const int64_t *slot_mapping,
                 int64_t n_tokens) {
  int err = 0;
  for (int64_t t = 0; t < n_tokens; ++t) {
    int64_t slot = slot_mapping[t];
    if (slot < 0) continue; /* padding token */
    int64_t block = slot / block_size;
    int64_t offset = slot % block_size;
    if (block >= num_blocks) {
      err |= ORC_ERR_SLOT_RANGE;
      continue;
    }
    for (int h = 0; h < hkv; ++h) {
      for (int e = 0; e < d; ++e) {
        int64_t dst = ((block * block_size + offset) * hkv + h) * d + e;
        key_cache[dst] = k[t * k_row_stride + (int64_t)h * d + e];
        value_cache[dst] = v[t * v_row_stride + (int64_t)h * d + e];
      }
    }
  }
  return err;
}

/* One int8 code: the reading stated in the header, in fp32. */
static int8_t quantize_int8(uint16_t bits, float scale) {
  uint32_t w = ((uint32_t)bits) << 16;
  float x;
  memcpy(&x, &w, sizeof x);
  float r = rintf(x / scale); /* fp32 division, round half to even */
  if (r != r) return 0;       /* NaN */
  if (r > 127.0f) r = 127.0f;
  if (r < -127.0f) r = -127.0f;
  return (int8_t)r;
}

/* The cache write into int8 caches: the same placement as oracle_write, each
 * element stored as its code. */
int oracle_write_int8(const uint16_t *k, int64_t k_row_stride, const uint16_t *v,
                      int64_t v_row_stride, int8_t *key_cache, int8_t *value_cache,
                      int64_t num_blocks, int block_size, int hkv, int d,
                      const int64_t *slot_mapping, int64_t n_tokens, float k_scale,
                      float v_scale) {
  int err = 0;
  for (int64_t t = 0; t < n_tokens; ++t) {
    int64_t slot = slot_mapping[t];
    if (slot < 0) continue; /* padding token */
    int64_t block = slot / block_size;
    int64_t offset = slot % block_size;
    if (block >= num_blocks) {
      err |= ORC_ERR_SLOT_RANGE;
      continue;
    }
    for (int h = 0; h < hkv; ++h) {
      for (int e = 0; e < d; ++e) {
        int64_t dst = ((block * block_size + offset) * hkv + h) * d + e;
        key_cache[dst] = quantize_int8(k[t * k_row_stride + (int64_t)h * d + e], k_scale);
        value_cache[dst] = quantize_int8(v[t * v_row_stride + (int64_t)h * d + e], v_scale);
      }
    }
  }
  return err;
}

/* Element idx of a cache: a bf16 value, or an int8 code times the scale. */
static double kv_value(const void *cache, int64_t idx, int kv_int8, double scale) {
  if (kv_int8) return (double)((const int8_t *)cache)[idx] * scale;
  return bf16_to_double(((const uint16_t *)cache)[idx]);
}

/* Checks one request against the contract; returns its error bits. */
static int check_request(const int32_t *qsl, const int32_t *seq_lens,
                         const int32_t *block_table, int64_t bt_row_stride,
                         int64_t bt_width, int64_t num_blocks, int block_size,
                         int64_t n_rows, int r) {
  int32_t q0 = qsl[r], q1 = qsl[r + 1], L = seq_lens[r];
  if (q0 < 0 || q1 < q0 || q1 > n_rows) return ORC_ERR_QSL;
  if (L < 0 || L < q1 - q0) return ORC_ERR_SEQ_LEN;
  int64_t nb = ((int64_t)L + block_size - 1) / block_size;
  if (nb > bt_width) return ORC_ERR_BT_WIDTH;
  for (int64_t b = 0; b < nb; ++b) {
    int32_t id = block_table[(int64_t)r * bt_row_stride + b];
    if (id < 0 || id >= num_blocks) return ORC_ERR_BLOCK_ID;
  }
  return 0;
}

/* One output row: request r, query row i (absolute position ctx + i),
 * query head h.  scores is scratch of at least ctx + i + 1 doubles. */
static void attend_one(const uint16_t *q, int64_t q_row_stride, int hq,
                       const void *key_cache, const void *value_cache, int kv_int8,
                       double k_scale, double v_scale,
                       int block_size, int hkv, int d, const int32_t *qsl,
                       const int32_t *seq_lens, const int32_t *block_table,
                       int64_t bt_row_stride, int r, int64_t i, int h,
                       double scale, double *scores, double *out_row) {
  int64_t q0 = qsl[r];
  int64_t n = (int64_t)qsl[r + 1] - q0;
  int64_t ctx = (int64_t)seq_lens[r] - n;
  int group = hq / hkv;
  int g = h / group;
  int64_t last = ctx + i; /* highest visible key position */
  const uint16_t *qrow = q + (q0 + i) * q_row_stride + (int64_t)h * d;

  double m = -INFINITY;
  for (int64_t j = 0; j <= last; ++j) {
    int64_t block = block_table[(int64_t)r * bt_row_stride + j / block_size];
    int64_t offset = j % block_size;
    int64_t krow = ((block * block_size + offset) * hkv + g) * d;
    double s = 0.0;
    for (int e = 0; e < d; ++e)
      s += bf16_to_double(qrow[e]) * kv_value(key_cache, krow + e, kv_int8, k_scale);
    s *= scale;
    scores[j] = s;
    if (s > m) m = s;
  }
  double l = 0.0;
  for (int64_t j = 0; j <= last; ++j) {
    scores[j] = exp(scores[j] - m);
    l += scores[j];
  }
  for (int e = 0; e < d; ++e) out_row[e] = 0.0;
  for (int64_t j = 0; j <= last; ++j) {
    int64_t block = block_table[(int64_t)r * bt_row_stride + j / block_size];
    int64_t offset = j % block_size;
    int64_t vrow = ((block * block_size + offset) * hkv + g) * d;
    double p = scores[j] / l;
    for (int e = 0; e < d; ++e)
      out_row[e] += p * kv_value(value_cache, vrow + e, kv_int8, v_scale);
  }
}

/* Attention over the paged cache for a packed batch.
 * q: [n_rows, hq, d] bf16 with row stride q_row_stride (elements);
 * caches: [num_blocks, block_size, hkv, d] bf16;
 * query_start_loc: int32 [num_reqs + 1]; seq_lens: int32 [num_reqs];
 * block_table: int32 [num_reqs, bt_width] with row stride bt_row_stride;
 * out: double [n_rows, hq, d] with row stride out_row_stride; rows that no
 * valid request covers are left as they are.  Returns the OR of the error
 * bits of the requests that were skipped. */
static int attention_impl(const uint16_t *q, int64_t q_row_stride, int64_t n_rows,
                          int hq, const void *key_cache, const void *value_cache,
                          int kv_int8, double k_scale, double v_scale, int64_t num_blocks,
                          int block_size, int hkv, int d,
                          const int32_t *query_start_loc, const int32_t *seq_lens,
                          const int32_t *block_table, int64_t bt_row_stride,
                          int64_t bt_width, int num_reqs, double scale, double *out,
                          int64_t out_row_stride) {
  if (hkv <= 0 || hq % hkv != 0) return -1;
  int err = 0;
  int *valid = (int *)malloc(sizeof(int) * (num_reqs > 0 ? num_reqs : 1));
  int64_t max_len = 1;
  for (int r = 0; r < num_reqs; ++r) {
    int e = check_request(query_start_loc, seq_lens, block_table,
                          bt_row_stride, bt_width, num_blocks, block_size,
                          n_rows, r);
    valid[r] = (e == 0);
    err |= e;
    if (e == 0 && seq_lens[r] > max_len) max_len = seq_lens[r];
  }
  int64_t tasks = (int64_t)num_reqs * hq;
#pragma omp parallel
  {
    double *scores = (double *)malloc(sizeof(double) * (size_t)max_len);
#pragma omp for schedule(dynamic, 1)
    for (int64_t task = 0; task < tasks; ++task) {
      int r = (int)(task / hq);
      int h = (int)(task % hq);
      if (!valid[r]) continue;
      int64_t n = (int64_t)query_start_loc[r + 1] - query_start_loc[r];
      for (int64_t i = 0; i < n; ++i) {
        double *orow = out + ((int64_t)query_start_loc[r] + i) * out_row_stride +
                       (int64_t)h * d;
        attend_one(q, q_row_stride, hq, key_cache, value_cache, kv_int8, k_scale,
                   v_scale, block_size, hkv, d, query_start_loc, seq_lens,
                   block_table, bt_row_stride, r, i, h, scale, scores, orow);
      }
    }
    free(scores);
  }
  free(valid);
  return err;
}

int oracle_attention(const uint16_t *q, int64_t q_row_stride, int64_t n_rows,
                     int hq, const uint16_t *key_cache,
                     const uint16_t *value_cache, int64_t num_blocks,
                     int block_size, int hkv, int d,
                     const int32_t *query_start_loc, const int32_t *seq_lens,
                     const int32_t *block_table, int64_t bt_row_stride,
                     int64_t bt_width, int num_reqs, double scale, double *out,
                     int64_t out_row_stride) {
  return attention_impl(q, q_row_stride, n_rows, hq, key_cache, value_cache, 0, 1.0, 1.0,
                        num_blocks, block_size, hkv, d, query_start_loc, seq_lens,
                        block_table, bt_row_stride, bt_width, num_reqs, scale, out,
                        out_row_stride);
}

/* The same attention over int8 caches: K = code * k_scale, V = code * v_scale. */
int oracle_attention_int8(const uint16_t *q, int64_t q_row_stride, int64_t n_rows,
                          int hq, const int8_t *key_cache, const int8_t *value_cache,
                          double k_scale, double v_scale, int64_t num_blocks,
                          int block_size, int hkv, int d,
                          const int32_t *query_start_loc, const int32_t *seq_lens,
                          const int32_t *block_table, int64_t bt_row_stride,
                          int64_t bt_width, int num_reqs, double scale, double *out,
                          int64_t out_row_stride) {
  return attention_impl(q, q_row_stride, n_rows, hq, key_cache, value_cache, 1, k_scale,
                        v_scale, num_blocks, block_size, hkv, d, query_start_loc,
                        seq_lens, block_table, bt_row_stride, bt_width, num_reqs, scale,
                        out, out_row_stride);
}

/* The same definition evaluated only at chosen (token row, query head)
 * pairs, for checks at sizes where the full batch would take too long.
 * rows[s], heads[s] select sample s; out: double [n_samples, d].  A sample
 * whose row belongs to no valid request is filled with NaN. */
int oracle_attention_sampled(const uint16_t *q, int64_t q_row_stride,
                             int64_t n_rows, int hq, const uint16_t *key_cache,
                             const uint16_t *value_cache, int64_t num_blocks,
                             int block_size, int hkv, int d,
                             const int32_t *query_start_loc,
                             const int32_t *seq_lens,
                             const int32_t *block_table, int64_t bt_row_stride,
                             int64_t bt_width, int num_reqs, double scale,
                             const int64_t *rows, const int32_t *heads,
                             int64_t n_samples, double *out) {
  if (hkv <= 0 || hq % hkv != 0) return -1;
  int err = 0;
  for (int r = 0; r < num_reqs; ++r)
    err |= check_request(query_start_loc, seq_lens, block_table, bt_row_stride,
                         bt_width, num_blocks, block_size, n_rows, r);
#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t s = 0; s < n_samples; ++s) {
    double *orow = out + s * d;
    int req = -1;
    for (int r = 0; r < num_reqs; ++r) {
      if (rows[s] >= query_start_loc[r] && rows[s] < query_start_loc[r + 1]) {
        req = r;
        break;
      }
    }
    if (req < 0 || heads[s] < 0 || heads[s] >= hq ||
        check_request(query_start_loc, seq_lens, block_table, bt_row_stride,
                      bt_width, num_blocks, block_size, n_rows, req) != 0) {
      for (int e = 0; e < d; ++e) orow[e] = NAN;
      continue;
    }
    double *scores = (double *)malloc(sizeof(double) * (size_t)(seq_lens[req] + 1));
    attend_one(q, q_row_stride, hq, key_cache, value_cache, 0, 1.0, 1.0, block_size, hkv,
               d, query_start_loc, seq_lens, block_table, bt_row_stride, req,
               rows[s] - query_start_loc[req], heads[s], scale, scores, orow);
    free(scores);
  }
  return err;
}
