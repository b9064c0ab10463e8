/*
 * attn_oracle.c -- fp64 CPU oracle for BSR paged-KV attention.
 *
 * TEST INFRASTRUCTURE ONLY (tests, smoke check, CPU-baseline timing); the
 * library path never links it. Plain single-threaded C, no BLAS, no blocking:
 * every output is the textbook definition evaluated in double precision.
 *
 * Sources (FlashInfer paper digest, modb.pro page):
 *  - "统一的 KV 缓存存储格式": the KV cache is a block-sparse row matrix; rows are
 *    requests, blocks are pages of a configurable size, and an index array maps
 *    logical blocks to physical pages. Its formula did not survive extraction;
 *    the reading used is in bsr_token_ptr() below.
 *  - "可组合格式" in the same section: several block-sparse formats take part in
 *    one attention computation; their partial states are combined by
 *    log-sum-exp merging (oracle_merge_states).
 * Attention itself is softmax(q K^T * sm_scale) V (yeyulingfeng.com page,
 * "FlashAttention 的遗产": the tiled form changes IO only, not the result).
 *
 * Parity pins: see the header comment of attn_oracle.h.
 */
#include "attn_oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>

double oracle_widen(uint16_t bits, int32_t dtype) {
  if (dtype == ORACLE_BF16) {
    /* bfloat16 is the top half of an IEEE binary32 word. */
    uint32_t u = (uint32_t)bits << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
  }
  /* IEEE binary16: 1 sign, 5 exponent (bias 15), 10 fraction bits. */
  int sign = bits >> 15;
  int e = (bits >> 10) & 0x1f;
  int m = bits & 0x3ff;
  double v;
  if (e == 0)
    v = ldexp((double)m, -24);               /* subnormal: m * 2^-24 */
  else if (e == 31)
    v = m ? NAN : INFINITY;
  else
    v = ldexp((double)(m | 0x400), e - 25);  /* (1024 + m) * 2^(e-15-10) */
  return sign ? -v : v;
}

double oracle_round(double v, int32_t dtype) {
  if (v == 0.0 || isnan(v) || isinf(v)) return v;
  /* significand bits (with the implicit one) and the smallest normal exponent */
  const int bits = dtype == ORACLE_BF16 ? 8 : 11;
  const int emin = dtype == ORACLE_BF16 ? -126 : -14;
  const double vmax = dtype == ORACLE_BF16 ? 0x1.fep127 : 65504.0;
  int e;
  frexp(v, &e); /* v = m 2^e, 0.5 <= |m| < 1: the leading bit has weight 2^(e-1) */
  int q = e - bits;            /* weight of the last kept bit */
  if (q < emin - bits + 1) q = emin - bits + 1; /* subnormals: fixed quantum */
  double r = ldexp(nearbyint(ldexp(v, -q)), q); /* default mode: ties to even */
  if (fabs(r) > vmax) return v > 0 ? INFINITY : -INFINITY;
  return r;
}

/* Rotary embedding of one D-vector at table row `pos` (see the header). */
static void rope_rotate(double* x, int32_t head_dim, const float* rope_cos,
                        const float* rope_sin, int64_t pos, int32_t dtype) {
  const int32_t half = head_dim / 2;
  for (int32_t d = 0; d < half; ++d) {
    const double c = rope_cos[pos * half + d], s = rope_sin[pos * half + d];
    const double a = x[d], b = x[d + half];
    x[d] = oracle_round(a * c - b * s, dtype);
    x[d + half] = oracle_round(b * c + a * s, dtype);
  }
}

/* Number of logical KV tokens of request r (BSR reading, see header). */
static int64_t bsr_kv_len(const int32_t* kv_indptr, const int32_t* last_page_len,
                          int32_t page_size, int32_t r) {
  int64_t n = (int64_t)kv_indptr[r + 1] - kv_indptr[r];
  if (n <= 0) return 0;
  return (n - 1) * page_size + last_page_len[r];
}

/* Address of the D-vector of logical token t, kv head hk, of request r. */
static const uint16_t* bsr_token_ptr(const uint16_t* pool, int32_t layout,
                                     const int32_t* kv_indptr,
                                     const int32_t* kv_indices, int32_t page_size,
                                     int32_t num_kv_heads, int32_t head_dim,
                                     int32_t r, int64_t t, int32_t hk) {
  int64_t page = kv_indices[kv_indptr[r] + t / page_size];
  int64_t slot = t % page_size;
  int64_t row;
  if (layout == ORACLE_HND)
    row = (page * num_kv_heads + hk) * page_size + slot;
  else
    row = (page * page_size + slot) * num_kv_heads + hk;
  return pool + row * head_dim;
}

static int32_t check_args(const int32_t* qo_indptr, int64_t num_pages,
                          int32_t layout, const int32_t* kv_indptr,
                          const int32_t* kv_indices, const int32_t* last_page_len,
                          int32_t batch, int32_t page_size, int32_t num_qo_heads,
                          int32_t num_kv_heads, int32_t head_dim, int32_t dtype) {
  if (batch < 0 || page_size <= 0 || num_qo_heads <= 0 || num_kv_heads <= 0 ||
      head_dim <= 0)
    return -1;
  if (num_qo_heads % num_kv_heads != 0) return -2;
  if (dtype != ORACLE_F16 && dtype != ORACLE_BF16) return -3;
  if (layout != ORACLE_HND && layout != ORACLE_NHD) return -4;
  for (int32_t r = 0; r < batch; ++r) {
    int32_t n = kv_indptr[r + 1] - kv_indptr[r];
    if (n < 0) return -5;
    if (n > 0 && (last_page_len[r] < 1 || last_page_len[r] > page_size)) return -6;
    for (int32_t k = kv_indptr[r]; k < kv_indptr[r + 1]; ++k)
      if (kv_indices[k] < 0 || kv_indices[k] >= num_pages) return -7;
    if (qo_indptr) {
      int64_t qo_len = (int64_t)qo_indptr[r + 1] - qo_indptr[r];
      if (qo_len < 0) return -8;
    }
  }
  return 0;
}

/*
 * One output row, restricted to logical kv positions [kv_lo, kv_hi) of the
 * visible set. Two passes: logits first (exact max), then the weighted sums,
 * all in logical kv order.
 */
static void attention_row(const uint16_t* q, const int32_t* qo_indptr,
                          const uint16_t* k_pool, const uint16_t* v_pool,
                          int32_t layout, const int32_t* kv_indptr,
                          const int32_t* kv_indices, const int32_t* last_page_len,
                          int32_t page_size, int32_t num_qo_heads,
                          int32_t num_kv_heads, int32_t head_dim, int32_t dtype,
                          int32_t causal, double sm_scale, int32_t r, int32_t i,
                          int32_t h, int64_t kv_lo, int64_t kv_hi, double* x_buf,
                          double* q_buf, const float* rope_cos, const float* rope_sin,
                          double* o, double* lse) {
  const int32_t group = num_qo_heads / num_kv_heads;
  const int32_t hk = h / group;
  const int64_t qo_start = qo_indptr ? qo_indptr[r] : r;
  const int64_t qo_len = qo_indptr ? (int64_t)qo_indptr[r + 1] - qo_indptr[r] : 1;
  const int64_t kv_len = bsr_kv_len(kv_indptr, last_page_len, page_size, r);

  /* Visible set J = [0, vis): causal rows see j <= kv_len - qo_len + i. */
  int64_t vis = kv_len;
  if (causal) {
    int64_t lim = kv_len - qo_len + i + 1;
    if (lim < vis) vis = lim;
  }
  if (vis < 0) vis = 0;
  int64_t lo = kv_lo < 0 ? 0 : kv_lo;
  int64_t hi = kv_hi < vis ? kv_hi : vis;

  const uint16_t* qrow = q + ((qo_start + i) * num_qo_heads + h) * head_dim;
  for (int32_t d = 0; d < head_dim; ++d) q_buf[d] = oracle_widen(qrow[d], dtype);
  double* k_buf = q_buf + head_dim; /* rotated key (RoPE only) */

  for (int32_t d = 0; d < head_dim; ++d) o[d] = 0.0;
  if (hi <= lo) {
    *lse = -INFINITY;
    return;
  }
  if (rope_cos) rope_rotate(q_buf, head_dim, rope_cos, rope_sin, kv_len - qo_len + i, dtype);

  double m = -INFINITY;
  for (int64_t j = lo; j < hi; ++j) {
    const uint16_t* krow = bsr_token_ptr(k_pool, layout, kv_indptr, kv_indices,
                                         page_size, num_kv_heads, head_dim, r, j, hk);
    double dot = 0.0;
    if (rope_cos) {
      for (int32_t d = 0; d < head_dim; ++d) k_buf[d] = oracle_widen(krow[d], dtype);
      rope_rotate(k_buf, head_dim, rope_cos, rope_sin, j, dtype);
      for (int32_t d = 0; d < head_dim; ++d) dot += q_buf[d] * k_buf[d];
    } else {
      for (int32_t d = 0; d < head_dim; ++d) dot += q_buf[d] * oracle_widen(krow[d], dtype);
    }
    double x = sm_scale * dot;
    x_buf[j - lo] = x;
    if (x > m) m = x;
  }
  double l = 0.0;
  for (int64_t j = lo; j < hi; ++j) {
    double p = exp(x_buf[j - lo] - m);
    l += p;
    const uint16_t* vrow = bsr_token_ptr(v_pool, layout, kv_indptr, kv_indices,
                                         page_size, num_kv_heads, head_dim, r, j, hk);
    for (int32_t d = 0; d < head_dim; ++d) o[d] += p * oracle_widen(vrow[d], dtype);
  }
  for (int32_t d = 0; d < head_dim; ++d) o[d] /= l;
  *lse = m + log(l);
}

static int64_t max_kv_len(const int32_t* kv_indptr, const int32_t* last_page_len,
                          int32_t page_size, int32_t batch) {
  int64_t mx = 1;
  for (int32_t r = 0; r < batch; ++r) {
    int64_t n = bsr_kv_len(kv_indptr, last_page_len, page_size, r);
    if (n > mx) mx = n;
  }
  return mx;
}

int32_t oracle_attention_row(const uint16_t* q, const int32_t* qo_indptr,
                             const uint16_t* k_pool, const uint16_t* v_pool,
                             int64_t num_pages, int32_t layout,
                             const int32_t* kv_indptr, const int32_t* kv_indices,
                             const int32_t* last_page_len, int32_t batch,
                             int32_t page_size, int32_t num_qo_heads,
                             int32_t num_kv_heads, int32_t head_dim,
                             int32_t dtype, int32_t causal, double sm_scale,
                             int32_t r, int32_t i, int32_t h,
                             double* o, double* lse) {
  if (r < 0 || r >= batch || h < 0 || h >= num_qo_heads || i < 0) return -1;
  int32_t rc = check_args(qo_indptr, num_pages, layout, kv_indptr, kv_indices,
                          last_page_len, batch, page_size, num_qo_heads,
                          num_kv_heads, head_dim, dtype);
  if (rc) return rc;
  int64_t qo_len = qo_indptr ? (int64_t)qo_indptr[r + 1] - qo_indptr[r] : 1;
  if (i >= qo_len) return -1;
  int64_t kv_len = bsr_kv_len(kv_indptr, last_page_len, page_size, r);
  double* x_buf = (double*)malloc(sizeof(double) * (size_t)(kv_len > 0 ? kv_len : 1));
  double* q_buf = (double*)malloc(sizeof(double) * 2 * (size_t)head_dim);
  if (!x_buf || !q_buf) {
    free(x_buf);
    free(q_buf);
    return -100;
  }
  attention_row(q, qo_indptr, k_pool, v_pool, layout, kv_indptr, kv_indices,
                last_page_len, page_size, num_qo_heads, num_kv_heads, head_dim,
                dtype, causal, sm_scale, r, i, h, 0, INT64_MAX, x_buf, q_buf, NULL, NULL,
                o, lse);
  free(x_buf);
  free(q_buf);
  return 0;
}

int32_t oracle_attention_row_rope(const uint16_t* q, const int32_t* qo_indptr,
                                  const uint16_t* k_pool, const uint16_t* v_pool,
                                  int64_t num_pages, int32_t layout,
                                  const int32_t* kv_indptr, const int32_t* kv_indices,
                                  const int32_t* last_page_len, int32_t batch,
                                  int32_t page_size, int32_t num_qo_heads,
                                  int32_t num_kv_heads, int32_t head_dim,
                                  int32_t dtype, int32_t causal, double sm_scale,
                                  const float* rope_cos, const float* rope_sin,
                                  int64_t rope_max_pos, int32_t r, int32_t i, int32_t h,
                                  double* o, double* lse) {
  if (!rope_cos || !rope_sin || head_dim % 2 != 0) return -1;
  if (r < 0 || r >= batch || h < 0 || h >= num_qo_heads || i < 0) return -1;
  int32_t rc = check_args(qo_indptr, num_pages, layout, kv_indptr, kv_indices,
                          last_page_len, batch, page_size, num_qo_heads,
                          num_kv_heads, head_dim, dtype);
  if (rc) return rc;
  int64_t qo_len = qo_indptr ? (int64_t)qo_indptr[r + 1] - qo_indptr[r] : 1;
  if (i >= qo_len) return -1;
  int64_t kv_len = bsr_kv_len(kv_indptr, last_page_len, page_size, r);
  /* this row's key positions (< kv_len) and query position must have table
     rows, and the query position must be >= 0 */
  if (kv_len > rope_max_pos || (kv_len > 0 && kv_len < qo_len)) return -9;
  double* x_buf = (double*)malloc(sizeof(double) * (size_t)(kv_len > 0 ? kv_len : 1));
  double* q_buf = (double*)malloc(sizeof(double) * 2 * (size_t)head_dim);
  if (!x_buf || !q_buf) {
    free(x_buf);
    free(q_buf);
    return -100;
  }
  attention_row(q, qo_indptr, k_pool, v_pool, layout, kv_indptr, kv_indices,
                last_page_len, page_size, num_qo_heads, num_kv_heads, head_dim,
                dtype, causal, sm_scale, r, i, h, 0, INT64_MAX, x_buf, q_buf, rope_cos,
                rope_sin, o, lse);
  free(x_buf);
  free(q_buf);
  return 0;
}

static int32_t batch_attention(const uint16_t* q, const int32_t* qo_indptr,
                               const uint16_t* k_pool, const uint16_t* v_pool,
                               int64_t num_pages, int32_t layout,
                               const int32_t* kv_indptr, const int32_t* kv_indices,
                               const int32_t* last_page_len, int32_t batch,
                               int32_t page_size, int32_t num_qo_heads,
                               int32_t num_kv_heads, int32_t head_dim,
                               int32_t dtype, int32_t causal, double sm_scale,
                               const int32_t* kv_begin, const int32_t* kv_end,
                               const float* rope_cos, const float* rope_sin,
                               double* o, double* lse) {
  int32_t rc = check_args(qo_indptr, num_pages, layout, kv_indptr, kv_indices,
                          last_page_len, batch, page_size, num_qo_heads,
                          num_kv_heads, head_dim, dtype);
  if (rc) return rc;
  int64_t mx = max_kv_len(kv_indptr, last_page_len, page_size, batch);
  double* x_buf = (double*)malloc(sizeof(double) * (size_t)mx);
  double* q_buf = (double*)malloc(sizeof(double) * 2 * (size_t)head_dim);
  if (!x_buf || !q_buf) {
    free(x_buf);
    free(q_buf);
    return -100;
  }
  for (int32_t r = 0; r < batch; ++r) {
    int64_t qo_start = qo_indptr ? qo_indptr[r] : r;
    int64_t qo_len = qo_indptr ? (int64_t)qo_indptr[r + 1] - qo_indptr[r] : 1;
    int64_t lo = kv_begin ? kv_begin[r] : 0;
    int64_t hi = kv_end ? kv_end[r] : INT64_MAX;
    for (int64_t i = 0; i < qo_len; ++i) {
      for (int32_t h = 0; h < num_qo_heads; ++h) {
        int64_t row = (qo_start + i) * num_qo_heads + h;
        attention_row(q, qo_indptr, k_pool, v_pool, layout, kv_indptr, kv_indices,
                      last_page_len, page_size, num_qo_heads, num_kv_heads,
                      head_dim, dtype, causal, sm_scale, r, (int32_t)i, h, lo, hi,
                      x_buf, q_buf, rope_cos, rope_sin, o + row * head_dim, lse + row);
      }
    }
  }
  free(x_buf);
  free(q_buf);
  return 0;
}

int32_t oracle_batch_attention(const uint16_t* q, const int32_t* qo_indptr,
                               const uint16_t* k_pool, const uint16_t* v_pool,
                               int64_t num_pages, int32_t layout,
                               const int32_t* kv_indptr, const int32_t* kv_indices,
                               const int32_t* last_page_len, int32_t batch,
                               int32_t page_size, int32_t num_qo_heads,
                               int32_t num_kv_heads, int32_t head_dim,
                               int32_t dtype, int32_t causal, double sm_scale,
                               const int32_t* kv_begin, const int32_t* kv_end,
                               double* o, double* lse) {
  return batch_attention(q, qo_indptr, k_pool, v_pool, num_pages, layout, kv_indptr,
                         kv_indices, last_page_len, batch, page_size, num_qo_heads,
                         num_kv_heads, head_dim, dtype, causal, sm_scale, kv_begin,
                         kv_end, NULL, NULL, o, lse);
}

int32_t oracle_batch_attention_rope(const uint16_t* q, const int32_t* qo_indptr,
                                    const uint16_t* k_pool, const uint16_t* v_pool,
                                    int64_t num_pages, int32_t layout,
                                    const int32_t* kv_indptr, const int32_t* kv_indices,
                                    const int32_t* last_page_len, int32_t batch,
                                    int32_t page_size, int32_t num_qo_heads,
                                    int32_t num_kv_heads, int32_t head_dim,
                                    int32_t dtype, int32_t causal, double sm_scale,
                                    const float* rope_cos, const float* rope_sin,
                                    int64_t rope_max_pos, double* o, double* lse) {
  if (!rope_cos || !rope_sin || head_dim % 2 != 0) return -1;
  /* every key position (< kv_len) and query position (kv_len - qo_len + i
     <= kv_len - 1) must have a table row */
  int64_t mx = max_kv_len(kv_indptr, last_page_len, page_size, batch);
  if (batch > 0 && mx > rope_max_pos) return -9;
  for (int32_t r = 0; r < batch; ++r) {
    int64_t kv_len = bsr_kv_len(kv_indptr, last_page_len, page_size, r);
    int64_t qo_len = qo_indptr ? (int64_t)qo_indptr[r + 1] - qo_indptr[r] : 1;
    if (kv_len > 0 && kv_len < qo_len) return -9; /* query positions must be >= 0 */
  }
  return batch_attention(q, qo_indptr, k_pool, v_pool, num_pages, layout, kv_indptr,
                         kv_indices, last_page_len, batch, page_size, num_qo_heads,
                         num_kv_heads, head_dim, dtype, causal, sm_scale, NULL, NULL,
                         rope_cos, rope_sin, o, lse);
}

double oracle_widen_e4m3(uint8_t bits) {
  /* FP8 E4M3 (the "fn" encoding: no infinities, S.1111.111 is NaN):
     1 sign, 4 exponent (bias 7), 3 fraction bits. */
  int sign = bits >> 7;
  int e = (bits >> 3) & 0xf;
  int m = bits & 7;
  double v;
  if (e == 15 && m == 7)
    v = NAN;
  else if (e == 0)
    v = ldexp((double)m, -9);             /* subnormal: (m / 8) * 2^-6 */
  else
    v = ldexp((double)(8 + m), e - 10);   /* (1 + m / 8) * 2^(e - 7) */
  return sign ? -v : v;
}

/*
 * One row with an FP8 (E4M3) K/V cache: the stored byte of kv head hk means
 * widen(byte) * k_scale[hk] (keys) or * v_scale[hk] (values); q is 16-bit.
 * Same definition and order as attention_row.
 */
static void attention_row_fp8(const uint16_t* q, const int32_t* qo_indptr,
                              const uint8_t* k_pool, const uint8_t* v_pool, int32_t layout,
                              const int32_t* kv_indptr, const int32_t* kv_indices,
                              const int32_t* last_page_len, int32_t page_size,
                              int32_t num_qo_heads, int32_t num_kv_heads, int32_t head_dim,
                              int32_t q_dtype, int32_t causal, double sm_scale,
                              const float* k_scale, const float* v_scale, int32_t r,
                              int32_t i, int32_t h, double* x_buf, double* q_buf, double* o,
                              double* lse) {
  const int32_t group = num_qo_heads / num_kv_heads;
  const int32_t hk = h / group;
  const int64_t qo_start = qo_indptr ? qo_indptr[r] : r;
  const int64_t qo_len = qo_indptr ? (int64_t)qo_indptr[r + 1] - qo_indptr[r] : 1;
  const int64_t kv_len = bsr_kv_len(kv_indptr, last_page_len, page_size, r);
  int64_t vis = kv_len;
  if (causal) {
    int64_t lim = kv_len - qo_len + i + 1;
    if (lim < vis) vis = lim;
  }
  if (vis < 0) vis = 0;
  const uint16_t* qrow = q + ((qo_start + i) * num_qo_heads + h) * head_dim;
  for (int32_t d = 0; d < head_dim; ++d) q_buf[d] = oracle_widen(qrow[d], q_dtype);
  for (int32_t d = 0; d < head_dim; ++d) o[d] = 0.0;
  if (vis <= 0) {
    *lse = -INFINITY;
    return;
  }
  const double ks = k_scale[hk], vs = v_scale[hk];
  double m = -INFINITY;
  for (int64_t j = 0; j < vis; ++j) {
    int64_t page = kv_indices[kv_indptr[r] + j / page_size];
    int64_t slot = j % page_size;
    int64_t row = layout == ORACLE_HND ? (page * num_kv_heads + hk) * page_size + slot
                                       : (page * page_size + slot) * num_kv_heads + hk;
    const uint8_t* krow = k_pool + row * head_dim;
    double dot = 0.0;
    for (int32_t d = 0; d < head_dim; ++d) dot += q_buf[d] * (oracle_widen_e4m3(krow[d]) * ks);
    double x = sm_scale * dot;
    x_buf[j] = x;
    if (x > m) m = x;
  }
  double l = 0.0;
  for (int64_t j = 0; j < vis; ++j) {
    int64_t page = kv_indices[kv_indptr[r] + j / page_size];
    int64_t slot = j % page_size;
    int64_t row = layout == ORACLE_HND ? (page * num_kv_heads + hk) * page_size + slot
                                       : (page * page_size + slot) * num_kv_heads + hk;
    const uint8_t* vrow = v_pool + row * head_dim;
    double p = exp(x_buf[j] - m);
    l += p;
    for (int32_t d = 0; d < head_dim; ++d) o[d] += p * (oracle_widen_e4m3(vrow[d]) * vs);
  }
  for (int32_t d = 0; d < head_dim; ++d) o[d] /= l;
  *lse = m + log(l);
}

int32_t oracle_batch_attention_fp8kv(const uint16_t* q, const int32_t* qo_indptr,
                                     const uint8_t* k_pool, const uint8_t* v_pool,
                                     int64_t num_pages, int32_t layout,
                                     const int32_t* kv_indptr, const int32_t* kv_indices,
                                     const int32_t* last_page_len, int32_t batch,
                                     int32_t page_size, int32_t num_qo_heads,
                                     int32_t num_kv_heads, int32_t head_dim, int32_t q_dtype,
                                     int32_t causal, double sm_scale, const float* k_scale,
                                     const float* v_scale, double* o, double* lse) {
  if (!k_scale || !v_scale) return -1;
  int32_t rc = check_args(qo_indptr, num_pages, layout, kv_indptr, kv_indices,
                          last_page_len, batch, page_size, num_qo_heads,
                          num_kv_heads, head_dim, q_dtype);
  if (rc) return rc;
  int64_t mx = max_kv_len(kv_indptr, last_page_len, page_size, batch);
  double* x_buf = (double*)malloc(sizeof(double) * (size_t)mx);
  double* q_buf = (double*)malloc(sizeof(double) * (size_t)head_dim);
  if (!x_buf || !q_buf) {
    free(x_buf);
    free(q_buf);
    return -100;
  }
  for (int32_t r = 0; r < batch; ++r) {
    int64_t qo_start = qo_indptr ? qo_indptr[r] : r;
    int64_t qo_len = qo_indptr ? (int64_t)qo_indptr[r + 1] - qo_indptr[r] : 1;
    for (int64_t i = 0; i < qo_len; ++i)
      for (int32_t h = 0; h < num_qo_heads; ++h) {
        int64_t row = (qo_start + i) * num_qo_heads + h;
        attention_row_fp8(q, qo_indptr, k_pool, v_pool, layout, kv_indptr, kv_indices,
                          last_page_len, page_size, num_qo_heads, num_kv_heads, head_dim,
                          q_dtype, causal, sm_scale, k_scale, v_scale, r, (int32_t)i, h,
                          x_buf, q_buf, o + row * head_dim, lse + row);
      }
  }
  free(x_buf);
  free(q_buf);
  return 0;
}

void oracle_merge_states(const double* o_in, const double* lse_in,
                         int32_t n_states, int64_t rows, int32_t head_dim,
                         double* o_out, double* lse_out) {
  for (int64_t row = 0; row < rows; ++row) {
    double m = -INFINITY;
    for (int32_t s = 0; s < n_states; ++s) {
      double v = lse_in[(int64_t)s * rows + row];
      if (v > m) m = v;
    }
    double* out = o_out + row * head_dim;
    for (int32_t d = 0; d < head_dim; ++d) out[d] = 0.0;
    if (m == -INFINITY) {
      lse_out[row] = -INFINITY;
      continue;
    }
    double sum = 0.0;
    for (int32_t s = 0; s < n_states; ++s)
      sum += exp(lse_in[(int64_t)s * rows + row] - m);
    double lse = m + log(sum);
    for (int32_t s = 0; s < n_states; ++s) {
      double w = exp(lse_in[(int64_t)s * rows + row] - lse);
      const double* in = o_in + ((int64_t)s * rows + row) * head_dim;
      for (int32_t d = 0; d < head_dim; ++d) out[d] += w * in[d];
    }
    lse_out[row] = lse;
  }
}
