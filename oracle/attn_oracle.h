/*
 * attn_oracle.h -- fp64 CPU oracle for attention over a block-sparse-row (BSR)
 * paged KV cache.
 *
 * TEST INFRASTRUCTURE ONLY. Nothing in the library path includes, links or
 * calls this code; only the tests, the package's smoke check and the
 * benchmark's CPU-baseline leg do. It shares no source with the CUDA path.
 *
 * What it computes follows "FlashInfer: Efficient and Customizable Attention
 * Engine for LLM Inference Serving" (arXiv 2501.01005) as summarised on the
 * modb.pro digest page, section "统一的 KV 缓存存储格式" (unified KV-cache storage
 * format: the BSR layout, composable formats) and "动态负载均衡调度" (split work
 * units), together with the IO-aware tiled softmax attention described on the
 * yeyulingfeng.com page, section "FlashAttention 的遗产". The tiling there is
 * an IO optimisation only; the oracle computes the untiled definition.
 *
 * Readings taken where the pages are silent:
 *  - the BSR index formula is missing from the digest: logical token t of
 *    request r lives in page kv_indices[kv_indptr[r] + t / P], slot t % P;
 *    kv_len_r = (n_r - 1) * P + last_page_len[r] with n_r pages (0 if n_r = 0);
 *  - grouped-query heads: query head h reads kv head h / (Hq / Hk);
 *  - LSE is the natural log-sum-exp of the scaled logits;
 *  - causal masking is aligned to the end of the sequence: query row i of a
 *    request with qo_len rows sees kv positions j <= kv_len - qo_len + i.
 *
 * Parity is pinned (tests/test_oracle_pins.py) by a library routine
 * (torch scaled_dot_product_attention in float64 on CPU), closed forms and the
 * invariants the pages imply (page-size / physical-order independence, split
 * + merge = unsplit, shared prefix + suffix = flat layout).
 */
#ifndef ATTN_ORACLE_H
#define ATTN_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Storage element types of q and the K/V pools (raw 16-bit words). */
enum { ORACLE_F16 = 0, ORACLE_BF16 = 1 };
/* Pool layouts: HND = [num_pages, Hk, P, D], NHD = [num_pages, P, Hk, D]. */
enum { ORACLE_HND = 0, ORACLE_NHD = 1 };

/* Exact widening of one stored 16-bit value to double. */
double oracle_widen(uint16_t bits, int32_t dtype);

/* Exact widening of one FP8 E4M3 byte (no infinities; 0x7f / 0xff are NaN). */
double oracle_widen_e4m3(uint8_t bits);

/*
 * All rows with an FP8 (E4M3) K/V cache and per-kv-head scales: the stored
 * byte b of kv head hk stands for widen_e4m3(b) * k_scale[hk] (keys) or
 * widen_e4m3(b) * v_scale[hk] (values); q is 16-bit (q_dtype). Pools are
 * bytes in `layout`. Same definition as oracle_batch_attention otherwise.
 */
int32_t oracle_batch_attention_fp8kv(const uint16_t* q, const int32_t* qo_indptr,
                                     const uint8_t* k_pool, const uint8_t* v_pool,
                                     int64_t num_pages, int32_t layout,
                                     const int32_t* kv_indptr, const int32_t* kv_indices,
                                     const int32_t* last_page_len, int32_t batch,
                                     int32_t page_size, int32_t num_qo_heads,
                                     int32_t num_kv_heads, int32_t head_dim, int32_t q_dtype,
                                     int32_t causal, double sm_scale, const float* k_scale,
                                     const float* v_scale, double* o, double* lse);

/*
 * Attention output of one (request r, query row i, query head h).
 *   q            : [total_qo, Hq, D] raw 16-bit words (decode: total_qo = batch)
 *   qo_indptr    : int32[batch + 1] or NULL for decode (one row per request)
 *   k_pool/v_pool: raw 16-bit words in `layout`
 *   o            : double[D] out; *lse: natural-log LSE out (-INFINITY if empty)
 * Returns 0 on success, a negative code on invalid input (nothing written).
 */
int32_t oracle_attention_row(const uint16_t* q, const int32_t* qo_indptr,
                             const uint16_t* k_pool, const uint16_t* v_pool,
                             int64_t num_pages, int32_t layout,
                             const int32_t* kv_indptr, const int32_t* kv_indices,
                             const int32_t* last_page_len, int32_t batch,
                             int32_t page_size, int32_t num_qo_heads,
                             int32_t num_kv_heads, int32_t head_dim,
                             int32_t dtype, int32_t causal, double sm_scale,
                             int32_t r, int32_t i, int32_t h,
                             double* o, double* lse);

/*
 * Every row of the batch: o is double[total_qo, Hq, D], lse double[total_qo, Hq].
 * Optional kv-range restriction: if kv_begin/kv_end are non-NULL, request r
 * attends only to logical positions [kv_begin[r], kv_end[r]) of its visible
 * set (used to build split-KV partial states). Returns 0 or a negative code.
 */
int32_t oracle_batch_attention(const uint16_t* q, const int32_t* qo_indptr,
                               const uint16_t* k_pool, const uint16_t* v_pool,
                               int64_t num_pages, int32_t layout,
                               const int32_t* kv_indptr, const int32_t* kv_indices,
                               const int32_t* last_page_len, int32_t batch,
                               int32_t page_size, int32_t num_qo_heads,
                               int32_t num_kv_heads, int32_t head_dim,
                               int32_t dtype, int32_t causal, double sm_scale,
                               const int32_t* kv_begin, const int32_t* kv_end,
                               double* o, double* lse);

/*
 * oracle_batch_attention with rotary position embedding applied to the
 * queries and keys first. The pages count LLaMA-style RoPE among the
 * supported features (gittoolsai.com README copy, feature list) and give it
 * as the example of a query / key transform that the attention template
 * applies inside the kernel (modb.pro digest, "可定制的注意力模板"). The
 * pages leave the pairing, positions and precision open; the readings taken:
 *  - LLaMA style = "rotate half": dims d and d + D/2 form a pair,
 *      x'_d       = x_d c - x_{d+D/2} s,   x'_{d+D/2} = x_{d+D/2} c + x_d s,
 *    with c = rope_cos[pos * (D/2) + d], s = rope_sin[pos * (D/2) + d];
 *  - key j of a request sits at position j; query row i of a request with
 *    qo_len rows at position kv_len - qo_len + i (decode: kv_len - 1);
 *  - the rotated q and k are rounded to the storage dtype (round to nearest,
 *    ties to even), as a kernel producing rotated 16-bit tensors would.
 *   rope_cos/rope_sin: float[rope_max_pos, D/2]; every position used must be
 *   < rope_max_pos (else -9 is returned). D must be even.
 */
/*
 * One row of oracle_batch_attention_rope (request r, query row i, query head
 * h), with the same tables and checks restricted to request r.
 */
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
                                  double* o, double* lse);

int32_t oracle_batch_attention_rope(const uint16_t* q, const int32_t* qo_indptr,
                                    const uint16_t* k_pool, const uint16_t* v_pool,
                                    int64_t num_pages, int32_t layout,
                                    const int32_t* kv_indptr, const int32_t* kv_indices,
                                    const int32_t* last_page_len, int32_t batch,
                                    int32_t page_size, int32_t num_qo_heads,
                                    int32_t num_kv_heads, int32_t head_dim,
                                    int32_t dtype, int32_t causal, double sm_scale,
                                    const float* rope_cos, const float* rope_sin,
                                    int64_t rope_max_pos, double* o, double* lse);

/* Round a double to the nearest value of the 16-bit storage type (ties to
 * even; overflow to +-inf). */
double oracle_round(double v, int32_t dtype);

/*
 * Log-sum-exp merge of n_states attention states per row:
 *   o_in  : double[n_states, rows, D], lse_in: double[n_states, rows]
 *   o_out : double[rows, D],           lse_out: double[rows]
 * m = max_i lse_i; lse = m + ln sum_i exp(lse_i - m); o = sum_i exp(lse_i - lse) o_i.
 * All states empty (lse = -inf): o = 0, lse = -inf.
 */
void oracle_merge_states(const double* o_in, const double* lse_in,
                         int32_t n_states, int64_t rows, int32_t head_dim,
                         double* o_out, double* lse_out);

#ifdef __cplusplus
}
#endif
#endif
