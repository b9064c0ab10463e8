/*
 * attn.h -- C ABI of libattn.so: attention over a block-sparse-row (BSR)
 * paged KV cache on one GB300 (sm_103a).
 *
 * The operations follow "FlashInfer: Efficient and Customizable Attention
 * Engine for LLM Inference Serving" (arXiv 2501.01005) as summarised on the
 * modb.pro digest page:
 *  - "统一的 KV 缓存存储格式" (unified KV-cache storage format): the cache of a
 *    batch is a block-sparse row matrix. Row r is request r; its blocks are
 *    pages of `page_size` tokens listed in kv_indices[kv_indptr[r] ..
 *    kv_indptr[r+1]); the last page holds last_page_len[r] tokens, so
 *    kv_len_r = (n_r - 1) * page_size + last_page_len[r] for n_r > 0 pages
 *    and 0 for n_r = 0. (The digest's formula did not survive extraction;
 *    this is the reading used.) Contiguous caches are the one-page case.
 *  - "可组合格式" (composable formats): several formats take part in one
 *    attention; their partial results are combined with attn_merge_states.
 *  - "动态负载均衡调度" (load-balanced scheduling): a CPU planning phase
 *    (attn_plan) splits the KV of every request into work units balanced
 *    across SMs; a persistent fixed-grid kernel (attn_*_run) follows the
 *    plan using a preallocated workspace, so runs can be captured in CUDA
 *    graphs.
 * Attention is softmax(q K^T * sm_scale) V per query head, with query head h
 * reading kv head h / (num_qo_heads / num_kv_heads) (grouped-query heads).
 * Decode has one query row per request (gittoolsai.com page, "基本用法":
 * q [num_qo_heads, head_dim] against k/v [kv_len, num_kv_heads, head_dim]).
 *
 * Conventions for every entry point:
 *  - The caller owns all memory. The library allocates nothing and keeps no
 *    state besides a per-device cache of attributes and per-thread error text.
 *  - Pointers documented as "device" are CUDA device memory of the current
 *    device; "host" pointers are CPU memory. Work is enqueued on `stream`
 *    (a cudaStream_t; NULL is the legacy default stream) and is asynchronous.
 *  - Every call returns an attn_status_t and never throws. On failure
 *    attn_last_error() returns a message for the calling thread, and nothing
 *    is enqueued. Argument checks happen on the host before any launch.
 *  - head_dim must be 128. num_qo_heads must be a multiple of num_kv_heads.
 *  - LSE outputs are natural-log log-sum-exp of the scaled logits, fp32;
 *    an empty visible set gives O = 0 and LSE = -inf.
 */
#ifndef PAGED_BSR_ATTN_H
#define PAGED_BSR_ATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  ATTN_OK = 0,
  ATTN_ERR_INVALID_ARG = 1,         /* a size, pointer or value is out of range  */
  ATTN_ERR_UNSUPPORTED = 2,         /* valid but not implemented (e.g. head_dim) */
  ATTN_ERR_WORKSPACE_TOO_SMALL = 3, /* a workspace is smaller than required      */
  ATTN_ERR_CUDA = 4,                /* a CUDA runtime/driver call failed         */
  ATTN_ERR_TIMEOUT = 5              /* a kernel gave up waiting (bounded waits)  */
} attn_status_t;

typedef enum { ATTN_F16 = 0, ATTN_BF16 = 1 } attn_dtype_t;

/* Pool layouts. HND: [num_pages, num_kv_heads, page_size, head_dim];
 * NHD: [num_pages, page_size, num_kv_heads, head_dim]. Both row-major. */
typedef enum { ATTN_LAYOUT_HND = 0, ATTN_LAYOUT_NHD = 1 } attn_kv_layout_t;

typedef enum { ATTN_MODE_DECODE = 0, ATTN_MODE_APPEND = 1, ATTN_MODE_CASCADE = 2 } attn_mode_t;

/*
 * A work plan: plain data produced by attn_plan. It records the shapes the
 * plan was made for and where the plan's tables live inside the device
 * workspace. Pass it unchanged to the matching run call.
 */
typedef struct attn_plan {
  int32_t mode;             /* attn_mode_t                                     */
  int32_t batch;
  int32_t page_size;
  int32_t num_qo_heads;
  int32_t num_kv_heads;
  int32_t head_dim;
  int32_t causal;
  int32_t num_ctas;         /* grid size of the persistent run kernel          */
  int32_t q_tile;           /* query tokens per item: 256 / group (append), 1  */
  int32_t rows_per_item;    /* packed rows of one item: group * q_tile         */
  int32_t num_items;        /* (request, kv head, query tile) triples          */
  int32_t num_units;        /* work units after the balanced cut               */
  int32_t num_split_items;  /* items cut into >= 2 units (merged after run)    */
  int32_t num_slots;        /* partial-state slots used by split items         */
  int32_t total_qo;         /* query rows (decode: batch)                      */
  int32_t max_qo_len;       /* longest query row count of a request (decode: 1) */
  int64_t total_weight;     /* sum over items of (pages + alpha): alpha 1 if
                               the few-row kernel runs the plan (decode,
                               short appends), else 16                       */
  int64_t max_cta_weight;   /* largest per-CTA share of the weights the cut
                               balances (cascade: tokens + 16 per segment)     */
  int64_t off_work_indptr;  /* byte offsets of the tables in the workspaces    */
  int64_t off_units;
  int64_t off_merge_indptr;
  int64_t off_merge_items;
  int64_t off_counters;     /* per split item arrival counters (zeroed by plan) */
  int64_t off_partial_o;
  int64_t off_partial_lse;
  int64_t table_bytes;      /* bytes [0, table_bytes) copied host -> device    */
  int64_t dev_bytes_needed; /* device workspace bytes this plan uses           */
  uint64_t fingerprint;     /* hash of the host inputs of the plan             */
  int64_t max_kv_len;       /* longest kv length of a request                  */
  int64_t min_kv_minus_qo;  /* smallest kv_len - qo_len over requests with kv
                               tokens (INT64_MAX if none)                      */
  int32_t page_size_suffix; /* cascade: page size of the suffix table (else 0) */
  int32_t reserved;         /* 0                                               */
} attn_plan_t;

/*
 * Workspace sizes able to hold any plan with at most max_batch requests,
 * max_total_qo query rows (append; pass max_batch for decode-only use) and
 * num_ctas CTAs. Pure host computation.
 *   dev_bytes         : device workspace (plan tables + partial states)
 *   pinned_host_bytes : host staging area for the plan tables (page-locked
 *                       memory, so the table copy is asynchronous)
 * Errors: INVALID_ARG for non-positive sizes or null outputs.
 */
attn_status_t attn_workspace_size(int32_t max_batch, int32_t max_total_qo,
                                  int32_t num_qo_heads, int32_t num_kv_heads,
                                  int32_t head_dim, int32_t num_ctas,
                                  size_t* dev_bytes, size_t* pinned_host_bytes);

/*
 * Default persistent grid for `mode` on CUDA device `device`: the number of
 * SMs times the CTAs of the run kernel that fit on one SM (cascade: one).
 * Errors: CUDA if the device cannot be queried; INVALID_ARG for bad mode.
 */
attn_status_t attn_default_num_ctas(int32_t device, int32_t mode, int32_t* num_ctas);

/*
 * Planning phase (host). Splits the work of a batch into units balanced over
 * num_ctas CTAs. Items are (request, kv head, query tile) triples in
 * request-major order, then kv head, then tile; an item weighs its visible
 * page count + 1, and W is the sum of the weights over all items.
 *  - decode: the weights are laid end to end and CTA c takes the positions
 *    [floor(c W / C), floor((c+1) W / C));
 *  - append: items are dealt in order to the CTA with the least weight so
 *    far (ties to the lowest index), each CTA capped at ceil(W / C) + 1; an
 *    item that does not fit is cut at the cap and continues on the next CTA.
 * An item cut into several units is "split": its units write partial states
 * that the run merges by log-sum-exp.
 *   qo_indptr_h     : host int32[batch+1] query row offsets (append, starting
 *                     at 0), or NULL for decode (one row per request)
 *   kv_indptr_h     : host int32[batch+1] page offsets into kv_indices
 *   last_page_len_h : host int32[batch]; 1..page_size when the request has pages
 *   causal          : 1 = query row i of a request with qo_len rows sees kv
 *                     positions j <= kv_len - qo_len + i (end-aligned);
 *                     0 = all positions. Ignored for decode.
 *   pinned_host_ws  : host staging buffer of pinned_bytes bytes. It must stay
 *                     untouched until the copy enqueued on `stream` has run.
 *   dev_ws          : device workspace of dev_bytes bytes, or NULL to only
 *                     compute the tables on the host (no CUDA call is made).
 *   plan_out        : receives the plan.
 * The tables are written to pinned_host_ws and copied to dev_ws on `stream`
 * in one go: by a small copy kernel that reads pinned_host_ws through its
 * device mapping when the memory is page-locked and mapped (so the run
 * kernel behind it waits on no copy engine), else by one cudaMemcpyAsync.
 * The copy also clears the workspace's error word. The plan depends only on
 * the host inputs and num_ctas and is identical run to run.
 * Errors: INVALID_ARG (negative lengths, last_page_len out of range, heads not
 * divisible, append with kv_len < qo_len), UNSUPPORTED (head_dim != 128,
 * group too large), WORKSPACE_TOO_SMALL, CUDA.
 */
attn_status_t attn_plan(const int32_t* qo_indptr_h, const int32_t* kv_indptr_h,
                        const int32_t* last_page_len_h, int32_t batch,
                        int32_t page_size, int32_t num_qo_heads,
                        int32_t num_kv_heads, int32_t head_dim, int32_t causal,
                        int32_t num_ctas, void* pinned_host_ws, size_t pinned_bytes,
                        void* dev_ws, size_t dev_bytes, void* stream,
                        attn_plan_t* plan_out);

/*
 * Batch decode over a paged cache (one query row per request), following a
 * decode plan. One persistent kernel with plan->num_ctas CTAs; the last unit
 * of a split item to finish merges the item's partial states (LSE weights).
 *   q          : device [batch, num_qo_heads, head_dim] of `dtype`
 *   k_pool,
 *   v_pool     : device pools of num_pages pages in `layout`, `dtype`
 *   kv_indptr, kv_indices, last_page_len : device copies of the BSR table
 *                (kv_indptr and last_page_len equal to the plan's host copies;
 *                every kv_indices entry in [0, num_pages))
 *   sm_scale   : logit scale (1/sqrt(head_dim) is the usual choice), finite
 *                and >= 0 (every run entry point rejects other values with
 *                INVALID_ARG); 0 weighs the visible keys equally
 *   o          : device [batch, num_qo_heads, head_dim] of `dtype` (out)
 *   lse        : device float[batch, num_qo_heads] (out) or NULL
 *   dev_ws     : the workspace given to attn_plan (holds the plan tables)
 * Supported: head_dim 128, group = num_qo_heads / num_kv_heads in 1..8,
 * any page_size >= 1, both layouts, fp16 and bf16. Groups 2, 4 and 8 run on
 * the tensor-core (tcgen05) decode kernel at any page size and either layout
 * (the group's query rows replicated over 32 MMA rows; 128-token K/V tiles
 * loaded by TMA in 16-row boxes when page_size % 16 == 0, else row by row
 * with gathers, down to one token per page); groups 1, 3, 5, 6 and 7 run on a
 * CUDA-core streaming kernel. Both merge split items inside the kernel.
 * Errors: INVALID_ARG (plan mode/shape mismatch, null pointers),
 * UNSUPPORTED, WORKSPACE_TOO_SMALL, CUDA (launch failure).
 */
attn_status_t attn_decode_run(const attn_plan_t* plan, const void* q,
                              const void* k_pool, const void* v_pool,
                              int64_t num_pages, int32_t layout,
                              const int32_t* kv_indptr, const int32_t* kv_indices,
                              const int32_t* last_page_len, int32_t dtype,
                              float sm_scale, void* o, float* lse, void* dev_ws,
                              size_t dev_bytes, void* stream);

/*
 * attn_decode_run over an FP8 KV cache: the pools hold FP8 E4M3 bytes (the
 * "fn" encoding: no infinities) with one scale per kv head, so a token row
 * is 128 bytes instead of 256 and a decode step reads half the bytes. The
 * pages list FP8 KV-cache support among the features (gittoolsai.com README
 * copy, feature list); the scale reading is this library's: the byte b of kv
 * head hk stands for e4m3(b) * k_scale[hk] in K and e4m3(b) * v_scale[hk] in
 * V. The kernel widens the bytes exactly as it reads them from shared memory,
 * folds k_scale into q and v_scale into the output.
 *   k_pool, v_pool   : device bytes, [num_pages, Hk, P, 128] (HND) or
 *                      [num_pages, P, Hk, 128] (NHD), 16-byte aligned
 *   k_scale, v_scale : device float[num_kv_heads]
 *   dtype            : the type of q and o (ATTN_F16 / ATTN_BF16)
 *   other arguments  : as attn_decode_run (same decode plan)
 * Supported: head_dim 128, group 1..8, any page size, both layouts. Groups
 * 2, 4 and 8 over HND pools with page_size % 16 == 0 run on the tensor-core
 * decode kernel: TMA stages the E4M3 tiles, four warps widen them to f16 in
 * shared memory, and the MMAs multiply f16 operands (a bf16 q is rounded to
 * f16 first: |q| must stay below 65504). The other shapes run on the
 * CUDA-core streaming kernel, which widens rows to fp32 as it reads them.
 * Errors: as attn_decode_run; INVALID_ARG for null scales.
 */
attn_status_t attn_decode_run_fp8(const attn_plan_t* plan, const void* q, const void* k_pool,
                                  const void* v_pool, int64_t num_pages, int32_t layout,
                                  const int32_t* kv_indptr, const int32_t* kv_indices,
                                  const int32_t* last_page_len, int32_t dtype,
                                  const float* k_scale, const float* v_scale, float sm_scale,
                                  void* o, float* lse, void* dev_ws, size_t dev_bytes,
                                  void* stream);

/*
 * attn_decode_run with rotary position embedding fused in: the kernel turns
 * q and each key as it streams the pages, so the cache keeps keys without
 * RoPE and no separate RoPE pass reads or writes them. The pages count
 * LLaMA-style RoPE, the LLaMA 3.1 variant included, among the supported
 * features (README copy on gittoolsai.com, feature list) and use it as their
 * example of a per-query / per-key transform that the attention template
 * applies inside the kernel (modb.pro digest, "可定制的注意力模板").
 * Readings: dims d and d + 64 form a pair ("rotate half"),
 *   x'_d = x_d cos - x_{d+64} sin,   x'_{d+64} = x_{d+64} cos + x_d sin,
 * with cos / sin = rope_cos / rope_sin[pos * 64 + d]; key j of a request sits
 * at position j and the query at position kv_len - 1; the turned q and k are
 * rounded to `dtype` before the products.
 *   rope_cos, rope_sin : device float[rope_max_pos, 64], row-major and
 *                        contiguous, 16-byte aligned, read only: the cos /
 *                        sin of the angles pos * theta_d for some per-pair
 *                        frequencies theta_d (plain LLaMA, or LLaMA 3.1 with
 *                        its rescaled frequencies); rope_max_pos must be at
 *                        least the plan's max_kv_len
 * The query reads its table row directly. Keys read a few rows per 128-key
 * tile and derive the others with the angle-sum identities
 * (cos((B + o) t) = cos(B t) cos(o t) - sin(B t) sin(o t), likewise for sin),
 * so tables that are not of that form (e.g. with a magnitude factor folded
 * in; fold such a factor into sm_scale instead) give other keys. The derived
 * values differ from direct rows by a few fp32 ulps.
 *   other arguments    : as attn_decode_run
 * Supported: the shapes attn_decode_run runs on the tensor-core kernel (2, 4
 * or 8 query heads per kv head, any page size, either layout); others return
 * UNSUPPORTED.
 * Errors: as attn_decode_run; INVALID_ARG for missing, misaligned or too
 * short tables.
 */
attn_status_t attn_decode_run_rope(const attn_plan_t* plan, const void* q,
                                   const void* k_pool, const void* v_pool,
                                   int64_t num_pages, int32_t layout,
                                   const int32_t* kv_indptr, const int32_t* kv_indices,
                                   const int32_t* last_page_len, int32_t dtype,
                                   float sm_scale, const float* rope_cos,
                                   const float* rope_sin, int64_t rope_max_pos,
                                   void* o, float* lse, void* dev_ws, size_t dev_bytes,
                                   void* stream);

/*
 * attn_append_run with rotary position embedding fused in (as
 * attn_decode_run_rope): query row i of a request with qo_len rows sits at
 * position kv_len - qo_len + i, key j at position j.
 *   rope_cos, rope_sin, rope_max_pos : as attn_decode_run_rope
 *   other arguments                  : as attn_append_run
 * Supported: every shape attn_append_run takes. Short appends (group x the
 * longest query count <= 16) run on the few-row kernel, whose rope warps
 * derive most key angles by the angle-sum identities (as in
 * attn_decode_run_rope); longer ones on the append kernel, whose two rope
 * warps turn each unit's query rows once and every K tile in shared memory,
 * reading a table row every 16 positions and stepping the angle by theta_d
 * (table row 1) in between -- so the tables must hold cos / sin of
 * pos * theta_d there too.
 * Errors: as attn_append_run and attn_decode_run_rope; INVALID_ARG if a
 * request with kv tokens has kv_len < qo_len (a query would sit before
 * position 0).
 */
attn_status_t attn_append_run_rope(const attn_plan_t* plan, const void* q,
                                   const int32_t* qo_indptr, const void* k_pool,
                                   const void* v_pool, int64_t num_pages, int32_t layout,
                                   const int32_t* kv_indptr, const int32_t* kv_indices,
                                   const int32_t* last_page_len, int32_t dtype,
                                   int32_t causal, float sm_scale, const float* rope_cos,
                                   const float* rope_sin, int64_t rope_max_pos, void* o,
                                   float* lse, void* dev_ws, size_t dev_bytes, void* stream);

/*
 * Append / prefill attention: many query rows per request (ragged, offsets
 * qo_indptr) against that request's paged KV, which already holds the new
 * tokens (kv_len >= qo_len), causal (end-aligned) or not, following an append
 * plan. Tensor-core kernel (tcgen05 MMA, TMEM accumulators, TMA-fed).
 *   q          : device [total_qo, num_qo_heads, head_dim] of `dtype`
 *   qo_indptr  : device int32[batch+1], equal to the plan's host copy
 *   other arguments as attn_decode_run; o is [total_qo, num_qo_heads, head_dim]
 *   and lse float[total_qo, num_qo_heads].
 * Supported: head_dim 128, bf16 or fp16, HND or NHD layout, any page_size
 * >= 1, group in {1, 2, 4, 8, 16}. Short appends (group x the longest query
 * count <= 16) run on the few-row tensor-core kernel; longer ones on the
 * append kernel. Both load K / V by TMA in 16-row boxes when
 * page_size % 16 == 0 and gather rows four at a time otherwise (down to one
 * token per page).
 * Errors: as attn_decode_run.
 */
attn_status_t attn_append_run(const attn_plan_t* plan, const void* q,
                              const int32_t* qo_indptr, const void* k_pool,
                              const void* v_pool, int64_t num_pages, int32_t layout,
                              const int32_t* kv_indptr, const int32_t* kv_indices,
                              const int32_t* last_page_len, int32_t dtype,
                              int32_t causal, float sm_scale, void* o, float* lse,
                              void* dev_ws, size_t dev_bytes, void* stream);

/*
 * Merge two attention states of the same rows by log-sum-exp ("可组合格式":
 * combining the partial results of composable formats / split KV):
 *   m = max(lse_a, lse_b); lse = m + ln(e^(lse_a - m) + e^(lse_b - m));
 *   o = e^(lse_a - lse) o_a + e^(lse_b - lse) o_b.
 * Both states empty (lse = -inf) gives o = 0, lse = -inf.
 *   o_a, o_b, o_out  : device [n, num_heads, head_dim] of `dtype`
 *   lse_a, lse_b     : device float[n, num_heads] (natural log)
 *   lse_out          : device float[n, num_heads] (out) or NULL
 * o_out may alias o_a or o_b. Any head_dim that is a multiple of 8.
 * Errors: INVALID_ARG, UNSUPPORTED, CUDA.
 */
attn_status_t attn_merge_states(const void* o_a, const float* lse_a,
                                const void* o_b, const float* lse_b, void* o_out,
                                float* lse_out, int32_t n, int32_t num_heads,
                                int32_t head_dim, int32_t dtype, void* stream);

/*
 * Composable formats in one launch ("可组合格式": a shared prefix stored once in
 * a table with large pages, each generation's own suffix in a second table
 * with small pages; the partial attention over the two is combined by
 * log-sum-exp). Decode shape: prompt p has n_p generations, rows
 * qo_indptr[p] .. qo_indptr[p+1] of q, one query row each. Generation b of
 * prompt p attends to the prompt's prefix (prefix table row p) followed by
 * its own suffix (suffix table row b); the result equals decode over the flat
 * layout prefix ++ suffix.
 *
 * attn_cascade_workspace_size: workspace sizes for any cascade plan with at
 * most max_prompts prompts, max_batch generations and num_ctas CTAs.
 *
 * attn_plan_cascade: items are (prompt, kv head) pairs; an item's segments are
 * its prefix row and then one suffix row per generation. A segment weighs
 * its tokens (pages x page size) + 16; the weights are laid end to end and
 * CTA c takes the positions [floor(c W / C), floor((c+1) W / C)), a page
 * going to the CTA that owns its first position (pages of one segment on one
 * CTA form a unit; segments without pages add none, and an item without any
 * page keeps one empty unit). The units of one item on one CTA run as a
 * chain that carries one online-softmax state per row (the prefix for all
 * n_p generations, a suffix only for its own generation's rows), so an item
 * on one CTA needs no merge; an item cut across CTAs writes one partial
 * state per chain and the last chain to finish merges them by log-sum-exp.
 * Within a CTA the chains of cut items run first.
 *   qo_indptr_h             : host int32[num_prompts+1], generations per
 *                             prompt, starting at 0 (batch = its last entry)
 *   kv_indptr_prefix_h,
 *   last_page_len_prefix_h  : host prefix table, num_prompts rows, pages of
 *                             page_size_prefix tokens
 *   kv_indptr_suffix_h,
 *   last_page_len_suffix_h  : host suffix table, batch rows, pages of
 *                             page_size_suffix tokens
 *   other arguments as attn_plan (dev_ws NULL plans on the host only).
 * group x (the largest n_p) must be at most 16 (rows of one MMA item).
 * Errors: INVALID_ARG, UNSUPPORTED (head_dim, group x n_p > 16),
 * WORKSPACE_TOO_SMALL, CUDA.
 *
 * attn_cascade_run: one persistent launch of the few-row tensor-core kernel
 * over both tables, merging inside the kernel.
 *   q                  : device [batch, num_qo_heads, head_dim] of `dtype`
 *   qo_indptr          : device copy of qo_indptr_h
 *   k_prefix, v_prefix : device pools of num_pages_prefix pages of
 *                        page_size_prefix tokens in `layout`, `dtype`
 *   kv_indptr_prefix, kv_indices_prefix, last_page_len_prefix : device copies
 *                        of the prefix table (indices in [0, num_pages_prefix))
 *   k_suffix ... last_page_len_suffix : the same for the suffix table
 *   o                  : device [batch, num_qo_heads, head_dim] (out)
 *   lse                : device float[batch, num_qo_heads] (out) or NULL
 *   layout             : ATTN_LAYOUT_HND or ATTN_LAYOUT_NHD (both pools)
 * Supported: any page sizes, both layouts, group 1..16 with group x n_p <= 16,
 * fp16 / bf16. K / V rows load in 16-row TMA boxes when the pools are HND
 * and both page sizes are multiples of 16, else row by row (cp.async).
 * ATTN_DEBUG_CHECKS applies to both tables.
 * Errors: INVALID_ARG, UNSUPPORTED, WORKSPACE_TOO_SMALL, CUDA.
 */
attn_status_t attn_cascade_workspace_size(int32_t max_prompts, int32_t max_batch,
                                          int32_t num_qo_heads, int32_t num_kv_heads,
                                          int32_t head_dim, int32_t num_ctas,
                                          size_t* dev_bytes, size_t* pinned_host_bytes);

attn_status_t attn_plan_cascade(const int32_t* qo_indptr_h, const int32_t* kv_indptr_prefix_h,
                                const int32_t* last_page_len_prefix_h, int32_t page_size_prefix,
                                const int32_t* kv_indptr_suffix_h,
                                const int32_t* last_page_len_suffix_h, int32_t page_size_suffix,
                                int32_t num_prompts, int32_t num_qo_heads, int32_t num_kv_heads,
                                int32_t head_dim, int32_t num_ctas, void* pinned_host_ws,
                                size_t pinned_bytes, void* dev_ws, size_t dev_bytes,
                                void* stream, attn_plan_t* plan_out);

attn_status_t attn_cascade_run(const attn_plan_t* plan, const void* q, const int32_t* qo_indptr,
                               const void* k_prefix, const void* v_prefix,
                               int64_t num_pages_prefix, const int32_t* kv_indptr_prefix,
                               const int32_t* kv_indices_prefix,
                               const int32_t* last_page_len_prefix, const void* k_suffix,
                               const void* v_suffix, int64_t num_pages_suffix,
                               const int32_t* kv_indptr_suffix, const int32_t* kv_indices_suffix,
                               const int32_t* last_page_len_suffix, int32_t layout,
                               int32_t dtype, float sm_scale, void* o, float* lse,
                               void* dev_ws, size_t dev_bytes, void* stream);

/*
 * Synchronises `stream`, then reads the error word that kernels set in a
 * workspace when a bounded wait expired. *code_out receives 0 if none.
 * Returns TIMEOUT if the word is set, CUDA on a runtime error, else OK.
 */
attn_status_t attn_workspace_status(const void* dev_ws, void* stream, int32_t* code_out);

/*
 * Failure-detection self-test (no counterpart on the pages; it checks this
 * library's bounded waits). Enqueues on `stream` one warp that waits, with
 * the same bounded wait every kernel here uses, on an mbarrier that nothing
 * arrives on. The wait gives up after limit_us microseconds and writes code
 * 0x1ff into dev_ws's error word (unless the word already holds a code, in
 * which case it gives up at once). The GPU never faults or hangs:
 * attn_workspace_status then returns TIMEOUT and the context stays usable;
 * the next attn_plan on the workspace clears the word.
 *   dev_ws   : a workspace given to attn_plan (or any 256-byte aligned
 *              device buffer of at least 4 bytes)
 *   limit_us : 1 .. 10^7
 * Errors: INVALID_ARG, CUDA.
 */
attn_status_t attn_wait_selftest(void* dev_ws, int32_t limit_us, void* stream);

/*
 * Batch decode for callers that cannot allocate device memory. The paper has
 * no counterpart: this is a deployment convenience of this library.
 *
 * Who needs it: code that may not call cudaMalloc or any allocator when it
 * runs attention -- e.g. inside an allocator-free region of a serving engine,
 * a plugin whose host application owns every device allocation, or a
 * latency-critical path that must not take allocator locks or grow a memory
 * pool. Such callers cannot provide the workspaces attn_plan and
 * attn_decode_run need, so this entry point plans and runs in one call using
 * a fixed 4 MiB scratch area that lives in the library's own device memory
 * (a file-scope __device__ array held on every device that loads the library
 * until the process exits). It calls no cudaMalloc, cudaFree or allocating
 * routine.
 *   kv_indptr_h, last_page_len_h : host copies of the page table (as attn_plan)
 *   other arguments              : as attn_decode_run (device inputs/outputs,
 *                                  q [batch, num_qo_heads, head_dim], ...)
 * Behaviour:
 *  - The first call on a device looks up the scratch array's address with that
 *    device current; make that first call before any stream capture.
 *  - All calls share the one scratch area (and one host staging area), which
 *    keeps the previous call's contents; each call re-initialises what must
 *    start at zero. Calls whose work overlaps on the GPU race with each other;
 *    calls ordered on one stream are safe. Host calls are serialised.
 *  - Batches whose plan tables and partial states exceed 4 MiB (roughly more
 *    than 60k (request, kv head) pairs at group 8, a few more at smaller
 *    groups) return ATTN_ERR_WORKSPACE_TOO_SMALL
 *    before any GPU work; use attn_plan + attn_decode_run instead.
 *  - The kernel's bounded waits report into an error word at the head of the
 *    scratch area; attn_decode_run_noalloc_status reads it. The next call's
 *    table upload clears the word, so read it before the next call.
 * Errors: as attn_plan and attn_decode_run.
 */
attn_status_t attn_decode_run_noalloc(const int32_t* kv_indptr_h,
                                      const int32_t* last_page_len_h, int32_t batch,
                                      int32_t page_size, int32_t num_qo_heads,
                                      int32_t num_kv_heads, int32_t head_dim, const void* q,
                                      const void* k_pool, const void* v_pool,
                                      int64_t num_pages, int32_t layout,
                                      const int32_t* kv_indptr, const int32_t* kv_indices,
                                      const int32_t* last_page_len, int32_t dtype,
                                      float sm_scale, void* o, float* lse, void* stream);

/*
 * Status of the no-allocation path on the current device (no counterpart in
 * the paper: this reads the library's own failure detection). Synchronises
 * `stream`, then reads the error word at the head of the scratch area that
 * attn_decode_run_noalloc uses; *code_out receives 0 if no kernel gave up a
 * bounded wait since the last attn_decode_run_noalloc call on this device.
 * Allocates nothing (the first call on a device looks up the scratch
 * address, like attn_decode_run_noalloc).
 * Returns TIMEOUT if the word is set, CUDA on a runtime error, else OK.
 */
attn_status_t attn_decode_run_noalloc_status(void* stream, int32_t* code_out);

/*
 * attn_wait_selftest aimed at the no-allocation scratch area (no counterpart
 * in the paper): one bounded wait that nothing completes, whose code 0x1ff
 * lands in the error word attn_decode_run_noalloc_status reads.
 *   limit_us : 1 .. 10^7
 * Errors: INVALID_ARG, CUDA.
 */
attn_status_t attn_wait_selftest_noalloc(int32_t limit_us, void* stream);

/* Message of the last failed call on this thread ("" if none). */
const char* attn_last_error(void);

#ifdef __cplusplus
}
#endif
#endif /* PAGED_BSR_ATTN_H */
