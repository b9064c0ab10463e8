// internal.h -- data shared between the host planner, the C ABI and the
// kernels of libattn.so (not part of the public interface).
#pragma once
#include <atomic>
#include <cstddef>
#include <cstdint>
#include <string>

#include <cuda_runtime.h>

#include "../../include/attn.h"

namespace attn {

constexpr int kHeadDim = 128;
constexpr int kTileRows = 128;      // packed query rows of one MMA tile (M = 128)
constexpr int kItemRows = 256;      // packed query rows of one append item (2 tiles)
constexpr int kMaxDecodeGroup = 8;  // query heads per kv head, decode kernel
constexpr int kTensorDecodeGroup = 2;  // decode groups >= this use the tensor-core kernel
constexpr int kUnitInts = 12;       // int32 words per work-unit record
constexpr int64_t kHeaderBytes = 256;

// One work unit of the plan (48 bytes = three int4, 16-byte aligned in the
// workspace). The request's geometry is copied in by the planner so that a
// kernel learns everything about a unit from three independent loads.
struct Unit {
  int32_t r;          // request
  int32_t hk;         // kv head
  int32_t t;          // query tile (append) / 0 (decode)
  int32_t p0;         // first page (index within the request's page list)
  int32_t p1;         // one past the last page
  int32_t slot;       // partial-state slot, -1 if the item is not split
  int32_t split;      // split-item index, -1 if not split
  int32_t page_base;  // kv_indptr[r]
  int32_t kv_len;     // the request's kv tokens
  int32_t qo_start;   // qo_indptr[r] (append) / r (decode)
  int32_t qo_len;     // the request's query rows (decode: 1)
  int32_t pad;
};
static_assert(sizeof(Unit) == kUnitInts * 4, "unit record size");

// Workspace header (first 256 bytes of the device workspace).
struct WsHeader {
  int32_t error;      // set by a kernel whose bounded wait expired (0 = none)
  int32_t reserved[63];
};

inline int64_t align_up(int64_t x, int64_t a) { return (x + a - 1) / a * a; }

// Pointers into a device workspace, derived from a plan.
struct WsView {
  int32_t* error;
  const int32_t* work_indptr;
  const Unit* units;
  const int32_t* merge_indptr;
  const int4* merge_items;  // (r, hk, t, n_units)
  int32_t* counters;        // arrivals per split item (0 between runs)
  float* partial_o;         // [slots, rows_per_item, D]
  float* partial_lse;       // [slots, rows_per_item] (log2 domain)
};

inline WsView ws_view(const attn_plan_t& p, void* ws) {
  char* b = static_cast<char*>(ws);
  WsView v;
  v.error = reinterpret_cast<int32_t*>(b);
  v.work_indptr = reinterpret_cast<const int32_t*>(b + p.off_work_indptr);
  v.units = reinterpret_cast<const Unit*>(b + p.off_units);
  v.merge_indptr = reinterpret_cast<const int32_t*>(b + p.off_merge_indptr);
  v.merge_items = reinterpret_cast<const int4*>(b + p.off_merge_items);
  v.counters = reinterpret_cast<int32_t*>(b + p.off_counters);
  v.partial_o = reinterpret_cast<float*>(b + p.off_partial_o);
  v.partial_lse = reinterpret_cast<float*>(b + p.off_partial_lse);
  return v;
}

// ------------------------------------------------------------------ planner
// Sizes of the tables for a given plan shape (host).
struct PlanLayout {
  int64_t off_work_indptr, off_units, off_merge_indptr, off_merge_items, off_counters;
  int64_t table_bytes, off_partial_o, off_partial_lse, dev_bytes;
};
PlanLayout plan_layout(int32_t num_ctas, int64_t num_units, int64_t num_split,
                       int64_t num_slots, int32_t rows_per_item, int32_t head_dim);

// Hash of a plan's host inputs (attn_plan_t::fingerprint); qo_indptr is NULL
// for decode.
uint64_t plan_fingerprint(const int32_t* qo_indptr, const int32_t* kv_indptr,
                          const int32_t* last_page_len, int32_t batch, int32_t page_size,
                          int32_t num_qo_heads, int32_t num_kv_heads, int32_t head_dim,
                          int32_t causal, int32_t num_ctas);

// Composable-format (cascade) plan over a prefix table (prompts rows, page
// size P0) and a suffix table (qo_indptr[prompts] rows, page size P1); unit
// t = -1 reads the prefix row of prompt r, t = j >= 0 the suffix row of its
// generation j (unit.pad bit 0: 0 prefix / 1 suffix; bit 1: the unit
// continues the previous unit's row state, bit 2: the next unit continues
// this one's). A segment weighs its tokens + kCascadeAlpha.
constexpr int64_t kCascadeAlpha = 16;
attn_status_t build_cascade_plan(const int32_t* qo_indptr, const int32_t* kv_indptr0,
                                 const int32_t* last0, int32_t page_size0,
                                 const int32_t* kv_indptr1, const int32_t* last1,
                                 int32_t page_size1, int32_t prompts, int32_t num_qo_heads,
                                 int32_t num_kv_heads, int32_t head_dim, int32_t num_ctas,
                                 void* host_tables, size_t host_bytes, attn_plan_t* plan,
                                 const char** msg);
uint64_t cascade_fingerprint(const int32_t* qo_indptr, const int32_t* kv_indptr0,
                             const int32_t* last0, int32_t page_size0, const int32_t* kv_indptr1,
                             const int32_t* last1, int32_t page_size1, int32_t prompts,
                             int32_t num_qo_heads, int32_t num_kv_heads, int32_t head_dim,
                             int32_t num_ctas);

// Cost of a unit beyond its pages, in pages, for the plan's balanced cut:
// plans the few-row kernel runs (decode, short appends), plans the append
// kernel runs (long appends, POD batches).
constexpr int64_t kDecodeAlpha = 1;
constexpr int64_t kAppendAlpha = 16;

// Builds the plan tables into `host_tables` (table_bytes of them).
// Returns ATTN_OK or an error with a message in *msg.
attn_status_t build_plan(const int32_t* qo_indptr, const int32_t* kv_indptr,
                         const int32_t* last_page_len, int32_t batch, int32_t page_size,
                         int32_t num_qo_heads, int32_t num_kv_heads, int32_t head_dim,
                         int32_t causal, int32_t num_ctas, void* host_tables,
                         size_t host_bytes, attn_plan_t* plan, const char** msg);

// ---------------------------------------------------------------- launchers
struct DecodeArgs {
  const void* q;
  const void* k_pool;
  const void* v_pool;
  const int32_t* kv_indptr;
  const int32_t* kv_indices;
  const int32_t* last_page_len;
  void* o;
  float* lse;
  WsView ws;
  int32_t num_ctas;
  int32_t num_units;
  int32_t num_split_items;
  int32_t layout;
  int32_t dtype;
  int32_t page_size;
  int32_t num_qo_heads;
  int32_t num_kv_heads;
  int32_t group;
  int32_t batch;
  float sm_scale;
  // FP8 E4M3 K/V pools (kv_fp8 = 1) and their per-kv-head scales
  // (device float[num_kv_heads]); q and o keep `dtype`
  int32_t kv_fp8;
  const float* k_scale;
  const float* v_scale;
};
cudaError_t launch_decode(const DecodeArgs& a, cudaStream_t stream);
int decode_ctas_per_sm();

struct AppendArgs {
  const void* q;
  const int32_t* qo_indptr;
  const void* k_pool;
  const void* v_pool;
  int64_t num_pages;
  const int32_t* kv_indptr;
  const int32_t* kv_indices;
  const int32_t* last_page_len;
  void* o;
  float* lse;
  WsView ws;
  int32_t num_ctas;
  int32_t num_units;
  int32_t num_split_items;
  int32_t dtype;
  int32_t page_size;
  int32_t num_qo_heads;
  int32_t num_kv_heads;
  int32_t group;
  int32_t q_tile;          // query tokens per item (1 in decode mode)
  int32_t tile_tokens;     // query tokens per 128-row MMA tile (1 in decode mode)
  int32_t rows_per_item;   // group * q_tile (<= 128)
  int32_t total_qo;
  int32_t max_qo_len;      // longest query count of a request
  int32_t causal;
  float sm_scale;
  // rotary position embedding of q and k (few-row kernel only): cos / sin
  // tables float[rope_rows, 64] of the angles pos * theta_i; NULL = none
  const float* rope_cos;
  const float* rope_sin;
  int64_t rope_rows;
  int32_t layout;  // KV pool layout (few-row kernel): ATTN_LAYOUT_HND or ATTN_LAYOUT_NHD
  // FP8 E4M3 K/V pools with per-kv-head scales (few-row decode, HND,
  // page_size % 16 == 0); q / o keep `dtype`
  int32_t kv_fp8;
  const float* k_scale;
  const float* v_scale;
  // composable formats in one launch (few-row kernel, HND, page sizes % 16
  // == 0): units with pad = 1 read the second table (suffix pool, page size
  // page_size2); query rows are the generations of a prompt
  int32_t cascade;
  int32_t page_size2;
  const void* k_pool2;
  const void* v_pool2;
  int64_t num_pages2;
  const int32_t* kv_indices2;
};
// qo_indptr == NULL runs the kernel in decode mode (one query row per
// request; q is [batch, Hq, D]). Returns cudaErrorNotSupported for shapes the
// kernel does not handle.
cudaError_t launch_append(const AppendArgs& a, cudaStream_t stream, const char** msg);
int append_ctas_per_sm();
// Few-row tensor-core kernel: items of at most kFewRowMax packed query rows
// (decode with qo_indptr == NULL: the group's heads; a short append: its
// tokens x heads), HND pools of any page size; merges split items
// itself. few_row_rows gives the rows per item it runs with (a power of two
// >= group x max_qo_len), or 0 if the shape needs more than kFewRowMax.
constexpr int kFewRowMax = 16;
int few_row_rows(int32_t group, int32_t max_qo_len);
cudaError_t launch_decode_tc(const AppendArgs& a, cudaStream_t stream, const char** msg);

// Merge of split items' partial states into o / lse (after a run).
struct SplitMergeArgs {
  WsView ws;
  int32_t num_split_items;
  int32_t rows_per_item;
  int32_t group;
  int32_t q_tile;
  int32_t num_qo_heads;
  const int32_t* qo_indptr;  // NULL for decode
  void* o;
  float* lse;
  int32_t dtype;
};
cudaError_t launch_split_merge(const SplitMergeArgs& a, cudaStream_t stream);

// One warp waits, with the kernels' bounded wait and the given limit, on an
// mbarrier nothing arrives on (attn_wait_selftest).
cudaError_t launch_wait_selftest(int32_t* error_word, uint64_t limit_ns, cudaStream_t stream);

// Sets the text attn_last_error() returns on this thread.
void set_last_error(const std::string& msg);

// Sets a kernel's dynamic shared-memory limit on the current device before
// its first launch there (the attribute belongs to a device context, so a
// process that runs on several devices sets it once per device). `done` is
// the kernel's bitmask of devices already set; devices 64 and up are set on
// every launch.
template <typename Kernel>
cudaError_t ensure_smem_limit(Kernel kernel, int bytes, std::atomic<uint64_t>& done) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const uint64_t bit = (dev >= 0 && dev < 64) ? (uint64_t(1) << dev) : 0;
  if (bit && (done.load(std::memory_order_acquire) & bit)) return cudaSuccess;
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess && bit) done.fetch_or(bit, std::memory_order_acq_rel);
  return e;
}

// Copies `bytes` (a multiple of 16) from `src_dev` -- pinned host memory
// seen through its device mapping -- to device memory, with a kernel: the
// run that follows on the stream then waits on no other engine.
cudaError_t launch_copy_tables(void* dst, const void* src_dev, size_t bytes,
                               cudaStream_t stream);

// Writes O = 0 and LSE = -inf for `rows` rows of num_heads x head_dim (a
// plan whose requests hold no kv tokens at all: every visible set is empty).
cudaError_t launch_fill_empty(void* o, float* lse, int64_t rows, int32_t dtype,
                              cudaStream_t stream);

cudaError_t launch_merge_states(const void* o_a, const float* lse_a, const void* o_b,
                                const float* lse_b, void* o_out, float* lse_out,
                                int64_t rows, int32_t head_dim, int32_t dtype,
                                cudaStream_t stream);

}  // namespace attn
