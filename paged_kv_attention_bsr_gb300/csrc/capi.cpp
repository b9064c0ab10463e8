// capi.cpp -- the extern "C" boundary of libattn.so: argument validation,
// workspace sizing, plan upload and kernel dispatch. Declarations and the
// contract of every entry point are in include/attn.h.
#include <algorithm>
#include <cfloat>
#include <cmath>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <string>
#include <vector>

#include <nvtx3/nvToolsExt.h>

#include "internal.h"

using namespace attn;

namespace {

thread_local std::string g_err;

attn_status_t fail(attn_status_t s, const std::string& msg) {
  g_err = msg;
  return s;
}

attn_status_t cuda_fail(cudaError_t e, const char* what) {
  return fail(ATTN_ERR_CUDA, std::string(what) + ": " + cudaGetErrorString(e));
}

// NVTX range around an entry point (free when no profiler is attached).
struct NvtxRange {
  explicit NvtxRange(const char* name) { nvtxRangePushA(name); }
  ~NvtxRange() { nvtxRangePop(); }
  NvtxRange(const NvtxRange&) = delete;
  NvtxRange& operator=(const NvtxRange&) = delete;
};

// ATTN_DEBUG_CHECKS=1: the run calls read the device page table back and
// check it on the host before launching (slow: a synchronising copy).
bool debug_checks_enabled() {
  static int on = [] {
    const char* v = std::getenv("ATTN_DEBUG_CHECKS");
    return (v && v[0] && v[0] != '0') ? 1 : 0;
  }();
  return on != 0;
}

bool log_enabled() {
  static int on = [] {
    const char* v = std::getenv("ATTN_LOG");
    return (v && v[0] && v[0] != '0') ? 1 : 0;
  }();
  return on != 0;
}

// Pages a plan's requests hold in total (each item weighs its pages + 1).
// (Sum over items of their visible pages: 0 exactly when no request holds kv.)
int64_t plan_pages(const attn_plan_t& p) { return p.total_weight - p.num_items; }

// A plan whose requests hold no kv tokens at all: every row gets O = 0 and
// LSE = -inf without touching the (possibly empty) pool.
attn_status_t run_empty(const attn_plan_t* plan, void* o, float* lse, int64_t rows,
                        int32_t dtype, void* stream, const char* fn) {
  cudaError_t e = launch_fill_empty(o, lse, rows * plan->num_qo_heads, dtype,
                                    static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, fn);
  return ATTN_OK;
}

attn_status_t check_plan_common(const attn_plan_t* plan, int32_t mode, const void* q,
                                const void* k_pool, const void* v_pool, int64_t num_pages,
                                int32_t layout, const int32_t* kv_indptr,
                                const int32_t* kv_indices, const int32_t* last_page_len,
                                int32_t dtype, const void* o, const void* dev_ws,
                                size_t dev_bytes, const char* fn) {
  std::string f(fn);
  if (!plan) return fail(ATTN_ERR_INVALID_ARG, f + ": plan is NULL");
  if (plan->mode != mode)
    return fail(ATTN_ERR_INVALID_ARG, f + ": plan was made for the other mode");
  if (plan->head_dim != kHeadDim)
    return fail(ATTN_ERR_UNSUPPORTED, f + ": only head_dim == 128 is implemented");
  if (dtype != ATTN_F16 && dtype != ATTN_BF16)
    return fail(ATTN_ERR_INVALID_ARG, f + ": dtype must be ATTN_F16 or ATTN_BF16");
  if (layout != ATTN_LAYOUT_HND && layout != ATTN_LAYOUT_NHD)
    return fail(ATTN_ERR_INVALID_ARG, f + ": unknown layout");
  if (plan->batch > 0 && plan->total_qo > 0 &&
      (!q || !o || !kv_indptr || !last_page_len))
    return fail(ATTN_ERR_INVALID_ARG, f + ": null device pointer");
  if (plan_pages(*plan) > 0 && (!k_pool || !v_pool || !kv_indices || num_pages < 1))
    return fail(ATTN_ERR_INVALID_ARG, f + ": null KV pool or kv_indices, or an empty pool");
  if (num_pages < 0) return fail(ATTN_ERR_INVALID_ARG, f + ": num_pages < 0");
  if (!dev_ws) return fail(ATTN_ERR_INVALID_ARG, f + ": dev_ws is NULL");
  if (size_t(plan->dev_bytes_needed) > dev_bytes)
    return fail(ATTN_ERR_WORKSPACE_TOO_SMALL, f + ": device workspace smaller than the plan needs");
  if (reinterpret_cast<uintptr_t>(dev_ws) % 256 != 0)
    return fail(ATTN_ERR_INVALID_ARG, f + ": dev_ws must be 256-byte aligned");
  const uintptr_t align_mask = 15;
  if ((reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(k_pool) |
       reinterpret_cast<uintptr_t>(v_pool) | reinterpret_cast<uintptr_t>(o)) & align_mask)
    return fail(ATTN_ERR_INVALID_ARG, f + ": q, k_pool, v_pool and o must be 16-byte aligned");
  return ATTN_OK;
}

// The device page table a run will read, checked on the host against the
// pool and the plan: kv_indptr, last_page_len (and qo_indptr for append) must
// be the arrays the plan was made from (same fingerprint), and every
// kv_indices entry the kernels will read must lie in [0, num_pages).
// Skipped while `stream` is being captured into a graph.
attn_status_t debug_check_table(const attn_plan_t* plan, const int32_t* qo_indptr,
                                const int32_t* kv_indptr, const int32_t* kv_indices,
                                const int32_t* last_page_len, int64_t num_pages, void* stream,
                                const char* fn) {
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(st, &cap) != cudaSuccess || cap != cudaStreamCaptureStatusNone)
    return ATTN_OK;
  const std::string f(fn);
  const int32_t B = plan->batch;
  if (B == 0) return ATTN_OK;
  std::vector<int32_t> indptr(static_cast<size_t>(B) + 1), last(static_cast<size_t>(B)), qo;
  cudaError_t e = cudaMemcpyAsync(indptr.data(), kv_indptr, 4 * (size_t(B) + 1),
                                  cudaMemcpyDeviceToHost, st);
  if (e == cudaSuccess)
    e = cudaMemcpyAsync(last.data(), last_page_len, 4 * size_t(B), cudaMemcpyDeviceToHost, st);
  if (e == cudaSuccess && qo_indptr) {
    qo.resize(size_t(B) + 1);
    e = cudaMemcpyAsync(qo.data(), qo_indptr, 4 * (size_t(B) + 1), cudaMemcpyDeviceToHost, st);
  }
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) return cuda_fail(e, (f + ": debug check: page table read").c_str());
  if (plan_fingerprint(qo_indptr ? qo.data() : nullptr, indptr.data(), last.data(), B,
                       plan->page_size, plan->num_qo_heads, plan->num_kv_heads, plan->head_dim,
                       plan->causal, plan->num_ctas) != plan->fingerprint)
    return fail(ATTN_ERR_INVALID_ARG, f + ": debug check: kv_indptr / last_page_len / qo_indptr "
                                          "on the device differ from the plan's host copies");
  const int64_t pages = int64_t(indptr[size_t(B)]) - indptr[0];
  if (pages <= 0) return ATTN_OK;
  std::vector<int32_t> idx(static_cast<size_t>(pages));
  e = cudaMemcpyAsync(idx.data(), kv_indices + indptr[0], 4 * size_t(pages),
                      cudaMemcpyDeviceToHost, st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) return cuda_fail(e, (f + ": debug check: kv_indices read").c_str());
  for (int64_t i = 0; i < pages; ++i)
    if (idx[size_t(i)] < 0 || idx[size_t(i)] >= num_pages) {
      char buf[160];
      std::snprintf(buf, sizeof buf,
                    ": debug check: kv_indices[%lld] = %d is outside [0, num_pages = %lld)",
                    (long long)(indptr[0] + i), idx[size_t(i)], (long long)num_pages);
      return fail(ATTN_ERR_INVALID_ARG, f + buf);
    }
  return ATTN_OK;
}

// debug_check_table for a composable-format run: both tables and qo_indptr
// must be the plan's (fingerprint), every index the run reads in range.
attn_status_t debug_check_cascade(const attn_plan_t* plan, const int32_t* qo_indptr,
                                  const int32_t* kv_indptr0, const int32_t* kv_indices0,
                                  const int32_t* last0, int64_t num_pages0,
                                  const int32_t* kv_indptr1, const int32_t* kv_indices1,
                                  const int32_t* last1, int64_t num_pages1, void* stream,
                                  const char* fn) {
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(st, &cap) != cudaSuccess || cap != cudaStreamCaptureStatusNone)
    return ATTN_OK;
  const std::string f(fn);
  const int32_t prompts = plan->batch, B = plan->total_qo;
  if (prompts == 0) return ATTN_OK;
  auto read = [&](std::vector<int32_t>& dst, const int32_t* src, int64_t n) -> cudaError_t {
    dst.resize(static_cast<size_t>(n));
    if (n == 0) return cudaSuccess;
    return cudaMemcpyAsync(dst.data(), src, 4 * size_t(n), cudaMemcpyDeviceToHost, st);
  };
  std::vector<int32_t> qo, ip0, l0, ip1, l1;
  cudaError_t e = read(qo, qo_indptr, int64_t(prompts) + 1);
  if (e == cudaSuccess) e = read(ip0, kv_indptr0, int64_t(prompts) + 1);
  if (e == cudaSuccess) e = read(l0, last0, prompts);
  if (e == cudaSuccess) e = read(ip1, kv_indptr1, int64_t(B) + 1);
  if (e == cudaSuccess) e = read(l1, last1, B);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) return cuda_fail(e, (f + ": debug check: page table read").c_str());
  if (qo[size_t(prompts)] != B ||
      cascade_fingerprint(qo.data(), ip0.data(), l0.data(), plan->page_size, ip1.data(),
                          l1.data(), plan->page_size_suffix, prompts, plan->num_qo_heads,
                          plan->num_kv_heads, plan->head_dim, plan->num_ctas) != plan->fingerprint)
    return fail(ATTN_ERR_INVALID_ARG, f + ": debug check: qo_indptr / kv_indptr / last_page_len "
                                          "on the device differ from the plan's host copies");
  const int32_t* tabs[2] = {kv_indices0, kv_indices1};
  const std::vector<int32_t>* ips[2] = {&ip0, &ip1};
  const int64_t lim[2] = {num_pages0, num_pages1};
  for (int t = 0; t < 2; ++t) {
    const std::vector<int32_t>& ip = *ips[t];
    const int64_t pages = int64_t(ip.back()) - ip.front();
    if (pages <= 0) continue;
    std::vector<int32_t> idx;
    e = read(idx, tabs[t] + ip.front(), pages);
    if (e == cudaSuccess) e = cudaStreamSynchronize(st);
    if (e != cudaSuccess) return cuda_fail(e, (f + ": debug check: kv_indices read").c_str());
    for (int64_t i = 0; i < pages; ++i)
      if (idx[size_t(i)] < 0 || idx[size_t(i)] >= lim[t]) {
        char buf[200];
        std::snprintf(buf, sizeof buf,
                      ": debug check: %s kv_indices[%lld] = %d is outside [0, num_pages = %lld)",
                      t == 0 ? "prefix" : "suffix", (long long)(ip.front() + i), idx[size_t(i)],
                      (long long)lim[t]);
        return fail(ATTN_ERR_INVALID_ARG, f + buf);
      }
  }
  return ATTN_OK;
}

// Copies a plan's tables from the pinned staging area into the device
// workspace (after the shared checks); dev_ws NULL = host-only planning.
attn_status_t upload_plan(const attn_plan_t* plan, const void* pinned_host_ws, void* dev_ws,
                          size_t dev_bytes, void* stream, const char* fn) {
  if (!dev_ws) return ATTN_OK;
  const std::string f(fn);
  if (size_t(plan->dev_bytes_needed) > dev_bytes)
    return fail(ATTN_ERR_WORKSPACE_TOO_SMALL, f + ": device workspace too small");
  if (reinterpret_cast<uintptr_t>(dev_ws) % 256 != 0)
    return fail(ATTN_ERR_INVALID_ARG, f + ": dev_ws must be 256-byte aligned");
  // Pinned memory that the device can address (every page-locked
  // allocation on a system with unified addressing, such as a Grace-Blackwell
  // node) is read by a copy kernel, so that the run kernel behind it on the
  // stream starts without a copy-engine -> compute hand-off (3 to 4 us per
  // run); other memory goes through cudaMemcpyAsync.
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const size_t bytes = size_t(plan->table_bytes);
  cudaPointerAttributes attr;
  const void* src_dev = nullptr;
  if (bytes % 16 == 0 && reinterpret_cast<uintptr_t>(pinned_host_ws) % 16 == 0 &&
      cudaPointerGetAttributes(&attr, pinned_host_ws) == cudaSuccess &&
      attr.type == cudaMemoryTypeHost && attr.devicePointer != nullptr)
    src_dev = attr.devicePointer;
  else
    cudaGetLastError();  // clear a lookup failure on unregistered memory
  cudaError_t e = src_dev ? launch_copy_tables(dev_ws, src_dev, bytes, st)
                          : cudaMemcpyAsync(dev_ws, pinned_host_ws, bytes,
                                            cudaMemcpyHostToDevice, st);
  if (e != cudaSuccess) return cuda_fail(e, (f + ": table upload").c_str());
  return ATTN_OK;
}

}  // namespace

namespace attn {
void set_last_error(const std::string& msg) { g_err = msg; }
}  // namespace attn

namespace {

// sm_scale as the kernels take it. The kernels scale a row's maximum over the
// unscaled scores, so the scale must be finite and >= 0. A zero scale (equal
// weights over the visible keys) runs as the smallest normal float: the same
// weights, while masked scores (-inf) still scale to -inf rather than NaN.
bool scale_for_kernels(float* sm_scale) {
  if (!std::isfinite(*sm_scale) || *sm_scale < 0.f) return false;
  if (*sm_scale == 0.f) *sm_scale = FLT_MIN;
  return true;
}

// Arguments of the few-row tensor-core kernel for a decode plan.
attn::AppendArgs decode_tc_args(const attn_plan_t* plan, const void* q, const void* k_pool,
                                const void* v_pool, int64_t num_pages, int32_t layout,
                                const int32_t* kv_indptr, const int32_t* kv_indices,
                                const int32_t* last_page_len, int32_t dtype, float sm_scale,
                                void* o, float* lse, void* dev_ws) {
  const int32_t group = plan->num_qo_heads / plan->num_kv_heads;
  attn::AppendArgs a;
  std::memset(&a, 0, sizeof a);
  a.q = q;
  a.qo_indptr = nullptr;
  a.k_pool = k_pool;
  a.v_pool = v_pool;
  a.num_pages = num_pages;
  a.kv_indptr = kv_indptr;
  a.kv_indices = kv_indices;
  a.last_page_len = last_page_len;
  a.o = o;
  a.lse = lse;
  a.ws = attn::ws_view(*plan, dev_ws);
  a.num_ctas = plan->num_ctas;
  a.num_units = plan->num_units;
  a.num_split_items = plan->num_split_items;
  a.dtype = dtype;
  a.page_size = plan->page_size;
  a.num_qo_heads = plan->num_qo_heads;
  a.num_kv_heads = plan->num_kv_heads;
  a.group = group;
  a.q_tile = 1;
  a.tile_tokens = 1;
  a.rows_per_item = group;
  a.total_qo = plan->batch;
  a.max_qo_len = 1;
  a.causal = 0;
  a.sm_scale = sm_scale;
  a.rope_cos = nullptr;
  a.rope_sin = nullptr;
  a.layout = layout;
  return a;
}

// Validation shared by the append entry points.
attn_status_t check_append(const attn_plan_t* plan, const void* q, const int32_t* qo_indptr,
                           const void* k_pool, const void* v_pool, int64_t num_pages,
                           int32_t layout, const int32_t* kv_indptr, const int32_t* kv_indices,
                           const int32_t* last_page_len, int32_t dtype, int32_t causal, void* o,
                           void* dev_ws, size_t dev_bytes, const char* fn) {
  attn_status_t s = check_plan_common(plan, ATTN_MODE_APPEND, q, k_pool, v_pool, num_pages,
                                      layout, kv_indptr, kv_indices, last_page_len, dtype, o,
                                      dev_ws, dev_bytes, fn);
  if (s != ATTN_OK) return s;
  if ((causal ? 1 : 0) != plan->causal)
    return fail(ATTN_ERR_INVALID_ARG, std::string(fn) + ": causal differs from the plan's");
  if (plan->batch > 0 && !qo_indptr)
    return fail(ATTN_ERR_INVALID_ARG, std::string(fn) + ": qo_indptr is NULL");
  return ATTN_OK;
}

// Kernel arguments of an append run (no RoPE).
attn::AppendArgs append_args(const attn_plan_t* plan, const void* q, const int32_t* qo_indptr,
                             const void* k_pool, const void* v_pool, int64_t num_pages,
                             int32_t layout, const int32_t* kv_indptr, const int32_t* kv_indices,
                             const int32_t* last_page_len, int32_t dtype, float sm_scale,
                             void* o, float* lse, void* dev_ws) {
  attn::AppendArgs a;
  std::memset(&a, 0, sizeof a);
  a.q = q;
  a.qo_indptr = qo_indptr;
  a.k_pool = k_pool;
  a.v_pool = v_pool;
  a.num_pages = num_pages;
  a.kv_indptr = kv_indptr;
  a.kv_indices = kv_indices;
  a.last_page_len = last_page_len;
  a.o = o;
  a.lse = lse;
  a.ws = ws_view(*plan, dev_ws);
  a.num_ctas = plan->num_ctas;
  a.num_units = plan->num_units;
  a.num_split_items = plan->num_split_items;
  a.dtype = dtype;
  a.page_size = plan->page_size;
  a.num_qo_heads = plan->num_qo_heads;
  a.num_kv_heads = plan->num_kv_heads;
  a.group = plan->num_qo_heads / plan->num_kv_heads;
  a.q_tile = plan->q_tile;
  a.tile_tokens = attn::kTileRows / a.group;
  a.rows_per_item = plan->rows_per_item;
  a.total_qo = plan->total_qo;
  a.max_qo_len = plan->max_qo_len;
  a.causal = plan->causal;
  a.sm_scale = sm_scale;
  a.layout = layout;
  return a;
}

// Checks of the cos / sin tables of a RoPE run.
attn_status_t check_rope(const attn_plan_t* plan, const float* rope_cos, const float* rope_sin,
                         int64_t rope_max_pos, const char* fn) {
  if (!rope_cos || !rope_sin)
    return fail(ATTN_ERR_INVALID_ARG, std::string(fn) + ": null cos / sin table");
  if ((reinterpret_cast<uintptr_t>(rope_cos) | reinterpret_cast<uintptr_t>(rope_sin)) & 15u)
    return fail(ATTN_ERR_INVALID_ARG, std::string(fn) + ": cos / sin tables must be 16-byte aligned");
  if (rope_max_pos < plan->max_kv_len)
    return fail(ATTN_ERR_INVALID_ARG,
                std::string(fn) + ": the cos / sin tables must cover every kv position "
                                  "(rope_max_pos >= the plan's longest kv length)");
  return ATTN_OK;
}

// An append run: short appends (group x longest query count <= 16 packed
// rows, e.g. the n generations of a shared prefix) on the few-row kernel,
// which keeps the softmax off the critical path of an HBM-bound pass and
// merges split items itself; longer ones on the append kernel, then the
// merge of its split items.
attn_status_t run_append_kernels(const attn_plan_t* plan, const attn::AppendArgs& a,
                                 const int32_t* qo_indptr, void* o, float* lse, int32_t dtype,
                                 void* stream, const char* fn) {
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const char* msg = "";
  const std::string f(fn);
  if (few_row_rows(a.group, a.max_qo_len) != 0) {
    cudaError_t e = launch_decode_tc(a, st, &msg);
    if (e == cudaErrorNotSupported) return fail(ATTN_ERR_UNSUPPORTED, msg);
    if (e != cudaSuccess) return cuda_fail(e, (f + ": few-row kernel launch").c_str());
    return ATTN_OK;
  }
  cudaError_t e = launch_append(a, st, &msg);
  if (e == cudaErrorNotSupported) return fail(ATTN_ERR_UNSUPPORTED, msg);
  if (e != cudaSuccess) return cuda_fail(e, (f + ": append kernel launch").c_str());
  if (plan->num_split_items > 0) {
    SplitMergeArgs m;
    m.ws = a.ws;
    m.num_split_items = plan->num_split_items;
    m.rows_per_item = plan->rows_per_item;
    m.group = a.group;
    m.q_tile = plan->q_tile;
    m.num_qo_heads = plan->num_qo_heads;
    m.qo_indptr = qo_indptr;
    m.o = o;
    m.lse = lse;
    m.dtype = dtype;
    e = launch_split_merge(m, st);
    if (e != cudaSuccess) return cuda_fail(e, (f + ": merge kernel launch").c_str());
  }
  return ATTN_OK;
}

// The few-row tensor-core kernel takes this decode shape.
bool decode_tc_shape(const attn_plan_t* plan, int32_t layout) {
  const int32_t group = plan->num_qo_heads / plan->num_kv_heads;
  return group >= attn::kTensorDecodeGroup && (group & (group - 1)) == 0 && group <= 8 &&
         (layout == ATTN_LAYOUT_HND || layout == ATTN_LAYOUT_NHD);
}

}  // namespace

extern "C" {

const char* attn_last_error(void) { return g_err.c_str(); }

attn_status_t attn_workspace_size(int32_t max_batch, int32_t max_total_qo,
                                  int32_t num_qo_heads, int32_t num_kv_heads,
                                  int32_t head_dim, int32_t num_ctas, size_t* dev_bytes,
                                  size_t* pinned_host_bytes) {
  if (!dev_bytes || !pinned_host_bytes)
    return fail(ATTN_ERR_INVALID_ARG, "attn_workspace_size: null output pointer");
  if (max_batch < 1 || max_total_qo < 0 || num_qo_heads < 1 || num_kv_heads < 1 ||
      num_ctas < 1)
    return fail(ATTN_ERR_INVALID_ARG, "attn_workspace_size: sizes must be positive");
  if (num_qo_heads % num_kv_heads)
    return fail(ATTN_ERR_INVALID_ARG,
                "attn_workspace_size: num_qo_heads must be a multiple of num_kv_heads");
  if (head_dim != kHeadDim)
    return fail(ATTN_ERR_UNSUPPORTED, "attn_workspace_size: only head_dim == 128");
  const int64_t group = num_qo_heads / num_kv_heads;
  const bool append_ok = (kTileRows % group == 0);
  const int64_t q_tile = append_ok ? kItemRows / group : 1;
  int64_t items = int64_t(max_batch) * num_kv_heads;
  if (append_ok)
    items = std::max<int64_t>(
        items, int64_t(num_kv_heads) * ((int64_t(max_total_qo) + q_tile - 1) / q_tile + max_batch));
  const int64_t C = num_ctas;
  // the cut adds at most C units; each extra unit cuts at most one item
  const int64_t units = items + C;
  const int64_t split = std::min<int64_t>(items, C);
  const int64_t slots = std::min<int64_t>(units, 2 * C);
  const int32_t rows = append_ok ? kItemRows : int32_t(group);
  const PlanLayout L = plan_layout(num_ctas, units, split, slots, rows, head_dim);
  *dev_bytes = size_t(L.dev_bytes);
  *pinned_host_bytes = size_t(L.table_bytes);
  return ATTN_OK;
}

attn_status_t attn_default_num_ctas(int32_t device, int32_t mode, int32_t* num_ctas) {
  if (!num_ctas) return fail(ATTN_ERR_INVALID_ARG, "attn_default_num_ctas: null output");
  if (mode != ATTN_MODE_DECODE && mode != ATTN_MODE_APPEND && mode != ATTN_MODE_CASCADE)
    return fail(ATTN_ERR_INVALID_ARG, "attn_default_num_ctas: unknown mode");
  int sms = 0;
  cudaError_t e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device);
  if (e != cudaSuccess) return cuda_fail(e, "attn_default_num_ctas");
  // cascade: the few-row kernel, one CTA per SM
  const int per_sm = mode == ATTN_MODE_DECODE   ? decode_ctas_per_sm()
                     : mode == ATTN_MODE_APPEND ? append_ctas_per_sm()
                                                : 1;
  *num_ctas = sms * per_sm;
  return ATTN_OK;
}

attn_status_t attn_plan(const int32_t* qo_indptr_h, const int32_t* kv_indptr_h,
                        const int32_t* last_page_len_h, int32_t batch, int32_t page_size,
                        int32_t num_qo_heads, int32_t num_kv_heads, int32_t head_dim,
                        int32_t causal, int32_t num_ctas, void* pinned_host_ws,
                        size_t pinned_bytes, void* dev_ws, size_t dev_bytes, void* stream,
                        attn_plan_t* plan_out) {
  NvtxRange nvtx("attn_plan");
  const char* msg = "";
  attn_status_t s = build_plan(qo_indptr_h, kv_indptr_h, last_page_len_h, batch, page_size,
                               num_qo_heads, num_kv_heads, head_dim, causal, num_ctas,
                               pinned_host_ws, pinned_bytes, plan_out, &msg);
  if (s != ATTN_OK) return fail(s, msg);
  if (log_enabled()) {
    const attn_plan_t& p = *plan_out;
    std::fprintf(stderr,
                 "[attn] plan mode=%s batch=%d items=%d units=%d split=%d slots=%d ctas=%d "
                 "W=%lld max_cta=%lld mean_cta=%.1f\n",
                 p.mode == ATTN_MODE_DECODE ? "decode" : "append", p.batch, p.num_items,
                 p.num_units, p.num_split_items, p.num_slots, p.num_ctas,
                 (long long)p.total_weight, (long long)p.max_cta_weight,
                 double(p.total_weight) / p.num_ctas);
  }
  return upload_plan(plan_out, pinned_host_ws, dev_ws, dev_bytes, stream, "attn_plan");
}

attn_status_t attn_cascade_workspace_size(int32_t max_prompts, int32_t max_batch,
                                          int32_t num_qo_heads, int32_t num_kv_heads,
                                          int32_t head_dim, int32_t num_ctas,
                                          size_t* dev_bytes, size_t* pinned_host_bytes) {
  if (!dev_bytes || !pinned_host_bytes)
    return fail(ATTN_ERR_INVALID_ARG, "attn_cascade_workspace_size: null output pointer");
  if (max_prompts < 1 || max_batch < 0 || num_qo_heads < 1 || num_kv_heads < 1 || num_ctas < 1)
    return fail(ATTN_ERR_INVALID_ARG, "attn_cascade_workspace_size: sizes must be positive");
  if (num_qo_heads % num_kv_heads)
    return fail(ATTN_ERR_INVALID_ARG, "attn_cascade_workspace_size: num_qo_heads must be a "
                                      "multiple of num_kv_heads");
  if (head_dim != kHeadDim)
    return fail(ATTN_ERR_UNSUPPORTED, "attn_cascade_workspace_size: only head_dim == 128");
  // a segment per (prompt, kv head) and per (generation, kv head); each CTA
  // boundary cuts at most one segment in two; every unit has a slot
  const int64_t items = int64_t(max_prompts) * num_kv_heads;
  const int64_t units = (int64_t(max_prompts) + max_batch) * num_kv_heads + num_ctas;
  const PlanLayout L = plan_layout(num_ctas, units, items, units, kFewRowMax, head_dim);
  *dev_bytes = size_t(L.dev_bytes);
  *pinned_host_bytes = size_t(L.table_bytes);
  return ATTN_OK;
}

attn_status_t attn_plan_cascade(const int32_t* qo_indptr_h, const int32_t* kv_indptr_prefix_h,
                                const int32_t* last_page_len_prefix_h, int32_t page_size_prefix,
                                const int32_t* kv_indptr_suffix_h,
                                const int32_t* last_page_len_suffix_h, int32_t page_size_suffix,
                                int32_t num_prompts, int32_t num_qo_heads, int32_t num_kv_heads,
                                int32_t head_dim, int32_t num_ctas, void* pinned_host_ws,
                                size_t pinned_bytes, void* dev_ws, size_t dev_bytes,
                                void* stream, attn_plan_t* plan_out) {
  NvtxRange nvtx("attn_plan_cascade");
  const char* msg = "";
  attn_status_t s = build_cascade_plan(
      qo_indptr_h, kv_indptr_prefix_h, last_page_len_prefix_h, page_size_prefix,
      kv_indptr_suffix_h, last_page_len_suffix_h, page_size_suffix, num_prompts, num_qo_heads,
      num_kv_heads, head_dim, num_ctas, pinned_host_ws, pinned_bytes, plan_out, &msg);
  if (s != ATTN_OK) return fail(s, msg);
  if (log_enabled()) {
    const attn_plan_t& p = *plan_out;
    std::fprintf(stderr,
                 "[attn] plan mode=cascade prompts=%d batch=%d items=%d units=%d rows=%d "
                 "ctas=%d max_cta_tokens=%lld\n",
                 p.batch, p.total_qo, p.num_items, p.num_units, p.rows_per_item, p.num_ctas,
                 (long long)p.max_cta_weight);
  }
  return upload_plan(plan_out, pinned_host_ws, dev_ws, dev_bytes, stream, "attn_plan_cascade");
}

attn_status_t attn_cascade_run(const attn_plan_t* plan, const void* q, const int32_t* qo_indptr,
                               const void* k_prefix, const void* v_prefix,
                               int64_t num_pages_prefix, const int32_t* kv_indptr_prefix,
                               const int32_t* kv_indices_prefix,
                               const int32_t* last_page_len_prefix, const void* k_suffix,
                               const void* v_suffix, int64_t num_pages_suffix,
                               const int32_t* kv_indptr_suffix, const int32_t* kv_indices_suffix,
                               const int32_t* last_page_len_suffix, int32_t layout,
                               int32_t dtype, float sm_scale, void* o, float* lse,
                               void* dev_ws, size_t dev_bytes, void* stream) {
  NvtxRange nvtx("attn_cascade_run");
  if (!scale_for_kernels(&sm_scale))
    return fail(ATTN_ERR_INVALID_ARG, "attn_cascade_run: sm_scale must be finite and >= 0");
  const char* fn = "attn_cascade_run";
  const std::string f(fn);
  attn_status_t s = check_plan_common(plan, ATTN_MODE_CASCADE, q, k_prefix, v_prefix,
                                      num_pages_prefix, layout, kv_indptr_prefix,
                                      kv_indices_prefix, last_page_len_prefix, dtype, o, dev_ws,
                                      dev_bytes, fn);
  if (s != ATTN_OK) return s;
  if (plan_pages(*plan) > 0 &&
      (!k_suffix || !v_suffix || !kv_indices_suffix || num_pages_suffix < 1))
    return fail(ATTN_ERR_INVALID_ARG, f + ": null suffix pool or kv_indices, or an empty pool");
  if (num_pages_suffix < 0) return fail(ATTN_ERR_INVALID_ARG, f + ": num_pages_suffix < 0");
  if ((reinterpret_cast<uintptr_t>(k_suffix) | reinterpret_cast<uintptr_t>(v_suffix)) & 15u)
    return fail(ATTN_ERR_INVALID_ARG, f + ": the suffix pools must be 16-byte aligned");
  if (plan->batch > 0 && plan->total_qo > 0 &&
      (!qo_indptr || !kv_indptr_suffix || !last_page_len_suffix))
    return fail(ATTN_ERR_INVALID_ARG, f + ": null device pointer");
  if (debug_checks_enabled()) {
    s = debug_check_cascade(plan, qo_indptr, kv_indptr_prefix, kv_indices_prefix,
                            last_page_len_prefix, num_pages_prefix, kv_indptr_suffix,
                            kv_indices_suffix, last_page_len_suffix, num_pages_suffix, stream,
                            fn);
    if (s != ATTN_OK) return s;
  }
  if (plan->batch == 0 || plan->total_qo == 0) return ATTN_OK;
  if (plan_pages(*plan) == 0)
    return run_empty(plan, o, lse, plan->total_qo, dtype, stream, fn);
  AppendArgs a = append_args(plan, q, qo_indptr, k_prefix, v_prefix, num_pages_prefix,
                             layout, kv_indptr_prefix, kv_indices_prefix,
                             last_page_len_prefix, dtype, sm_scale, o, lse, dev_ws);
  a.cascade = 1;
  a.page_size2 = plan->page_size_suffix;
  a.k_pool2 = k_suffix;
  a.v_pool2 = v_suffix;
  a.num_pages2 = num_pages_suffix;
  a.kv_indices2 = kv_indices_suffix;
  const char* msg = "";
  cudaError_t e = launch_decode_tc(a, static_cast<cudaStream_t>(stream), &msg);
  if (e == cudaErrorNotSupported) return fail(ATTN_ERR_UNSUPPORTED, msg);
  if (e != cudaSuccess) return cuda_fail(e, "attn_cascade_run: kernel launch");
  return ATTN_OK;
}

attn_status_t attn_decode_run(const attn_plan_t* plan, const void* q, const void* k_pool,
                              const void* v_pool, int64_t num_pages, int32_t layout,
                              const int32_t* kv_indptr, const int32_t* kv_indices,
                              const int32_t* last_page_len, int32_t dtype, float sm_scale,
                              void* o, float* lse, void* dev_ws, size_t dev_bytes,
                              void* stream) {
  NvtxRange nvtx("attn_decode_run");
  if (!scale_for_kernels(&sm_scale))
    return fail(ATTN_ERR_INVALID_ARG, "attn_decode_run: sm_scale must be finite and >= 0");
  attn_status_t s = check_plan_common(plan, ATTN_MODE_DECODE, q, k_pool, v_pool, num_pages,
                                      layout, kv_indptr, kv_indices, last_page_len, dtype, o,
                                      dev_ws, dev_bytes, "attn_decode_run");
  if (s != ATTN_OK) return s;
  if (debug_checks_enabled()) {
    s = debug_check_table(plan, nullptr, kv_indptr, kv_indices, last_page_len, num_pages,
                          stream, "attn_decode_run");
    if (s != ATTN_OK) return s;
  }
  const int32_t group = plan->num_qo_heads / plan->num_kv_heads;
  if (group > kMaxDecodeGroup)
    return fail(ATTN_ERR_UNSUPPORTED, "attn_decode_run: group > 8 is not implemented");
  if (plan->batch == 0) return ATTN_OK;
  if (plan_pages(*plan) == 0)
    return run_empty(plan, o, lse, plan->batch, dtype, stream, "attn_decode_run");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (decode_tc_shape(plan, layout)) {
    // Tensor-core decode: Q K^T and P V run as M = 128 MMAs over 128-token
    // tiles gathered by TMA, the softmax on one warp (query heads replicated
    // across the MMA rows so that each thread handles a slice of the tile).
    const AppendArgs a = decode_tc_args(plan, q, k_pool, v_pool, num_pages, layout, kv_indptr,
                                        kv_indices, last_page_len, dtype, sm_scale, o, lse,
                                        dev_ws);
    const char* msg = "";
    cudaError_t e = launch_decode_tc(a, st, &msg);  // merges split items itself
    if (e == cudaErrorNotSupported) return fail(ATTN_ERR_UNSUPPORTED, msg);
    if (e != cudaSuccess) return cuda_fail(e, "attn_decode_run: tensor-core decode launch");
    return ATTN_OK;
  }
  DecodeArgs a;
  a.q = q;
  a.k_pool = k_pool;
  a.v_pool = v_pool;
  a.kv_indptr = kv_indptr;
  a.kv_indices = kv_indices;
  a.last_page_len = last_page_len;
  a.o = o;
  a.lse = lse;
  a.ws = ws_view(*plan, dev_ws);
  a.num_ctas = plan->num_ctas;
  a.num_units = plan->num_units;
  a.num_split_items = plan->num_split_items;
  a.layout = layout;
  a.dtype = dtype;
  a.page_size = plan->page_size;
  a.num_qo_heads = plan->num_qo_heads;
  a.num_kv_heads = plan->num_kv_heads;
  a.group = group;
  a.batch = plan->batch;
  a.sm_scale = sm_scale;
  a.kv_fp8 = 0;
  a.k_scale = nullptr;
  a.v_scale = nullptr;
  cudaError_t e = launch_decode(a, st);  // split items are merged inside the kernel
  if (e != cudaSuccess) return cuda_fail(e, "attn_decode_run: decode kernel launch");
  return ATTN_OK;
}

attn_status_t attn_decode_run_fp8(const attn_plan_t* plan, const void* q, const void* k_pool,
                                  const void* v_pool, int64_t num_pages, int32_t layout,
                                  const int32_t* kv_indptr, const int32_t* kv_indices,
                                  const int32_t* last_page_len, int32_t dtype,
                                  const float* k_scale, const float* v_scale, float sm_scale,
                                  void* o, float* lse, void* dev_ws, size_t dev_bytes,
                                  void* stream) {
  NvtxRange nvtx("attn_decode_run_fp8");
  if (!scale_for_kernels(&sm_scale))
    return fail(ATTN_ERR_INVALID_ARG, "attn_decode_run_fp8: sm_scale must be finite and >= 0");
  attn_status_t s = check_plan_common(plan, ATTN_MODE_DECODE, q, k_pool, v_pool, num_pages,
                                      layout, kv_indptr, kv_indices, last_page_len, dtype, o,
                                      dev_ws, dev_bytes, "attn_decode_run_fp8");
  if (s != ATTN_OK) return s;
  if (debug_checks_enabled()) {
    s = debug_check_table(plan, nullptr, kv_indptr, kv_indices, last_page_len, num_pages,
                          stream, "attn_decode_run_fp8");
    if (s != ATTN_OK) return s;
  }
  if (plan->num_qo_heads / plan->num_kv_heads > kMaxDecodeGroup)
    return fail(ATTN_ERR_UNSUPPORTED, "attn_decode_run_fp8: group > 8 is not implemented");
  if (plan_pages(*plan) > 0 && (!k_scale || !v_scale))
    return fail(ATTN_ERR_INVALID_ARG, "attn_decode_run_fp8: null k_scale / v_scale");
  if (plan->batch == 0) return ATTN_OK;
  if (plan_pages(*plan) == 0)
    return run_empty(plan, o, lse, plan->batch, dtype, stream, "attn_decode_run_fp8");
  if (decode_tc_shape(plan, layout) && layout == ATTN_LAYOUT_HND && plan->page_size % 16 == 0) {
    // Tensor cores: TMA stages the E4M3 tiles, warps widen them to f16 in
    // shared memory, the MMAs multiply f16 (q converted when bf16).
    AppendArgs t = decode_tc_args(plan, q, k_pool, v_pool, num_pages, layout, kv_indptr,
                                  kv_indices, last_page_len, dtype, sm_scale, o, lse, dev_ws);
    t.kv_fp8 = 1;
    t.k_scale = k_scale;
    t.v_scale = v_scale;
    const char* msg = "";
    cudaError_t e = launch_decode_tc(t, static_cast<cudaStream_t>(stream), &msg);
    if (e == cudaErrorNotSupported) return fail(ATTN_ERR_UNSUPPORTED, msg);
    if (e != cudaSuccess) return cuda_fail(e, "attn_decode_run_fp8: tensor-core kernel launch");
    return ATTN_OK;
  }
  DecodeArgs a;
  a.q = q;
  a.k_pool = k_pool;
  a.v_pool = v_pool;
  a.kv_indptr = kv_indptr;
  a.kv_indices = kv_indices;
  a.last_page_len = last_page_len;
  a.o = o;
  a.lse = lse;
  a.ws = ws_view(*plan, dev_ws);
  a.num_ctas = plan->num_ctas;
  a.num_units = plan->num_units;
  a.num_split_items = plan->num_split_items;
  a.layout = layout;
  a.dtype = dtype;
  a.page_size = plan->page_size;
  a.num_qo_heads = plan->num_qo_heads;
  a.num_kv_heads = plan->num_kv_heads;
  a.group = plan->num_qo_heads / plan->num_kv_heads;
  a.batch = plan->batch;
  a.sm_scale = sm_scale;
  a.kv_fp8 = 1;
  a.k_scale = k_scale;
  a.v_scale = v_scale;
  cudaError_t e = launch_decode(a, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "attn_decode_run_fp8: decode kernel launch");
  return ATTN_OK;
}

attn_status_t attn_decode_run_rope(const attn_plan_t* plan, const void* q, const void* k_pool,
                                   const void* v_pool, int64_t num_pages, int32_t layout,
                                   const int32_t* kv_indptr, const int32_t* kv_indices,
                                   const int32_t* last_page_len, int32_t dtype, float sm_scale,
                                   const float* rope_cos, const float* rope_sin,
                                   int64_t rope_max_pos, void* o, float* lse, void* dev_ws,
                                   size_t dev_bytes, void* stream) {
  NvtxRange nvtx("attn_decode_run_rope");
  if (!scale_for_kernels(&sm_scale))
    return fail(ATTN_ERR_INVALID_ARG, "attn_decode_run_rope: sm_scale must be finite and >= 0");
  attn_status_t s = check_plan_common(plan, ATTN_MODE_DECODE, q, k_pool, v_pool, num_pages,
                                      layout, kv_indptr, kv_indices, last_page_len, dtype, o,
                                      dev_ws, dev_bytes, "attn_decode_run_rope");
  if (s != ATTN_OK) return s;
  if (debug_checks_enabled()) {
    s = debug_check_table(plan, nullptr, kv_indptr, kv_indices, last_page_len, num_pages,
                          stream, "attn_decode_run_rope");
    if (s != ATTN_OK) return s;
  }
  s = check_rope(plan, rope_cos, rope_sin, rope_max_pos, "attn_decode_run_rope");
  if (s != ATTN_OK) return s;
  if (!decode_tc_shape(plan, layout))
    return fail(ATTN_ERR_UNSUPPORTED,
                "attn_decode_run_rope: fused RoPE needs 2, 4 or 8 query heads per kv head");
  if (plan->batch == 0) return ATTN_OK;
  if (plan_pages(*plan) == 0)
    return run_empty(plan, o, lse, plan->batch, dtype, stream, "attn_decode_run_rope");
  AppendArgs a = decode_tc_args(plan, q, k_pool, v_pool, num_pages, layout, kv_indptr,
                                kv_indices, last_page_len, dtype, sm_scale, o, lse, dev_ws);
  a.rope_cos = rope_cos;
  a.rope_sin = rope_sin;
  a.rope_rows = rope_max_pos;
  const char* msg = "";
  cudaError_t e = launch_decode_tc(a, static_cast<cudaStream_t>(stream), &msg);
  if (e == cudaErrorNotSupported) return fail(ATTN_ERR_UNSUPPORTED, msg);
  if (e != cudaSuccess) return cuda_fail(e, "attn_decode_run_rope: kernel launch");
  return ATTN_OK;
}

attn_status_t attn_append_run(const attn_plan_t* plan, const void* q,
                              const int32_t* qo_indptr, const void* k_pool,
                              const void* v_pool, int64_t num_pages, int32_t layout,
                              const int32_t* kv_indptr, const int32_t* kv_indices,
                              const int32_t* last_page_len, int32_t dtype, int32_t causal,
                              float sm_scale, void* o, float* lse, void* dev_ws,
                              size_t dev_bytes, void* stream) {
  NvtxRange nvtx("attn_append_run");
  if (!scale_for_kernels(&sm_scale))
    return fail(ATTN_ERR_INVALID_ARG, "attn_append_run: sm_scale must be finite and >= 0");
  attn_status_t s = check_append(plan, q, qo_indptr, k_pool, v_pool, num_pages, layout,
                                 kv_indptr, kv_indices, last_page_len, dtype, causal, o,
                                 dev_ws, dev_bytes, "attn_append_run");
  if (s != ATTN_OK) return s;
  if (debug_checks_enabled()) {
    s = debug_check_table(plan, qo_indptr, kv_indptr, kv_indices, last_page_len, num_pages,
                          stream, "attn_append_run");
    if (s != ATTN_OK) return s;
  }
  if (plan->batch == 0 || plan->total_qo == 0) return ATTN_OK;
  if (plan_pages(*plan) == 0)
    return run_empty(plan, o, lse, plan->total_qo, dtype, stream, "attn_append_run");
  AppendArgs a = append_args(plan, q, qo_indptr, k_pool, v_pool, num_pages, layout, kv_indptr,
                             kv_indices, last_page_len, dtype, sm_scale, o, lse, dev_ws);
  return run_append_kernels(plan, a, qo_indptr, o, lse, dtype, stream, "attn_append_run");
}

attn_status_t attn_append_run_rope(const attn_plan_t* plan, const void* q,
                                   const int32_t* qo_indptr, const void* k_pool,
                                   const void* v_pool, int64_t num_pages, int32_t layout,
                                   const int32_t* kv_indptr, const int32_t* kv_indices,
                                   const int32_t* last_page_len, int32_t dtype,
                                   int32_t causal, float sm_scale, const float* rope_cos,
                                   const float* rope_sin, int64_t rope_max_pos, void* o,
                                   float* lse, void* dev_ws, size_t dev_bytes, void* stream) {
  NvtxRange nvtx("attn_append_run_rope");
  if (!scale_for_kernels(&sm_scale))
    return fail(ATTN_ERR_INVALID_ARG, "attn_append_run_rope: sm_scale must be finite and >= 0");
  attn_status_t s = check_append(plan, q, qo_indptr, k_pool, v_pool, num_pages, layout,
                                 kv_indptr, kv_indices, last_page_len, dtype, causal, o,
                                 dev_ws, dev_bytes, "attn_append_run_rope");
  if (s != ATTN_OK) return s;
  if (debug_checks_enabled()) {
    s = debug_check_table(plan, qo_indptr, kv_indptr, kv_indices, last_page_len, num_pages,
                          stream, "attn_append_run_rope");
    if (s != ATTN_OK) return s;
  }
  s = check_rope(plan, rope_cos, rope_sin, rope_max_pos, "attn_append_run_rope");
  if (s != ATTN_OK) return s;
  if (plan->min_kv_minus_qo < 0)
    return fail(ATTN_ERR_INVALID_ARG,
                "attn_append_run_rope: a request has fewer kv tokens than queries, so a "
                "query would sit before position 0");
  if (plan->batch == 0 || plan->total_qo == 0) return ATTN_OK;
  if (plan_pages(*plan) == 0)
    return run_empty(plan, o, lse, plan->total_qo, dtype, stream, "attn_append_run_rope");
  AppendArgs a = append_args(plan, q, qo_indptr, k_pool, v_pool, num_pages, layout, kv_indptr,
                             kv_indices, last_page_len, dtype, sm_scale, o, lse, dev_ws);
  a.rope_cos = rope_cos;
  a.rope_sin = rope_sin;
  a.rope_rows = rope_max_pos;
  return run_append_kernels(plan, a, qo_indptr, o, lse, dtype, stream, "attn_append_run_rope");
}

attn_status_t attn_merge_states(const void* o_a, const float* lse_a, const void* o_b,
                                const float* lse_b, void* o_out, float* lse_out, int32_t n,
                                int32_t num_heads, int32_t head_dim, int32_t dtype,
                                void* stream) {
  NvtxRange nvtx("attn_merge_states");
  if (n < 0 || num_heads < 1 || head_dim < 1)
    return fail(ATTN_ERR_INVALID_ARG, "attn_merge_states: sizes must be positive");
  if (head_dim % 8 != 0)
    return fail(ATTN_ERR_UNSUPPORTED, "attn_merge_states: head_dim must be a multiple of 8");
  if (dtype != ATTN_F16 && dtype != ATTN_BF16)
    return fail(ATTN_ERR_INVALID_ARG, "attn_merge_states: dtype must be ATTN_F16 or ATTN_BF16");
  if (n == 0) return ATTN_OK;
  if (!o_a || !o_b || !lse_a || !lse_b || !o_out)
    return fail(ATTN_ERR_INVALID_ARG, "attn_merge_states: null device pointer");
  if ((reinterpret_cast<uintptr_t>(o_a) | reinterpret_cast<uintptr_t>(o_b) |
       reinterpret_cast<uintptr_t>(o_out)) & 15)
    return fail(ATTN_ERR_INVALID_ARG, "attn_merge_states: o pointers must be 16-byte aligned");
  cudaError_t e = launch_merge_states(o_a, lse_a, o_b, lse_b, o_out, lse_out,
                                      int64_t(n) * num_heads, head_dim, dtype,
                                      static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "attn_merge_states: launch");
  return ATTN_OK;
}

attn_status_t attn_wait_selftest(void* dev_ws, int32_t limit_us, void* stream) {
  if (!dev_ws) return fail(ATTN_ERR_INVALID_ARG, "attn_wait_selftest: dev_ws is NULL");
  if (limit_us < 1 || limit_us > 10000000)
    return fail(ATTN_ERR_INVALID_ARG, "attn_wait_selftest: limit_us must be in [1, 10^7]");
  cudaError_t e = launch_wait_selftest(static_cast<int32_t*>(dev_ws), uint64_t(limit_us) * 1000u,
                                       static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "attn_wait_selftest: launch");
  return ATTN_OK;
}

attn_status_t attn_workspace_status(const void* dev_ws, void* stream, int32_t* code_out) {
  if (!dev_ws || !code_out)
    return fail(ATTN_ERR_INVALID_ARG, "attn_workspace_status: null pointer");
  int32_t code = 0;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) return cuda_fail(e, "attn_workspace_status: stream");
  e = cudaMemcpy(&code, dev_ws, sizeof code, cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_fail(e, "attn_workspace_status: read");
  *code_out = code;
  if (code != 0) {
    char buf[96];
    std::snprintf(buf, sizeof buf, "a kernel gave up a bounded wait (code 0x%x)", code);
    return fail(ATTN_ERR_TIMEOUT, buf);
  }
  return ATTN_OK;
}

}  // extern "C"
