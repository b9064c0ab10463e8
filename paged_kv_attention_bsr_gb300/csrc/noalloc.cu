// noalloc.cu -- batch decode for callers that cannot allocate memory.
//
// Some callers may not call cudaMalloc (or any allocator) at the point where
// they run attention: code inside an allocator-free region of a serving
// engine, a plugin whose host owns every device allocation, or a real-time
// path that must not touch the allocator's locks or grow the memory pool.
// attn_decode_run_noalloc serves them: it plans and runs a decode batch
// using a fixed scratch area that lives in this library's own device memory
// (a file-scope __device__ array, created when the library is loaded on a
// device and kept until the process exits). The caller passes only inputs
// and outputs.
//
// Rules of use:
//  * the first call on a device looks up the scratch array's device address
//    (cudaGetSymbolAddress with that device current); make that first call
//    before any stream capture;
//  * all calls share the one scratch area and the one host staging area, so
//    calls whose work overlaps on the GPU (different streams, or a second
//    call issued while the first is still running on another stream) race;
//    calls on a single stream are ordered and safe;
//  * the plan tables, partial states and arrival counters must fit in
//    kNoAllocScratchBytes; larger batches are rejected before any GPU work.
#include <cfloat>
#include <cmath>
#include <cstring>
#include <mutex>
#include <string>

#include "internal.h"

namespace attn {
namespace {

constexpr size_t kNoAllocScratchBytes = size_t(4) << 20;  // 4 MiB per device
constexpr int kMaxDevices = 64;

// Device-side scratch: plan tables, split partial states, counters.
static __device__ __align__(256) uint8_t g_noalloc_scratch[kNoAllocScratchBytes];

// Host-side staging for the plan tables (static storage, not allocated).
alignas(256) static uint8_t g_noalloc_host_tables[kNoAllocScratchBytes];
std::mutex g_noalloc_mutex;
void* g_scratch_ptr[kMaxDevices] = {};

attn_status_t noalloc_fail(attn_status_t s, const std::string& msg) {
  set_last_error(msg);  // reported by attn_last_error()
  return s;
}

// Device address of the scratch array on the current device, looked up on
// the first use there (with that device current). The caller holds the mutex.
attn_status_t scratch_of_current_device(void** ws, const char* fn) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess || dev < 0 || dev >= kMaxDevices)
    return noalloc_fail(ATTN_ERR_CUDA, std::string(fn) + ": no usable current device");
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess || !p)
      return noalloc_fail(ATTN_ERR_CUDA, std::string(fn) + ": cudaGetSymbolAddress: " +
                                             cudaGetErrorString(e));
    g_scratch_ptr[dev] = p;
  }
  *ws = g_scratch_ptr[dev];
  return ATTN_OK;
}

}  // namespace
}  // namespace attn

using namespace attn;

extern "C" attn_status_t attn_decode_run_noalloc(
    const int32_t* kv_indptr_h, const int32_t* last_page_len_h, int32_t batch,
    int32_t page_size, int32_t num_qo_heads, int32_t num_kv_heads, int32_t head_dim,
    const void* q, const void* k_pool, const void* v_pool, int64_t num_pages, int32_t layout,
    const int32_t* kv_indptr, const int32_t* kv_indices, const int32_t* last_page_len,
    int32_t dtype, float sm_scale, void* o, float* lse, void* stream) {
  std::lock_guard<std::mutex> lock(g_noalloc_mutex);
  // the scale rule of the other run entry points: finite and >= 0, zero run
  // as the smallest normal float (equal weights, masked scores stay -inf)
  if (!std::isfinite(sm_scale) || sm_scale < 0.f)
    return noalloc_fail(ATTN_ERR_INVALID_ARG,
                        "attn_decode_run_noalloc: sm_scale must be finite and >= 0");
  if (sm_scale == 0.f) sm_scale = FLT_MIN;
  if (dtype != ATTN_F16 && dtype != ATTN_BF16)
    return noalloc_fail(ATTN_ERR_INVALID_ARG, "attn_decode_run_noalloc: bad dtype");
  if (layout != ATTN_LAYOUT_HND && layout != ATTN_LAYOUT_NHD)
    return noalloc_fail(ATTN_ERR_INVALID_ARG, "attn_decode_run_noalloc: bad layout");
  if (num_pages < 0)
    return noalloc_fail(ATTN_ERR_INVALID_ARG, "attn_decode_run_noalloc: num_pages < 0");
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess || dev < 0 || dev >= kMaxDevices)
    return noalloc_fail(ATTN_ERR_CUDA, "attn_decode_run_noalloc: no usable current device");
  int sms = 0;
  e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess)
    return noalloc_fail(ATTN_ERR_CUDA, "attn_decode_run_noalloc: cannot query the SM count");
  const int32_t num_ctas = sms * decode_ctas_per_sm();

  // Plan on the host into the static staging area (validates every input).
  attn_plan_t plan;
  const char* msg = "";
  attn_status_t s = build_plan(nullptr, kv_indptr_h, last_page_len_h, batch, page_size,
                               num_qo_heads, num_kv_heads, head_dim, 0, num_ctas,
                               g_noalloc_host_tables, sizeof g_noalloc_host_tables, &plan,
                               &msg);
  if (s == ATTN_ERR_WORKSPACE_TOO_SMALL)
    return noalloc_fail(ATTN_ERR_WORKSPACE_TOO_SMALL,
                        "attn_decode_run_noalloc: the batch's plan tables exceed the 4 MiB "
                        "scratch area; use attn_plan + attn_decode_run with a caller workspace");
  if (s != ATTN_OK) return noalloc_fail(s, msg);
  if (size_t(plan.dev_bytes_needed) > kNoAllocScratchBytes)
    return noalloc_fail(ATTN_ERR_WORKSPACE_TOO_SMALL,
                        "attn_decode_run_noalloc: the batch needs more than the 4 MiB scratch "
                        "area; use attn_plan + attn_decode_run with a caller workspace");
  if (plan.num_qo_heads / plan.num_kv_heads > kMaxDecodeGroup)
    return noalloc_fail(ATTN_ERR_UNSUPPORTED, "attn_decode_run_noalloc: group > 8");
  if (batch > 0 && (!q || !o || !kv_indptr || !last_page_len))
    return noalloc_fail(ATTN_ERR_INVALID_ARG, "attn_decode_run_noalloc: null device pointer");
  if (plan.total_weight > plan.num_items && (!k_pool || !v_pool || !kv_indices))
    return noalloc_fail(ATTN_ERR_INVALID_ARG,
                        "attn_decode_run_noalloc: null KV pool or kv_indices");
  if ((reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(k_pool) |
       reinterpret_cast<uintptr_t>(v_pool) | reinterpret_cast<uintptr_t>(o)) & 15)
    return noalloc_fail(ATTN_ERR_INVALID_ARG,
                        "attn_decode_run_noalloc: q, k_pool, v_pool and o must be 16-byte aligned");
  if (batch == 0) return ATTN_OK;

  // One-time set-up per device: the device address of the scratch array.
  void* ws = nullptr;
  s = scratch_of_current_device(&ws, "attn_decode_run_noalloc");
  if (s != ATTN_OK) return s;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  // The table copy also zeroes the error word and the split-item counters.
  // The source is pageable static memory, so the call returns only once the
  // bytes are staged: the next call may reuse the host area immediately.
  e = cudaMemcpyAsync(ws, g_noalloc_host_tables, size_t(plan.table_bytes),
                      cudaMemcpyHostToDevice, st);
  if (e != cudaSuccess)
    return noalloc_fail(ATTN_ERR_CUDA, std::string("attn_decode_run_noalloc: table upload: ") +
                                           cudaGetErrorString(e));
  DecodeArgs a;
  a.q = q;
  a.k_pool = k_pool;
  a.v_pool = v_pool;
  a.kv_indptr = kv_indptr;
  a.kv_indices = kv_indices;
  a.last_page_len = last_page_len;
  a.o = o;
  a.lse = lse;
  a.ws = ws_view(plan, ws);
  a.num_ctas = plan.num_ctas;
  a.num_units = plan.num_units;
  a.num_split_items = plan.num_split_items;
  a.layout = layout;
  a.dtype = dtype;
  a.page_size = plan.page_size;
  a.num_qo_heads = plan.num_qo_heads;
  a.num_kv_heads = plan.num_kv_heads;
  a.group = plan.num_qo_heads / plan.num_kv_heads;
  a.batch = plan.batch;
  a.sm_scale = sm_scale;
  a.kv_fp8 = 0;
  a.k_scale = nullptr;
  a.v_scale = nullptr;
  e = launch_decode(a, st);
  if (e != cudaSuccess)
    return noalloc_fail(ATTN_ERR_CUDA, std::string("attn_decode_run_noalloc: launch: ") +
                                           cudaGetErrorString(e));
  return ATTN_OK;
}

// Reads the error word at the head of the current device's scratch area.
extern "C" attn_status_t attn_decode_run_noalloc_status(void* stream, int32_t* code_out) {
  std::lock_guard<std::mutex> lock(g_noalloc_mutex);
  if (!code_out)
    return noalloc_fail(ATTN_ERR_INVALID_ARG, "attn_decode_run_noalloc_status: null output");
  void* ws = nullptr;
  attn_status_t s = scratch_of_current_device(&ws, "attn_decode_run_noalloc_status");
  if (s != ATTN_OK) return s;
  cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess)
    return noalloc_fail(ATTN_ERR_CUDA, std::string("attn_decode_run_noalloc_status: stream: ") +
                                           cudaGetErrorString(e));
  int32_t code = 0;
  e = cudaMemcpy(&code, ws, sizeof code, cudaMemcpyDeviceToHost);
  if (e != cudaSuccess)
    return noalloc_fail(ATTN_ERR_CUDA, std::string("attn_decode_run_noalloc_status: read: ") +
                                           cudaGetErrorString(e));
  *code_out = code;
  if (code != 0)
    return noalloc_fail(ATTN_ERR_TIMEOUT,
                        "attn_decode_run_noalloc: a kernel gave up a bounded wait (code " +
                            std::to_string(code) + ")");
  return ATTN_OK;
}

// The failure-detection self-test of attn_wait_selftest, aimed at the
// no-allocation scratch area's error word.
extern "C" attn_status_t attn_wait_selftest_noalloc(int32_t limit_us, void* stream) {
  std::lock_guard<std::mutex> lock(g_noalloc_mutex);
  if (limit_us < 1 || limit_us > 10000000)
    return noalloc_fail(ATTN_ERR_INVALID_ARG,
                        "attn_wait_selftest_noalloc: limit_us must be in [1, 10^7]");
  void* ws = nullptr;
  attn_status_t s = scratch_of_current_device(&ws, "attn_wait_selftest_noalloc");
  if (s != ATTN_OK) return s;
  cudaError_t e = launch_wait_selftest(static_cast<int32_t*>(ws), uint64_t(limit_us) * 1000u,
                                       static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess)
    return noalloc_fail(ATTN_ERR_CUDA, std::string("attn_wait_selftest_noalloc: launch: ") +
                                           cudaGetErrorString(e));
  return ATTN_OK;
}
