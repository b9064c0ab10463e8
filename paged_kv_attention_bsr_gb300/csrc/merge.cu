// merge.cu -- log-sum-exp merging of attention states.
//
// FlashInfer paper digest (modb.pro), "可组合格式": one attention may combine
// several block-sparse formats (e.g. a shared prefix stored with large pages
// plus per-request suffixes with small pages); the partial results are
// combined through their log-sum-exp. The same merge joins the units of an
// item that the plan split across CTAs ("动态负载均衡调度").
//
//   m = max_i lse_i,  lse = m + ln sum_i e^(lse_i - m),  o = sum_i e^(lse_i - lse) o_i
//
// Both kernels are HBM-streaming: each thread owns 8 (public merge) or one
// (split merge) contiguous element(s) of a row and reads every state once.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "internal.h"
#include "ptx.cuh"

namespace attn {
namespace {

template <bool BF16>
__device__ __forceinline__ void load8(const void* base, int64_t idx, float (&f)[8]) {
  const uint4 raw = __ldg(reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(base) + idx));
  const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    if constexpr (BF16) {
      f[2 * i] = __uint_as_float(w[i] << 16);
      f[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    } else {
      float2 t = __half22float2(*reinterpret_cast<const __half2*>(&w[i]));
      f[2 * i] = t.x;
      f[2 * i + 1] = t.y;
    }
  }
}

template <bool BF16>
__device__ __forceinline__ void store8(void* base, int64_t idx, const float (&f)[8]) {
  uint32_t w[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    if constexpr (BF16) {
      __nv_bfloat162 b = __floats2bfloat162_rn(f[2 * i], f[2 * i + 1]);
      w[i] = *reinterpret_cast<uint32_t*>(&b);
    } else {
      __half2 h = __floats2half2_rn(f[2 * i], f[2 * i + 1]);
      w[i] = *reinterpret_cast<uint32_t*>(&h);
    }
  }
  *reinterpret_cast<uint4*>(static_cast<uint16_t*>(base) + idx) = make_uint4(w[0], w[1], w[2], w[3]);
}

template <bool BF16>
__global__ void __launch_bounds__(256) merge_states_kernel(
    const void* __restrict__ o_a, const float* __restrict__ lse_a, const void* __restrict__ o_b,
    const float* __restrict__ lse_b, void* o_out, float* lse_out, int64_t rows, int32_t head_dim) {
  const int chunks = head_dim / 8;
  const int64_t total = rows * chunks;
  for (int64_t i = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; i < total;
       i += int64_t(gridDim.x) * blockDim.x) {
    const int64_t row = i / chunks;
    const int c = int(i - row * chunks);
    const float la = __ldg(lse_a + row), lb = __ldg(lse_b + row);
    const float m = fmaxf(la, lb);
    float out[8];
    float lse = -INFINITY;
    if (m == -INFINITY) {
#pragma unroll
      for (int j = 0; j < 8; ++j) out[j] = 0.f;
    } else {
      const float wa = ex2((la - m) * kLog2e);
      const float wb = ex2((lb - m) * kLog2e);
      const float inv = 1.f / (wa + wb);
      float xa[8], xb[8];
      load8<BF16>(o_a, row * head_dim + c * 8, xa);
      load8<BF16>(o_b, row * head_dim + c * 8, xb);
#pragma unroll
      for (int j = 0; j < 8; ++j) out[j] = (wa * xa[j] + wb * xb[j]) * inv;
      lse = m + lg2(wa + wb) * kLn2;
    }
    store8<BF16>(o_out, row * head_dim + c * 8, out);
    if (c == 0 && lse_out) lse_out[row] = lse;
  }
}

// One warp per (split item, row): the warps of the whole grid share the
// items' rows; lane owns 4 of the 128 dims. Each partial row is read once.
template <bool BF16>
__global__ void __launch_bounds__(256) split_merge_kernel(const SplitMergeArgs a) {
  const int64_t gw = (int64_t(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (gw >= int64_t(a.num_split_items) * a.rows_per_item) return;
  const int s = int(gw / a.rows_per_item);
  const int rho = int(gw - int64_t(s) * a.rows_per_item);
  const int4 item = __ldg(a.ws.merge_items + s);
  const int r = item.x, hk = item.y, t = item.z;
  int64_t qo_start = r, qo_len = 1;
  if (a.qo_indptr) {
    qo_start = __ldg(a.qo_indptr + r);
    qo_len = int64_t(__ldg(a.qo_indptr + r + 1)) - qo_start;
  }
  const int tok = rho / a.group, hh = rho - tok * a.group;
  const int64_t qi = int64_t(t) * a.q_tile + tok;
  if (qi >= qo_len) return;
  const int slot0 = __ldg(a.ws.merge_indptr + s), slot1 = __ldg(a.ws.merge_indptr + s + 1);
  float lse_s[8];
  float M = -INFINITY;
  const int ns = slot1 - slot0;
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    lse_s[k] = k < ns ? __ldcg(a.ws.partial_lse + int64_t(slot0 + k) * a.rows_per_item + rho)
                      : -INFINITY;
    M = fmaxf(M, lse_s[k]);
  }
  for (int sl = slot0 + 8; sl < slot1; ++sl)
    M = fmaxf(M, __ldcg(a.ws.partial_lse + int64_t(sl) * a.rows_per_item + rho));
  float acc[4] = {0.f, 0.f, 0.f, 0.f};
  float lse2 = -INFINITY;
  if (M != -INFINITY) {
    float L = 0.f;
    for (int sl = slot0; sl < slot1; ++sl) {
      const int64_t prow = int64_t(sl) * a.rows_per_item + rho;
      const float ls = sl - slot0 < 8 ? lse_s[(sl - slot0) & 7] : __ldcg(a.ws.partial_lse + prow);
      const float f = ex2(ls - M);
      L += f;
      const float4 x = __ldcg(reinterpret_cast<const float4*>(a.ws.partial_o + prow * kHeadDim) + lane);
      acc[0] += f * x.x;
      acc[1] += f * x.y;
      acc[2] += f * x.z;
      acc[3] += f * x.w;
    }
    const float inv = 1.f / L;
#pragma unroll
    for (int j = 0; j < 4; ++j) acc[j] *= inv;
    lse2 = M + lg2(L);
  }
  const int64_t orow = (qo_start + qi) * a.num_qo_heads + int64_t(hk) * a.group + hh;
  uint32_t w[2];
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    if constexpr (BF16) {
      __nv_bfloat162 b = __floats2bfloat162_rn(acc[2 * i], acc[2 * i + 1]);
      w[i] = *reinterpret_cast<uint32_t*>(&b);
    } else {
      __half2 h = __floats2half2_rn(acc[2 * i], acc[2 * i + 1]);
      w[i] = *reinterpret_cast<uint32_t*>(&h);
    }
  }
  *reinterpret_cast<uint2*>(static_cast<uint16_t*>(a.o) + orow * kHeadDim + lane * 4) =
      make_uint2(w[0], w[1]);
  if (lane == 0 && a.lse) a.lse[orow] = lse2 * kLn2;
}

// O = 0 and LSE = -inf for rows whose visible set is empty: 16 bytes of a
// row (8 elements) per thread.
__global__ void __launch_bounds__(256) fill_empty_kernel(void* o, float* lse, int64_t rows) {
  const int64_t total = rows * (kHeadDim / 8);
  for (int64_t i = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; i < total;
       i += int64_t(gridDim.x) * blockDim.x) {
    reinterpret_cast<uint4*>(o)[i] = make_uint4(0, 0, 0, 0);
    if (lse && i % (kHeadDim / 8) == 0) lse[i / (kHeadDim / 8)] = -INFINITY;
  }
}

// Plan-table upload: 16 bytes per thread from device-mapped pinned host
// memory into the workspace.
__global__ void __launch_bounds__(256) copy_tables_kernel(uint4* dst, const uint4* src,
                                                          int64_t n16) {
  for (int64_t i = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; i < n16;
       i += int64_t(gridDim.x) * blockDim.x)
    dst[i] = src[i];
}

}  // namespace

cudaError_t launch_copy_tables(void* dst, const void* src_dev, size_t bytes,
                               cudaStream_t stream) {
  const int64_t n16 = int64_t(bytes / 16);
  if (n16 <= 0) return cudaSuccess;
  int64_t blocks = (n16 + 255) / 256;
  if (blocks > 152) blocks = 152;
  copy_tables_kernel<<<int(blocks), 256, 0, stream>>>(static_cast<uint4*>(dst),
                                                      static_cast<const uint4*>(src_dev), n16);
  return cudaGetLastError();
}

cudaError_t launch_fill_empty(void* o, float* lse, int64_t rows, int32_t /*dtype: both 16-bit*/,
                              cudaStream_t stream) {
  if (rows <= 0) return cudaSuccess;
  int64_t blocks = (rows * (kHeadDim / 8) + 255) / 256;
  if (blocks > 152 * 16) blocks = 152 * 16;
  fill_empty_kernel<<<int(blocks), 256, 0, stream>>>(o, lse, rows);
  return cudaGetLastError();
}

cudaError_t launch_merge_states(const void* o_a, const float* lse_a, const void* o_b,
                                const float* lse_b, void* o_out, float* lse_out, int64_t rows,
                                int32_t head_dim, int32_t dtype, cudaStream_t stream) {
  const int64_t total = rows * (head_dim / 8);
  const int threads = 256;
  int64_t blocks = (total + threads - 1) / threads;
  if (blocks > 152 * 16) blocks = 152 * 16;
  if (blocks < 1) blocks = 1;
  if (dtype == ATTN_BF16)
    merge_states_kernel<true><<<int(blocks), threads, 0, stream>>>(o_a, lse_a, o_b, lse_b, o_out,
                                                                    lse_out, rows, head_dim);
  else
    merge_states_kernel<false><<<int(blocks), threads, 0, stream>>>(o_a, lse_a, o_b, lse_b, o_out,
                                                                     lse_out, rows, head_dim);
  return cudaGetLastError();
}

cudaError_t launch_split_merge(const SplitMergeArgs& a, cudaStream_t stream) {
  if (a.num_split_items <= 0) return cudaSuccess;
  const int64_t warps = int64_t(a.num_split_items) * a.rows_per_item;
  const int64_t blocks = (warps + 7) / 8;
  if (a.dtype == ATTN_BF16)
    split_merge_kernel<true><<<unsigned(blocks), 256, 0, stream>>>(a);
  else
    split_merge_kernel<false><<<unsigned(blocks), 256, 0, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace attn
