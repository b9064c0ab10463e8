// tc.cuh -- 5th-generation tensor core building blocks shared by the
// append and the decode kernels: shared-memory matrix descriptors, tcgen05
// MMA / commit / fence, tensor-memory loads and stores, packed fp32 math,
// and the host-side TMA tensor maps of the paged K/V pools.
//
// Operand conventions (all MMAs M = N = 128, 16-bit inputs, fp32 accumulate):
//  * shared-memory tiles are 128 rows of 128 x 16-bit, stored as two 64-column
//    halves of 128 rows x 128 B with the 128-byte swizzle (16-byte chunk j of
//    row r at chunk j ^ (r & 7)); 8-row groups are 1024 B apart;
//  * a K-major operand advances 32 B per 16-wide k-step inside a half; an
//    MN-major V operand steps 16 rows (2048 B) per k-step, its halves 16 KB apart;
//  * tensor memory row m of an accumulator is TMEM lane m; warp w may access
//    lanes 32 (w % 4) .. 32 (w % 4) + 31.
#pragma once
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <cstdint>
#include <mutex>

#include "internal.h"
#include "ptx.cuh"

namespace attn {

constexpr int kTcTile = 128;            // tokens per K/V tile, rows per query tile
constexpr int kTcChunk = 16;            // kv rows per TMA box
constexpr int kTcHalf = kTcTile * 128;  // 128 rows x 128 B (64 x 16-bit)
constexpr int kTcTileBytes = 2 * kTcHalf;

// ------------------------------------------------------------ tcgen05 PTX
__device__ __forceinline__ uint64_t smem_desc(uint32_t addr, uint32_t lbo, uint32_t sbo) {
  // start address, leading / stride byte offsets (>> 4), version 1, SWIZZLE_128B
  return uint64_t((addr & 0x3FFFFu) >> 4) | (uint64_t((lbo >> 4) & 0x3FFFu) << 16) |
         (uint64_t((sbo >> 4) & 0x3FFFu) << 32) | (1ull << 46) | (2ull << 61);
}

__device__ __forceinline__ void mma_f16(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc,
                                        uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a), "l"(b), "r"(idesc), "r"(acc)
      : "memory");
}
// D[tmem] (+)= A[tmem] * B[smem]: A read from tensor memory (K-major, two
// 16-bit elements per 32-bit column, row m in lane m).
__device__ __forceinline__ void mma_f16_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b,
                                           uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b), "r"(idesc), "r"(acc)
      : "memory");
}
__device__ __forceinline__ void mma_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                   bar)
               : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// 32 consecutive fp32 columns of this thread's TMEM lane (load + wait).
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
      "%11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, "
      "%28, %29, %30, %31}, [%32];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
        "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),
        "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
        "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]),
        "=r"(r[31])
      : "r"(taddr)
      : "memory");
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

// All 128 fp32 columns of this thread's TMEM lane: one load, one wait.
__device__ __forceinline__ void tmem_ld128(uint32_t taddr, float (&v)[128]) {
  uint32_t r[128];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x128.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32, %33, %34, %35, %36, %37, %38, %39, %40, %41, %42, %43, %44, %45, %46, %47, %48, %49, %50, %51, %52, %53, %54, %55, %56, %57, %58, %59, %60, %61, %62, %63, %64, %65, %66, %67, %68, %69, %70, %71, %72, %73, %74, %75, %76, %77, %78, %79, %80, %81, %82, %83, %84, %85, %86, %87, %88, %89, %90, %91, %92, %93, %94, %95, %96, %97, %98, %99, %100, %101, %102, %103, %104, %105, %106, %107, %108, %109, %110, %111, %112, %113, %114, %115, %116, %117, %118, %119, %120, %121, %122, %123, %124, %125, %126, %127}, [%128];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31]), "=r"(r[32]), "=r"(r[33]), "=r"(r[34]), "=r"(r[35]), "=r"(r[36]), "=r"(r[37]), "=r"(r[38]), "=r"(r[39]), "=r"(r[40]), "=r"(r[41]), "=r"(r[42]), "=r"(r[43]), "=r"(r[44]), "=r"(r[45]), "=r"(r[46]), "=r"(r[47]), "=r"(r[48]), "=r"(r[49]), "=r"(r[50]), "=r"(r[51]), "=r"(r[52]), "=r"(r[53]), "=r"(r[54]), "=r"(r[55]), "=r"(r[56]), "=r"(r[57]), "=r"(r[58]), "=r"(r[59]), "=r"(r[60]), "=r"(r[61]), "=r"(r[62]), "=r"(r[63]), "=r"(r[64]), "=r"(r[65]), "=r"(r[66]), "=r"(r[67]), "=r"(r[68]), "=r"(r[69]), "=r"(r[70]), "=r"(r[71]), "=r"(r[72]), "=r"(r[73]), "=r"(r[74]), "=r"(r[75]), "=r"(r[76]), "=r"(r[77]), "=r"(r[78]), "=r"(r[79]), "=r"(r[80]), "=r"(r[81]), "=r"(r[82]), "=r"(r[83]), "=r"(r[84]), "=r"(r[85]), "=r"(r[86]), "=r"(r[87]), "=r"(r[88]), "=r"(r[89]), "=r"(r[90]), "=r"(r[91]), "=r"(r[92]), "=r"(r[93]), "=r"(r[94]), "=r"(r[95]), "=r"(r[96]), "=r"(r[97]), "=r"(r[98]), "=r"(r[99]), "=r"(r[100]), "=r"(r[101]), "=r"(r[102]), "=r"(r[103]), "=r"(r[104]), "=r"(r[105]), "=r"(r[106]), "=r"(r[107]), "=r"(r[108]), "=r"(r[109]), "=r"(r[110]), "=r"(r[111]), "=r"(r[112]), "=r"(r[113]), "=r"(r[114]), "=r"(r[115]), "=r"(r[116]), "=r"(r[117]), "=r"(r[118]), "=r"(r[119]), "=r"(r[120]), "=r"(r[121]), "=r"(r[122]), "=r"(r[123]), "=r"(r[124]), "=r"(r[125]), "=r"(r[126]), "=r"(r[127])
      : "r"(taddr)
      : "memory");
#pragma unroll
  for (int i = 0; i < 128; ++i) v[i] = __uint_as_float(r[i]);
}

// 16 consecutive 32-bit columns of this thread's TMEM lane (no wait).
__device__ __forceinline__ void tmem_st16_nowait(uint32_t taddr, const uint32_t (&v)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
      "%11, %12, %13, %14, %15, %16};" ::"r"(taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]),
      "r"(v[8]), "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]),
      "r"(v[15])
      : "memory");
}
__device__ __forceinline__ void tmem_wait_st() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const float (&v)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
      "%11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, "
      "%28, %29, %30, %31, %32};\n\t"
      "tcgen05.wait::st.sync.aligned;" ::"r"(taddr),
      "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])),
      "r"(__float_as_uint(v[3])), "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])),
      "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])), "r"(__float_as_uint(v[8])),
      "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])), "r"(__float_as_uint(v[11])),
      "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])), "r"(__float_as_uint(v[14])),
      "r"(__float_as_uint(v[15])), "r"(__float_as_uint(v[16])), "r"(__float_as_uint(v[17])),
      "r"(__float_as_uint(v[18])), "r"(__float_as_uint(v[19])), "r"(__float_as_uint(v[20])),
      "r"(__float_as_uint(v[21])), "r"(__float_as_uint(v[22])), "r"(__float_as_uint(v[23])),
      "r"(__float_as_uint(v[24])), "r"(__float_as_uint(v[25])), "r"(__float_as_uint(v[26])),
      "r"(__float_as_uint(v[27])), "r"(__float_as_uint(v[28])), "r"(__float_as_uint(v[29])),
      "r"(__float_as_uint(v[30])), "r"(__float_as_uint(v[31]))
      : "memory");
}

__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}
__device__ __forceinline__ float2 ffma2(float2 a, float2 b, float2 c) {
  float2 d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;"
      : "=l"(*reinterpret_cast<unsigned long long*>(&d))
      : "l"(*reinterpret_cast<const unsigned long long*>(&a)),
        "l"(*reinterpret_cast<const unsigned long long*>(&b)),
        "l"(*reinterpret_cast<const unsigned long long*>(&c)));
  return d;
}
__device__ __forceinline__ float2 fmul2(float2 a, float2 b) {
  float2 d;
  asm("mul.rn.f32x2 %0, %1, %2;"
      : "=l"(*reinterpret_cast<unsigned long long*>(&d))
      : "l"(*reinterpret_cast<const unsigned long long*>(&a)),
        "l"(*reinterpret_cast<const unsigned long long*>(&b)));
  return d;
}
__device__ __forceinline__ float2 fadd2(float2 a, float2 b) {
  float2 d;
  asm("add.rn.f32x2 %0, %1, %2;"
      : "=l"(*reinterpret_cast<unsigned long long*>(&d))
      : "l"(*reinterpret_cast<const unsigned long long*>(&a)),
        "l"(*reinterpret_cast<const unsigned long long*>(&b)));
  return d;
}

template <bool BF16>
__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
  if constexpr (BF16) {
    __nv_bfloat162 b = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&b);
  } else {
    __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&h);
  }
}

// ------------------------------------------------------------------- host
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

inline EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

inline uint32_t make_idesc(bool bf16, bool b_mn_major) {
  const uint32_t fmt = bf16 ? 1u : 0u;
  return (1u << 4)                 // D = f32
         | (fmt << 7) | (fmt << 10)  // A, B = bf16 / f16
         | (0u << 15)              // A K-major
         | ((b_mn_major ? 1u : 0u) << 16) | ((128u >> 3) << 17)  // N = 128
         | ((128u >> 4) << 24);                                 // M = 128
}


// Element types of the K / V pools: 16-bit (f16, bf16) or FP8 bytes.
constexpr int kKvElemF16 = 0;
constexpr int kKvElemBF16 = 1;
constexpr int kKvElemU8 = 2;

// The paged K and V pools as 2-D tensors [pages * kv heads * page_size, 128]
// with 16-row x 64-column boxes and the 128-byte swizzle (FP8 bytes: 128-byte
// rows, a box is 16 whole rows). Returns false when the driver cannot
// describe them (message in *msg).
// box_rows: 16 (16-row boxes within a page) or 1 (rows gathered one by one
// with tile::gather4: the append kernel at page sizes that are not a
// multiple of 16). Rows are
// the 256-byte (token, head) vectors: HND [pages, Hk, P, 128] and NHD
// [pages, P, Hk, 128] pools are both [pages * Hk * P, 128] row arrays, and
// 16-row boxes of one head in NHD take a 3-D map [tokens, Hk, 128] (box
// 16 x 1 x 64), which lands the same 16 swizzled rows.
inline bool encode_kv_maps(const void* k_pool, const void* v_pool, int64_t num_pages,
                         int32_t num_kv_heads, int32_t page_size, int elem, uint32_t box_rows,
                         bool nhd, CUtensorMap* tm_k, CUtensorMap* tm_v, const char** msg) {
  const cuuint64_t rows = cuuint64_t(num_pages) * num_kv_heads * page_size;
  if (rows == 0 || rows > 0x7fffffffull) {
    *msg = "attn: the pool has no rows or more than 2^31 (page, head, slot) rows (32-bit TMA "
           "row coordinates)";
    return false;
  }
  EncodeTiledFn enc = encode_fn();
  if (!enc) {
    *msg = "attn: cuTensorMapEncodeTiled is unavailable";
    return false;
  }
  const CUtensorMapDataType dt = elem == kKvElemU8     ? CU_TENSOR_MAP_DATA_TYPE_UINT8
                                 : elem == kKvElemBF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                                       : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  const cuuint64_t esz = elem == kKvElemU8 ? 1 : 2;
  const cuuint32_t box_in = elem == kKvElemU8 ? 128u : 64u;  // 128 bytes either way
  const bool three_d = nhd && box_rows > 1;
  for (int which = 0; which < 2; ++which) {
    const cuuint64_t dims2[2] = {cuuint64_t(kHeadDim), rows};
    const cuuint64_t strides2[1] = {cuuint64_t(kHeadDim) * esz};
    const cuuint32_t box2[2] = {box_in, box_rows};
    const cuuint64_t dims3[3] = {cuuint64_t(kHeadDim), cuuint64_t(num_kv_heads),
                                 cuuint64_t(num_pages) * page_size};
    const cuuint64_t strides3[2] = {cuuint64_t(kHeadDim) * esz,
                                    cuuint64_t(kHeadDim) * esz * cuuint64_t(num_kv_heads)};
    const cuuint32_t box3[3] = {box_in, 1u, box_rows};
    const cuuint32_t es[3] = {1, 1, 1};
    CUtensorMap* tm = which == 0 ? tm_k : tm_v;
    void* ptr = const_cast<void*>(which == 0 ? k_pool : v_pool);
    if (enc(tm, dt, three_d ? 3 : 2, ptr, three_d ? dims3 : dims2,
            three_d ? strides3 : strides2, three_d ? box3 : box2, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS) {
      *msg = "attn: cannot describe the KV pool for TMA";
      return false;
    }
  }
  return true;
}

// encode_kv_maps, remembering the last pools described on this thread (a
// serving loop runs over the same pools step after step).
inline bool make_kv_maps(const void* k_pool, const void* v_pool, int64_t num_pages,
                         int32_t num_kv_heads, int32_t page_size, int elem, uint32_t box_rows,
                         bool nhd, CUtensorMap* tm_k, CUtensorMap* tm_v, const char** msg) {
  // two entries per thread: a composable-format run encodes two pools per call
  struct Key {
    const void *k, *v;
    int64_t pages;
    int32_t heads, page_size, elem;
    uint32_t box_rows;
    int32_t nhd;
    bool operator==(const Key& o) const {
      return k == o.k && v == o.v && pages == o.pages && heads == o.heads &&
             page_size == o.page_size && elem == o.elem && box_rows == o.box_rows && nhd == o.nhd;
    }
  };
  struct Entry {
    Key key;
    CUtensorMap k, v;
  };
  thread_local Entry cache[2] = {{{nullptr, nullptr, -1, 0, 0, 0, 0, 0}, {}, {}},
                                 {{nullptr, nullptr, -1, 0, 0, 0, 0, 0}, {}, {}}};
  thread_local int oldest = 0;
  const Key key = {k_pool, v_pool, num_pages, num_kv_heads, page_size, elem, box_rows,
                   nhd ? 1 : 0};
  for (int i = 0; i < 2; ++i)
    if (cache[i].key == key) {
      *tm_k = cache[i].k;
      *tm_v = cache[i].v;
      oldest = 1 - i;
      return true;
    }
  if (!encode_kv_maps(k_pool, v_pool, num_pages, num_kv_heads, page_size, elem, box_rows, nhd,
                      tm_k, tm_v, msg))
    return false;
  cache[oldest] = {key, *tm_k, *tm_v};
  oldest = 1 - oldest;
  return true;
}

// Number of SMs of the current device (cached per device on this thread).
inline cudaError_t current_sm_count(int* sms) {
  thread_local int cache[64] = {0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev >= 0 && dev < 64 && cache[dev] > 0) {
    *sms = cache[dev];
    return cudaSuccess;
  }
  e = cudaDeviceGetAttribute(sms, cudaDevAttrMultiProcessorCount, dev);
  if (e == cudaSuccess && dev >= 0 && dev < 64) cache[dev] = *sms;
  return e;
}

}  // namespace attn
