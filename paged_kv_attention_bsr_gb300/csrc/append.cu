// append.cu -- append / prefill attention over a BSR paged KV cache on the
// 5th-generation tensor cores (tcgen05 MMA, TMEM accumulators, TMA loads).
//
// Method: many new query rows of a request attend to that request's paged KV
// (which already holds the new tokens), with the causal mask aligned to the
// end of the sequence (FlashInfer README copy on gittoolsai.com, "解码、预填充
// 与追加"; paged KV per the modb.pro digest, "统一的 KV 缓存存储格式"). Work
// follows the CPU plan of "动态负载均衡调度" in a persistent fixed grid.
//
// Tile shapes. A work unit is (request r, query tile t, kv head hk, pages
// [p0, p1)). Its query tile packs 128 rows: tq = 128 / group query tokens x
// the group's query heads (row = token * group + head), so one K/V tile feeds
// every head of the GQA group. K/V tiles hold 128 kv tokens, gathered from the
// page table in 16-row TMA boxes (page_size % 16 == 0).
//
// Per KV tile j (all MMAs M = 128, N = 128, bf16/fp16 in, fp32 accumulate):
//   S_j = Q K_j^T          tcgen05.mma, A = Q (smem, K-major), B = K (smem,
//                          K-major), D = TMEM S buffer j % 2
//   P_j = exp2(S_j*c - m)  4 softmax warps, one TMEM lane (= row) per thread
//   O  += P_j V_j          A = P (smem, K-major), B = V (smem, MN-major), D =
//                          TMEM O
// Warp roles (192 threads, one CTA per SM): warp 0 issues TMA loads, warp 1
// allocates TMEM and issues MMAs from one thread, warps 2-5 run the softmax,
// the lazy O rescale (only when a row max grows by more than 2^8) and the
// epilogue. S is double-buffered in TMEM so S_{j+1} runs under softmax_j.
// Every wait is bounded; TMEM is freed on every path.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <cstring>
#include <mutex>

#include "internal.h"
#include "ptx.cuh"

namespace attn {
namespace {

constexpr int kTile = 128;
constexpr int kChunk = 16;                  // kv rows per TMA box
constexpr int kHalf = kTile * 128;          // 128 rows x 128 B (64 x 16-bit)
constexpr int kTileBytes = 2 * kHalf;       // 128 x 128 x 16-bit
constexpr int kThreads = 192;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColS = 0;    // S buffers at columns 0 and 128
constexpr uint32_t kColO = 256;  // O at columns 256..383

// Shared memory map (offsets from a 1024-byte aligned base). K and V tiles
// travel through one ring of kSlots 32 KB slots: tile j's K takes slot use
// 2j and its V use 2j + 1 (slot = use % kSlots), so 2.5 tiles are in flight.
constexpr int kSlots = 5;
constexpr int kOffQ = 0;                               // query tile
constexpr int kOffRing = kOffQ + kTileBytes;           // K/V ring
constexpr int kOffP = kOffRing + kSlots * kTileBytes;  // probabilities
constexpr int kOffBar = kOffP + kTileBytes;
constexpr int kSmemBytes = kOffBar + 256 + 1024;  // + barriers + alignment slack

struct Bars {
  uint64_t q_full, q_empty;
  uint64_t slot_full[kSlots], slot_empty[kSlots];
  uint64_t s_full[2], s_empty[2];
  uint64_t p_full, o_done, o_free, drain;
  uint32_t tmem_base;
};
static_assert(sizeof(Bars) <= 256, "barrier block");

struct AppendParams {
  CUtensorMap tm_q;
  CUtensorMap tm_k;
  CUtensorMap tm_v;
  AppendArgs a;
  float scale_log2;
  uint32_t idesc_s;
  uint32_t idesc_pv;
};

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

// --------------------------------------------------------- unit geometry
struct AGeo {
  int32_t r, hk, t, slot, page_base;
  int64_t qo_start, qo_len, kv_len;
  int64_t tok_begin, tok_end;
  int32_t ntiles;
};

__device__ __forceinline__ AGeo append_geo(const AppendArgs& a, int ui) {
  const int4* rec = reinterpret_cast<const int4*>(a.ws.units + ui);
  const int4 x = __ldg(rec);
  const int4 y = __ldg(rec + 1);
  AGeo g;
  g.r = x.x;
  g.t = x.z;
  g.hk = x.y;
  g.slot = y.y;
  g.qo_start = __ldg(a.qo_indptr + g.r);
  g.qo_len = int64_t(__ldg(a.qo_indptr + g.r + 1)) - g.qo_start;
  g.page_base = __ldg(a.kv_indptr + g.r);
  const int64_t n = int64_t(__ldg(a.kv_indptr + g.r + 1)) - g.page_base;
  g.kv_len = n > 0 ? (n - 1) * a.page_size + __ldg(a.last_page_len + g.r) : 0;
  int64_t vis = g.kv_len;
  if (a.causal) {
    const int64_t last_row = min(int64_t(g.t + 1) * a.q_tile, g.qo_len) - 1;
    vis = min(g.kv_len, max(int64_t(0), g.kv_len - g.qo_len + last_row + 1));
  }
  g.tok_begin = int64_t(x.w) * a.page_size;
  g.tok_end = min(int64_t(y.x) * a.page_size, vis);
  const int64_t nt = g.tok_end - g.tok_begin;
  g.ntiles = nt > 0 ? int32_t((nt + kTile - 1) / kTile) : 0;
  return g;
}

template <bool BF16>
__global__ void __launch_bounds__(kThreads, 1) append_kernel(const __grid_constant__ AppendParams prm) {
  extern __shared__ uint8_t smem_raw[];
  const AppendArgs& a = prm.a;
  const uint32_t raw_base = smem_u32(smem_raw);
  const uint32_t base = (raw_base + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (base - raw_base);
  Bars& bars = *reinterpret_cast<Bars*>(gbase + kOffBar);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  volatile int32_t* err = a.ws.error;

  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bars.q_full), 1);
    mbar_init(smem_u32(&bars.q_empty), 1);
    for (int i = 0; i < kSlots; ++i) {
      mbar_init(smem_u32(&bars.slot_full[i]), 1);
      mbar_init(smem_u32(&bars.slot_empty[i]), 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(smem_u32(&bars.s_full[i]), 1);
      mbar_init(smem_u32(&bars.s_empty[i]), 128);
    }
    mbar_init(smem_u32(&bars.p_full), 128);
    mbar_init(smem_u32(&bars.o_done), 1);
    mbar_init(smem_u32(&bars.o_free), 128);
    mbar_init(smem_u32(&bars.drain), 1);
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&prm.tm_q);
    prefetch_tmap(&prm.tm_k);
    prefetch_tmap(&prm.tm_v);
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(&bars.tmem_base)),
                 "r"(kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars.tmem_base;

  const int u_begin = __ldg(a.ws.work_indptr + blockIdx.x);
  const int u_end = __ldg(a.ws.work_indptr + blockIdx.x + 1);
  const int group = a.group;

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    // The whole warp runs the loop; lane c fetches the page index of the
    // tile's 16-row chunk c and issues that chunk's boxes, so the eight index
    // loads of a tile overlap instead of serialising.
    uint32_t ua = 0, uses = 0;
    const int P = a.page_size;
    bool ok = true;
    auto wait0 = [&](uint32_t bar, uint32_t parity) -> bool {
      bool r = true;
      if (lane == 0) r = mbar_wait(bar, parity, err, ERR_WAIT_EMPTY);
      return __shfl_sync(0xffffffffu, r ? 1 : 0, 0) != 0;
    };
    for (int ui = u_begin; ui < u_end && ok; ++ui) {
      const AGeo g = append_geo(a, ui);
      if (g.ntiles == 0) continue;
      if (!wait0(smem_u32(&bars.q_empty), (ua & 1u) ^ 1u)) break;
      if (lane == 0) {
        const uint32_t qf = smem_u32(&bars.q_full);
        mbar_arrive_expect_tx(qf, kTileBytes);
        const int32_t qrow = int32_t(g.qo_start + int64_t(g.t) * a.q_tile);
        tma_load_3d(base + kOffQ, &prm.tm_q, 0, g.hk * group, qrow, qf);
        tma_load_3d(base + kOffQ + kHalf, &prm.tm_q, 64, g.hk * group, qrow, qf);
      }
      ++ua;
      for (int i = 0; i < g.ntiles && ok; ++i) {
        const int64_t kv0 = g.tok_begin + int64_t(i) * kTile;
        const int ntt = int(min(int64_t(kTile), g.tok_end - kv0));
        const int nch = (ntt + kChunk - 1) / kChunk;
        int32_t row = 0;
        if (lane < nch) {
          const int64_t kvt = kv0 + int64_t(lane) * kChunk;
          const int64_t pg = kvt / P;
          const int64_t phys = __ldg(a.kv_indices + g.page_base + pg);
          row = int32_t((phys * a.num_kv_heads + g.hk) * P + (kvt - pg * P));
        }
        for (int kv = 0; kv < 2; ++kv, ++uses) {  // K then V
          const int slot = int(uses % kSlots);
          if (!wait0(smem_u32(&bars.slot_empty[slot]), ((uses / kSlots) & 1u) ^ 1u)) {
            ok = false;
            break;
          }
          const uint32_t full = smem_u32(&bars.slot_full[slot]);
          if (lane == 0) mbar_arrive_expect_tx(full, uint32_t(nch) * kChunk * 256u);
          __syncwarp();
          if (lane < nch) {
            const uint32_t dst = base + kOffRing + slot * kTileBytes + uint32_t(lane) * kChunk * 128u;
            const void* tm = kv == 0 ? static_cast<const void*>(&prm.tm_k)
                                     : static_cast<const void*>(&prm.tm_v);
            tma_load_2d(dst, tm, 0, row, full);
            tma_load_2d(dst + kHalf, tm, 64, row, full);
          }
        }
      }
    }
    // drain: every issued copy has landed before the CTA can exit
    if (lane == 0) {
      if (ua > 0) mbar_wait(smem_u32(&bars.q_full), (ua - 1) & 1u, err, ERR_WAIT_DRAIN);
      for (uint32_t sl = 0; sl < uint32_t(kSlots) && sl < uses; ++sl) {
        const uint32_t last = uses - 1 - ((uses - 1 - sl) % kSlots);
        mbar_wait(smem_u32(&bars.slot_full[sl]), (last / kSlots) & 1u, err, ERR_WAIT_DRAIN);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      uint32_t ua = 0, jt = 0;
      bool ok = true;
      auto issue_pv = [&](uint32_t jt_pv, bool first) -> bool {
        const uint32_t use = 2 * jt_pv + 1;
        const int slot = int(use % kSlots);
        if (!mbar_wait(smem_u32(&bars.p_full), jt_pv & 1u, err, ERR_WAIT_SOFTMAX)) return false;
        if (first && !mbar_wait(smem_u32(&bars.o_free), (ua & 1u) ^ 1u, err, ERR_WAIT_SOFTMAX))
          return false;
        if (!mbar_wait(smem_u32(&bars.slot_full[slot]), (use / kSlots) & 1u, err, ERR_WAIT_FULL))
          return false;
        tc_fence_after();
        const uint32_t pbase = base + kOffP;
        const uint32_t vbase = base + kOffRing + slot * kTileBytes;
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const uint64_t ad = smem_desc(pbase + (k >> 2) * kHalf + (k & 3) * 32, 16, 1024);
          const uint64_t bd = smem_desc(vbase + k * kChunk * 128, kHalf, 1024);
          mma_f16(tmem + kColO, ad, bd, prm.idesc_pv, (first && k == 0) ? 0u : 1u);
        }
        mma_commit(smem_u32(&bars.o_done));
        mma_commit(smem_u32(&bars.slot_empty[slot]));
        return true;
      };
      for (int ui = u_begin; ui < u_end && ok; ++ui) {
        const AGeo g = append_geo(a, ui);
        if (g.ntiles == 0) continue;
        if (!mbar_wait(smem_u32(&bars.q_full), ua & 1u, err, ERR_WAIT_FULL)) break;
        const uint32_t qbase = base + kOffQ;
        for (int i = 0; i < g.ntiles; ++i, ++jt) {
          const uint32_t use = 2 * jt;
          const int slot = int(use % kSlots);
          const int sb = jt & 1;
          if (!mbar_wait(smem_u32(&bars.slot_full[slot]), (use / kSlots) & 1u, err,
                         ERR_WAIT_FULL) ||
              !mbar_wait(smem_u32(&bars.s_empty[sb]), ((jt >> 1) & 1u) ^ 1u, err,
                         ERR_WAIT_SOFTMAX)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t kbase = base + kOffRing + slot * kTileBytes;
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            const uint32_t koff = (k >> 2) * kHalf + (k & 3) * 32;
            mma_f16(tmem + kColS + sb * 128, smem_desc(qbase + koff, 16, 1024),
                    smem_desc(kbase + koff, 16, 1024), prm.idesc_s, k > 0 ? 1u : 0u);
          }
          mma_commit(smem_u32(&bars.s_full[sb]));
          mma_commit(smem_u32(&bars.slot_empty[slot]));
          if (i == g.ntiles - 1) mma_commit(smem_u32(&bars.q_empty));
          if (i > 0 && !issue_pv(jt - 1, i == 1)) {
            ok = false;
            break;
          }
        }
        if (ok && !issue_pv(jt - 1, g.ntiles == 1)) ok = false;
        ++ua;
      }
      // drain: no MMA may still be writing TMEM when it is freed
      mma_commit(smem_u32(&bars.drain));
      mbar_wait(smem_u32(&bars.drain), 0, err, ERR_WAIT_DRAIN);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------- softmax / epilogue
    const int quarter = warp & 3;            // TMEM lanes this warp may access
    const int rho = quarter * 32 + lane;     // row of the query tile
    const uint32_t lane_off = uint32_t(quarter * 32) << 16;
    const int tok = rho / group;
    const int hh = rho - tok * group;
    const float c2 = prm.scale_log2;
    uint8_t* pbuf = gbase + kOffP;
    uint32_t ua = 0, jt = 0;
    bool ok = true;
    for (int ui = u_begin; ui < u_end && ok; ++ui) {
      const AGeo g = append_geo(a, ui);
      const int64_t qi = int64_t(g.t) * a.q_tile + tok;
      const bool row_ok = (tok < a.q_tile) && (qi < g.qo_len);
      const int64_t orow = (g.qo_start + qi) * a.num_qo_heads + int64_t(g.hk) * group + hh;
      const int64_t limit = a.causal ? (g.kv_len - g.qo_len + qi) : (g.kv_len - 1);
      const int64_t row_end = row_ok ? min(g.tok_end, limit + 1) : g.tok_begin;
      if (g.ntiles == 0) {
        if (row_ok) {
          if (g.slot < 0) {
            uint4* dst = reinterpret_cast<uint4*>(static_cast<uint16_t*>(a.o) + orow * kHeadDim);
            for (int i = 0; i < 16; ++i) dst[i] = make_uint4(0, 0, 0, 0);
            if (a.lse) a.lse[orow] = -INFINITY;
          } else {
            const int64_t prow = int64_t(g.slot) * kTile + rho;
            float4* dst = reinterpret_cast<float4*>(a.ws.partial_o + prow * kHeadDim);
            for (int i = 0; i < 32; ++i) dst[i] = make_float4(0.f, 0.f, 0.f, 0.f);
            a.ws.partial_lse[prow] = -INFINITY;
          }
        }
        continue;
      }
      float m_ref = -INFINITY, l = 0.f;
      for (int i = 0; i < g.ntiles; ++i, ++jt) {
        const int sb = jt & 1;
        // waits are made warp-uniform: tcgen05.ld/st below are .sync.aligned
        if (!__all_sync(0xffffffffu,
                        mbar_wait(smem_u32(&bars.s_full[sb]), (jt >> 1) & 1u, err, ERR_WAIT_MMA))) {
          ok = false;
          break;
        }
        tc_fence_after();
        float s[kTile];
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          float tmp[32];
          tmem_ld32(tmem + lane_off + kColS + sb * 128 + c * 32, tmp);
#pragma unroll
          for (int x = 0; x < 32; ++x) s[c * 32 + x] = tmp[x];
        }
        tc_fence_before();
        mbar_arrive(smem_u32(&bars.s_empty[sb]));

        const int64_t kv0 = g.tok_begin + int64_t(i) * kTile;
        const int nvalid = int(max(int64_t(0), min(int64_t(kTile), row_end - kv0)));
        float mx = -INFINITY;
#pragma unroll
        for (int c = 0; c < kTile; ++c) {
          s[c] = (c < nvalid) ? s[c] : -INFINITY;
          mx = fmaxf(mx, s[c]);
        }
        const float m_tile = mx * c2;  // -inf stays -inf
        float alpha = 1.f;
        bool rescale_o = false;
        if (m_tile > m_ref + 8.f) {
          alpha = ex2(m_ref - m_tile);  // 0 when m_ref = -inf
          rescale_o = (i > 0) && (m_ref != -INFINITY);
          l *= alpha;
          m_ref = m_tile;
        }
        // probabilities, packed to the MMA input type right away (2 per word)
        float lsum = 0.f;
        uint32_t pk[kTile / 2];
        if (m_ref != -INFINITY) {
#pragma unroll
          for (int c = 0; c < kTile; c += 2) {
            const float p0 = ex2(fmaf(s[c], c2, -m_ref));
            const float p1 = ex2(fmaf(s[c + 1], c2, -m_ref));
            lsum += p0 + p1;
            pk[c / 2] = pack2<BF16>(p0, p1);
          }
        } else {
#pragma unroll
          for (int c = 0; c < kTile / 2; ++c) pk[c] = 0u;
        }
        l += lsum;
        // P_{j-1}'s MMA must be done before P is overwritten and O rescaled.
        if (i > 0) {
          if (!__all_sync(0xffffffffu,
                          mbar_wait(smem_u32(&bars.o_done), (jt - 1) & 1u, err, ERR_WAIT_MMA))) {
            ok = false;
            break;
          }
          tc_fence_after();
        }
        // warp-uniform: tcgen05.ld/st are .sync.aligned
        if (__any_sync(0xffffffffu, rescale_o)) {
#pragma unroll 1
          for (int c = 0; c < 4; ++c) {
            float o[32];
            const uint32_t ta = tmem + lane_off + kColO + c * 32;
            tmem_ld32(ta, o);
            const float f = rescale_o ? alpha : 1.f;
#pragma unroll
            for (int x = 0; x < 32; ++x) o[x] *= f;
            tmem_st32(ta, o);
          }
        }
        // P row -> shared memory, 128B-swizzled K-major layout
#pragma unroll
        for (int ch = 0; ch < 16; ++ch) {
          const int half = ch >> 3, cc = ch & 7;
          *reinterpret_cast<uint4*>(pbuf + half * kHalf + rho * 128 + ((cc ^ (rho & 7)) << 4)) =
              make_uint4(pk[ch * 4], pk[ch * 4 + 1], pk[ch * 4 + 2], pk[ch * 4 + 3]);
        }
        // kv rows past the unit's end hold whatever the pool had: zero them in V
        const int ntt = int(min(int64_t(kTile), g.tok_end - kv0));
        if (ntt < kTile) {
          // wait for this tile's V to land before overwriting its tail rows
          const uint32_t vuse = 2 * jt + 1;
          if (!__all_sync(0xffffffffu, mbar_wait(smem_u32(&bars.slot_full[vuse % kSlots]),
                                                 (vuse / kSlots) & 1u, err, ERR_WAIT_FULL))) {
            ok = false;
            break;
          }
        }
        if (ntt < kTile && rho >= ntt) {
          uint8_t* vrow = gbase + kOffRing + (2 * jt + 1) % kSlots * kTileBytes + rho * 128;
#pragma unroll
          for (int x = 0; x < 8; ++x) {
            *reinterpret_cast<uint4*>(vrow + x * 16) = make_uint4(0, 0, 0, 0);
            *reinterpret_cast<uint4*>(vrow + kHalf + x * 16) = make_uint4(0, 0, 0, 0);
          }
        }
        fence_proxy_async_smem();
        tc_fence_before();
        mbar_arrive(smem_u32(&bars.p_full));
      }
      if (!ok) break;
      // ---- epilogue: O / l
      if (!__all_sync(0xffffffffu,
                      mbar_wait(smem_u32(&bars.o_done), (jt - 1) & 1u, err, ERR_WAIT_MMA))) {
        ok = false;
        break;
      }
      tc_fence_after();
      const bool any = l > 0.f;
      const float inv = any ? 1.f / l : 0.f;
      const float lse2 = any ? m_ref + lg2(l) : -INFINITY;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        float o[32];
        tmem_ld32(tmem + lane_off + kColO + c * 32, o);
        if (row_ok) {
          if (g.slot < 0) {
            uint4* dst = reinterpret_cast<uint4*>(static_cast<uint16_t*>(a.o) + orow * kHeadDim + c * 32);
#pragma unroll
            for (int x = 0; x < 4; ++x) {
              uint4 v;
              v.x = pack2<BF16>(o[x * 8 + 0] * inv, o[x * 8 + 1] * inv);
              v.y = pack2<BF16>(o[x * 8 + 2] * inv, o[x * 8 + 3] * inv);
              v.z = pack2<BF16>(o[x * 8 + 4] * inv, o[x * 8 + 5] * inv);
              v.w = pack2<BF16>(o[x * 8 + 6] * inv, o[x * 8 + 7] * inv);
              dst[x] = v;
            }
          } else {
            const int64_t prow = int64_t(g.slot) * kTile + rho;
            float4* dst = reinterpret_cast<float4*>(a.ws.partial_o + prow * kHeadDim + c * 32);
#pragma unroll
            for (int x = 0; x < 8; ++x)
              dst[x] = make_float4(o[x * 4] * inv, o[x * 4 + 1] * inv, o[x * 4 + 2] * inv,
                                   o[x * 4 + 3] * inv);
          }
        }
      }
      if (row_ok) {
        if (g.slot < 0) {
          if (a.lse) a.lse[orow] = lse2 * kLn2;
        } else {
          a.ws.partial_lse[int64_t(g.slot) * kTile + rho] = lse2;
        }
      }
      tc_fence_before();
      mbar_arrive(smem_u32(&bars.o_free));
      ++ua;
    }
  }

  // ---------------------------------------------------------------- teardown
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                 "r"(kTmemCols)
                 : "memory");
  }
}

// ------------------------------------------------------------------- host
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
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

uint32_t make_idesc(bool bf16, bool b_mn_major) {
  const uint32_t fmt = bf16 ? 1u : 0u;
  return (1u << 4)                 // D = f32
         | (fmt << 7) | (fmt << 10)  // A, B = bf16 / f16
         | (0u << 15)              // A K-major
         | ((b_mn_major ? 1u : 0u) << 16) | ((128u >> 3) << 17)  // N = 128
         | ((128u >> 4) << 24);                                 // M = 128
}

template <bool BF16>
cudaError_t launch_t(AppendParams& prm, int ctas, cudaStream_t stream) {
  static bool configured = false;
  if (!configured) {
    cudaError_t e = cudaFuncSetAttribute(append_kernel<BF16>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    if (e != cudaSuccess) return e;
    configured = true;
  }
  append_kernel<BF16><<<ctas, kThreads, kSmemBytes, stream>>>(prm);
  return cudaGetLastError();
}

}  // namespace

int append_ctas_per_sm() { return 1; }

cudaError_t launch_append(const AppendArgs& a, cudaStream_t stream, const char** msg) {
  if (a.group * a.q_tile != kTile) {
    *msg = "attn_append_run: num_qo_heads / num_kv_heads must divide 128";
    return cudaErrorNotSupported;
  }
  if (a.page_size % kChunk != 0) {
    *msg = "attn_append_run: page_size must be a multiple of 16";
    return cudaErrorNotSupported;
  }
  if (a.num_ctas <= 0 || a.num_units == 0) return cudaSuccess;
  EncodeTiledFn enc = encode_fn();
  if (!enc) {
    *msg = "attn_append_run: cuTensorMapEncodeTiled is unavailable";
    return cudaErrorNotSupported;
  }
  const bool bf16 = a.dtype == ATTN_BF16;
  const CUtensorMapDataType dt = bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  AppendParams prm;
  std::memset(&prm, 0, sizeof prm);
  prm.a = a;
  prm.scale_log2 = a.sm_scale * kLog2e;
  prm.idesc_s = make_idesc(bf16, false);
  prm.idesc_pv = make_idesc(bf16, true);
  {
    const cuuint64_t dims[3] = {cuuint64_t(kHeadDim), cuuint64_t(a.num_qo_heads),
                                cuuint64_t(a.total_qo)};
    const cuuint64_t strides[2] = {cuuint64_t(kHeadDim) * 2,
                                   cuuint64_t(kHeadDim) * 2 * a.num_qo_heads};
    const cuuint32_t box[3] = {64u, cuuint32_t(a.group), cuuint32_t(a.q_tile)};
    const cuuint32_t es[3] = {1, 1, 1};
    if (enc(&prm.tm_q, dt, 3, const_cast<void*>(a.q), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS) {
      *msg = "attn_append_run: cannot describe q for TMA";
      return cudaErrorInvalidValue;
    }
  }
  const cuuint64_t rows = cuuint64_t(a.num_pages) * a.num_kv_heads * a.page_size;
  if (rows == 0 || rows > 0x7fffffffull) {
    *msg = "attn_append_run: pool too large for 32-bit TMA row coordinates";
    return cudaErrorNotSupported;
  }
  for (int which = 0; which < 2; ++which) {
    const cuuint64_t dims[2] = {cuuint64_t(kHeadDim), rows};
    const cuuint64_t strides[1] = {cuuint64_t(kHeadDim) * 2};
    const cuuint32_t box[2] = {64u, cuuint32_t(kChunk)};
    const cuuint32_t es[2] = {1, 1};
    CUtensorMap* tm = which == 0 ? &prm.tm_k : &prm.tm_v;
    void* ptr = const_cast<void*>(which == 0 ? a.k_pool : a.v_pool);
    if (enc(tm, dt, 2, ptr, dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS) {
      *msg = "attn_append_run: cannot describe the KV pool for TMA";
      return cudaErrorInvalidValue;
    }
  }
  return bf16 ? launch_t<true>(prm, a.num_ctas, stream) : launch_t<false>(prm, a.num_ctas, stream);
}

}  // namespace attn
