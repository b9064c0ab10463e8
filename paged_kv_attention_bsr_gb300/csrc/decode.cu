// decode.cu -- persistent batch-decode kernel over a BSR paged KV cache.
//
// Method (FlashInfer paper digest, modb.pro): requests' KV live in pages
// addressed through a block-sparse row table ("统一的 KV 缓存存储格式"); a CPU
// plan cuts the (request, kv head) items into units balanced across SMs and a
// fixed-grid persistent kernel follows it ("动态负载均衡调度"). Attention is
// the IO-aware tiled softmax of the yeyulingfeng.com page ("FlashAttention
// 的遗产"): K/V stream through on-chip memory once, with a running max / sum.
//
// GB300 design:
//  * one producer warp streams K/V rows of the unit's pages into a 3-stage
//    shared-memory ring with bulk async copies (TMA engine, 1-D), completing on
//    mbarriers; each stage holds 64 tokens (32 KB of K+V) plus the group's q;
//  * four consumer warps each take 16 of the stage's tokens. A half-warp owns
//    one token: each of its 16 lanes holds 8 of the 128 dims (128-bit shared
//    loads, conflict-free). Every K/V row read from HBM serves all `group`
//    query heads of the GQA group (q and the accumulators of all heads sit in
//    registers), so HBM traffic is the KV bytes once;
//  * q.k partial dots are reduced over the 16 lanes with a transposing
//    butterfly (log2(group) exchanges that halve the live values, then plain
//    xor steps), leaving each lane with one head's score;
//  * online softmax in base 2 (q pre-scaled by sm_scale * log2 e), fp32 state;
//  * at the end of a unit the four warps' (m, l, acc) are combined in the
//    stage's own shared memory; unsplit items write o / lse directly, split
//    items write an fp32 partial state (o, log2-LSE) to the workspace slot
//    the plan assigned; the last of an item's units to finish (an atomic
//    arrival count in the workspace) merges them, so a run is one launch;
//  * K/V may be stored as FP8 E4M3 with a scale per kv head (half the bytes
//    per token): rows are widened to floats as they are read from shared
//    memory, the key scale is folded into q and the value scale into the
//    output;
//  * every wait is bounded (ptx.cuh) and reports through the workspace
//    error word instead of hanging.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include "internal.h"
#include "ptx.cuh"

namespace attn {
namespace {

constexpr int kConsumerWarps = 4;
constexpr int kThreads = (kConsumerWarps + 1) * 32;
constexpr int kStageTok = 64;
constexpr int kTokPerWarp = kStageTok / kConsumerWarps;  // 16
constexpr int kQRowBytes = kHeadDim * 2;                 // one q / o row, 16-bit

// K/V storage: 16-bit (a token row is 256 B) or FP8 E4M3 (128 B, with a
// scale per kv head). An FP8 stage holds half the bytes, so the ring has
// twice the stages and keeps as many bytes in flight.
template <bool FP8>
struct Kv {
  static constexpr int kRowBytes = FP8 ? kHeadDim : kHeadDim * 2;
  static constexpr int kStages = FP8 ? 6 : 3;
};

template <bool FP8>
struct __align__(128) Stage {
  uint8_t k[kStageTok * Kv<FP8>::kRowBytes];
  uint8_t v[kStageTok * Kv<FP8>::kRowBytes];
  uint16_t q[kMaxDecodeGroup * kHeadDim];
};

template <bool FP8>
struct __align__(128) Smem {
  Stage<FP8> st[Kv<FP8>::kStages];
  float pbuf[kConsumerWarps][kTokPerWarp * kMaxDecodeGroup];
  float sbuf[kConsumerWarps][kMaxDecodeGroup];
  uint64_t full[Kv<FP8>::kStages];
  uint64_t empty[Kv<FP8>::kStages];
  uint64_t cbar;
};

template <bool BF16>
__device__ __forceinline__ void cvt8(const uint4 raw, float (&f)[8]) {
  const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    if constexpr (BF16) {
      f[2 * i] = __uint_as_float(w[i] << 16);
      f[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    } else {
      __half2 h = *reinterpret_cast<const __half2*>(&w[i]);
      float2 t = __half22float2(h);
      f[2 * i] = t.x;
      f[2 * i + 1] = t.y;
    }
  }
}

// Eight consecutive dims of a K / V row at `p` (shared memory) as floats:
// 16-byte loads of 16-bit values, or 8-byte loads of E4M3 bytes widened
// through f16 (exact: every E4M3 value is an f16 value).
template <bool BF16, bool FP8>
__device__ __forceinline__ void load_kv8(const uint8_t* p, float (&f)[8]) {
  if constexpr (FP8) {
    const uint2 raw = *reinterpret_cast<const uint2*>(p);
    const uint32_t w[2] = {raw.x, raw.y};
#pragma unroll
    for (int i = 0; i < 2; ++i) {
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        const __nv_fp8x2_storage_t pair =
            static_cast<__nv_fp8x2_storage_t>((w[i] >> (16 * hh)) & 0xffffu);
        const __half2_raw h = __nv_cvt_fp8x2_to_halfraw2(pair, __NV_E4M3);
        const float2 t = __half22float2(*reinterpret_cast<const __half2*>(&h));
        f[4 * i + 2 * hh] = t.x;
        f[4 * i + 2 * hh + 1] = t.y;
      }
    }
  } else {
    cvt8<BF16>(*reinterpret_cast<const uint4*>(p), f);
  }
}

template <bool BF16>
__device__ __forceinline__ void store_out(void* o, int64_t idx, float x) {
  if constexpr (BF16)
    static_cast<__nv_bfloat16*>(o)[idx] = __float2bfloat16_rn(x);
  else
    static_cast<__half*>(o)[idx] = __float2half_rn(x);
}

template <int N>
struct Log2 {
  static constexpr int value = 1 + Log2<N / 2>::value;
};
template <>
struct Log2<1> {
  static constexpr int value = 0;
};

// Sum of v[h] over the 16 lanes of a half-warp, for h = li >> (4 - log2 GM).
template <int GM>
__device__ __forceinline__ float reduce_heads16(float (&v)[GM], int li) {
  constexpr int LG = Log2<GM>::value;
  int n = GM;
#pragma unroll
  for (int step = 0; step < LG; ++step) {
    const int mask = 8 >> step;
    const bool upper = (li & mask) != 0;
    n >>= 1;
#pragma unroll
    for (int k = 0; k < GM / 2; ++k) {
      if (k < n) {
        const float send = upper ? v[k] : v[k + n];
        const float keep = upper ? v[k + n] : v[k];
        v[k] = keep + __shfl_xor_sync(0xffffffffu, send, mask);
      }
    }
  }
  float s = v[0];
#pragma unroll
  for (int mask = 8 >> LG; mask >= 1; mask >>= 1) s += __shfl_xor_sync(0xffffffffu, s, mask);
  return s;
}

struct Geo {
  int32_t r, hk, slot, split, page_base;
  int64_t tok_begin;
  int32_t ntok, nst;
};

__device__ __forceinline__ Geo unit_geo(const DecodeArgs& a, int ui) {
  const int4* rec = reinterpret_cast<const int4*>(a.ws.units + ui);
  const int4 x = __ldg(rec);
  const int4 y = __ldg(rec + 1);
  const int4 z = __ldg(rec + 2);
  Geo g;
  g.r = x.x;
  g.hk = x.y;
  g.slot = y.y;
  g.split = y.z;
  const int64_t kv_len = z.x;  // the request's geometry, copied in by the planner
  g.page_base = y.w;
  g.tok_begin = int64_t(x.w) * a.page_size;  // p0 * P
  const int64_t te = min(int64_t(y.x) * a.page_size, kv_len);
  const int64_t nt = te - g.tok_begin;
  g.ntok = nt > 0 ? int32_t(nt) : 0;
  g.nst = g.ntok > 0 ? (g.ntok + kStageTok - 1) / kStageTok : 1;
  return g;
}

template <int GM, bool BF16, bool FP8>
__global__ void __launch_bounds__(kThreads, 2) decode_kernel(const DecodeArgs a) {
  constexpr int kStages = Kv<FP8>::kStages;
  constexpr int kRowBytes = Kv<FP8>::kRowBytes;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  Smem<FP8>& sm = *reinterpret_cast<Smem<FP8>*>(smem_raw);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  volatile int32_t* err = a.ws.error;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(smem_u32(&sm.full[s]), 1);
      mbar_init(smem_u32(&sm.empty[s]), kConsumerWarps);
    }
    mbar_init(smem_u32(&sm.cbar), kConsumerWarps * 32);
    fence_mbar_init();
  }
  __syncthreads();

  const int u_begin = __ldg(a.ws.work_indptr + blockIdx.x);
  const int u_end = __ldg(a.ws.work_indptr + blockIdx.x + 1);
  const int group = a.group;

  if (warp == kConsumerWarps) {
    // ------------------------------------------------------------ producer
    const uint64_t policy = policy_evict_first();
    const char* kb = static_cast<const char*>(a.k_pool);
    const char* vb = static_cast<const char*>(a.v_pool);
    const int P = a.page_size;
    const int Hk = a.num_kv_heads;
    uint32_t it = 0;
    for (int ui = u_begin; ui < u_end; ++ui) {
      const Geo g = unit_geo(a, ui);
      for (int s = 0; s < g.nst; ++s, ++it) {
        const int stage = it % kStages;
        const uint32_t ph = (it / kStages) & 1u;
        const int tok0 = s * kStageTok;
        const int nt = min(kStageTok, g.ntok - tok0);
        // HND: the page index of the stage's page (lane), loaded before the
        // slot is free so that its latency hides behind the wait
        int64_t phys_l = 0;
        if (a.layout == ATTN_LAYOUT_HND && nt > 0) {
          const int64_t pg = (g.tok_begin + tok0) / P + lane;
          if (pg <= (g.tok_begin + tok0 + nt - 1) / P)
            phys_l = __ldg(a.kv_indices + g.page_base + pg);
        }
        if (!mbar_wait(smem_u32(&sm.empty[stage]), ph ^ 1u, err, ERR_WAIT_EMPTY)) goto drain;
        const uint32_t full = smem_u32(&sm.full[stage]);
        const uint32_t bytes = uint32_t(max(nt, 0)) * 2u * kRowBytes +
                               (s == 0 ? uint32_t(group) * kQRowBytes : 0u);
        if (lane == 0) mbar_arrive_expect_tx(full, bytes);
        __syncwarp();
        Stage<FP8>& S = sm.st[stage];
        if (s == 0 && lane == 0) {
          const char* qsrc = static_cast<const char*>(a.q) +
                             (int64_t(g.r) * a.num_qo_heads + int64_t(g.hk) * group) * kQRowBytes;
          bulk_g2s(smem_u32(S.q), qsrc, uint32_t(group) * kQRowBytes, full);
        }
        if (nt > 0) {
          const int64_t t_lo_all = g.tok_begin + tok0;
          const int64_t t_hi_all = t_lo_all + nt;
          if (a.layout == ATTN_LAYOUT_HND) {
            const int64_t pg_a = t_lo_all / P;
            const int64_t pg_b = (t_hi_all - 1) / P;
            for (int64_t pg = pg_a + lane; pg <= pg_b; pg += 32) {
              const int64_t t_lo = max(pg * P, t_lo_all);
              const int64_t t_hi = min((pg + 1) * P, t_hi_all);
              const int64_t phys =
                  pg - pg_a < 32 ? phys_l : int64_t(__ldg(a.kv_indices + g.page_base + pg));
              const int64_t row = (phys * Hk + g.hk) * P + (t_lo - pg * P);
              const uint32_t off = uint32_t(t_lo - t_lo_all) * kRowBytes;
              const uint32_t nb = uint32_t(t_hi - t_lo) * kRowBytes;
              bulk_g2s_hint(smem_u32(S.k) + off, kb + row * kRowBytes, nb, full, policy);
              bulk_g2s_hint(smem_u32(S.v) + off, vb + row * kRowBytes, nb, full, policy);
            }
          } else {
            for (int j = lane; j < nt; j += 32) {
              const int64_t t = t_lo_all + j;
              const int64_t pg = t / P;
              const int64_t phys = __ldg(a.kv_indices + g.page_base + pg);
              const int64_t row = (phys * P + (t - pg * P)) * Hk + g.hk;
              const uint32_t off = uint32_t(j) * kRowBytes;
              bulk_g2s_hint(smem_u32(S.k) + off, kb + row * kRowBytes, kRowBytes, full, policy);
              bulk_g2s_hint(smem_u32(S.v) + off, vb + row * kRowBytes, kRowBytes, full, policy);
            }
          }
        }
      }
    }
  drain:
    // Make sure no copy into this CTA's shared memory is still in flight.
    if (lane == 0) {
      const uint32_t total = it;
      for (int s = 0; s < kStages; ++s) {
        if (uint32_t(s) >= total) break;
        const uint32_t last = total - 1 - ((total - 1 - s) % kStages);
        mbar_wait(smem_u32(&sm.full[s]), (last / kStages) & 1u, err, ERR_WAIT_DRAIN);
      }
    }
    return;
  }

  // -------------------------------------------------------------- consumers
  constexpr int LG = Log2<GM>::value;
  constexpr int R = 16 / GM;  // lanes of a half-warp holding the same head
  const int hf = lane >> 4;
  const int li = lane & 15;
  const int hsel = li >> (4 - LG);
  // FP8: the key scale of the unit's kv head folds into q, the value scale
  // into the output (o = v_scale * sum p widen(v) / l)
  const float qscale0 = a.sm_scale * kLog2e;
  const int wt0 = warp * kTokPerWarp;
  uint32_t it = 0;
  uint32_t cph = 0;

  for (int ui = u_begin; ui < u_end; ++ui) {
    const Geo g = unit_geo(a, ui);
    float m_run = -INFINITY, l_run = 0.f;
    float acc[GM][8];
    float qf[GM][8];
#pragma unroll
    for (int h = 0; h < GM; ++h)
#pragma unroll
      for (int j = 0; j < 8; ++j) acc[h][j] = 0.f;

    const float qscale = FP8 ? qscale0 * __ldg(a.k_scale + g.hk) : qscale0;
    for (int s = 0; s < g.nst; ++s, ++it) {
      const int stage = it % kStages;
      const uint32_t ph = (it / kStages) & 1u;
      if (!mbar_wait(smem_u32(&sm.full[stage]), ph, err, ERR_WAIT_FULL)) return;
      const Stage<FP8>& S = sm.st[stage];
      if (s == 0) {
#pragma unroll
        for (int h = 0; h < GM; ++h) {
          if (h < group) {
            const uint4 raw = *reinterpret_cast<const uint4*>(&S.q[h * kHeadDim + li * 8]);
            cvt8<BF16>(raw, qf[h]);
#pragma unroll
            for (int j = 0; j < 8; ++j) qf[h][j] *= qscale;
          } else {
#pragma unroll
            for (int j = 0; j < 8; ++j) qf[h][j] = 0.f;
          }
        }
      }
      const int nt = min(kStageTok, g.ntok - s * kStageTok);

      if (wt0 < nt) {
        // ---- scores of this warp's 16 tokens (pair p: token 2p + hf)
        float sc[kTokPerWarp / 2];
#pragma unroll
        for (int p = 0; p < kTokPerWarp / 2; ++p) {
          const int tt = wt0 + 2 * p + hf;
          float kf[8];
          load_kv8<BF16, FP8>(S.k + tt * kRowBytes + li * 8 * (kRowBytes / kHeadDim), kf);
          float part[GM];
#pragma unroll
          for (int h = 0; h < GM; ++h) {
            float d = qf[h][0] * kf[0];
#pragma unroll
            for (int j = 1; j < 8; ++j) d = fmaf(qf[h][j], kf[j], d);
            part[h] = d;
          }
          const float tot = reduce_heads16<GM>(part, li);
          sc[p] = (tt < nt) ? tot : -INFINITY;
        }
        // ---- online softmax for head `hsel`
        float mt = sc[0];
#pragma unroll
        for (int p = 1; p < kTokPerWarp / 2; ++p) mt = fmaxf(mt, sc[p]);
        mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, 16));
        const float m_new = fmaxf(m_run, mt);
        float scale = 1.f;
        float ls = 0.f;
        if (m_new != -INFINITY) {
          scale = ex2(m_run - m_new);
#pragma unroll
          for (int p = 0; p < kTokPerWarp / 2; ++p) {
            sc[p] = ex2(sc[p] - m_new);
            ls += sc[p];
          }
        } else {
#pragma unroll
          for (int p = 0; p < kTokPerWarp / 2; ++p) sc[p] = 0.f;
        }
        ls += __shfl_xor_sync(0xffffffffu, ls, 16);
        l_run = l_run * scale + ls;
        m_run = m_new;
        // ---- publish probabilities and rescale factors to the warp
        float* pb = sm.pbuf[warp];
        if ((li & (R - 1)) == 0) {
#pragma unroll
          for (int p = 0; p < kTokPerWarp / 2; ++p) pb[(2 * p + hf) * GM + hsel] = sc[p];
          if (hf == 0) sm.sbuf[warp][hsel] = scale;
        }
        __syncwarp();
#pragma unroll
        for (int h = 0; h < GM; ++h) {
          const float sh = sm.sbuf[warp][h];
#pragma unroll
          for (int j = 0; j < 8; ++j) acc[h][j] *= sh;
        }
        // ---- acc += p * v
#pragma unroll
        for (int p = 0; p < kTokPerWarp / 2; ++p) {
          const int tt = wt0 + 2 * p + hf;
          if (tt < nt) {
            float vf[8];
            load_kv8<BF16, FP8>(S.v + tt * kRowBytes + li * 8 * (kRowBytes / kHeadDim), vf);
            float pr[GM];
#pragma unroll
            for (int h = 0; h < GM; ++h) pr[h] = pb[(2 * p + hf) * GM + h];
#pragma unroll
            for (int h = 0; h < GM; ++h)
#pragma unroll
              for (int j = 0; j < 8; ++j) acc[h][j] = fmaf(pr[h], vf[j], acc[h][j]);
          }
        }
        __syncwarp();
      }

      if (s == g.nst - 1) {
        // ---- combine the two half-warps, then the four warps
#pragma unroll
        for (int h = 0; h < GM; ++h)
#pragma unroll
          for (int j = 0; j < 8; ++j) acc[h][j] += __shfl_xor_sync(0xffffffffu, acc[h][j], 16);
        const uint32_t cbar = smem_u32(&sm.cbar);
        mbar_arrive(cbar);  // everyone is done with this stage's K/V
        if (!mbar_wait(cbar, cph, err, ERR_WAIT_CONSUMER)) return;
        cph ^= 1u;
        // the stage's K (and, for FP8, V) bytes hold the warps' accumulators
        // [4][GM][128] floats; the row states [4][GM][2] and a flag follow in
        // V (16-bit) or in the stage's q rows (FP8; q already sits in registers)
        static_assert(sizeof(float) * kConsumerWarps * kMaxDecodeGroup * kHeadDim <=
                          sizeof(S.k) + (FP8 ? sizeof(S.v) : 0),
                      "combine buffer fits the stage");
        float* comb = reinterpret_cast<float*>(const_cast<uint8_t*>(S.k));
        float* ml = FP8 ? reinterpret_cast<float*>(const_cast<uint16_t*>(S.q))
                        : reinterpret_cast<float*>(const_cast<uint8_t*>(S.v));
        const float out_scale = FP8 ? __ldg(a.v_scale + g.hk) : 1.f;
        if (hf == 0) {
#pragma unroll
          for (int h = 0; h < GM; ++h) {
            float4* dst = reinterpret_cast<float4*>(comb + (warp * GM + h) * kHeadDim + li * 8);
            dst[0] = make_float4(acc[h][0], acc[h][1], acc[h][2], acc[h][3]);
            dst[1] = make_float4(acc[h][4], acc[h][5], acc[h][6], acc[h][7]);
          }
          if ((li & (R - 1)) == 0) {
            ml[(warp * GM + hsel) * 2] = m_run;
            ml[(warp * GM + hsel) * 2 + 1] = l_run;
          }
        }
        mbar_arrive(cbar);
        if (!mbar_wait(cbar, cph, err, ERR_WAIT_CONSUMER)) return;
        cph ^= 1u;
        const int d = threadIdx.x;  // 0..127
        for (int h = 0; h < group; ++h) {
          float M = -INFINITY;
#pragma unroll
          for (int w = 0; w < kConsumerWarps; ++w) M = fmaxf(M, ml[(w * GM + h) * 2]);
          float out = 0.f, lse2 = -INFINITY;
          if (M != -INFINITY) {
            float L = 0.f, acc_d = 0.f;
#pragma unroll
            for (int w = 0; w < kConsumerWarps; ++w) {
              const float f = ex2(ml[(w * GM + h) * 2] - M);
              L += f * ml[(w * GM + h) * 2 + 1];
              acc_d += f * comb[(w * GM + h) * kHeadDim + d];
            }
            out = acc_d / L;
            lse2 = M + lg2(L);
          }
          if (g.slot < 0) {
            const int64_t row = int64_t(g.r) * a.num_qo_heads + int64_t(g.hk) * group + h;
            store_out<BF16>(a.o, row * kHeadDim + d, out * out_scale);
            if (d == 0 && a.lse) a.lse[row] = lse2 * kLn2;
          } else {
            const int64_t row = int64_t(g.slot) * group + h;
            a.ws.partial_o[row * kHeadDim + d] = out;
            if (d == 0) a.ws.partial_lse[row] = lse2;
          }
        }
        if (g.slot >= 0) {
          // Split item: the last of its units to finish merges every partial
          // state (log-sum-exp weights) and resets the item's counter.
          __threadfence();
          mbar_arrive(cbar);
          if (!mbar_wait(cbar, cph, err, ERR_WAIT_CONSUMER)) return;
          cph ^= 1u;
          volatile int* last_flag = reinterpret_cast<volatile int*>(ml + 2 * kConsumerWarps * GM);
          if (threadIdx.x == 0) {
            const int4 mi = __ldg(a.ws.merge_items + g.split);
            const int old = atomicAdd(a.ws.counters + g.split, 1);
            *last_flag = (old == mi.w - 1) ? 1 : 0;
          }
          mbar_arrive(cbar);
          if (!mbar_wait(cbar, cph, err, ERR_WAIT_CONSUMER)) return;
          cph ^= 1u;
          if (*last_flag) {
            __threadfence();
            const int s0 = __ldg(a.ws.merge_indptr + g.split);
            const int s1 = __ldg(a.ws.merge_indptr + g.split + 1);
            // loads in batches of kB slots (a few L2 round trips, not one per
            // slot); with one head per kv head and up to kB1 slots, LSEs
            // and O values come in one batch
            constexpr int kB = 16, kB1 = 16;
            for (int h = 0; h < group; ++h) {
              if (GM == 1 && s1 - s0 <= kB1) {  // (one head: registers to spare)
                float ls[kB1], ov[kB1];
#pragma unroll
                for (int k = 0; k < kB1; ++k) {
                  const int64_t prow = int64_t(s0 + k) * group + h;
                  ls[k] = s0 + k < s1 ? __ldcg(a.ws.partial_lse + prow) : -INFINITY;
                  ov[k] = s0 + k < s1 ? __ldcg(a.ws.partial_o + prow * kHeadDim + d) : 0.f;
                }
                float M = -INFINITY;
#pragma unroll
                for (int k = 0; k < kB1; ++k) M = fmaxf(M, ls[k]);
                float out = 0.f, lse2 = -INFINITY;
                if (M != -INFINITY) {
                  float L = 0.f, acc_d = 0.f;
#pragma unroll
                  for (int k = 0; k < kB1; ++k) {
                    const float f = ex2(ls[k] - M);
                    L += f;
                    acc_d += f * ov[k];
                  }
                  out = acc_d / L;
                  lse2 = M + lg2(L);
                }
                const int64_t row = int64_t(g.r) * a.num_qo_heads + int64_t(g.hk) * group + h;
                store_out<BF16>(a.o, row * kHeadDim + d, out * out_scale);
                if (d == 0 && a.lse) a.lse[row] = lse2 * kLn2;
                continue;
              }
              float M = -INFINITY;
              for (int b0 = s0; b0 < s1; b0 += kB) {
                float x[kB];
#pragma unroll
                for (int k = 0; k < kB; ++k)
                  x[k] = b0 + k < s1 ? __ldcg(a.ws.partial_lse + int64_t(b0 + k) * group + h)
                                     : -INFINITY;
#pragma unroll
                for (int k = 0; k < kB; ++k) M = fmaxf(M, x[k]);
              }
              float out = 0.f, lse2 = -INFINITY;
              if (M != -INFINITY) {
                float L = 0.f, acc_d = 0.f;
                for (int b0 = s0; b0 < s1; b0 += kB) {
                  float ls[kB], ov[kB];
#pragma unroll
                  for (int k = 0; k < kB; ++k) {
                    const int64_t prow = int64_t(b0 + k) * group + h;
                    ls[k] = b0 + k < s1 ? __ldcg(a.ws.partial_lse + prow) : -INFINITY;
                    ov[k] = b0 + k < s1 ? __ldcg(a.ws.partial_o + prow * kHeadDim + d) : 0.f;
                  }
#pragma unroll
                  for (int k = 0; k < kB; ++k) {
                    const float f = ex2(ls[k] - M);
                    L += f;
                    acc_d += f * ov[k];
                  }
                }
                out = acc_d / L;
                lse2 = M + lg2(L);
              }
              const int64_t row = int64_t(g.r) * a.num_qo_heads + int64_t(g.hk) * group + h;
              store_out<BF16>(a.o, row * kHeadDim + d, out * out_scale);
              if (d == 0 && a.lse) a.lse[row] = lse2 * kLn2;
            }
            if (threadIdx.x == 0) a.ws.counters[g.split] = 0;
          }
        }
        fence_proxy_async_smem();  // generic writes above precede later bulk copies
        mbar_arrive(cbar);
        if (!mbar_wait(cbar, cph, err, ERR_WAIT_CONSUMER)) return;
        cph ^= 1u;
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&sm.empty[stage]));
    }
  }
}

template <int GM, bool BF16, bool FP8>
cudaError_t launch_t(const DecodeArgs& a, cudaStream_t stream) {
  const size_t smem = sizeof(Smem<FP8>);
  static std::atomic<uint64_t> configured{0};
  cudaError_t e = ensure_smem_limit(decode_kernel<GM, BF16, FP8>, int(smem), configured);
  if (e != cudaSuccess) return e;
  decode_kernel<GM, BF16, FP8><<<a.num_ctas, kThreads, smem, stream>>>(a);
  return cudaGetLastError();
}

template <bool BF16, bool FP8>
cudaError_t launch_dtype(const DecodeArgs& a, cudaStream_t stream) {
  if (a.group <= 1) return launch_t<1, BF16, FP8>(a, stream);
  if (a.group <= 2) return launch_t<2, BF16, FP8>(a, stream);
  if (a.group <= 4) return launch_t<4, BF16, FP8>(a, stream);
  return launch_t<8, BF16, FP8>(a, stream);
}

}  // namespace

int decode_ctas_per_sm() { return 2; }

cudaError_t launch_decode(const DecodeArgs& a, cudaStream_t stream) {
  if (a.num_ctas <= 0) return cudaSuccess;
  if (a.kv_fp8)
    return a.dtype == ATTN_BF16 ? launch_dtype<true, true>(a, stream)
                                : launch_dtype<false, true>(a, stream);
  return a.dtype == ATTN_BF16 ? launch_dtype<true, false>(a, stream)
                              : launch_dtype<false, false>(a, stream);
}

}  // namespace attn
