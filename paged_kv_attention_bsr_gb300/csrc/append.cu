// append.cu -- append / prefill attention over a BSR paged KV cache on the
// 5th-generation tensor cores (tcgen05 MMA, TMEM accumulators, TMA loads).
//
// Method: many new query rows of a request attend to that request's paged KV
// (which already holds the new tokens), with the causal mask aligned to the
// end of the sequence (FlashInfer README copy on gittoolsai.com, "解码、预填充
// 与追加"; paged KV per the modb.pro digest, "统一的 KV 缓存存储格式"). Work
// follows the CPU plan of "动态负载均衡调度" in a persistent fixed grid.
//
// Tile shapes. A work unit is (request r, kv head hk, item t, pages [p0, p1)).
// An item packs 256 query rows (token x GQA head, row = token * group + head)
// as two 128-row query tiles A and B, so every K/V tile read from L2/HBM
// feeds both tiles and every head of the GQA group. K/V tiles hold 128 kv
// tokens, gathered from the page table in 16-row TMA boxes when
// page_size % 16 == 0, else four rows at a time with TMA gathers (any page
// size down to one token per page: vector-level sparsity); HND or NHD pools.
//
// Per KV tile j (all MMAs M = N = 128, bf16/fp16 in, fp32 accumulate), for
// each query tile x:
//   S_x = Q_x K_j^T          A = Q_x (smem, K-major), B = K (smem, K-major),
//                            D = TMEM S_x
//   P_x = exp2(S_x*c - m)    softmax warpgroup x, one TMEM lane (= row) per
//                            thread; P_x (bf16/fp16) written over S_x in TMEM
//   O_x += P_x V_j           A = P_x (TMEM), B = V (smem, MN-major), D = TMEM O_x
// Keeping P in tensor memory halves the shared-memory traffic of P.V (only V
// is read from shared memory) and removes P's shared-memory writes; with
// both MMA operands in shared memory the kernel would be bound by shared
// memory bandwidth well before the tensor core.
// Warp roles (320 threads, one CTA per SM): warps 0-3 and 4-7 are the softmax
// warpgroups of tiles A and B (lazy O rescale only when a row max grows by
// more than 2^8, epilogue from TMEM); warp 8 issues TMA loads through a ring
// of 32 KB K/V slots; warp 9 allocates TMEM and issues the MMAs from one
// thread (P_x(j).V then S_x(j+1) per tile x), so the tensor core works on one
// query tile while the other tile's softmax runs.
// Every wait is bounded; TMEM is freed on every path.
//
// Decode mode (no qo_indptr): one query row per request; an item is the
// group's query heads of one request (group rows of tile A).
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <cstring>
#include <mutex>

#include "internal.h"
#include "ptx.cuh"
#include "tc.cuh"

namespace attn {
namespace {

constexpr int kTile = 128;
constexpr int kChunk = 16;                  // kv rows per TMA box
constexpr int kHalf = kTile * 128;          // 128 rows x 128 B (64 x 16-bit)
constexpr int kTileBytes = 2 * kHalf;       // 128 x 128 x 16-bit
constexpr int kWarpSoftmax0 = 0;            // warps 0-3: tile A, 4-7: tile B
constexpr int kWarpLoad = 8;                // warps 8-11: load, MMA, 2 idle
constexpr int kWarpMma = 9;
constexpr int kWarpRope0 = 10;              // RoPE: warps 10-11 turn q and K rows
constexpr int kThreads = 384;
// Register split (setmaxnreg): launched at 168 per thread (384 x 168 =
// 64512); the load/MMA/rope warpgroup drops to 104 (frees 128 x 64 = 8192)
// and the two softmax warpgroups rise to 192 (take 256 x 24 = 6144). Per
// scheduler: 192 + 192 + 104 registers x 32 lanes <= 16384.
constexpr int kRegsLaunch = 168;
constexpr int kRegsControl = 104;
constexpr int kRegsSoftmax = 192;
static_assert(128 * kRegsControl + 256 * kRegsSoftmax <= kThreads * kRegsLaunch,
              "register split exceeds the launch allocation");
// K tiles in flight between the TMA and the S MMA are at most three (the
// ring holds at most 2.5 K/V tile pairs), so three k_rot barriers, used by
// K tile kt as k_rot[kt % 3] with parity (kt / 3) & 1, never run ahead of
// their waiter.
constexpr int kKRot = 3;
constexpr uint32_t kTmemCols = 512;
// TMEM columns of query tile x: S_x (then P_x, packed 16-bit, over its first
// 64 columns) at 256 x, O_x at 256 x + 128.
constexpr uint32_t kColS = 0;
constexpr uint32_t kColO = 128;
constexpr uint32_t kColTile = 256;

// Shared memory map (offsets from a 1024-byte aligned base) for NQ query
// tiles per item. K and V tiles travel through one ring of SLOTS 32 KB slots:
// KV tile j's K takes slot use 2j and its V use 2j + 1 (slot = use % SLOTS).
// P never touches shared memory: it is written over S in TMEM and the P.V
// MMA reads it from there.
constexpr int kMaxSlots = 6;
template <int NQ>
struct Layout {
  static constexpr int SLOTS = NQ == 2 ? 5 : 6;
  static constexpr int OFF_Q = 0;                            // query tiles
  static constexpr int OFF_RING = OFF_Q + NQ * kTileBytes;   // K/V ring
  static constexpr int OFF_BAR = OFF_RING + SLOTS * kTileBytes;
  static constexpr int SMEM = OFF_BAR + 256 + 1024;         // + barriers + alignment slack
};
static_assert(Layout<1>::OFF_BAR == Layout<2>::OFF_BAR, "both layouts fill 224 KB");

struct Bars {
  uint64_t q_full, q_empty;
  uint64_t slot_full[kMaxSlots], slot_empty[kMaxSlots];
  uint64_t s_full[2];
  uint64_t p_full[2], o_done[2], o_free[2];
  uint64_t drain;
  uint64_t q_rot;          // RoPE: the unit's query rows are turned (count 64)
  uint64_t k_rot[kKRot];   // RoPE: K tile kt is turned in its slot (count 64)
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
  int32_t gather;  // K / V rows gathered 4 at a time (page_size % 16 != 0)
  int32_t nhd;     // pools are NHD [pages, P, Hk, 128] (else HND [pages, Hk, P, 128])
};

// The two 16-bit values of a word as floats.
template <bool BF16>
__device__ __forceinline__ float2 unpack2(uint32_t w) {
  if constexpr (BF16) {
    return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
  } else {
    return __half22float2(*reinterpret_cast<const __half2*>(&w));
  }
}

// Rotary embedding of 4 pairs (dims d..d+3 with d+64..d+67) of a row: x / y
// hold the lower / upper dims, c / s the cos / sin of the pairs' angles at
// the row's position; x' = x cos - y sin, y' = y cos + x sin in fp32, then
// rounded to the storage type.
template <bool BF16>
__device__ __forceinline__ void rope_pairs4(uint2& x, uint2& y, const float4 c, const float4 s) {
  const float2 x0 = unpack2<BF16>(x.x), x1 = unpack2<BF16>(x.y);
  const float2 y0 = unpack2<BF16>(y.x), y1 = unpack2<BF16>(y.y);
  const float2 c0 = make_float2(c.x, c.y), c1 = make_float2(c.z, c.w);
  const float2 s0 = make_float2(s.x, s.y), s1 = make_float2(s.z, s.w);
  const float2 ns0 = make_float2(-s.x, -s.y), ns1 = make_float2(-s.z, -s.w);
  // packed fp32x2: x' = x cos - y sin, y' = y cos + x sin
  const float2 xr0 = ffma2(y0, ns0, fmul2(x0, c0)), xr1 = ffma2(y1, ns1, fmul2(x1, c1));
  const float2 yr0 = ffma2(x0, s0, fmul2(y0, c0)), yr1 = ffma2(x1, s1, fmul2(y1, c1));
  x = make_uint2(pack2<BF16>(xr0.x, xr0.y), pack2<BF16>(xr1.x, xr1.y));
  y = make_uint2(pack2<BF16>(yr0.x, yr0.y), pack2<BF16>(yr1.x, yr1.y));
}

// --------------------------------------------------------- unit geometry
struct AGeo {
  int32_t r, hk, t, slot, page_base;
  int32_t ntiles;  // 128-token KV tiles of the unit
  int32_t nq;      // 128-row query tiles of the item that hold queries (1 or 2)
  int64_t qo_start, qo_len, kv_len;
  int64_t tok_begin, tok_end;
};

// Every role prefetches the next unit's records into L1 when it starts a
// unit, so that their global-load latency is spent under the current unit's
// work and not between two units, where it would delay the next first tile.
__device__ __forceinline__ AGeo append_geo(const AppendArgs& a, int ui) {
  const int4* rec = reinterpret_cast<const int4*>(a.ws.units + ui);
  prefetch_l1(rec + 3);
  prefetch_l1(rec + 5);
  const int4 x = __ldg(rec);
  const int4 y = __ldg(rec + 1);
  const int4 z = __ldg(rec + 2);
  AGeo g;
  g.r = x.x;
  g.hk = x.y;
  g.t = x.z;
  g.slot = y.y;
  g.page_base = y.w;  // the request's geometry, copied in by the planner
  g.kv_len = z.x;
  g.qo_start = z.y;
  g.qo_len = z.z;
  int64_t vis = g.kv_len;
  if (a.causal) {
    const int64_t last_row = min(int64_t(g.t + 1) * a.q_tile, g.qo_len) - 1;
    vis = min(g.kv_len, max(int64_t(0), g.kv_len - g.qo_len + last_row + 1));
  }
  g.tok_begin = int64_t(x.w) * a.page_size;
  g.tok_end = min(int64_t(y.x) * a.page_size, vis);
  const int64_t nt = g.tok_end - g.tok_begin;
  g.ntiles = nt > 0 ? int32_t((nt + kTile - 1) / kTile) : 0;
  const int64_t rem = g.qo_len - int64_t(g.t) * a.q_tile;  // queries left for this item
  g.nq = (a.q_tile > a.tile_tokens && rem > a.tile_tokens) ? 2 : 1;  // capped by NQ at use
  return g;
}

// K / V producer modes: 16-row boxes of HND pools, 16-row boxes of NHD pools
// (a 3-D map [tokens, Hk, 128] whose box is 16 tokens of one head), rows
// gathered four at a time (page sizes that are not a multiple of 16).
constexpr int kModeHndBox = 0;
constexpr int kModeNhdBox = 1;
constexpr int kModeGather = 2;

// The TMA producer warp: per KV tile of each unit, K then V into the next
// ring slots, and after tile 0's K / V the unit's query tile(s) once the
// previous unit's last S MMA has read the query buffer. Boxes: lane c
// fetches the page index of the tile's 16-row chunk c and issues that
// chunk's boxes, so the tile's index loads overlap. Gathers: lane c fetches
// the rows of tokens 4c .. 4c+3 with one tile::gather4 per 64-dim half,
// tokens past the unit's end repeating its last token (every row read lies
// in the pool; those K columns are masked, those V rows zeroed).
struct ProducerEnd {
  uint32_t ua;    // units whose query tiles were loaded
  uint32_t uses;  // ring slot uses (K and V tiles) issued
  bool ok;        // no wait gave up
};

template <int NQ, int MODE>
__device__ __forceinline__ ProducerEnd produce_kv(const AppendParams& prm, Bars& bars,
                                                  uint32_t base, int lane,
                                                  volatile int32_t* err) {
  uint32_t ua = 0, uses = 0;
  bool ok = true;
  constexpr int kSlots = Layout<NQ>::SLOTS;
  constexpr int kOffQ = Layout<NQ>::OFF_Q;
  constexpr int kOffRing = Layout<NQ>::OFF_RING;
  constexpr uint32_t kRowsPerLd = MODE == kModeGather ? 4u : uint32_t(kChunk);
  const AppendArgs& a = prm.a;
  const int P = a.page_size;
  const int Hk = a.num_kv_heads;
  const int group = a.group;
  const uint32_t tile_rows = uint32_t(group * a.tile_tokens);
  auto wait0 = [&](uint32_t bar, uint32_t parity) -> bool {
    bool r = true;
    if (lane == 0) r = mbar_wait(bar, parity, err, ERR_WAIT_EMPTY);
    return __shfl_sync(0xffffffffu, r ? 1 : 0, 0) != 0;
  };
  for (int vc = blockIdx.x; vc < a.num_ctas && ok; vc += gridDim.x)
  for (int ui = __ldg(a.ws.work_indptr + vc); ui < __ldg(a.ws.work_indptr + vc + 1) && ok; ++ui) {
    AGeo g = append_geo(a, ui);
    g.nq = min(g.nq, NQ);
    if (g.ntiles == 0) continue;
    for (int i = 0; i < g.ntiles && ok; ++i) {
      const int64_t kv0 = g.tok_begin + int64_t(i) * kTile;
      const int ntt = int(min(int64_t(kTile), g.tok_end - kv0));
      const int nld = MODE == kModeGather ? (ntt + 3) / 4 : (ntt + kChunk - 1) / kChunk;
      int32_t row[MODE == kModeGather ? 4 : 1];
#pragma unroll
      for (int u = 0; u < int(sizeof(row) / sizeof(row[0])); ++u) row[u] = 0;
      if (lane < nld) {
        if constexpr (MODE == kModeGather) {
          const int64_t t0 = kv0 + 4 * lane;
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const int64_t t = min(t0 + u, g.tok_end - 1);
            const int64_t pg = t / P;
            const int64_t sl = t - pg * P;
            const int64_t phys = __ldg(a.kv_indices + g.page_base + pg);
            row[u] = prm.nhd ? int32_t((phys * P + sl) * Hk + g.hk)
                             : int32_t((phys * Hk + g.hk) * P + sl);
          }
        } else {
          const int64_t kvt = kv0 + int64_t(lane) * kChunk;
          const int64_t pg = kvt / P;
          const int64_t phys = __ldg(a.kv_indices + g.page_base + pg);
          row[0] = MODE == kModeNhdBox ? int32_t(phys * P + (kvt - pg * P))  // token row
                                       : int32_t((phys * Hk + g.hk) * P + (kvt - pg * P));
        }
      }
      for (int kv = 0; kv < 2; ++kv, ++uses) {  // K then V
        const int slot = int(uses % kSlots);
        if (!wait0(smem_u32(&bars.slot_empty[slot]), ((uses / kSlots) & 1u) ^ 1u)) {
          ok = false;
          break;
        }
        const uint32_t full = smem_u32(&bars.slot_full[slot]);
        if (lane == 0) mbar_arrive_expect_tx(full, uint32_t(nld) * kRowsPerLd * 256u);
        __syncwarp();
        if (lane < nld) {
          const uint32_t dst =
              base + kOffRing + slot * kTileBytes + uint32_t(lane) * kRowsPerLd * 128u;
          const void* tm = kv == 0 ? static_cast<const void*>(&prm.tm_k)
                                   : static_cast<const void*>(&prm.tm_v);
          if constexpr (MODE == kModeGather) {
            tma_gather4(dst, tm, 0, row[0], row[1], row[2], row[3], full);
            tma_gather4(dst + kHalf, tm, 64, row[0], row[1], row[2], row[3], full);
          } else if constexpr (MODE == kModeNhdBox) {
            tma_load_3d(dst, tm, 0, g.hk, row[0], full);
            tma_load_3d(dst + kHalf, tm, 64, g.hk, row[0], full);
          } else {
            tma_load_2d(dst, tm, 0, row[0], full);
            tma_load_2d(dst + kHalf, tm, 64, row[0], full);
          }
        }
      }
      if (i == 0 && ok) {
        // the unit's query tile(s), once the previous unit's last S MMA is done
        if (!wait0(smem_u32(&bars.q_empty), (ua & 1u) ^ 1u)) {
          ok = false;
          break;
        }
        if (lane == 0) {
          const uint32_t qf = smem_u32(&bars.q_full);
          mbar_arrive_expect_tx(qf, 256u * tile_rows * uint32_t(g.nq));
          for (int x = 0; x < g.nq; ++x) {
            const int32_t qrow =
                int32_t(g.qo_start + int64_t(g.t) * a.q_tile + x * a.tile_tokens);
            const uint32_t dst = base + kOffQ + x * kTileBytes;
            tma_load_3d(dst, &prm.tm_q, 0, g.hk * group, qrow, qf);
            tma_load_3d(dst + kHalf, &prm.tm_q, 64, g.hk * group, qrow, qf);
          }
        }
        ++ua;
      }
    }
  }
  return {ua, uses, ok};
}

template <int NQ, int MODE>
__device__ __noinline__ ProducerEnd produce_kv_outlined(const AppendParams& prm, Bars& bars,
                                                        uint32_t base, int lane,
                                                        volatile int32_t* err) {
  return produce_kv<NQ, MODE>(prm, bars, base, lane, err);
}

template <bool BF16, int NQ, bool ROPE>
__global__ void __launch_bounds__(kThreads, 1) append_kernel(const __grid_constant__ AppendParams prm) {
  constexpr int kSlots = Layout<NQ>::SLOTS;
  constexpr int kOffQ = Layout<NQ>::OFF_Q;
  constexpr int kOffRing = Layout<NQ>::OFF_RING;
  constexpr int kOffBar = Layout<NQ>::OFF_BAR;
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
      mbar_init(smem_u32(&bars.p_full[i]), 128);
      mbar_init(smem_u32(&bars.o_done[i]), 1);
      mbar_init(smem_u32(&bars.o_free[i]), 128);
    }
    mbar_init(smem_u32(&bars.drain), 1);
    mbar_init(smem_u32(&bars.q_rot), 64);
    for (int i = 0; i < kKRot; ++i) mbar_init(smem_u32(&bars.k_rot[i]), 64);
    fence_mbar_init();
  }
  if (warp == kWarpLoad && lane == 0) {
    prefetch_tmap(&prm.tm_q);
    prefetch_tmap(&prm.tm_k);
    prefetch_tmap(&prm.tm_v);
  }
  if (warp == kWarpMma) {
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
  const int group = a.group;

  // TMEM columns. Two query tiles: tile x has S_x/P_x at 256 x and O_x at
  // 256 x + 128. One query tile: S/P double-buffered at 0 and 128 (KV tile k
  // uses buffer k & 1, so S of tile k+1 runs under the softmax of tile k), O
  // at 256.
  auto col_s = [](int x, uint32_t k) -> uint32_t {
    return NQ == 2 ? uint32_t(x) * kColTile + kColS : (k & 1u) * 128u;
  };
  auto col_o = [](int x) -> uint32_t { return NQ == 2 ? uint32_t(x) * kColTile + kColO : 256u; };

  // A CTA runs the unit lists of plan CTAs blockIdx.x, blockIdx.x + gridDim.x,
  // ... (the grid is at most one CTA per SM; a plan may have more CTAs).
  if (warp >= kWarpLoad) {
  // warpgroup 2: TMA loads, MMA issue, two warps idle (or turning q and K rows
  // with RoPE); gives registers away
  asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegsControl));
  if (warp == kWarpLoad) {
    // ------------------------------------------------------------ TMA producer
    // HND pools at page sizes that are a multiple of 16 (the common case)
    // inline; NHD pools and gathered rows out of line, so that the kernel
    // body the softmax warps run from stays as compact as without them.
    const ProducerEnd pe =
        prm.gather ? produce_kv_outlined<NQ, kModeGather>(prm, bars, base, lane, err)
        : prm.nhd  ? produce_kv_outlined<NQ, kModeNhdBox>(prm, bars, base, lane, err)
                   : produce_kv<NQ, kModeHndBox>(prm, bars, base, lane, err);
    const uint32_t ua = pe.ua, uses = pe.uses;
    // drain: every issued copy has landed before the CTA can exit
    if (lane == 0) {
      if (ua > 0) mbar_wait(smem_u32(&bars.q_full), (ua - 1) & 1u, err, ERR_WAIT_DRAIN);
      for (uint32_t sl = 0; sl < uint32_t(kSlots) && sl < uses; ++sl) {
        const uint32_t last = uses - 1 - ((uses - 1 - sl) % kSlots);
        mbar_wait(smem_u32(&bars.slot_full[sl]), (last / kSlots) & 1u, err, ERR_WAIT_DRAIN);
      }
    }
    __syncwarp();
  } else if (warp == kWarpMma) {
    // ------------------------------------------------------------ MMA issuer
    // Per KV tile i of a unit, for each live query tile x (0 = A, 1 = B), in
    // issue order: O_x += P_x(i) V_i once softmax x has written P_x(i) into
    // TMEM, then S_x(i+1) = Q_x K_{i+1}^T into the same columns. The tensor
    // core runs in issue order, so S_x(i+1) completing (s_full) also means
    // P_x(i) has been consumed and O_x is up to date. While tile A's softmax
    // runs, the tensor core works on tile B's P.V and S, and vice versa.
    if (lane == 0) {
      uint32_t ua = 0, jt = 0;
      uint32_t n_p[2] = {0, 0}, n_u[2] = {0, 0};
      bool ok = true;
      auto slot_of = [&](uint32_t use) { return use % kSlots; };
      auto wait_slot = [&](uint32_t use) -> bool {
        return mbar_wait(smem_u32(&bars.slot_full[slot_of(use)]), (use / kSlots) & 1u, err,
                         ERR_WAIT_FULL);
      };
      // K tile kt (slot use 2 kt) has landed and, with RoPE, been turned
      auto wait_k = [&](uint32_t kt) -> bool {
        if constexpr (ROPE)
          return mbar_wait(smem_u32(&bars.k_rot[kt % kKRot]), (kt / kKRot) & 1u, err,
                           ERR_WAIT_FULL);
        else
          return wait_slot(2 * kt);
      };
      // S for query tile x and KV tile k (global count) from the K in kslot
      auto issue_s = [&](int x, uint32_t kslot, uint32_t k) {
        const uint32_t qbase = base + kOffQ + x * kTileBytes;
        const uint32_t kbase = base + kOffRing + kslot * kTileBytes;
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const uint32_t koff = (kk >> 2) * kHalf + (kk & 3) * 32;
          mma_f16(tmem + col_s(x, k), smem_desc(qbase + koff, 16, 1024),
                  smem_desc(kbase + koff, 16, 1024), prm.idesc_s, kk > 0 ? 1u : 0u);
        }
        mma_commit(smem_u32(&bars.s_full[NQ == 2 ? x : int(k & 1u)]));
      };
      // O_x += P_x(k) V once softmax x has written P_x(k) into TMEM
      auto issue_pv = [&](int x, uint32_t vslot, uint32_t k, bool first) -> bool {
        // one query tile: the softmax of tile k+1 may finish before P(k).V is
        // issued (S(k+1) precedes it), so tile k signals p_full[k & 1]
        const int pb = NQ == 2 ? x : int(k & 1u);
        const uint32_t ppar = NQ == 2 ? (n_p[x] & 1u) : ((k >> 1) & 1u);
        if (!mbar_wait(smem_u32(&bars.p_full[pb]), ppar, err, ERR_WAIT_SOFTMAX)) return false;
        if (first &&
            !mbar_wait(smem_u32(&bars.o_free[x]), (n_u[x] & 1u) ^ 1u, err, ERR_WAIT_SOFTMAX))
          return false;
        tc_fence_after();
        const uint32_t vbase = base + kOffRing + vslot * kTileBytes;
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const uint64_t bd = smem_desc(vbase + kk * kChunk * 128, kHalf, 1024);
          mma_f16_ts(tmem + col_o(x), tmem + col_s(x, k) + kk * 8, bd, prm.idesc_pv,
                     (first && kk == 0) ? 0u : 1u);
        }
        mma_commit(smem_u32(&bars.o_done[NQ == 2 ? x : int(k & 1u)]));
        ++n_p[x];
        return true;
      };
      for (int vc = blockIdx.x; vc < a.num_ctas && ok; vc += gridDim.x)
      for (int ui = __ldg(a.ws.work_indptr + vc); ui < __ldg(a.ws.work_indptr + vc + 1) && ok; ++ui) {
        AGeo g = append_geo(a, ui);
        g.nq = min(g.nq, NQ);
        if (g.ntiles == 0) continue;
        const int n = g.ntiles;
        if (!mbar_wait(smem_u32(ROPE ? &bars.q_rot : &bars.q_full), ua & 1u, err,
                       ERR_WAIT_FULL) ||
            !wait_k(jt)) {
          ok = false;
          break;
        }
        tc_fence_after();
        if constexpr (NQ == 2) {
          // S_A(0), S_B(0); then per KV tile i: P_A(i).V, S_A(i+1), P_B(i).V, S_B(i+1)
#pragma unroll
          for (int x = 0; x < 2; ++x)
            if (x < g.nq) issue_s(x, slot_of(2 * jt), jt);
          mma_commit(smem_u32(&bars.slot_empty[slot_of(2 * jt)]));
          if (n == 1) mma_commit(smem_u32(&bars.q_empty));
          for (int i = 0; i < n && ok; ++i) {
            const uint32_t k = jt + i;
            const bool more = i + 1 < n;
            if (!wait_slot(2 * k + 1)) {
              ok = false;
              break;
            }
#pragma unroll
            for (int x = 0; x < 2; ++x) {
              if (x < g.nq && ok) {
                ok = issue_pv(x, slot_of(2 * k + 1), k, i == 0);
                if (ok && more) {
                  if (x == 0 && !wait_k(k + 1)) {
                    ok = false;
                    break;
                  }
                  tc_fence_after();
                  issue_s(x, slot_of(2 * k + 2), k + 1);
                }
              }
            }
            if (!ok) break;
            if (more) {
              mma_commit(smem_u32(&bars.slot_empty[slot_of(2 * k + 2)]));
              if (i + 2 == n) mma_commit(smem_u32(&bars.q_empty));  // last S issued
            }
            mma_commit(smem_u32(&bars.slot_empty[slot_of(2 * k + 1)]));
          }
        } else {
          // S(0), S(1) into the two S buffers; then per KV tile i: P(i).V, S(i+2)
          issue_s(0, slot_of(2 * jt), jt);
          mma_commit(smem_u32(&bars.slot_empty[slot_of(2 * jt)]));
          if (n > 1) {
            if (!wait_k(jt + 1)) {
              ok = false;
              break;
            }
            tc_fence_after();
            issue_s(0, slot_of(2 * jt + 2), jt + 1);
            mma_commit(smem_u32(&bars.slot_empty[slot_of(2 * jt + 2)]));
          }
          if (n <= 2) mma_commit(smem_u32(&bars.q_empty));
          for (int i = 0; i < n && ok; ++i) {
            const uint32_t k = jt + i;
            if (!wait_slot(2 * k + 1)) {
              ok = false;
              break;
            }
            ok = issue_pv(0, slot_of(2 * k + 1), k, i == 0);
            if (ok && i + 2 < n) {
              if (!wait_k(k + 2)) {
                ok = false;
                break;
              }
              tc_fence_after();
              issue_s(0, slot_of(2 * k + 4), k + 2);
              mma_commit(smem_u32(&bars.slot_empty[slot_of(2 * k + 4)]));
              if (i + 3 == n) mma_commit(smem_u32(&bars.q_empty));  // last S issued
            }
            mma_commit(smem_u32(&bars.slot_empty[slot_of(2 * k + 1)]));
          }
        }
        if (!ok) break;
#pragma unroll
        for (int x = 0; x < 2; ++x)
          if (x < g.nq) ++n_u[x];
        jt += n;
        ++ua;
      }
      // drain: no MMA may still be writing TMEM when it is freed
      mma_commit(smem_u32(&bars.drain));
      mbar_wait(smem_u32(&bars.drain), 0, err, ERR_WAIT_DRAIN);
    }
    __syncwarp();
  } else if (ROPE && warp >= kWarpRope0) {
    // ------------------------------------------------------------ rope warps
    // Warps 10-11 turn each unit's query rows once (between the query TMA
    // and the unit's first S MMA; query i of a request at position
    // kv_len - qo_len + i) and every K tile in its ring slot (between its
    // TMA and the S MMAs that read it; key j at position j). A half-warp
    // takes a row: lane l holds the pairs (d, d + 64), d = 4 (l % 16) .. + 3,
    // one 8-byte piece in each 64-dim half of the 128B-swizzled tile, at the
    // same offset in both halves. The tables hold cos / sin of pos * theta_d,
    // so a half-warp walks consecutive positions by turning its (cos, sin)
    // by theta_d (table row 1) at each step and reloads the table every 8-16
    // positions: one table row per 8 K rows and per 16 query tokens. The MMA warp waits on
    // q_rot / k_rot instead of the TMA barriers.
    const int hq = (warp - kWarpRope0) * 2 + (lane >> 4);  // half-warp 0..3
    const int l16 = lane & 15;
    const int kbyte = ((l16 >> 1) << 4) | ((l16 & 1) << 3);  // piece, byte in it
    auto table_row = [&](int64_t pos, float4& c, float4& sn) {
      c = __ldg(reinterpret_cast<const float4*>(a.rope_cos + pos * (kHeadDim / 2) + 4 * l16));
      sn = __ldg(reinterpret_cast<const float4*>(a.rope_sin + pos * (kHeadDim / 2) + 4 * l16));
    };
    float4 ct = make_float4(1.f, 1.f, 1.f, 1.f), stt = make_float4(0.f, 0.f, 0.f, 0.f);
    if (a.rope_rows > 1) table_row(1, ct, stt);  // cos / sin of theta_d
    // (c, sn) at position p -> at p + 1
    const float2 ct0 = make_float2(ct.x, ct.y), ct1 = make_float2(ct.z, ct.w);
    const float2 st0 = make_float2(stt.x, stt.y), st1 = make_float2(stt.z, stt.w);
    const float2 nst0 = make_float2(-stt.x, -stt.y), nst1 = make_float2(-stt.z, -stt.w);
    auto step = [&](float4& c, float4& sn) {  // packed fp32x2 angle sums
      const float2 c0 = make_float2(c.x, c.y), c1 = make_float2(c.z, c.w);
      const float2 s0 = make_float2(sn.x, sn.y), s1 = make_float2(sn.z, sn.w);
      const float2 cn0 = ffma2(s0, nst0, fmul2(c0, ct0)), cn1 = ffma2(s1, nst1, fmul2(c1, ct1));
      const float2 sn0 = ffma2(c0, st0, fmul2(s0, ct0)), sn1 = ffma2(c1, st1, fmul2(s1, ct1));
      c = make_float4(cn0.x, cn0.y, cn1.x, cn1.y);
      sn = make_float4(sn0.x, sn0.y, sn1.x, sn1.y);
    };
    auto turn = [&](uint8_t* tile, int row, const float4 c, const float4 sn) {
      const int off = row * 128 + (kbyte ^ ((row & 7) << 4));
      uint2 x = *reinterpret_cast<const uint2*>(tile + off);
      uint2 y = *reinterpret_cast<const uint2*>(tile + kHalf + off);
      rope_pairs4<BF16>(x, y, c, sn);
      *reinterpret_cast<uint2*>(tile + off) = x;
      *reinterpret_cast<uint2*>(tile + kHalf + off) = y;
    };
    uint32_t ua = 0, jt = 0;
    bool ok = true;
    for (int vc = blockIdx.x; vc < a.num_ctas && ok; vc += gridDim.x)
    for (int ui = __ldg(a.ws.work_indptr + vc); ui < __ldg(a.ws.work_indptr + vc + 1) && ok; ++ui) {
      AGeo g = append_geo(a, ui);
      g.nq = min(g.nq, NQ);
      if (g.ntiles == 0) continue;
      // ---- query rows: tile x, token tau (row tau * group + head) at
      // position kv_len - qo_len + t * q_tile + x * tile_tokens + tau; a
      // half-warp takes a quarter of each tile's tokens, all their heads
      if (!mbar_wait(smem_u32(&bars.q_full), ua & 1u, err, ERR_WAIT_FULL)) {
        ok = false;
        break;
      }
      const int T = a.tile_tokens;
      for (int x = 0; x < g.nq; ++x) {
        uint8_t* qt = gbase + kOffQ + x * kTileBytes;
        const int64_t qi0 = int64_t(g.t) * a.q_tile + int64_t(x) * T;
        const int tau1 = min((hq + 1) * T / 4, int(max(int64_t(0), g.qo_len - qi0)));
        float4 c, sn;
        for (int tau = hq * T / 4; tau < tau1; ++tau) {
          if ((tau - hq * T / 4) % 16 == 0) table_row(g.kv_len - g.qo_len + qi0 + tau, c, sn);
#pragma unroll 1
          for (int h = 0; h < group; ++h) turn(qt, tau * group + h, c, sn);
          step(c, sn);
        }
      }
      fence_proxy_async_smem();  // generic stores -> the MMA's operand reads
      mbar_arrive(smem_u32(&bars.q_rot));
      ++ua;
      // ---- K tiles: half-warp hq takes rows [32 hq, 32 hq + 32), two at a time
      for (int i = 0; i < g.ntiles && ok; ++i) {
        const uint32_t kt = jt + i, use = 2 * kt;
        if (!mbar_wait(smem_u32(&bars.slot_full[use % kSlots]), (use / kSlots) & 1u, err,
                       ERR_WAIT_FULL)) {
          ok = false;
          break;
        }
        const int64_t kv0 = g.tok_begin + int64_t(i) * kTile;
        const int ntt = int(min(int64_t(kTile), g.tok_end - kv0));
        uint8_t* kt_tile = gbase + kOffRing + (use % kSlots) * kTileBytes;
        // four runs of 8 consecutive rows, one row of each per step: the
        // four rows' shared-memory loads are in flight together
        const int r0 = 32 * hq;
        float4 cg[4], sg[4];
#pragma unroll
        for (int q = 0; q < 4; ++q)
          if (r0 + 8 * q < ntt) table_row(kv0 + r0 + 8 * q, cg[q], sg[q]);
#pragma unroll 1
        for (int k = 0; k < 8; ++k) {
          uint2 x[4], y[4];
          int off[4];
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const int row = r0 + 8 * q + k;
            off[q] = row * 128 + (kbyte ^ ((row & 7) << 4));
            if (row < ntt) {
              x[q] = *reinterpret_cast<const uint2*>(kt_tile + off[q]);
              y[q] = *reinterpret_cast<const uint2*>(kt_tile + kHalf + off[q]);
            }
          }
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            if (r0 + 8 * q + k < ntt) {
              rope_pairs4<BF16>(x[q], y[q], cg[q], sg[q]);
              *reinterpret_cast<uint2*>(kt_tile + off[q]) = x[q];
              *reinterpret_cast<uint2*>(kt_tile + kHalf + off[q]) = y[q];
              step(cg[q], sg[q]);
            }
          }
        }
        fence_proxy_async_smem();
        mbar_arrive(smem_u32(&bars.k_rot[kt % kKRot]));
      }
      jt += g.ntiles;
    }
  }
  } else {
    // ------------------------------------------------- softmax / epilogue
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kRegsSoftmax));
    const int x = (warp - kWarpSoftmax0) / 4;  // query tile of this warpgroup
    const int quarter = warp & 3;               // TMEM lanes this warp may access
    const int rho_t = quarter * 32 + lane;      // row within the query tile
    const int rho = x * kTile + rho_t;          // row within the item
    const uint32_t lane_off = uint32_t(quarter * 32) << 16;
    const uint32_t col_ox = col_o(x);
    const int tok = rho / group;
    const int hh = rho - tok * group;
    const float c2 = prm.scale_log2;
    uint32_t jt = 0, n_t = 0;
    bool ok = x < NQ;  // a one-tile kernel leaves the second warpgroup idle
    for (int vc = blockIdx.x; vc < a.num_ctas && ok; vc += gridDim.x)
    for (int ui = __ldg(a.ws.work_indptr + vc); ui < __ldg(a.ws.work_indptr + vc + 1) && ok; ++ui) {
      AGeo g = append_geo(a, ui);
      g.nq = min(g.nq, NQ);
      const int64_t qi = int64_t(g.t) * a.q_tile + tok;
      const bool row_ok = (rho < a.rows_per_item) && (qi < g.qo_len);
      // warps whose 32 rows hold no query (short query tiles, decode mode)
      // only keep the barrier protocol: their P rows feed O rows that are
      // never stored
      const bool warp_live = __any_sync(0xffffffffu, row_ok);
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
            const int64_t prow = int64_t(g.slot) * a.rows_per_item + rho;
            float4* dst = reinterpret_cast<float4*>(a.ws.partial_o + prow * kHeadDim);
            for (int i = 0; i < 32; ++i) dst[i] = make_float4(0.f, 0.f, 0.f, 0.f);
            a.ws.partial_lse[prow] = -INFINITY;
          }
        }
        continue;
      }
      const uint32_t jt0 = jt;
      jt += g.ntiles;
      if (x >= g.nq) continue;  // this query tile holds no queries for the item
      float m_ref = -INFINITY, l = 0.f;
      for (int i = 0; i < g.ntiles; ++i, ++n_t) {
        // waits are made warp-uniform: tcgen05.ld/st below are .sync.aligned
        // S of this tile: barrier s_full[x] (two tiles) or s_full[n_t & 1] (one
        // tile, S double-buffered: the buffer's uses alternate phases)
        const int sb = NQ == 2 ? x : int(n_t & 1u);
        const uint32_t sparity = NQ == 2 ? (n_t & 1u) : ((n_t >> 1) & 1u);
        const uint32_t col_sx = col_s(x, n_t);
        if (!__all_sync(0xffffffffu, mbar_wait(smem_u32(&bars.s_full[sb]), sparity, err,
                                               ERR_WAIT_MMA))) {
          ok = false;
          break;
        }
        tc_fence_after();
        const int64_t kv0 = g.tok_begin + int64_t(i) * kTile;
        const int nvalid = int(max(int64_t(0), min(int64_t(kTile), row_end - kv0)));
        if (warp_live) {
          float v[kTile];
          tmem_ld128(tmem + lane_off + col_sx, v);
          // Tiles with masked columns (the causal diagonal, the unit's last
          // tile) first set those scores to -inf with selects, no branches
          // (nvalid differs from row to row on the diagonal); every tile then
          // takes the same path. Rows without a query may skip the masking
          // (their P row only feeds their own O row, which is never stored).
          const bool full = __all_sync(0xffffffffu, !row_ok || nvalid == kTile);
          if (!full) {
#pragma unroll
            for (int c = 0; c < kTile; ++c) v[c] = (c < nvalid) ? v[c] : -INFINITY;
          }
          float mx;
          {
            float m0 = fmax3(v[0], v[1], v[2]), m1 = fmax3(v[3], v[4], v[5]);
#pragma unroll
            for (int c = 6; c + 3 < kTile; c += 4) {
              m0 = fmax3(m0, v[c], v[c + 1]);
              m1 = fmax3(m1, v[c + 2], v[c + 3]);
            }
            mx = fmax3(m0, m1, fmaxf(v[kTile - 2], v[kTile - 1]));
          }
          const float m_tile = mx * c2;  // -inf stays -inf
          float alpha = 1.f;
          bool rescale_o = false;
          if (m_tile > m_ref + 8.f) {
            alpha = ex2(m_ref - m_tile);  // 0 when m_ref = -inf
            rescale_o = row_ok && (i > 0) && (m_ref != -INFINITY);
            l *= alpha;
            m_ref = m_tile;
          }
          // O_x must hold every earlier tile before it is rescaled. With two
          // query tiles S_x(i) completing implies P_x(i-1).V is done; with one
          // (S double-buffered) wait for that P.V explicitly.
          if (__any_sync(0xffffffffu, rescale_o)) {
            if (NQ == 1 && i > 0 &&
                !__all_sync(0xffffffffu, mbar_wait(smem_u32(&bars.o_done[(n_t - 1) & 1u]),
                                                   ((n_t - 1) >> 1) & 1u, err, ERR_WAIT_MMA))) {
              ok = false;
              break;
            }
            tc_fence_after();
#pragma unroll 1
            for (int c = 0; c < 4; ++c) {
              float o[32];
              const uint32_t ta = tmem + lane_off + col_ox + c * 32;
              tmem_ld32(ta, o);
              const float f = rescale_o ? alpha : 1.f;
#pragma unroll
              for (int q = 0; q < 32; ++q) o[q] *= f;
              tmem_st32(ta, o);
            }
          }
          // probabilities, packed to the MMA input type, written over S_x in
          // TMEM (column c holds elements 2c, 2c+1 of the row)
          // (a row with no unmasked score yet keeps m_ref = -inf: its scores
          // are all -inf and come out as 0 with a zero offset)
          float2 lsum2 = make_float2(0.f, 0.f);
          {
            const float2 c2x2 = make_float2(c2, c2);
            const float nm = m_ref == -INFINITY ? 0.f : -m_ref;
            const float2 negm = make_float2(nm, nm);
#pragma unroll
            for (int c = 0; c < 4; ++c) {
              uint32_t pk[16];
#pragma unroll
              for (int q = 0; q < 32; q += 2) {
                const float2 t = ffma2(make_float2(v[c * 32 + q], v[c * 32 + q + 1]), c2x2, negm);
                const float2 pr = make_float2(ex2(t.x), ex2(t.y));
                lsum2 = fadd2(lsum2, pr);
                pk[q / 2] = pack2<BF16>(pr.x, pr.y);
              }
              tmem_st16_nowait(tmem + lane_off + col_sx + c * 16, pk);
            }
          }
          tmem_wait_st();
          l += lsum2.x + lsum2.y;
        }
        // kv rows past the unit's end hold whatever the pool had: tile A's
        // warpgroup zeroes them in V once this tile's V has landed
        const int ntt = int(min(int64_t(kTile), g.tok_end - kv0));
        if (x == 0 && ntt < kTile) {
          const uint32_t vuse = 2 * (jt0 + i) + 1;
          if (!__all_sync(0xffffffffu, mbar_wait(smem_u32(&bars.slot_full[vuse % kSlots]),
                                                 (vuse / kSlots) & 1u, err, ERR_WAIT_FULL))) {
            ok = false;
            break;
          }
          if (rho_t >= ntt) {
            uint8_t* vrow = gbase + kOffRing + (vuse % kSlots) * kTileBytes + rho_t * 128;
#pragma unroll
            for (int q = 0; q < 8; ++q) {
              *reinterpret_cast<uint4*>(vrow + q * 16) = make_uint4(0, 0, 0, 0);
              *reinterpret_cast<uint4*>(vrow + kHalf + q * 16) = make_uint4(0, 0, 0, 0);
            }
          }
          fence_proxy_async_smem();
        }
        tc_fence_before();
        mbar_arrive(smem_u32(&bars.p_full[NQ == 2 ? x : int(n_t & 1u)]));
      }
      if (!ok) break;
      // ---- epilogue: O / l
      // P.V of the last tile: with two query tiles S_x(last) completing put
      // O_x one P.V behind; with one, S(last) only follows P.V(last - 2), so
      // P.V of tile k signals o_done[k & 1] and no wait is two phases behind.
      const int od = NQ == 2 ? x : int((n_t - 1) & 1u);
      const uint32_t opar = NQ == 2 ? ((n_t - 1) & 1u) : (((n_t - 1) >> 1) & 1u);
      if (!__all_sync(0xffffffffu, mbar_wait(smem_u32(&bars.o_done[od]), opar, err,
                                             ERR_WAIT_MMA))) {
        ok = false;
        break;
      }
      tc_fence_after();
      const bool any = l > 0.f;
      const float inv = any ? 1.f / l : 0.f;
      const float lse2 = any ? m_ref + lg2(l) : -INFINITY;
#pragma unroll
      for (int c = 0; c < 4 && warp_live; ++c) {
        float o[32];
        tmem_ld32(tmem + lane_off + col_ox + c * 32, o);
        if (row_ok) {
          if (g.slot < 0) {
            uint4* dst =
                reinterpret_cast<uint4*>(static_cast<uint16_t*>(a.o) + orow * kHeadDim + c * 32);
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              uint4 w;
              w.x = pack2<BF16>(o[q * 8 + 0] * inv, o[q * 8 + 1] * inv);
              w.y = pack2<BF16>(o[q * 8 + 2] * inv, o[q * 8 + 3] * inv);
              w.z = pack2<BF16>(o[q * 8 + 4] * inv, o[q * 8 + 5] * inv);
              w.w = pack2<BF16>(o[q * 8 + 6] * inv, o[q * 8 + 7] * inv);
              dst[q] = w;
            }
          } else {
            const int64_t prow = int64_t(g.slot) * a.rows_per_item + rho;
            float4* dst = reinterpret_cast<float4*>(a.ws.partial_o + prow * kHeadDim + c * 32);
#pragma unroll
            for (int q = 0; q < 8; ++q)
              dst[q] = make_float4(o[q * 4] * inv, o[q * 4 + 1] * inv, o[q * 4 + 2] * inv,
                                   o[q * 4 + 3] * inv);
          }
        }
      }
      if (row_ok) {
        if (g.slot < 0) {
          if (a.lse) a.lse[orow] = lse2 * kLn2;
        } else {
          a.ws.partial_lse[int64_t(g.slot) * a.rows_per_item + rho] = lse2;
        }
      }
      tc_fence_before();
      mbar_arrive(smem_u32(&bars.o_free[x]));
    }
  }

  // ---------------------------------------------------------------- teardown
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == kWarpMma) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                 "r"(kTmemCols)
                 : "memory");
  }
}

// ------------------------------------------------------------------- host
template <bool BF16, int NQ, bool ROPE>
cudaError_t launch_t(AppendParams& prm, int ctas, cudaStream_t stream) {
  static std::atomic<uint64_t> configured{0};
  cudaError_t e =
      ensure_smem_limit(append_kernel<BF16, NQ, ROPE>, Layout<NQ>::SMEM, configured);
  if (e != cudaSuccess) return e;
  append_kernel<BF16, NQ, ROPE><<<ctas, kThreads, Layout<NQ>::SMEM, stream>>>(prm);
  return cudaGetLastError();
}

template <bool BF16, bool ROPE>
cudaError_t launch_nq(AppendParams& prm, int ctas, bool one_tile, cudaStream_t stream) {
  return one_tile ? launch_t<BF16, 1, ROPE>(prm, ctas, stream)
                  : launch_t<BF16, 2, ROPE>(prm, ctas, stream);
}

}  // namespace

int append_ctas_per_sm() { return 1; }

cudaError_t launch_append(const AppendArgs& a, cudaStream_t stream, const char** msg) {
  const bool decode_mode = a.qo_indptr == nullptr;
  if (a.group * a.tile_tokens > kTile || a.rows_per_item != a.group * a.q_tile ||
      (!decode_mode && (a.group * a.tile_tokens != kTile || a.q_tile != 2 * a.tile_tokens)) ||
      (decode_mode && (a.q_tile != 1 || a.tile_tokens != 1))) {
    *msg = "attn_append_run: num_qo_heads / num_kv_heads must divide 128";
    return cudaErrorNotSupported;
  }
  if (a.page_size <= 0) {
    *msg = "attn_append_run: page_size must be positive";
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
  prm.gather = a.page_size % kChunk != 0 ? 1 : 0;
  prm.nhd = a.layout == ATTN_LAYOUT_NHD ? 1 : 0;
  {
    const cuuint64_t dims[3] = {cuuint64_t(kHeadDim), cuuint64_t(a.num_qo_heads),
                                cuuint64_t(a.total_qo)};
    const cuuint64_t strides[2] = {cuuint64_t(kHeadDim) * 2,
                                   cuuint64_t(kHeadDim) * 2 * a.num_qo_heads};
    const cuuint32_t box[3] = {64u, cuuint32_t(a.group), cuuint32_t(a.tile_tokens)};
    const cuuint32_t es[3] = {1, 1, 1};
    if (enc(&prm.tm_q, dt, 3, const_cast<void*>(a.q), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS) {
      *msg = "attn_append_run: cannot describe q for TMA";
      return cudaErrorInvalidValue;
    }
  }
  if (!make_kv_maps(a.k_pool, a.v_pool, a.num_pages, a.num_kv_heads, a.page_size,
                    bf16 ? kKvElemBF16 : kKvElemF16, prm.gather ? 1u : uint32_t(kTcChunk),
                    prm.nhd != 0, &prm.tm_k, &prm.tm_v, msg))
    return cudaErrorNotSupported;  // *msg says why
  // at most one CTA per SM (shared memory); extra plan CTAs are run in turn
  int sms = 0;
  cudaError_t e = current_sm_count(&sms);
  if (e != cudaSuccess) return e;
  const int grid = a.num_ctas < sms ? a.num_ctas : sms;
  // one query tile per item suffices when no request has more queries than a tile
  const bool one_tile = decode_mode || a.max_qo_len <= a.tile_tokens;
  const bool rope = a.rope_cos != nullptr;
  if (rope && decode_mode) {
    *msg = "attn_append_run: fused RoPE in the append kernel needs query rows (qo_indptr)";
    return cudaErrorNotSupported;
  }
  if (bf16)
    return rope ? launch_nq<true, true>(prm, grid, one_tile, stream)
                : launch_nq<true, false>(prm, grid, one_tile, stream);
  return rope ? launch_nq<false, true>(prm, grid, one_tile, stream)
              : launch_nq<false, false>(prm, grid, one_tile, stream);
}

}  // namespace attn
