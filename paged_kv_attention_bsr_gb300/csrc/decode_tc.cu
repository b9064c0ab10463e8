// decode_tc.cu -- batch decode over a BSR paged KV cache on the tensor cores
// (tcgen05 MMA with TMEM accumulators, TMA gathers of the K/V pages).
//
// Method: one new query token per request attends to that request's paged
// KV (FlashInfer README copy on gittoolsai.com, "解码、预填充与追加"; pages
// addressed through a block-sparse row table, modb.pro digest,
// "统一的 KV 缓存存储格式"); the CPU plan of "动态负载均衡调度" cuts the
// (request, kv head) items into page ranges balanced across a persistent
// fixed grid, and split items are joined afterwards by their log-sum-exp.
//
// A unit (request r, kv head hk, pages [p0, p1)) multiplies the R packed
// query rows of its item (row rho = token i x group + head h: the GQA group's
// heads in decode, R = group; a few new tokens per request in a short
// append, R >= qo_len x group) with 128-token K/V tiles:
//   S = Q K^T     A = Q (smem, K-major), B = K (smem, K-major), D = TMEM
//   P = exp2(S c - m) over each row, written over S in TMEM (16-bit)
//   O += P V      A = P (TMEM), B = V (smem, MN-major), D = TMEM
// Only R of the 128 MMA rows would hold queries, and one thread per row
// would exponentiate all 128 scores of a tile. Instead the R rows are
// replicated C = 32 / R times in query rows 0..31 (row rho + R c is copy c of
// row rho) and copy c owns kv columns [W c, W c + W) of every tile
// (W = 128 / C = 4 R). One warp runs the softmax with one TMEM lane per
// thread, W exponentials per thread and tile; the copies of a row share the
// running max through shuffles, write P only in their own columns (zeros
// elsewhere), and their O rows -- partial sums over disjoint tokens at a
// common scale -- are added in the epilogue. Rows 32..127 carry no queries
// and are never read back. A causal short append masks each row at its own
// end-aligned limit (token i of qo_len sees kv positions <= kv_len - qo_len + i).
//
// Warps (256 threads, one CTA per SM): 0 softmax; 1 producer of the K/V
// ring (six 32 KB slots; TMA 16-row boxes by page index when the page size is
// a multiple of 16, else rows copied one by one with cp.async, down to one
// token per page, together with warps 5-7 in the kernels without RoPE);
// 2 TMEM
// allocation and the MMAs (one thread: S of tile k+1 runs under the softmax
// of tile k, S double-buffered in TMEM); 3 query loader (plain loads of the
// next unit's R query rows into registers, stored into the swizzled query
// tile as soon as the last S of the current unit is done); 4 epilogue. O is
// double-buffered in TMEM (unit u accumulates into O[u & 1]), so while the
// epilogue warp reads one unit's O, sums the copies, writes the output and
// merges split items, the softmax warp is already on the next unit's tiles;
// the softmax hands over each row's max and sum through shared memory.
// With rotary position embedding fused in (288 threads), the query loader
// turns each query row at its position, and warps 5-8 turn every K tile in
// shared memory between its TMA landing and the S MMA.
// Every wait is bounded; TMEM is freed on every path.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <cstring>

#include "internal.h"
#include "ptx.cuh"
#include "tc.cuh"

namespace attn {
namespace {

constexpr int kTile = kTcTile;
constexpr int kChunk = kTcChunk;
constexpr int kHalf = kTcHalf;
constexpr int kTileBytes = kTcTileBytes;
constexpr int kWarpSoftmax = 0;
constexpr int kWarpLoad = 1;
constexpr int kWarpMma = 2;
constexpr int kWarpQ = 3;
constexpr int kWarpEpi = 4;  // TMEM lanes 0-31, like the softmax warp
constexpr int kWarpRope0 = 5;  // warps 5-8 turn K tiles when RoPE is fused in
// warps 5-8 turn K tiles (RoPE); warps 5-7 widen FP8 tiles (eight warps in
// all, two per scheduler: the register budget stays at 255 per thread)
// warps 5-7: FP8 converters, or (page sizes that are not a multiple of 16)
// copiers of gathered rows beside warp 1; idle otherwise. Eight warps keep
// the register budget at 255 a thread.
template <bool ROPE, bool FP8 = false>
constexpr int block_threads() { return ROPE ? 288 : 256; }
constexpr int kConvThreads = 96;  // FP8 converter warps 5-7

// Two E4M3 values (the low byte first) as an f16x2 word (exact).
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t pair) {
  uint32_t d;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(d) : "h"(static_cast<unsigned short>(pair)));
  return d;
}
constexpr int kSlots = 6;
// FP8 K/V (E4M3 bytes): TMA lands a 128-row tile of 128-byte rows (128B
// swizzle, the same row pattern as one 64-dim half of a 16-bit tile) in the
// upper 64-dim half of its own 16-bit slot, and warps 5-7 widen it there in
// place: row r's E4M3 bytes occupy exactly the bytes of row r's upper f16
// half, and a warp reads whole rows before it writes them. So FP8 keeps
// the six-slot ring of 16-bit pools, with up to six tiles of E4M3 bytes in
// flight (a separate four-slot staging ring beside four 16-bit slots held
// it to about 0.48 of the HBM peak).
constexpr int kF8TileBytes = kTcTile * 128;
template <bool FP8>
constexpr int ring_slots() { return kSlots; }
constexpr int kOffQ = 0;
// RoPE key angles: cos / sin of the offset rows o = 0, 2, .., 14 (8 x 64
// floats each) in query-tile rows 32-63 of the lower half, which hold no
// query (the few-row kernel's queries sit in rows 0-31; the MMA's output
// lanes of rows 32-127 are never read)
constexpr int kOffRopeCos = kOffQ + 32 * 128;
constexpr int kOffRopeSin = kOffRopeCos + 8 * 64 * 4;
static_assert(kOffRopeSin + 8 * 64 * 4 <= kOffQ + 64 * 128, "RoPE offset rows fit query rows 32-63");
// Gathered rows: the pool row of each token of a tile (128 int32), stored
// kRowLead - 1 tiles ahead into a ring of kRowSlots tiles (the slot being
// read is never the one being written) in query-tile rows 64-127 of the
// lower half.
constexpr int kRowLead = 4;
constexpr int kRowSlots = kRowLead + 1;
constexpr int kOffRowRing = kOffQ + 64 * 128;
static_assert(kOffRowRing + kRowSlots * kTcTile * 4 <= kOffQ + kTcHalf, "row ring fits the spare query rows");
constexpr int kOffRing = kTileBytes;
constexpr int kOffBar = kOffRing + kSlots * kTileBytes;
static_assert(kF8TileBytes == kHalf, "an E4M3 tile fills the upper half of a 16-bit slot");
constexpr int kOffHand = kOffBar + 512;         // softmax -> epilogue row state
constexpr int kSmem = kOffHand + 512 + 1024;    // + alignment slack
constexpr uint32_t kTmemCols = 512;  // S buffers at 0 and 128, O buffers at 256 and 384
constexpr uint32_t kColO = 256;

struct Bars {
  uint64_t q_full, q_empty;
  uint64_t slot_full[kSlots], slot_empty[kSlots];
  uint64_t s_full[2], p_full[2], o_done[2];
  uint64_t o_free[2];   // epilogue read O[b] (count 32)
  uint64_t ounit[2];    // a unit's last P.V into O[b] is done (commit)
  uint64_t ep_full[2];  // softmax wrote the row state of a unit with O[b] (count 32)
  uint64_t k_rot[kSlots / 2];  // RoPE: K tile k is turned in its slot (count 128)
  uint64_t f8_full[kSlots];    // FP8: a tile's E4M3 bytes have landed (TMA bytes)
  uint64_t drain;
  uint32_t tmem_base;
};
static_assert(sizeof(Bars) <= 512, "barrier block");
struct Hand {
  float m[2][32];  // per O buffer and TMEM lane: running max (log2 units)
  float l[2][32];  // and the copy's partial sum
};

struct DecodeTcParams {
  CUtensorMap tm_k;
  CUtensorMap tm_v;
  CUtensorMap tm_k2;  // composable formats: the suffix pool
  CUtensorMap tm_v2;
  AppendArgs a;
  float scale_log2;
  uint32_t idesc_s;
  uint32_t idesc_pv;
  int32_t gather;  // K / V rows gathered 4 at a time (page_size % 16 != 0)
  int32_t nhd;     // pools are NHD [pages, P, Hk, 128] (else HND [pages, Hk, P, 128])
};

// f16 bits of two bf16 values (FP8 kernels multiply in f16: the MMA's two
// operands share one type, and every E4M3 value is an f16 value)
__device__ __forceinline__ uint32_t bf16x2_to_f16x2(uint32_t w) {
  const float lo = __uint_as_float(w << 16), hi = __uint_as_float(w & 0xffff0000u);
  const __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&h);
}

struct DGeo {
  int32_t r, hk, t, slot, split, page_base, ntiles;
  int32_t pad;           // composable formats: 1 = the unit reads the suffix table
  bool cprev, cnext;     // chain: continues the previous unit / continued by the next
  int64_t qo_start, qo_len, kv_len;
  int64_t tok_begin, tok_end;
};

// DEC: decode (one query row per request, the whole kv visible).
template <bool DEC>
__device__ __forceinline__ DGeo decode_geo(const AppendArgs& a, int ui) {
  const int4* rec = reinterpret_cast<const int4*>(a.ws.units + ui);
  const int4 x = __ldg(rec);
  const int4 y = __ldg(rec + 1);
  const int4 z = __ldg(rec + 2);
  DGeo g;
  g.r = x.x;
  g.hk = x.y;
  g.t = x.z;
  g.slot = y.y;
  g.split = y.z;
  g.page_base = y.w;  // the request's geometry, copied in by the planner
  g.kv_len = z.x;
  g.qo_start = z.y;
  g.qo_len = DEC ? 1 : z.z;
  // composable formats: table bit and chain flags (0 in other plans)
  const int32_t flags = (!DEC && a.cascade) ? z.w : 0;
  g.pad = flags & 1;
  g.cprev = (flags & 2) != 0;
  g.cnext = (flags & 4) != 0;
  int64_t vis = g.kv_len;
  if (!DEC && a.causal) {  // the item's last query row sees the most
    const int64_t last_row = min(int64_t(g.t + 1) * a.q_tile, g.qo_len) - 1;
    vis = min(g.kv_len, max(int64_t(0), g.kv_len - g.qo_len + last_row + 1));
  }
  const int64_t P = g.pad ? a.page_size2 : a.page_size;
  g.tok_begin = int64_t(x.w) * P;
  g.tok_end = min(int64_t(y.x) * P, vis);
  const int64_t nt = g.tok_end - g.tok_begin;
  g.ntiles = nt > 0 ? int32_t((nt + kTile - 1) / kTile) : 0;
  return g;
}

// Packed query row rho of a unit: its token and head, output row and the
// last kv position it may see (ok = false for rows past the request's queries).
struct QRow {
  bool ok;
  int64_t orow;   // row of q / o / lse ([tokens, Hq] flattened)
  int64_t limit;  // last visible kv position
  int64_t pos;    // the query's own position (RoPE): kv_len - qo_len + i
};
template <bool DEC, int R>
__device__ __forceinline__ QRow qrow(const AppendArgs& a, const DGeo& g, int rho) {
  QRow q;
  if constexpr (DEC) {  // rows are the group's heads (group = R)
    q.ok = true;
    q.orow = int64_t(g.r) * a.num_qo_heads + int64_t(g.hk) * R + rho;
    q.limit = g.kv_len - 1;
    q.pos = g.kv_len - 1;
  } else if (a.cascade) {
    // composable formats: rows are the generations of prompt r (token tok =
    // generation tok); a prefix unit (t < 0) serves every generation, a
    // suffix unit only its own (t): the other rows see nothing
    const int tok = rho / a.group, hh = rho - tok * a.group;
    q.ok = tok < g.qo_len;
    q.orow = (g.qo_start + tok) * a.num_qo_heads + int64_t(g.hk) * a.group + hh;
    q.limit = (g.t < 0 || g.t == tok) ? g.kv_len - 1 : -1;
    q.pos = 0;
  } else {
    const int tok = rho / a.group, hh = rho - tok * a.group;
    const int64_t qi = int64_t(g.t) * a.q_tile + tok;
    q.ok = qi < g.qo_len;
    q.orow = (g.qo_start + qi) * a.num_qo_heads + int64_t(g.hk) * a.group + hh;
    q.limit = a.causal ? g.kv_len - g.qo_len + qi : g.kv_len - 1;
    q.pos = g.kv_len - g.qo_len + qi;
  }
  return q;
}

template <int N>
struct ILog2 {
  static constexpr int value = 1 + ILog2<N / 2>::value;
};
template <>
struct ILog2<1> {
  static constexpr int value = 0;
};

// N consecutive outputs (N = 1, 2, 4 or a multiple of 8) of one row,
// scaled: 16-bit or fp32.
template <bool BF16, int N>
__device__ __forceinline__ void store_out16(void* o, int64_t idx, const float* v, float scale) {
  static_assert(N == 1 || N == 2 || N == 4 || N % 8 == 0, "output run length");
  uint16_t* dst = static_cast<uint16_t*>(o) + idx;
  if constexpr (N == 1) {
    if constexpr (BF16)
      *reinterpret_cast<__nv_bfloat16*>(dst) = __float2bfloat16_rn(v[0] * scale);
    else
      *reinterpret_cast<__half*>(dst) = __float2half_rn(v[0] * scale);
  } else {
    uint32_t w[N / 2];
#pragma unroll
    for (int i = 0; i < N / 2; ++i) w[i] = pack2<BF16>(v[2 * i] * scale, v[2 * i + 1] * scale);
    if constexpr (N == 2) *reinterpret_cast<uint32_t*>(dst) = w[0];
    if constexpr (N == 4) *reinterpret_cast<uint2*>(dst) = make_uint2(w[0], w[1]);
    if constexpr (N % 8 == 0) {
#pragma unroll
      for (int i = 0; i < N / 8; ++i)
        reinterpret_cast<uint4*>(dst)[i] =
            make_uint4(w[4 * i], w[4 * i + 1], w[4 * i + 2], w[4 * i + 3]);
    }
  }
}
template <int N>
__device__ __forceinline__ void store_out32(float* dst, const float* v, float scale) {
  static_assert(N == 1 || N == 2 || N % 4 == 0, "output run length");
  if constexpr (N == 1) dst[0] = v[0] * scale;
  if constexpr (N == 2) *reinterpret_cast<float2*>(dst) = make_float2(v[0] * scale, v[1] * scale);
  if constexpr (N >= 4) {
#pragma unroll
    for (int i = 0; i < N; i += 4)
      *reinterpret_cast<float4*>(dst + i) =
          make_float4(v[i] * scale, v[i + 1] * scale, v[i + 2] * scale, v[i + 3] * scale);
  }
}

// Split item: after this unit's partial state is written, the last of the
// item's units to arrive (atomic count in the workspace) merges every
// partial state of the item by log-sum-exp and resets the count to 0.
// One warp: lane = row rho * (32 / R) + dl, dims [4 R dl, 4 R dl + 4 R).
// The merge is a chain of L2 round trips (about 1.7 us each while the other
// SMs stream K / V), so the loads are issued in batches. With `land` (shared
// memory nothing else uses any more, land_cap bytes) every slot's O rows
// are copied there by cp.async in one round trip, the LSEs loaded
// meanwhile; rows are stored with their 16-byte pieces XOR-swizzled by the
// reading lane (R >= 4) so the reads are free of bank conflicts.
template <bool BF16, int R, bool DEC>
__device__ __forceinline__ bool merge_split_impl(const AppendArgs& a, const DGeo& g,
                                                 uint8_t* land = nullptr,
                                                 uint32_t land_cap = 0) {
  constexpr int LP = 32 / R, DL = 4 * R, kS = DL < 8 ? DL : 8;
  constexpr bool kSw = R >= 4;
  const int lane = threadIdx.x & 31;
  __threadfence();  // every lane's partial stores before the arrival
  __syncwarp();
  int last = 0;
  if (lane == 0) {
    const int4 mi = __ldg(a.ws.merge_items + g.split);
    last = atomicAdd(a.ws.counters + g.split, 1) == mi.w - 1;
  }
  if (!__shfl_sync(0xffffffffu, last, 0)) return true;
  __threadfence();  // the other units' partial states
  const int rho = lane / LP, dl = lane % LP;
  const QRow qr = qrow<DEC, R>(a, g, rho);
  const int s0 = __ldg(a.ws.merge_indptr + g.split), s1 = __ldg(a.ws.merge_indptr + g.split + 1);
  const uint32_t obytes = uint32_t(s1 - s0) * R * kHeadDim * 4;
  const bool staged = land != nullptr && obytes <= land_cap;
  if (staged) {
    // row k of the landing area = (slot s0 + k / R, row k % R) (a slot's
    // rows start every rows_per_item rows); this lane copies piece `lane`
    // (bytes 16 lane ..) of every row
    const char* src = reinterpret_cast<const char*>(a.ws.partial_o) + lane * 16;
    const uint32_t dst = smem_u32(land);
    const int nrows = (s1 - s0) * R;
    for (int k = 0; k < nrows; ++k) {
      const int sl = s0 + k / R, rr = k % R;
      const uint32_t key = kSw ? uint32_t((rr * LP + (lane * 4) / DL) & 7) : 0u;
      cp_async16_cg(dst + uint32_t(k) * 512u + ((uint32_t(lane) * 16u) ^ (key << 4)),
                    src + (int64_t(sl) * a.rows_per_item + rr) * (kHeadDim * 4));
    }
    cp_async_commit();
  }
  // The first kKeep slots' LSEs at once (kept in registers); without the
  // landing area, the O rows kBo slots at a time (8 float4 loads in flight
  // per lane).
  constexpr int kKeep = 16;
  constexpr int kBo = DL >= 32 ? 1 : 32 / DL;
  auto lse_at = [&](int sl) {
    return __ldcg(a.ws.partial_lse + int64_t(sl) * a.rows_per_item + rho);
  };
  float keep[kKeep];
#pragma unroll
  for (int k = 0; k < kKeep; ++k) keep[k] = s0 + k < s1 ? lse_at(s0 + k) : -INFINITY;
  float M = -INFINITY;
#pragma unroll
  for (int k = 0; k < kKeep; ++k) M = fmaxf(M, keep[k]);
  for (int sl = s0 + kKeep; sl < s1; ++sl) M = fmaxf(M, lse_at(sl));
  auto lse_of = [&](int sl) {
    float ls = -INFINITY;
#pragma unroll
    for (int k = 0; k < kKeep; ++k) ls = (sl - s0 == k) ? keep[k] : ls;
    if (sl - s0 >= kKeep) ls = lse_at(sl);
    return ls;
  };
  float acc[DL];
#pragma unroll
  for (int j = 0; j < DL; ++j) acc[j] = 0.f;
  float L = 0.f;
  if (staged) {
    cp_async_wait<0>();
    __syncwarp();  // every lane's pieces have landed
    if (M != -INFINITY) {
      const uint32_t key = kSw ? uint32_t(lane & 7) : 0u;
      for (int sl = s0; sl < s1; ++sl) {
        const float f = ex2(lse_of(sl) - M);
        L += f;
        const uint8_t* row = land + (uint32_t(sl - s0) * R + rho) * 512u;
#pragma unroll
        for (int j = 0; j < DL / 4; ++j) {
          const float4 x = *reinterpret_cast<const float4*>(
              row + ((uint32_t(DL * dl + 4 * j) * 4u) ^ (key << 4)));
          acc[4 * j] += f * x.x;
          acc[4 * j + 1] += f * x.y;
          acc[4 * j + 2] += f * x.z;
          acc[4 * j + 3] += f * x.w;
        }
      }
    }
  } else if (M != -INFINITY) {
    for (int b0 = s0; b0 < s1; b0 += kBo) {
      float4 x[kBo][DL / 4];
      float f[kBo];
#pragma unroll
      for (int u = 0; u < kBo; ++u) {
        const int sl = b0 + u;
        f[u] = 0.f;
        if (sl < s1) {
          const int64_t prow = int64_t(sl) * a.rows_per_item + rho;
          const float4* src =
              reinterpret_cast<const float4*>(a.ws.partial_o + prow * kHeadDim + DL * dl);
#pragma unroll
          for (int j = 0; j < DL / 4; ++j) x[u][j] = __ldcg(src + j);
          f[u] = ex2(lse_of(sl) - M);
        }
      }
#pragma unroll
      for (int u = 0; u < kBo; ++u) {
        if (b0 + u < s1) {
          L += f[u];
#pragma unroll
          for (int j = 0; j < DL / 4; ++j) {
            acc[4 * j] += f[u] * x[u][j].x;
            acc[4 * j + 1] += f[u] * x[u][j].y;
            acc[4 * j + 2] += f[u] * x[u][j].z;
            acc[4 * j + 3] += f[u] * x[u][j].w;
          }
        }
      }
    }
  }
  if (qr.ok) {
    const float inv = L > 0.f ? 1.f / L : 0.f;
#pragma unroll
    for (int j = 0; j < DL; j += kS)
      store_out16<BF16, kS>(a.o, qr.orow * kHeadDim + DL * dl + j, acc + j, inv);
    if (dl == 0 && a.lse) a.lse[qr.orow] = L > 0.f ? (M + lg2(L)) * kLn2 : -INFINITY;
  }
  if (lane == 0) a.ws.counters[g.split] = 0;
  return true;
}

// Rotary embedding of one 32-bit word (two consecutive dims) of a row:
// `mine` holds dims (d, d + 1) of one half of the row, `other` the same dims
// of the other half; first: mine is the lower half (x' = x cos - y sin), else
// the upper (y' = y cos + x sin). Products and sums in fp32, then rounded to
// the storage type.
template <bool BF16>
__device__ __forceinline__ uint32_t rope_word(uint32_t mine, uint32_t other, bool first, float c0,
                                              float c1, float s0, float s1) {
  float m0, m1, o0, o1;
  if constexpr (BF16) {
    m0 = __uint_as_float(mine << 16);
    m1 = __uint_as_float(mine & 0xffff0000u);
    o0 = __uint_as_float(other << 16);
    o1 = __uint_as_float(other & 0xffff0000u);
  } else {
    const float2 mf = __half22float2(*reinterpret_cast<const __half2*>(&mine));
    const float2 of = __half22float2(*reinterpret_cast<const __half2*>(&other));
    m0 = mf.x, m1 = mf.y, o0 = of.x, o1 = of.y;
  }
  const float sg = first ? -1.f : 1.f;
  return pack2<BF16>(fmaf(sg * o0, s0, m0 * c0), fmaf(sg * o1, s1, m1 * c1));
}

// 8 consecutive dims (one 16-byte piece); c0 / c1, s0 / s1: their cos / sin
template <bool BF16>
__device__ __forceinline__ uint4 rope8(uint4 mine, uint4 other, bool first, const float4 c0,
                                       const float4 c1, const float4 s0, const float4 s1) {
  return make_uint4(rope_word<BF16>(mine.x, other.x, first, c0.x, c0.y, s0.x, s0.y),
                    rope_word<BF16>(mine.y, other.y, first, c0.z, c0.w, s0.z, s0.w),
                    rope_word<BF16>(mine.z, other.z, first, c1.x, c1.y, s1.x, s1.y),
                    rope_word<BF16>(mine.w, other.w, first, c1.z, c1.w, s1.z, s1.w));
}

// 4 consecutive dims (8 bytes); c / s: their cos / sin
template <bool BF16>
__device__ __forceinline__ uint2 rope4(uint2 mine, uint2 other, bool first, const float4 c,
                                       const float4 s) {
  return make_uint2(rope_word<BF16>(mine.x, other.x, first, c.x, c.y, s.x, s.y),
                    rope_word<BF16>(mine.y, other.y, first, c.z, c.w, s.z, s.w));
}

// The two 16-bit values of a word as floats.
template <bool BF16>
__device__ __forceinline__ float2 unpack2(uint32_t w) {
  if constexpr (BF16) {
    return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
  } else {
    return __half22float2(*reinterpret_cast<const __half2*>(&w));
  }
}

// Key rotation of 4 pairs (dims d..d+3 with d+64..d+67) at an angle B + o:
// x / y hold the lower / upper dims, (cb, sb, nsb) = (cos, sin, -sin) of
// B theta and (oc, os) = (cos, sin) of o theta for the 4 pairs. The angle
// sums and the turn run on packed fp32x2 arithmetic.
template <bool BF16>
__device__ __forceinline__ void rope_key4(uint2& x, uint2& y, float4 cb, float4 sb, float4 nsb,
                                          float4 oc, float4 os) {
  const float2 oc0 = make_float2(oc.x, oc.y), oc1 = make_float2(oc.z, oc.w);
  const float2 os0 = make_float2(os.x, os.y), os1 = make_float2(os.z, os.w);
  // cos((B + o) t) = cos B cos o - sin B sin o;  sin((B + o) t) = sin B cos o + cos B sin o
  const float2 c0 = ffma2(make_float2(cb.x, cb.y), oc0, fmul2(make_float2(nsb.x, nsb.y), os0));
  const float2 c1 = ffma2(make_float2(cb.z, cb.w), oc1, fmul2(make_float2(nsb.z, nsb.w), os1));
  const float2 s0 = ffma2(make_float2(sb.x, sb.y), oc0, fmul2(make_float2(cb.x, cb.y), os0));
  const float2 s1 = ffma2(make_float2(sb.z, sb.w), oc1, fmul2(make_float2(cb.z, cb.w), os1));
  const float2 x0 = unpack2<BF16>(x.x), x1 = unpack2<BF16>(x.y);
  const float2 y0 = unpack2<BF16>(y.x), y1 = unpack2<BF16>(y.y);
  const float2 ns0 = make_float2(-s0.x, -s0.y), ns1 = make_float2(-s1.x, -s1.y);
  // x' = x cos - y sin;  y' = y cos + x sin
  const float2 xr0 = ffma2(x0, c0, fmul2(y0, ns0)), xr1 = ffma2(x1, c1, fmul2(y1, ns1));
  const float2 yr0 = ffma2(y0, c0, fmul2(x0, s0)), yr1 = ffma2(y1, c1, fmul2(x1, s1));
  x = make_uint2(pack2<BF16>(xr0.x, xr0.y), pack2<BF16>(xr1.x, xr1.y));
  y = make_uint2(pack2<BF16>(yr0.x, yr0.y), pack2<BF16>(yr1.x, yr1.y));
}

// Producer of gathered rows (page sizes that are not a multiple of 16, down
// to one token per page): the rows are copied with 16-byte cp.async (the
// load-store unit, not the TMA engine: a TMA gather moves four 128-byte rows
// per instruction, and at one token per page its per-instruction cost, not
// DRAM, set the pace) straight into the slot's 128B-swizzled layout. NW
// warps share the work, warp cw taking rows [cw RW, cw RW + RW) of every
// tile (RW = 128 / NW): the copies of random rows are issue-bound in one
// warp (address translation per row), so the plain decode kernel spreads
// them over four warps, one per scheduler.
//  - Pool rows: lane c loads the page indices of the warp's tokens
//    c TPL .. c TPL + TPL - 1 (TPL = RW / 32) of tile i + kRowLead at tile
//    i and, one tile later (the load has landed meanwhile), stores their
//    pool rows (-1 past the unit's end) into the warp's shared ring of
//    kRowSlots tiles x RW rows.
//  - Copies: per 16-byte piece of a row, lanes 0-15 take one row and 16-31
//    the next; a lane reads 8 rows' pool indices from the ring, then issues
//    their 8 copies.
//  - Every lane arrives on the slot's full barrier (count 32 NW) through
//    cp.async.mbarrier.arrive, i.e. once its copies have landed; the MMA
//    thread fences into the async proxy after its wait. Nothing here waits
//    for its own copies, so the whole ring stays in flight.
//  - Rows past a unit's end are not copied: the softmax masks those keys
//    and zeroes those V rows.
// Kept out of line: the kernel body stays as compact as without this mode.
template <bool DEC, int NW>
__device__ __noinline__ void produce_gather(const DecodeTcParams& prm, Bars& bars, uint32_t base,
                                            uint8_t* gbase, int lane, int cw,
                                            volatile int32_t* err, uint32_t& uses, bool& ok) {
  constexpr int RW = kTile / NW;  // rows of a tile this warp copies
  constexpr int TPL = RW / 32;    // tokens whose pool rows a lane looks up
  static_assert(RW % 32 == 0 && RW % 16 == 0, "rows per warp");
  const AppendArgs& a = prm.a;
  int32_t* ring = reinterpret_cast<int32_t*>(gbase + kOffRowRing) + cw * (kRowSlots * RW);
  // a unit's table (composable formats: pad = 1 reads the suffix table)
  uint32_t P = 1;
  const char* pools[2] = {nullptr, nullptr};
  const int32_t* indices = nullptr;
  auto table_of = [&](const DGeo& g) {
    const bool second = g.pad != 0;
    P = uint32_t(second ? a.page_size2 : a.page_size);
    pools[0] = static_cast<const char*>(second ? a.k_pool2 : a.k_pool);
    pools[1] = static_cast<const char*>(second ? a.v_pool2 : a.v_pool);
    indices = second ? a.kv_indices2 : a.kv_indices;
  };
  // page indices of lane's tokens of tile i (positions < 2^31: 32-bit
  // division); tokens past the unit's end load nothing
  auto load_pages = [&](const DGeo& g, int i, int32_t (&ph)[TPL]) {
    const int64_t kv0 = g.tok_begin + int64_t(i) * kTile + cw * RW + lane * TPL;
#pragma unroll
    for (int u = 0; u < TPL; ++u) {
      ph[u] = 0;
      if (i < g.ntiles && kv0 + u < g.tok_end)
        ph[u] = __ldg(indices + g.page_base + uint32_t(kv0 + u) / P);
    }
  };
  // their pool rows into ring slot i % kRowSlots
  auto store_rows = [&](const DGeo& g, int i, const int32_t (&ph)[TPL]) {
    const int64_t kv0 = g.tok_begin + int64_t(i) * kTile + cw * RW + lane * TPL;
#pragma unroll
    for (int u = 0; u < TPL; ++u) {
      int32_t rw = -1;
      if (i < g.ntiles && kv0 + u < g.tok_end) {
        const uint32_t sl = uint32_t(kv0 + u) % P;
        const int64_t phys = ph[u];
        rw = prm.nhd ? int32_t((phys * P + sl) * a.num_kv_heads + g.hk)
                     : int32_t((phys * a.num_kv_heads + g.hk) * P + sl);
      }
      ring[(i % kRowSlots) * RW + lane * TPL + u] = rw;
    }
  };
  const int hb = lane >> 4, pc = lane & 15;  // row of the pair, 16-byte piece
  const uint32_t piece_off = uint32_t(pc >> 3) * kHalf;
  for (int vc = blockIdx.x; vc < a.num_ctas && ok; vc += gridDim.x)
    for (int ui = __ldg(a.ws.work_indptr + vc); ui < __ldg(a.ws.work_indptr + vc + 1) && ok;
         ++ui) {
      const DGeo g = decode_geo<DEC>(a, ui);
      if (g.ntiles == 0) continue;
      table_of(g);
      int32_t ph[TPL];
      for (int j = 0; j + 1 < kRowLead; ++j) {  // the first tiles' rows, directly
        load_pages(g, j, ph);
        store_rows(g, j, ph);
      }
      load_pages(g, kRowLead - 1, ph);
      for (int i = 0; i < g.ntiles && ok; ++i) {
        store_rows(g, i + kRowLead - 1, ph);  // loaded a tile ago
        load_pages(g, i + kRowLead, ph);
        __syncwarp();  // the ring rows of tile i (stored kRowLead - 1 tiles ago)
        const int64_t kv0 = g.tok_begin + int64_t(i) * kTile;
        // rows of this warp's share that hold tokens
        const int nr = int(max(int64_t(0), min(int64_t(RW), g.tok_end - kv0 - cw * RW)));
        const int32_t* rows = ring + (i % kRowSlots) * RW;
        for (int kv = 0; kv < 2; ++kv, ++uses) {  // K then V
          const int slot = int(uses % kSlots);
          bool r = true;
          if (lane == 0)
            r = mbar_wait(smem_u32(&bars.slot_empty[slot]), ((uses / kSlots) & 1u) ^ 1u, err,
                          ERR_WAIT_EMPTY);
          if (__shfl_sync(0xffffffffu, r ? 1 : 0, 0) == 0) {
            ok = false;
            break;
          }
          const char* pool = pools[kv] + pc * 16;
          const uint32_t dst0 = base + kOffRing + slot * kTileBytes + piece_off;
          for (int r0 = 0; r0 < nr; r0 += 16) {  // rows r0 .. r0 + 15, two per step
            int32_t gr[8];
#pragma unroll
            for (int k = 0; k < 8; ++k) gr[k] = rows[r0 + 2 * k + hb];
#pragma unroll
            for (int k = 0; k < 8; ++k) {
              const int rl = r0 + 2 * k + hb;  // row within the share
              const int row = cw * RW + rl;    // row within the tile
              if (rl < nr && gr[k] >= 0)
                cp_async16_cg(dst0 + uint32_t(row) * 128u + (uint32_t((pc & 7) ^ (row & 7)) << 4),
                              pool + int64_t(gr[k]) * (kHeadDim * 2));
            }
          }
          cp_async_mbar_arrive_noinc(smem_u32(&bars.slot_full[slot]));
        }
      }
    }
  cp_async_wait<0>();  // every copy has landed before the CTA can exit
}

// Producer of 16-row boxes from NHD pools (page sizes that are a multiple of
// 16): as the HND box producer, with a 3-D map [tokens, Hk, 128] whose box is
// 16 tokens x 1 head x 64 dims, so the tile rows land as in HND. Kept out of
// line like produce_gather.
template <bool DEC>
__device__ __noinline__ void produce_nhd_box(const DecodeTcParams& prm, Bars& bars, uint32_t base,
                                             int lane, volatile int32_t* err, uint32_t& uses,
                                             bool& ok) {
  const AppendArgs& a = prm.a;
  const int P = a.page_size;
  // token row (phys * P + slot) of the tile's 16-row chunk c = lane
  auto chunk_tok = [&](const DGeo& g, int i) -> int32_t {
    const int64_t kvt = g.tok_begin + int64_t(i) * kTile + int64_t(lane) * kChunk;
    if (kvt >= g.tok_end) return 0;
    const int64_t pg = kvt / P;
    const int64_t phys = __ldg(a.kv_indices + g.page_base + pg);
    return int32_t(phys * P + (kvt - pg * P));
  };
  for (int vc = blockIdx.x; vc < a.num_ctas && ok; vc += gridDim.x)
    for (int ui = __ldg(a.ws.work_indptr + vc); ui < __ldg(a.ws.work_indptr + vc + 1) && ok;
         ++ui) {
      const DGeo g = decode_geo<DEC>(a, ui);
      if (g.ntiles == 0) continue;
      int32_t tok = chunk_tok(g, 0);
      for (int i = 0; i < g.ntiles && ok; ++i) {
        const int64_t kv0 = g.tok_begin + int64_t(i) * kTile;
        const int ntt = int(min(int64_t(kTile), g.tok_end - kv0));
        const int nch = (ntt + kChunk - 1) / kChunk;
        const int32_t tok_next = i + 1 < g.ntiles ? chunk_tok(g, i + 1) : 0;
        for (int kv = 0; kv < 2; ++kv, ++uses) {  // K then V
          const int slot = int(uses % kSlots);
          bool r = true;
          if (lane == 0)
            r = mbar_wait(smem_u32(&bars.slot_empty[slot]), ((uses / kSlots) & 1u) ^ 1u, err,
                          ERR_WAIT_EMPTY);
          if (__shfl_sync(0xffffffffu, r ? 1 : 0, 0) == 0) {
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
            tma_load_3d(dst, tm, 0, g.hk, tok, full);
            tma_load_3d(dst + kHalf, tm, 64, g.hk, tok, full);
          }
        }
        tok = tok_next;
      }
    }
}

template <bool BF16, int R, bool DEC, bool ROPE, bool FP8 = false>
__global__ void __launch_bounds__(block_threads<ROPE, FP8>(), 1)
    decode_tc_kernel(const __grid_constant__ DecodeTcParams prm) {
  constexpr int C = 32 / R;     // copies of each query row
  constexpr int W = kTile / C;  // kv columns per copy and tile
  constexpr int LC = ILog2<C>::value;
  constexpr int kRing = ring_slots<FP8>();  // 16-bit K/V slots
  constexpr bool kMmaBF16 = FP8 ? false : BF16;  // operand type of the MMAs (and of P)
  static_assert(!(FP8 && ROPE), "FP8 K/V and fused RoPE are separate kernels");
  extern __shared__ uint8_t smem_raw[];
  const AppendArgs& a = prm.a;
  const uint32_t raw_base = smem_u32(smem_raw);
  const uint32_t base = (raw_base + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (base - raw_base);
  Bars& bars = *reinterpret_cast<Bars*>(gbase + kOffBar);
  Hand& hand = *reinterpret_cast<Hand*>(gbase + kOffHand);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  volatile int32_t* err = a.ws.error;

  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bars.q_full), 32);
    mbar_init(smem_u32(&bars.q_empty), 1);
    for (int i = 0; i < kRing; ++i) {
      // FP8: the converters fill it; gathered rows: each producer lane's
      // copies arrive on it; else one TMA arrival with its byte count
      mbar_init(smem_u32(&bars.slot_full[i]),
                FP8 ? kConvThreads : prm.gather ? (ROPE ? 32 : 4 * 32) : 1);
      mbar_init(smem_u32(&bars.slot_empty[i]), 1);
    }
    if (FP8)
      for (int i = 0; i < kSlots; ++i) mbar_init(smem_u32(&bars.f8_full[i]), 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(smem_u32(&bars.s_full[i]), 1);
      mbar_init(smem_u32(&bars.p_full[i]), 32);
      mbar_init(smem_u32(&bars.o_done[i]), 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(smem_u32(&bars.o_free[i]), 32);
      mbar_init(smem_u32(&bars.ounit[i]), 1);
      mbar_init(smem_u32(&bars.ep_full[i]), 32);
    }
    for (int i = 0; i < kSlots / 2; ++i) mbar_init(smem_u32(&bars.k_rot[i]), 128);
    mbar_init(smem_u32(&bars.drain), 1);
    fence_mbar_init();
  }
  if (warp == kWarpLoad && lane == 0 && !prm.gather) {
    prefetch_tmap(&prm.tm_k);
    prefetch_tmap(&prm.tm_v);
    if (!DEC && a.cascade) {
      prefetch_tmap(&prm.tm_k2);
      prefetch_tmap(&prm.tm_v2);
    }
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

  // A CTA runs the unit lists of plan CTAs blockIdx.x, blockIdx.x + gridDim.x,
  // ... (the grid is at most one CTA per SM; a plan may have more CTAs).
  if (warp == kWarpLoad) {
    // ------------------------------------------------------------ TMA producer
    // Page sizes that are a multiple of 16: lane c fetches the page index of
    // the tile's 16-row chunk c and issues that chunk's boxes; the next
    // tile's indices are loaded before this tile's slots are awaited, so
    // their latency hides behind the wait. Other page sizes: produce_gather.
    uint32_t uses = 0;
    bool ok = true;
    if (!FP8 && prm.gather) {
      if constexpr (ROPE)  // (warps 5-8 turn K tiles)
        produce_gather<DEC, 1>(prm, bars, base, gbase, lane, 0, err, uses, ok);
      else  // with warps 5-7: a quarter of every tile's rows each
        produce_gather<DEC, 4>(prm, bars, base, gbase, lane, 0, err, uses, ok);
    } else if (!FP8 && prm.nhd) {
      produce_nhd_box<DEC>(prm, bars, base, lane, err, uses, ok);
    } else {
      // composable formats: a unit with pad = 1 reads the suffix table / pool
      auto chunk_row = [&](const DGeo& g, int i) -> int32_t {
        const int64_t kvt = g.tok_begin + int64_t(i) * kTile + int64_t(lane) * kChunk;
        if (kvt >= g.tok_end) return 0;
        const bool second = g.pad != 0;
        const int P = second ? a.page_size2 : a.page_size;
        const int64_t pg = kvt / P;
        const int64_t phys = __ldg((second ? a.kv_indices2 : a.kv_indices) + g.page_base + pg);
        return int32_t((phys * a.num_kv_heads + g.hk) * P + (kvt - pg * P));
      };
      for (int vc = blockIdx.x; vc < a.num_ctas && ok; vc += gridDim.x)
        for (int ui = __ldg(a.ws.work_indptr + vc); ui < __ldg(a.ws.work_indptr + vc + 1) && ok;
             ++ui) {
          const DGeo g = decode_geo<DEC>(a, ui);
          if (g.ntiles == 0) continue;
          int32_t row = chunk_row(g, 0);
          for (int i = 0; i < g.ntiles && ok; ++i) {
            const int64_t kv0 = g.tok_begin + int64_t(i) * kTile;
            const int ntt = int(min(int64_t(kTile), g.tok_end - kv0));
            const int nch = (ntt + kChunk - 1) / kChunk;
            const int32_t row_next = i + 1 < g.ntiles ? chunk_row(g, i + 1) : 0;
            for (int kv = 0; kv < 2; ++kv, ++uses) {  // K then V
              // a ring slot (FP8: its upper half receives the 128-byte rows)
              const int nslot = kRing;
              const int slot = int(uses % nslot);
              bool r = true;
              if (lane == 0)
                r = mbar_wait(smem_u32(&bars.slot_empty[slot]),
                              ((uses / nslot) & 1u) ^ 1u, err, ERR_WAIT_EMPTY);
              if (__shfl_sync(0xffffffffu, r ? 1 : 0, 0) == 0) {
                ok = false;
                break;
              }
              const uint32_t full = smem_u32(FP8 ? &bars.f8_full[slot] : &bars.slot_full[slot]);
              if (lane == 0)
                mbar_arrive_expect_tx(full, uint32_t(nch) * kChunk * (FP8 ? 128u : 256u));
              __syncwarp();
              if (lane < nch) {
                const bool second = g.pad != 0;
                const void* tm = kv == 0 ? (second ? static_cast<const void*>(&prm.tm_k2)
                                                   : static_cast<const void*>(&prm.tm_k))
                                         : (second ? static_cast<const void*>(&prm.tm_v2)
                                                   : static_cast<const void*>(&prm.tm_v));
                if constexpr (FP8) {
                  tma_load_2d(base + kOffRing + slot * kTileBytes + kHalf +
                                  uint32_t(lane) * kChunk * 128u,
                              tm, 0, row, full);
                } else {
                  const uint32_t dst =
                      base + kOffRing + slot * kTileBytes + uint32_t(lane) * kChunk * 128u;
                  tma_load_2d(dst, tm, 0, row, full);
                  tma_load_2d(dst + kHalf, tm, 64, row, full);
                }
              }
            }
            row = row_next;
          }
        }
    }
    // drain: every issued copy has landed before the CTA can exit
    cp_async_wait<0>();  // this lane's index copies (they always complete)
    if (lane == 0) {
      const uint32_t nslot = kRing;
      for (uint32_t sl = 0; sl < nslot && sl < uses; ++sl) {
        const uint32_t last = uses - 1 - ((uses - 1 - sl) % nslot);
        mbar_wait(smem_u32(FP8 ? &bars.f8_full[sl] : &bars.slot_full[sl]), (last / nslot) & 1u,
                  err, ERR_WAIT_DRAIN);
      }
    }
    __syncwarp();
  } else if (warp == kWarpQ) {
    // ------------------------------------------------------------ query loader
    // The R query rows of a unit (R x 256 B) are read with plain loads one
    // unit ahead and stored C times into the swizzled query tile (rows past
    // the request's queries as zeros).
    constexpr int kVec = R * 16;            // 16-byte pieces of the R rows
    constexpr int kPer = (kVec + 31) / 32;  // pieces per lane
    uint4 qr[kPer];
    int32_t qpos[kPer];  // RoPE position of the piece's row (< 2^31); -1: not turned
    uint32_t ua = 0;
    auto fetch = [&](const DGeo& g) {
#pragma unroll
      for (int j = 0; j < kPer; ++j) {
        const int idx = lane + 32 * j;
        qr[j] = make_uint4(0, 0, 0, 0);
        qpos[j] = -1;
        if (idx < kVec) {
          const QRow q = qrow<DEC, R>(a, g, idx >> 4);
          if constexpr (ROPE)
            if (q.ok && q.pos >= 0 && q.pos < a.rope_rows) qpos[j] = int32_t(q.pos);
          if (q.ok)
            qr[j] = __ldg(reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(a.q) +
                                                         q.orow * kHeadDim) +
                          (idx & 15));
        }
      }
    };
    // the units of this CTA that have kv tokens, in order
    int vc = blockIdx.x, ui = vc < a.num_ctas ? __ldg(a.ws.work_indptr + vc) : 0;
    // (a chain of units shares its first unit's query tile)
    auto next_unit = [&](DGeo& g) -> bool {
      while (vc < a.num_ctas) {
        if (ui < __ldg(a.ws.work_indptr + vc + 1)) {
          g = decode_geo<DEC>(a, ui++);
          if (g.ntiles > 0 && !g.cprev) return true;
        } else {
          vc += gridDim.x;
          if (vc < a.num_ctas) ui = __ldg(a.ws.work_indptr + vc);
        }
      }
      return false;
    };
    DGeo g;
    bool have = next_unit(g);
    if (have) fetch(g);
    while (have) {
      bool r = true;
      if (lane == 0)
        r = mbar_wait(smem_u32(&bars.q_empty), (ua & 1u) ^ 1u, err, ERR_WAIT_EMPTY);
      if (__shfl_sync(0xffffffffu, r ? 1 : 0, 0) == 0) break;
#pragma unroll
      for (int j = 0; j < kPer; ++j) {
        const int idx = lane + 32 * j;
        uint4 val = qr[j];
        if constexpr (ROPE) {
          // the query at position kv_len - 1: dims d and d + 64 sit in the
          // pieces ch and ch + 8 of a row, i.e. in lanes l and l ^ 8
          uint4 oth;
          oth.x = __shfl_xor_sync(0xffffffffu, val.x, 8);
          oth.y = __shfl_xor_sync(0xffffffffu, val.y, 8);
          oth.z = __shfl_xor_sync(0xffffffffu, val.z, 8);
          oth.w = __shfl_xor_sync(0xffffffffu, val.w, 8);
          if (idx < kVec && qpos[j] >= 0) {
            const int ch = idx & 15;
            const int64_t pos = qpos[j];
            const float4* cp =
                reinterpret_cast<const float4*>(a.rope_cos + pos * (kHeadDim / 2) + 8 * (ch & 7));
            const float4* sp =
                reinterpret_cast<const float4*>(a.rope_sin + pos * (kHeadDim / 2) + 8 * (ch & 7));
            val = rope8<BF16>(val, oth, ch < 8, __ldg(cp), __ldg(cp + 1), __ldg(sp), __ldg(sp + 1));
          }
        }
        if constexpr (FP8 && BF16)
          val = make_uint4(bf16x2_to_f16x2(val.x), bf16x2_to_f16x2(val.y),
                           bf16x2_to_f16x2(val.z), bf16x2_to_f16x2(val.w));
        if (idx < kVec) {
          const int rho = idx >> 4, ch = idx & 15;
          const int half = ch >> 3, j8 = ch & 7;
#pragma unroll
          for (int c = 0; c < C; ++c) {
            const int row = rho + R * c;
            const int off = kOffQ + half * kHalf + row * 128 + ((j8 ^ (row & 7)) << 4);
            *reinterpret_cast<uint4*>(gbase + off) = val;
          }
        }
      }
      fence_proxy_async_smem();  // generic stores -> the MMA's operand reads
      mbar_arrive(smem_u32(&bars.q_full));
      ++ua;
      have = next_unit(g);
      if (have) fetch(g);
    }
  } else if (warp == kWarpMma) {
    // ------------------------------------------------------------ MMA issuer
    // Per unit: S(0), S(1) into the two S buffers; then per KV tile k:
    // O += P(k) V once the softmax has written P(k), then S(k+2). The tensor
    // core runs in issue order, so S(k+2) overwrites P(k) only after P(k).V.
    if (lane == 0) {
      uint32_t ua = 0, jt = 0, n_u = 0;
      bool ok = true;
      auto slot_of = [](uint32_t use) { return use % kRing; };
      // (gathered rows land through cp.async, i.e. the generic proxy: fence
      // them into the async proxy before the MMAs read the slot)
      auto wait_slot = [&](uint32_t use) -> bool {
        const bool r = mbar_wait(smem_u32(&bars.slot_full[slot_of(use)]), (use / kRing) & 1u,
                                 err, ERR_WAIT_FULL);
        if (prm.gather) fence_proxy_async_smem();
        return r;
      };
      // K tile k in its slot (and, with RoPE, turned by the rope warps)
      auto wait_k = [&](uint32_t k) -> bool {
        if constexpr (ROPE)
          return mbar_wait(smem_u32(&bars.k_rot[k % (kSlots / 2)]), (k / (kSlots / 2)) & 1u, err,
                           ERR_WAIT_FULL);
        else
          return wait_slot(2 * k);
      };
      auto issue_s = [&](uint32_t k) {
        const uint32_t qbase = base + kOffQ;
        const uint32_t kbase = base + kOffRing + slot_of(2 * k) * kTileBytes;
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const uint32_t koff = (kk >> 2) * kHalf + (kk & 3) * 32;
          mma_f16(tmem + (k & 1u) * 128u, smem_desc(qbase + koff, 16, 1024),
                  smem_desc(kbase + koff, 16, 1024), prm.idesc_s, kk > 0 ? 1u : 0u);
        }
        mma_commit(smem_u32(&bars.s_full[k & 1u]));
        mma_commit(smem_u32(&bars.slot_empty[slot_of(2 * k)]));
      };
      // O += P(k) V over the tile's nk 16-token chunks (chunks past the
      // unit's end are skipped: their V rows were never loaded)
      auto issue_pv = [&](uint32_t k, int nk, bool first) -> bool {
        if (!mbar_wait(smem_u32(&bars.p_full[k & 1u]), (k >> 1) & 1u, err, ERR_WAIT_SOFTMAX))
          return false;
        // O[n_u & 1] is free once the epilogue read it for unit n_u - 2
        if (first && !mbar_wait(smem_u32(&bars.o_free[n_u & 1u]), ((n_u >> 1) & 1u) ^ 1u, err,
                                ERR_WAIT_SOFTMAX))
          return false;
        tc_fence_after();
        const uint32_t vbase = base + kOffRing + slot_of(2 * k + 1) * kTileBytes;
        for (int kk = 0; kk < nk; ++kk) {
          const uint64_t bd = smem_desc(vbase + kk * kChunk * 128, kHalf, 1024);
          mma_f16_ts(tmem + kColO + 128u * (n_u & 1u), tmem + (k & 1u) * 128u + kk * 8, bd,
                     prm.idesc_pv, (first && kk == 0) ? 0u : 1u);
        }
        mma_commit(smem_u32(&bars.o_done[k & 1u]));
        mma_commit(smem_u32(&bars.slot_empty[slot_of(2 * k + 1)]));
        return true;
      };
      for (int vc = blockIdx.x; vc < a.num_ctas && ok; vc += gridDim.x)
        for (int ui = __ldg(a.ws.work_indptr + vc); ui < __ldg(a.ws.work_indptr + vc + 1) && ok;
             ++ui) {
          const DGeo g = decode_geo<DEC>(a, ui);
          if (g.ntiles == 0) continue;
          const int n = g.ntiles;
          // a chain (composable formats) keeps its query tile and O buffer:
          // the query is awaited at its first unit and released after its
          // last S, O is overwritten only by its first P.V
          if ((!g.cprev && !mbar_wait(smem_u32(&bars.q_full), ua & 1u, err, ERR_WAIT_FULL)) ||
              !wait_k(jt)) {
            ok = false;
            break;
          }
          tc_fence_after();
          issue_s(jt);
          if (n > 1) {
            if (!wait_k(jt + 1)) {
              ok = false;
              break;
            }
            tc_fence_after();
            issue_s(jt + 1);
          }
          if (n <= 2 && !g.cnext) mma_commit(smem_u32(&bars.q_empty));  // last S issued
          for (int i = 0; i < n && ok; ++i) {
            const uint32_t k = jt + i;
            const int64_t kv0 = g.tok_begin + int64_t(i) * kTile;
            const int ntt = int(min(int64_t(kTile), g.tok_end - kv0));
            if (!wait_slot(2 * k + 1)) {
              ok = false;
              break;
            }
            ok = issue_pv(k, (ntt + kChunk - 1) / kChunk, i == 0 && !g.cprev);
            if (ok && i + 2 < n) {
              if (!wait_k(k + 2)) {
                ok = false;
                break;
              }
              tc_fence_after();
              issue_s(k + 2);
              if (i + 3 == n && !g.cnext) mma_commit(smem_u32(&bars.q_empty));  // last S issued
            }
          }
          if (!ok) break;
          jt += n;
          if (g.cnext) continue;  // the chain goes on in the next unit
          mma_commit(smem_u32(&bars.ounit[n_u & 1u]));  // the unit's O is complete
          ++n_u;
          ++ua;
        }
      // drain: no MMA may still be writing TMEM when it is freed
      mma_commit(smem_u32(&bars.drain));
      mbar_wait(smem_u32(&bars.drain), 0, err, ERR_WAIT_DRAIN);
    }
    __syncwarp();
  } else if (warp == kWarpSoftmax) {
    // ------------------------------------------------- softmax / epilogue
    // Thread (rho, c) = lane (rho = lane % R, c = lane / R) owns TMEM lane
    // `lane`: copy c of query row rho, kv columns [W c, W c + W) of every
    // tile. Waits are made warp-uniform: the tcgen05.ld/st after them are
    // .sync.aligned.
    const int rho = lane % R;
    const int c = lane / R;
    uint32_t n_t = 0, n_u = 0;  // tiles and units with tiles so far
    bool ok = true;
    float m_ref = -INFINITY, l = 0.f;  // row state (carried along a chain)
    for (int vc = blockIdx.x; vc < a.num_ctas && ok; vc += gridDim.x)
      for (int ui = __ldg(a.ws.work_indptr + vc); ui < __ldg(a.ws.work_indptr + vc + 1) && ok;
           ++ui) {
        const DGeo g = decode_geo<DEC>(a, ui);
        const QRow qr = qrow<DEC, R>(a, g, rho);
        // log2-domain logit scale (FP8: the kv head's key scale folded in)
        const float c2 = FP8 ? prm.scale_log2 * __ldg(a.k_scale + g.hk) : prm.scale_log2;
        const uint32_t ob = n_u & 1u;  // this unit's O buffer
        const uint32_t col_o = kColO + 128u * ob;
        const int64_t orow = qr.orow;
        const int64_t prow = int64_t(g.slot) * a.rows_per_item + rho;  // split items
        if (g.ntiles == 0) {  // no kv: o = 0, lse = -inf
          if (!qr.ok) {
          } else if (g.slot < 0) {
            constexpr int kS = W < 8 ? W : 8;
            float z[kS];
#pragma unroll
            for (int j = 0; j < kS; ++j) z[j] = 0.f;
#pragma unroll
            for (int j = 0; j < W; j += kS)
              store_out16<BF16, kS>(a.o, orow * kHeadDim + W * c + j, z, 1.f);
            if (c == 0 && a.lse) a.lse[orow] = -INFINITY;
          } else {
            float* dst = a.ws.partial_o + prow * kHeadDim + W * c;
            for (int j = 0; j < W; ++j) dst[j] = 0.f;
            if (c == 0) a.ws.partial_lse[prow] = -INFINITY;
          }
          if (g.slot >= 0) merge_split_impl<BF16, R, DEC>(a, g);
          continue;
        }
        // kv positions this row sees: [tok_begin, row_end)
        const int64_t row_end = qr.ok ? min(g.tok_end, qr.limit + 1) : g.tok_begin;
        if (!g.cprev) {
          m_ref = -INFINITY;
          l = 0.f;
        }
        for (int i = 0; i < g.ntiles; ++i, ++n_t) {
          if (!__all_sync(0xffffffffu, mbar_wait(smem_u32(&bars.s_full[n_t & 1u]),
                                                 (n_t >> 1) & 1u, err, ERR_WAIT_MMA))) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t col_s = (n_t & 1u) * 128u;
          const int64_t kv0 = g.tok_begin + int64_t(i) * kTile;
          const int nvalid = int(max(int64_t(0), min(int64_t(kTile), row_end - kv0)));
          // this thread's W scores: columns [W c, W c + W) of its row
          float s[W];
          if constexpr (ROPE) {
            // nine warps leave 168 registers a thread: 32 columns at a time
#pragma unroll
            for (int j = 0; j < W; ++j) s[j] = 0.f;
#pragma unroll
            for (int q4 = 0; q4 < kTile / 32; ++q4) {
              float v[32];
              tmem_ld32(tmem + col_s + 32u * q4, v);
#pragma unroll
              for (int b = 0; b < C; ++b) {
                const bool mine = c == b;
#pragma unroll
                for (int j = 0; j < W; ++j)
                  if (W * b + j >= 32 * q4 && W * b + j < 32 * q4 + 32)
                    s[j] = mine ? v[W * b + j - 32 * q4] : s[j];
              }
            }
          } else {
            float v[kTile];
            tmem_ld128(tmem + col_s, v);
#pragma unroll
            for (int j = 0; j < W; ++j) s[j] = v[j];
#pragma unroll
            for (int b = 1; b < C; ++b) {
              const bool mine = c == b;
#pragma unroll
              for (int j = 0; j < W; ++j) s[j] = mine ? v[W * b + j] : s[j];
            }
          }
          // (decode: every row sees the same columns)
          const bool full = DEC ? nvalid == kTile : __all_sync(0xffffffffu, nvalid == kTile);
          float mx = -INFINITY;
          if (full) {
#pragma unroll
            for (int j = 0; j < W; ++j) mx = fmaxf(mx, s[j]);
          } else {
#pragma unroll
            for (int j = 0; j < W; ++j) mx = fmaxf(mx, (W * c + j < nvalid) ? s[j] : -INFINITY);
          }
#pragma unroll
          for (int st = 0; st < LC; ++st) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, R << st));
          const float m_tile = mx * c2;  // -inf stays -inf
          float alpha = 1.f;
          bool rescale_o = false;
          if (m_tile > m_ref + 8.f) {
            alpha = ex2(m_ref - m_tile);  // 0 when m_ref = -inf
            rescale_o = (i > 0 || g.cprev) && (m_ref != -INFINITY);
            l *= alpha;
            m_ref = m_tile;
          }
          if (__any_sync(0xffffffffu, rescale_o)) {
            // O must hold every earlier tile: S(k) completing only implies
            // P(k-2).V, so wait for P(k-1).V explicitly
            if (!__all_sync(0xffffffffu, mbar_wait(smem_u32(&bars.o_done[(n_t - 1) & 1u]),
                                                   ((n_t - 1) >> 1) & 1u, err, ERR_WAIT_MMA))) {
              ok = false;
              break;
            }
            tc_fence_after();
#pragma unroll 1
            for (int b = 0; b < 4; ++b) {
              float o[32];
              tmem_ld32(tmem + col_o + b * 32, o);
              const float f = rescale_o ? alpha : 1.f;
#pragma unroll
              for (int q = 0; q < 32; ++q) o[q] *= f;
              tmem_st32(tmem + col_o + b * 32, o);
            }
          }
          // probabilities of this thread's W columns, packed to 16-bit
          uint32_t pk[W / 2];
          float lsum = 0.f;
          const bool live = m_ref != -INFINITY;
#pragma unroll
          for (int j = 0; j < W; j += 2) {
            float p0 = ex2(fmaf(s[j], c2, -m_ref));
            float p1 = ex2(fmaf(s[j + 1], c2, -m_ref));
            if (!full || !live) {
              p0 = (live && W * c + j < nvalid) ? p0 : 0.f;
              p1 = (live && W * c + j + 1 < nvalid) ? p1 : 0.f;
            }
            lsum += p0 + p1;
            pk[j / 2] = pack2<kMmaBF16>(p0, p1);
          }
          l += lsum;
          // the P row: this thread's W/2 packed columns at (W/2) c, zeros elsewhere
#pragma unroll
          for (int b = 0; b < 4; ++b) {
            uint32_t blk[16];
#pragma unroll
            for (int q = 0; q < 16; ++q) {
              constexpr int HW = W / 2;
              const int pc = 16 * b + q;
              blk[q] = (pc / HW == c) ? pk[pc % HW] : 0u;
            }
            tmem_st16_nowait(tmem + col_s + 16 * b, blk);
          }
          tmem_wait_st();
          // V rows past the unit's end inside its last 16-row chunk hold
          // whatever the pool had there: zero them once the tile's V has
          // landed (whole chunks past the end are skipped by the P.V MMA)
          const int ntt = int(min(int64_t(kTile), g.tok_end - kv0));
          const int nrow = ((ntt + kChunk - 1) / kChunk) * kChunk;
          if (ntt < nrow) {
            const uint32_t vuse = 2 * n_t + 1;
            if (!__all_sync(0xffffffffu, mbar_wait(smem_u32(&bars.slot_full[vuse % kRing]),
                                                   (vuse / kRing) & 1u, err, ERR_WAIT_FULL))) {
              ok = false;
              break;
            }
            uint8_t* vslot = gbase + kOffRing + (vuse % kRing) * kTileBytes;
            for (int e = lane; e < (nrow - ntt) * 16; e += 32) {
              const int rr = ntt + (e >> 4), q = e & 15;
              *reinterpret_cast<uint4*>(vslot + (q >> 3) * kHalf + rr * 128 + (q & 7) * 16) =
                  make_uint4(0, 0, 0, 0);
            }
            fence_proxy_async_smem();
          }
          tc_fence_before();
          mbar_arrive(smem_u32(&bars.p_full[n_t & 1u]));
        }
        if (!ok) break;
        if (g.cnext) continue;  // the chain goes on: keep the row state
        // ---- hand the row state to the epilogue warp; the slot of O[ob]
        // is free once the epilogue has finished unit n_u - 2
        if (!__all_sync(0xffffffffu, mbar_wait(smem_u32(&bars.o_free[ob]),
                                               ((n_u >> 1) & 1u) ^ 1u, err, ERR_WAIT_MMA))) {
          ok = false;
          break;
        }
        hand.m[ob][lane] = m_ref;
        hand.l[ob][lane] = l;
        mbar_arrive(smem_u32(&bars.ep_full[ob]));
        ++n_u;
      }
  } else if (warp == kWarpEpi) {
    // ------------------------------------------------------------ epilogue
    // Per unit with kv tiles, in order: once the softmax handed over the row
    // state and the unit's last P.V is done, sum the copies of every row out
    // of O[u & 1], write o / lse (or the split item's partial state), free
    // the buffer, and merge the item if this unit arrives last.
    const int rho = lane % R;
    const int c = lane / R;
    uint32_t n_u = 0;
    bool ok = true;
    for (int vc = blockIdx.x; vc < a.num_ctas && ok; vc += gridDim.x)
      for (int ui = __ldg(a.ws.work_indptr + vc); ui < __ldg(a.ws.work_indptr + vc + 1) && ok;
           ++ui) {
        const DGeo g = decode_geo<DEC>(a, ui);
        if (g.ntiles == 0) continue;  // written by the softmax warp
        if (g.cnext) continue;        // not the end of its chain
        const QRow qr = qrow<DEC, R>(a, g, rho);
        const int64_t orow = qr.orow;
        const int64_t prow = int64_t(g.slot) * a.rows_per_item + rho;  // split items
        const uint32_t ob = n_u & 1u;
        const uint32_t col_o = kColO + 128u * ob;
        const uint32_t ph = (n_u >> 1) & 1u;
        if (!__all_sync(0xffffffffu,
                        mbar_wait(smem_u32(&bars.ep_full[ob]), ph, err, ERR_WAIT_SOFTMAX) &&
                            mbar_wait(smem_u32(&bars.ounit[ob]), ph, err, ERR_WAIT_MMA))) {
          ok = false;
          break;
        }
        tc_fence_after();
        const float m_ref = hand.m[ob][lane];
        float lt = hand.l[ob][lane];
#pragma unroll
        for (int st = 0; st < LC; ++st) lt += __shfl_xor_sync(0xffffffffu, lt, R << st);
        const bool any = lt > 0.f;
        // 1 / l (FP8: times the kv head's value scale)
        const float inv = any ? (FP8 ? __ldg(a.v_scale + g.hk) : 1.f) / lt : 0.f;
        const float lse2 = any ? m_ref + lg2(lt) : -INFINITY;
        // first dim (within a 32-column chunk) that this thread holds after
        // the transposing reduction, and how many
        int doff = 0;
#pragma unroll
        for (int st = 0; st < LC; ++st) doff += ((c >> st) & 1) * (16 >> st);
        constexpr int NF = 32 / C;
#pragma unroll 1
        for (int b = 0; b < 4; ++b) {
          float o[32];
          tmem_ld32(tmem + col_o + b * 32, o);
          // transposing butterfly over the copies: each step halves the
          // values a thread keeps and adds the partner's matching half
          int n = 32;
#pragma unroll
          for (int st = 0; st < LC; ++st) {
            n >>= 1;
            const bool upper = (c >> st) & 1;
#pragma unroll
            for (int k = 0; k < 16; ++k) {
              if (k < n) {
                const float send = upper ? o[k] : o[k + n];
                const float keep = upper ? o[k + n] : o[k];
                o[k] = keep + __shfl_xor_sync(0xffffffffu, send, R << st);
              }
            }
          }
          const int d0 = 32 * b + doff;
          if (!qr.ok) {
          } else if (g.slot < 0) {
            store_out16<BF16, NF>(a.o, orow * kHeadDim + d0, o, inv);
          } else {
            store_out32<NF>(a.ws.partial_o + prow * kHeadDim + d0, o, inv);
          }
        }
        if (c == 0 && qr.ok) {
          if (g.slot < 0) {
            if (a.lse) a.lse[orow] = lse2 * kLn2;
          } else {
            a.ws.partial_lse[prow] = lse2;
          }
        }
        tc_fence_before();
        mbar_arrive(smem_u32(&bars.o_free[ob]));
        ++n_u;
        // the CTA's last unit: every tile has been consumed, so the K / V
        // ring is idle and serves as the merge's landing area
        const bool final_unit = vc + int(gridDim.x) >= a.num_ctas &&
                                ui + 1 == __ldg(a.ws.work_indptr + vc + 1);
        if (g.slot >= 0 &&
            !merge_split_impl<BF16, R, DEC>(a, g, final_unit ? gbase + kOffRing : nullptr,
                                            final_unit ? 4u * kTileBytes : 0u)) {
          ok = false;
          break;
        }
      }
  }

  if constexpr (!ROPE && !FP8) {
    if (prm.gather && warp >= kWarpRope0 && warp < kWarpRope0 + 3) {
      // ------------------------------------------------- gathered-row copies
      // (quarters 1-3 of every tile; warp 1 copies quarter 0)
      uint32_t uses = 0;
      bool ok = true;
      produce_gather<DEC, 4>(prm, bars, base, gbase, lane, warp - kWarpRope0 + 1, err, uses, ok);
    }
  }

  if constexpr (FP8) {
    if (warp >= kWarpRope0 && warp < kWarpRope0 + kConvThreads / 32) {
      // ------------------------------------------------------- FP8 converters
      // Warps 5-7 widen every K / V tile in place: its 128 rows of 128 E4M3
      // bytes (128B-swizzled) sit in the upper half of the slot, and become
      // two 128B-swizzled 64-dim halves of f16 for the MMAs. Thread t takes
      // the 16-byte pieces t, t + 96, ... (row = piece / 8, dims
      // 16 (piece % 8) .. + 15): a warp holds whole rows, reads all of its
      // pieces, syncs, then writes (the upper f16 half of a row overwrites
      // that row's E4M3 bytes). E4M3 -> f16 is exact (one cvt per pair).
      // Rows past a unit's end are widened too: the softmax masks those keys
      // and zeroes those V rows, as it does for 16-bit pools.
      const int t = threadIdx.x - kWarpRope0 * 32;  // 0..95
      int vc = blockIdx.x, ui = vc < a.num_ctas ? __ldg(a.ws.work_indptr + vc) : 0;
      auto next_unit = [&](DGeo& g) -> bool {
        while (vc < a.num_ctas) {
          if (ui < __ldg(a.ws.work_indptr + vc + 1)) {
            g = decode_geo<DEC>(a, ui++);
            if (g.ntiles > 0) return true;
          } else {
            vc += gridDim.x;
            if (vc < a.num_ctas) ui = __ldg(a.ws.work_indptr + vc);
          }
        }
        return false;
      };
      uint32_t use = 0;
      bool ok = true;
      DGeo g;
      while (ok && next_unit(g)) {
        for (int i = 0; i < 2 * g.ntiles && ok; ++i, ++use) {  // K then V of each tile
          const uint32_t rs = use % kRing;
          // (the producer loads a slot only once it is free)
          if (!mbar_wait(smem_u32(&bars.f8_full[rs]), (use / kRing) & 1u, err, ERR_WAIT_FULL)) {
            ok = false;
            break;
          }
          uint8_t* dst = gbase + kOffRing + rs * kTileBytes;
          const uint8_t* src = dst + kHalf;
          constexpr int kPieces = kTile * 8;  // 16-byte pieces of an E4M3 tile
          constexpr int kPer = (kPieces + kConvThreads - 1) / kConvThreads;
          // all of this thread's pieces are loaded before any is widened
          uint4 raws[kPer];
#pragma unroll
          for (int k = 0; k < kPer; ++k) {
            const int piece = t + kConvThreads * k;
            const int row = piece >> 3, c = piece & 7;
            if (piece < kPieces)
              raws[k] = *reinterpret_cast<const uint4*>(src + row * 128 + ((c ^ (row & 7)) << 4));
          }
          __syncwarp();  // the warp's rows are read before any is overwritten
#pragma unroll
          for (int k = 0; k < kPer; ++k) {
            const int piece = t + kConvThreads * k;
            if (piece >= kPieces) break;
            const int row = piece >> 3, c = piece & 7;
            const uint4 raw = raws[k];
            const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
            uint32_t h[8];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              h[2 * q] = e4m3x2_to_f16x2(w[q] & 0xffffu);
              h[2 * q + 1] = e4m3x2_to_f16x2(w[q] >> 16);
            }
            // dims 16 c .. 16 c + 15: half c / 4, 8-dim chunks 2 (c % 4) and + 1
            uint8_t* rowp = dst + (c >> 2) * kHalf + row * 128;
            const int j0 = 2 * (c & 3);
            *reinterpret_cast<uint4*>(rowp + ((j0 ^ (row & 7)) << 4)) =
                make_uint4(h[0], h[1], h[2], h[3]);
            *reinterpret_cast<uint4*>(rowp + (((j0 + 1) ^ (row & 7)) << 4)) =
                make_uint4(h[4], h[5], h[6], h[7]);
          }
          fence_proxy_async_smem();  // generic stores -> the MMA's operand reads
          mbar_arrive(smem_u32(&bars.slot_full[rs]));
        }
      }
    }
  }

  if constexpr (ROPE) {
    if (warp >= kWarpRope0 && warp < kWarpRope0 + 4) {
      // ------------------------------------------------------------ rope warps
      // Warp w turns rows [32 w, 32 w + 32) of every K tile in place once the
      // tile has landed, then releases it to the MMA warp: a half-warp per
      // row, lane l on pairs 4 (l % 16) .. + 3. The angles are pos * theta_i,
      // so the cos / sin of row B + o follow from those of rows B and o by
      // the angle-sum identities. A lane's rows are B_h + 2 it (it < 8) for
      // two bases B_h per tile: the 8 offset rows o = 2 it sit in shared
      // memory (written once by the rope warps), and a lane loads a tile's
      // two base rows (512 B per half-warp) one tile ahead, so no table read
      // waits on a tile. The rotation itself runs on packed fp32x2 math in
      // a rolled loop of two-row steps (code size matters with nine warps).
      const int wr = warp - kWarpRope0;
      const int hrow = lane >> 4, p0 = 4 * (lane & 15);
      const int kbyte = (((lane & 15) >> 1) << 4) | ((lane & 1) << 3);  // piece, byte in it
      int vc = blockIdx.x, ui = vc < a.num_ctas ? __ldg(a.ws.work_indptr + vc) : 0;
      auto next_unit = [&](DGeo& g) -> bool {
        while (vc < a.num_ctas) {
          if (ui < __ldg(a.ws.work_indptr + vc + 1)) {
            g = decode_geo<DEC>(a, ui++);
            if (g.ntiles > 0) return true;
          } else {
            vc += gridDim.x;
            if (vc < a.num_ctas) ui = __ldg(a.ws.work_indptr + vc);
          }
        }
        return false;
      };
      constexpr int kIt = 8;  // row pairs per warp and half tile
      auto row_c = [&](int64_t pos) {
        return __ldg(reinterpret_cast<const float4*>(a.rope_cos + pos * (kHeadDim / 2) + p0));
      };
      auto row_s = [&](int64_t pos) {
        return __ldg(reinterpret_cast<const float4*>(a.rope_sin + pos * (kHeadDim / 2) + p0));
      };
      // offset rows 2 it into shared memory (only those below the table's
      // length can be needed: a row B + 2 it in use is below it and B >= 0)
      {
        const int t = threadIdx.x - kWarpRope0 * 32;
        float* oc_s = reinterpret_cast<float*>(gbase + kOffRopeCos);
        float* os_s = reinterpret_cast<float*>(gbase + kOffRopeSin);
        for (int idx = t; idx < 8 * 64; idx += 128) {
          const int o = 2 * (idx >> 6);
          const bool ok_row = o < a.rope_rows;
          oc_s[idx] = ok_row ? __ldg(a.rope_cos + o * (kHeadDim / 2) + (idx & 63)) : 1.f;
          os_s[idx] = ok_row ? __ldg(a.rope_sin + o * (kHeadDim / 2) + (idx & 63)) : 0.f;
        }
        asm volatile("bar.sync 1, 128;" ::: "memory");  // the four rope warps
      }
      // base rows of tile i of unit g: B_h = kv0 + 32 w + 16 h + (l >> 4)
      float4 bc[2], bs[2], nbc[2], nbs[2];
#pragma unroll
      for (int h = 0; h < 2; ++h) bc[h] = bs[h] = nbc[h] = nbs[h] = make_float4(0.f, 0.f, 0.f, 0.f);
      auto fetch = [&](const DGeo& g, int i, float4 (&c)[2], float4 (&sn)[2]) {
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int64_t base = g.tok_begin + int64_t(i) * kTile + 32 * wr + 2 * kIt * h + hrow;
          if (base < g.tok_end) {
            c[h] = row_c(base);
            sn[h] = row_s(base);
          }
        }
      };
      DGeo g, gn;
      int i = 0, in = 0;
      bool have = next_unit(g), have_n = false;
      auto advance = [&]() {  // (gn, in) = the tile after (g, i)
        if (i + 1 < g.ntiles) {
          gn = g;
          in = i + 1;
          have_n = true;
        } else {
          in = 0;
          have_n = next_unit(gn);
        }
      };
      if (have) {
        fetch(g, 0, bc, bs);
        advance();
      }
      for (uint32_t k = 0; have; ++k) {
        const uint32_t use = 2 * k, slot = use % kSlots;
        if (!mbar_wait(smem_u32(&bars.slot_full[slot]), (use / kSlots) & 1u, err, ERR_WAIT_FULL))
          break;
        if (have_n) fetch(gn, in, nbc, nbs);
        const int64_t kv0 = g.tok_begin + int64_t(i) * kTile;
        uint8_t* tile = gbase + kOffRing + slot * kTileBytes;
        // a compact loop (the block's nine warps run six different loops, so
        // code size matters): kStep rows per step, all read before any is
        // written back
        constexpr int kStep = 2;
#pragma unroll 1
        for (int st = 0; st < 2 * kIt / kStep; ++st) {
          const int h = st / (kIt / kStep);  // half tile
          const float4 cb = h ? bc[1] : bc[0], sb = h ? bs[1] : bs[0];
          const float4 nsb = make_float4(-sb.x, -sb.y, -sb.z, -sb.w);
          uint2 x[kStep], y[kStep];
          float4 oci[kStep], osi[kStep];
          int off[kStep];
          bool use[kStep];
#pragma unroll
          for (int u = 0; u < kStep; ++u) {
            const int it = kStep * (st % (kIt / kStep)) + u;  // offset row 2 it
            const int row = 32 * wr + 2 * kIt * h + 2 * it + hrow;
            off[u] = row * 128 + (kbyte ^ ((row & 7) << 4));
            use[u] = kv0 + row < g.tok_end;
            if (use[u]) {
              x[u] = *reinterpret_cast<const uint2*>(tile + off[u]);
              y[u] = *reinterpret_cast<const uint2*>(tile + kHalf + off[u]);
              oci[u] = *reinterpret_cast<const float4*>(gbase + kOffRopeCos + it * 256 + p0 * 4);
              osi[u] = *reinterpret_cast<const float4*>(gbase + kOffRopeSin + it * 256 + p0 * 4);
            }
          }
#pragma unroll
          for (int u = 0; u < kStep; ++u) {
            if (use[u]) {
              rope_key4<BF16>(x[u], y[u], cb, sb, nsb, oci[u], osi[u]);
              *reinterpret_cast<uint2*>(tile + off[u]) = x[u];
              *reinterpret_cast<uint2*>(tile + kHalf + off[u]) = y[u];
            }
          }
        }
        fence_proxy_async_smem();  // generic stores -> the MMA's operand reads
        mbar_arrive(smem_u32(&bars.k_rot[k % (kSlots / 2)]));
        have = have_n;
        if (have) {
          g = gn;
          i = in;
          bc[0] = nbc[0], bc[1] = nbc[1], bs[0] = nbs[0], bs[1] = nbs[1];
          advance();
        }
      }
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

template <bool BF16, int R, bool DEC, bool ROPE = false, bool FP8 = false>
cudaError_t launch_k(const DecodeTcParams& prm, int grid, cudaStream_t stream) {
  static std::atomic<uint64_t> configured{0};
  cudaError_t e =
      ensure_smem_limit(decode_tc_kernel<BF16, R, DEC, ROPE, FP8>, kSmem, configured);
  if (e != cudaSuccess) return e;
  decode_tc_kernel<BF16, R, DEC, ROPE, FP8>
      <<<grid, block_threads<ROPE, FP8>(), kSmem, stream>>>(prm);
  return cudaGetLastError();
}
// decode runs with R = group in {2, 4, 8}; short appends with R in {1..16}
template <bool BF16>
cudaError_t launch_dt(const DecodeTcParams& prm, int rows, int grid, cudaStream_t stream) {
  if (prm.a.kv_fp8) {  // decode over an FP8 cache (HND, page_size % 16 == 0)
    switch (rows) {
      case 2: return launch_k<BF16, 2, true, false, true>(prm, grid, stream);
      case 4: return launch_k<BF16, 4, true, false, true>(prm, grid, stream);
      default: return launch_k<BF16, 8, true, false, true>(prm, grid, stream);
    }
  }
  if (!prm.a.qo_indptr && prm.a.rope_cos) {  // decode with fused RoPE
    switch (rows) {
      case 2: return launch_k<BF16, 2, true, true>(prm, grid, stream);
      case 4: return launch_k<BF16, 4, true, true>(prm, grid, stream);
      default: return launch_k<BF16, 8, true, true>(prm, grid, stream);
    }
  }
  if (prm.a.rope_cos) {  // short append with fused RoPE
    switch (rows) {
      case 1: return launch_k<BF16, 1, false, true>(prm, grid, stream);
      case 2: return launch_k<BF16, 2, false, true>(prm, grid, stream);
      case 4: return launch_k<BF16, 4, false, true>(prm, grid, stream);
      case 8: return launch_k<BF16, 8, false, true>(prm, grid, stream);
      default: return launch_k<BF16, 16, false, true>(prm, grid, stream);
    }
  }
  if (!prm.a.qo_indptr) {
    switch (rows) {
      case 2: return launch_k<BF16, 2, true>(prm, grid, stream);
      case 4: return launch_k<BF16, 4, true>(prm, grid, stream);
      default: return launch_k<BF16, 8, true>(prm, grid, stream);
    }
  }
  switch (rows) {
    case 1: return launch_k<BF16, 1, false>(prm, grid, stream);
    case 2: return launch_k<BF16, 2, false>(prm, grid, stream);
    case 4: return launch_k<BF16, 4, false>(prm, grid, stream);
    case 8: return launch_k<BF16, 8, false>(prm, grid, stream);
    default: return launch_k<BF16, 16, false>(prm, grid, stream);
  }
}

}  // namespace

int few_row_rows(int32_t group, int32_t max_qo_len) {
  const int64_t need = int64_t(group) * (max_qo_len > 0 ? max_qo_len : 1);
  for (int r = 1; r <= kFewRowMax; r *= 2)
    if (need <= r) return r;
  return 0;
}

cudaError_t launch_decode_tc(const AppendArgs& a, cudaStream_t stream, const char** msg) {
  const int rows = few_row_rows(a.group, a.qo_indptr ? a.max_qo_len : 1);
  if (rows == 0 || (!a.qo_indptr && (rows < 2 || rows > 8 || rows != a.group))) {
    *msg = "attn: the few-row tensor-core kernel takes 2, 4 or 8 heads per kv head in decode "
           "and at most 16 packed query rows per item in append";
    return cudaErrorNotSupported;
  }
  if (a.page_size <= 0) {
    *msg = "attn: page_size must be positive";
    return cudaErrorNotSupported;
  }
  if (a.num_ctas <= 0 || a.num_units == 0) return cudaSuccess;
  const bool bf16 = a.dtype == ATTN_BF16;
  DecodeTcParams prm;
  std::memset(&prm, 0, sizeof prm);
  prm.a = a;
  prm.scale_log2 = a.sm_scale * kLog2e;
  // FP8 K/V: the MMAs multiply f16 operands (q is converted when it is bf16)
  prm.idesc_s = make_idesc(bf16 && !a.kv_fp8, false);
  prm.idesc_pv = make_idesc(bf16 && !a.kv_fp8, true);
  prm.gather = a.page_size % kChunk != 0 ? 1 : 0;
  prm.nhd = a.layout == ATTN_LAYOUT_NHD ? 1 : 0;
  // composable formats: 16-row boxes when both tables allow them (HND, page
  // sizes that are multiples of 16), else rows copied one by one for both
  if (a.cascade && (prm.nhd || a.page_size2 % kChunk != 0)) prm.gather = 1;
  if (a.kv_fp8 && (prm.gather || prm.nhd || a.qo_indptr || a.rope_cos)) {
    *msg = "attn: the tensor-core FP8 decode takes HND pools with page_size % 16 == 0";
    return cudaErrorNotSupported;
  }
  if (a.cascade && (!a.qo_indptr || a.page_size2 <= 0 || a.kv_fp8 || a.rope_cos || a.causal)) {
    *msg = "attn: composable formats in one launch take 16-bit pools without RoPE";
    return cudaErrorNotSupported;
  }
  // gathered rows are addressed by 32-bit (page, head, slot) row indices
  if (prm.gather) {
    const int64_t rows1 = a.num_pages * a.num_kv_heads * int64_t(a.page_size);
    const int64_t rows2 = a.cascade ? a.num_pages2 * a.num_kv_heads * int64_t(a.page_size2) : 0;
    if (rows1 >= (int64_t(1) << 31) || rows2 >= (int64_t(1) << 31)) {
      *msg = "attn: the pool has 2^31 or more (page, head, slot) rows";
      return cudaErrorNotSupported;
    }
  }
  const int elem = a.kv_fp8 ? kKvElemU8 : (bf16 ? kKvElemBF16 : kKvElemF16);
  // (gathered rows are copied with cp.async: no tensor map)
  if (!prm.gather &&
      !make_kv_maps(a.k_pool, a.v_pool, a.num_pages, a.num_kv_heads, a.page_size, elem,
                    uint32_t(kChunk), prm.nhd != 0, &prm.tm_k, &prm.tm_v, msg))
    return cudaErrorNotSupported;  // *msg says why
  if (a.cascade && !prm.gather &&
      !make_kv_maps(a.k_pool2, a.v_pool2, a.num_pages2, a.num_kv_heads, a.page_size2, elem,
                    uint32_t(kChunk), false, &prm.tm_k2, &prm.tm_v2, msg))
    return cudaErrorNotSupported;
  int sms = 0;
  cudaError_t e = current_sm_count(&sms);
  if (e != cudaSuccess) return e;
  const int grid = a.num_ctas < sms ? a.num_ctas : sms;
  return bf16 ? launch_dt<true>(prm, rows, grid, stream)
              : launch_dt<false>(prm, rows, grid, stream);
}

}  // namespace attn
