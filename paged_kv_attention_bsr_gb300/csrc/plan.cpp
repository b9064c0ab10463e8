// plan.cpp -- host planning phase: balanced split of attention work over a
// fixed persistent grid.
//
// FlashInfer paper digest (modb.pro), section "动态负载均衡调度": scheduling is
// Stream-K inspired and runs in two phases -- a CPU phase that analyses the
// length distribution and emits a work assignment, and a GPU phase whose
// persistent kernel (fixed grid, preallocated workspace) follows it. The page
// gives no algorithm; the cut used here:
//   * items (request, kv head, query tile) in request-major order, then kv
//     head, then tile; an item's cost is its visible page count n plus one
//     overhead slot; W = the sum of all costs;
//   * decode: the costs are laid end to end and CTA c takes the contiguous
//     positions [floor(c W / C), floor((c+1) W / C)) (Stream-K's equal cut);
//     an item crossed by a boundary becomes several units;
//   * append: the items of requests with at most 16 query rows (group x
//     qo_len; decode-like) and the rest are interleaved by weight (prefill
//     and decode requests of one batch run side by side, POD-style). Items
//     are then dealt in that order to the CTA with the least work so far
//     (ties to the lowest index), each CTA capped at ceil(W / C) + 1; an
//     item that does not fit is cut at the cap and continues on the next
//     CTA. CTAs run items in roughly the order of the list, so the query
//     tiles of a kv head are in flight together and share its K/V pages
//     through L2, while every CTA gets an equal share;
//   * units of an item cut in several ("split") write partial (o, lse)
//     states that are merged by log-sum-exp.
// Every CTA gets at most ceil(W/C) + 1 of the cost and the cut adds at most
// C extra units. The result depends only on the inputs and is deterministic.
#include <algorithm>
#include <climits>
#include <cstring>
#include <functional>
#include <queue>
#include <utility>
#include <vector>

#include "internal.h"

namespace attn {

PlanLayout plan_layout(int32_t num_ctas, int64_t num_units, int64_t num_split,
                       int64_t num_slots, int32_t rows_per_item, int32_t head_dim) {
  PlanLayout L;
  int64_t at = kHeaderBytes;
  L.off_work_indptr = at;
  at = align_up(at + 4 * (int64_t(num_ctas) + 1), 256);
  L.off_units = at;
  at = align_up(at + int64_t(sizeof(Unit)) * num_units, 256);
  L.off_merge_indptr = at;
  at = align_up(at + 4 * (num_split + 1), 256);
  L.off_merge_items = at;
  at = align_up(at + 16 * num_split, 256);
  L.off_counters = at;
  at = align_up(at + 4 * num_split, 256);
  L.table_bytes = at;
  L.off_partial_o = at;
  at = align_up(at + 4 * num_slots * rows_per_item * int64_t(head_dim), 256);
  L.off_partial_lse = at;
  at = align_up(at + 4 * num_slots * rows_per_item, 256);
  L.dev_bytes = at;
  return L;
}

namespace {

// An item and its request's geometry (copied into each of its units).
struct Item {
  int32_t r, hk, t, n;
  int32_t page_base, kv_len, qo_start, qo_len;
  int32_t few;  // the request has at most kFewRowMax query rows: decode-like
};

// Per-thread scratch reused across calls (a plan runs every step). One
// thread_local object, bound to a reference once per call: in a shared
// library every access to a thread_local may otherwise go through a TLS
// lookup call.
struct Scratch {
  std::vector<Item> items;
  std::vector<int64_t> bounds;   // floor(c W / C), c = 0 .. C (decode cut)
  std::vector<Unit> gen;         // units in generation order
  std::vector<int32_t> gen_cta;  // and their CTA and item
  std::vector<int32_t> gen_item;
  std::vector<int64_t> load;
  std::vector<int32_t> n_units, split_of, merge_indptr, next, work_indptr, at, order;
  std::vector<int4> merge_items;
  std::vector<Unit> units;       // CTA order (append)
};
Scratch& scratch() {
  thread_local Scratch s;
  return s;
}

uint64_t fnv1a(uint64_t h, const void* data, size_t bytes) {
  const unsigned char* p = static_cast<const unsigned char*>(data);
  for (size_t i = 0; i < bytes; ++i) {
    h ^= p[i];
    h *= 1099511628211ull;
  }
  return h;
}

// Within each CTA's range of `v` (bounds in indptr), the units of split
// items (slot >= 0) first, each group in its order; `tmp` is scratch. One
// pass per CTA with no allocation (std::stable_partition may allocate on
// every call).
void split_units_first(std::vector<Unit>& v, const std::vector<int32_t>& indptr, int64_t C,
                       std::vector<Unit>& tmp) {
  for (int64_t c = 0; c < C; ++c) {
    const size_t b = size_t(indptr[size_t(c)]), e = size_t(indptr[size_t(c) + 1]);
    bool need = false;  // an unsplit unit before a split one
    for (size_t i = b, seen_unsplit = 0; i < e; ++i) {
      if (v[i].slot < 0) seen_unsplit = 1;
      else if (seen_unsplit) need = true;
    }
    if (!need) continue;
    tmp.clear();
    for (size_t i = b; i < e; ++i)
      if (v[i].slot >= 0) tmp.push_back(v[i]);
    for (size_t i = b; i < e; ++i)
      if (v[i].slot < 0) tmp.push_back(v[i]);
    std::copy(tmp.begin(), tmp.end(), v.begin() + std::ptrdiff_t(b));
  }
}

}  // namespace

uint64_t plan_fingerprint(const int32_t* qo_indptr, const int32_t* kv_indptr,
                          const int32_t* last_page_len, int32_t batch, int32_t page_size,
                          int32_t num_qo_heads, int32_t num_kv_heads, int32_t head_dim,
                          int32_t causal, int32_t num_ctas) {
  uint64_t h = 1469598103934665603ull;
  h = fnv1a(h, kv_indptr, 4 * (size_t(batch) + 1));
  if (batch) h = fnv1a(h, last_page_len, 4 * size_t(batch));
  if (qo_indptr) h = fnv1a(h, qo_indptr, 4 * (size_t(batch) + 1));
  const int32_t shape[6] = {page_size, num_qo_heads, num_kv_heads, head_dim, causal, num_ctas};
  return fnv1a(h, shape, sizeof shape);
}

attn_status_t build_plan(const int32_t* qo_indptr, const int32_t* kv_indptr,
                         const int32_t* last_page_len, int32_t batch, int32_t page_size,
                         int32_t num_qo_heads, int32_t num_kv_heads, int32_t head_dim,
                         int32_t causal, int32_t num_ctas, void* host_tables,
                         size_t host_bytes, attn_plan_t* plan, const char** msg) {
  *msg = "";
  if (!kv_indptr || !plan || !host_tables || (batch > 0 && !last_page_len)) {
    *msg = "attn_plan: null pointer argument";
    return ATTN_ERR_INVALID_ARG;
  }
  if (batch < 0 || page_size < 1 || num_qo_heads < 1 || num_kv_heads < 1 || num_ctas < 1) {
    *msg = "attn_plan: batch, page_size, head counts and num_ctas must be positive";
    return ATTN_ERR_INVALID_ARG;
  }
  if (num_qo_heads % num_kv_heads != 0) {
    *msg = "attn_plan: num_qo_heads must be a multiple of num_kv_heads";
    return ATTN_ERR_INVALID_ARG;
  }
  if (head_dim != kHeadDim) {
    *msg = "attn_plan: only head_dim == 128 is implemented";
    return ATTN_ERR_UNSUPPORTED;
  }
  const bool decode = (qo_indptr == nullptr);
  const int32_t group = num_qo_heads / num_kv_heads;
  if (decode && group > kMaxDecodeGroup) {
    *msg = "attn_plan: decode supports num_qo_heads / num_kv_heads <= 8";
    return ATTN_ERR_UNSUPPORTED;
  }
  if (!decode && (group > kTileRows || kTileRows % group != 0)) {  // a tile holds whole tokens
    *msg = "attn_plan: append needs num_qo_heads / num_kv_heads to divide 128";
    return ATTN_ERR_UNSUPPORTED;
  }
  const int32_t q_tile = decode ? 1 : kItemRows / group;
  const int32_t rows_per_item = group * q_tile;

  // ---- validate the table and build items
  if (kv_indptr[0] < 0) {
    *msg = "attn_plan: kv_indptr must start at a non-negative offset";
    return ATTN_ERR_INVALID_ARG;
  }
  if (!decode && qo_indptr[0] != 0) {
    *msg = "attn_plan: qo_indptr must start at 0 (q rows are indexed from the tensor start)";
    return ATTN_ERR_INVALID_ARG;
  }
  Scratch& sc = scratch();
  std::vector<Item>& items = sc.items;
  items.clear();
  items.reserve(size_t(batch) * num_kv_heads);
  int64_t max_qo_len = decode ? 1 : 0;
  int64_t max_kv_len = 0;
  int64_t min_kv_minus_qo = INT64_MAX;  // over requests with kv tokens
  for (int32_t r = 0; r < batch; ++r) {
    const int64_t n_pages = int64_t(kv_indptr[r + 1]) - kv_indptr[r];
    if (n_pages < 0) {
      *msg = "attn_plan: kv_indptr must be non-decreasing";
      return ATTN_ERR_INVALID_ARG;
    }
    if (n_pages > 0 && (last_page_len[r] < 1 || last_page_len[r] > page_size)) {
      *msg = "attn_plan: last_page_len must be in [1, page_size] for a request with pages";
      return ATTN_ERR_INVALID_ARG;
    }
    const int64_t kv_len = n_pages > 0 ? (n_pages - 1) * page_size + last_page_len[r] : 0;
    if (kv_len > INT32_MAX) {
      *msg = "attn_plan: a request's kv length must fit in 31 bits";
      return ATTN_ERR_INVALID_ARG;
    }
    max_kv_len = std::max(max_kv_len, kv_len);
    int64_t qo_len = 1;
    if (!decode) {
      qo_len = int64_t(qo_indptr[r + 1]) - qo_indptr[r];
      if (qo_len < 0) {
        *msg = "attn_plan: qo_indptr must be non-decreasing";
        return ATTN_ERR_INVALID_ARG;
      }
      max_qo_len = std::max(max_qo_len, qo_len);
      if (causal && kv_len < qo_len) {
        *msg = "attn_plan: causal append needs kv_len >= qo_len for every request";
        return ATTN_ERR_INVALID_ARG;
      }
    }
    if (kv_len > 0) min_kv_minus_qo = std::min(min_kv_minus_qo, kv_len - qo_len);
    const int64_t tiles = decode ? 1 : (qo_len + q_tile - 1) / q_tile;
    for (int32_t hk = 0; hk < num_kv_heads; ++hk) {
      for (int64_t t = 0; t < tiles; ++t) {
        int64_t vis = kv_len;
        if (causal && !decode) {
          const int64_t last_row = std::min<int64_t>((t + 1) * q_tile, qo_len) - 1;
          vis = std::min<int64_t>(kv_len, std::max<int64_t>(0, kv_len - qo_len + last_row + 1));
        }
        const int64_t n = (vis + page_size - 1) / page_size;
        items.push_back({r, hk, int32_t(t), int32_t(n), kv_indptr[r], int32_t(kv_len),
                         decode ? r : qo_indptr[r], int32_t(qo_len),
                         int64_t(group) * qo_len <= kFewRowMax ? 1 : 0});
      }
    }
  }

  // ---- cut the work into units
  // cost of a unit beyond its pages, in pages: a unit of the few-row kernel
  // (decode, short appends) starts and ends cheaply next to its pages; an
  // append-kernel unit's epilogue (O out of tensor memory) and next-unit
  // start cost about two KV tiles of MMAs
  const bool few_kernel = decode || int64_t(group) * max_qo_len <= kFewRowMax;
  const int64_t kAlpha = few_kernel ? kDecodeAlpha : kAppendAlpha;
  int64_t W = 0;
  for (const Item& it : items) W += it.n + kAlpha;
  const int64_t C = num_ctas;
  std::vector<int64_t>& bounds = sc.bounds;
  if (decode) {
    // floor(c W / C) by a running quotient and remainder (one division)
    bounds.resize(size_t(C) + 1);
    const int64_t dq = W / C, dr = W % C;
    int64_t q = 0, rem = 0;
    for (int64_t c = 0; c <= C; ++c) {
      bounds[size_t(c)] = q;
      q += dq;
      rem += dr;
      if (rem >= C) {
        ++q;
        rem -= C;
      }
    }
  }
  const int64_t* const bnd = bounds.data();
  auto bound = [bnd](int64_t c) -> int64_t { return bnd[c]; };

  // units in generation order (decode: already CTA order), with their CTA
  // and item, and the request's geometry filled in
  std::vector<Unit>& gen = sc.gen;
  std::vector<int32_t>& gen_cta = sc.gen_cta;
  std::vector<int32_t>& gen_item = sc.gen_item;
  // at most one unit per item plus one per CTA boundary (either cut)
  const size_t max_units = items.size() + size_t(C);
  if (gen.size() < max_units) {
    gen.resize(max_units);
    gen_cta.resize(max_units);
    gen_item.resize(max_units);
  }
  size_t num_units = 0;
  bool overflow = false;
  auto emit = [&](const Item& it, size_t k, int64_t p0, int64_t p1, int64_t cta) {
    if (num_units >= max_units) {
      overflow = true;
      return;
    }
    Unit& u = gen[num_units];
    u.r = it.r;
    u.hk = it.hk;
    u.t = it.t;
    u.p0 = int32_t(p0);
    u.p1 = int32_t(p1);
    u.slot = -1;
    u.split = -1;
    u.page_base = it.page_base;
    u.kv_len = it.kv_len;
    u.qo_start = it.qo_start;
    u.qo_len = it.qo_len;
    u.pad = 0;
    gen_cta[num_units] = int32_t(cta);
    gen_item[num_units] = int32_t(k);
    ++num_units;
  };
  std::vector<int64_t>& load = sc.load;
  load.assign(size_t(C), 0);

  if (decode) {
    // Contiguous balanced cut of the cost line (Stream-K style).
    int64_t c = 0;
    int64_t base = 0;
    for (size_t k = 0; k < items.size(); ++k) {
      const Item& it = items[k];
      const int64_t w = it.n + kAlpha;
      while (c + 1 < C && bound(c + 1) <= base) ++c;  // CTA owning position `base`
      for (int64_t cc = c; cc < C && bound(cc) < base + w; ++cc) {
        const int64_t lo = bound(cc), hi = bound(cc + 1);
        if (hi <= lo) continue;
        if (it.n == 0) {
          if (lo <= base && base < hi) emit(it, k, 0, 0, cc);
          continue;
        }
        const int64_t p0 = std::max<int64_t>(0, lo - base - kAlpha);
        const int64_t p1 = std::min<int64_t>(it.n, hi - base - kAlpha);
        if (p1 > p0) emit(it, k, p0, p1, cc);
      }
      base += w;
    }
    for (int64_t i = 0; i < C; ++i) load[size_t(i)] = bound(i + 1) - bound(i);
  } else {
    // Visiting order (prefill and decode in one plan, POD-style): the items
    // of requests with at most kFewRowMax query rows (decode-like,
    // memory-bound) and the other items (tensor-bound) keep their own order
    // and are interleaved by weight -- the next item comes from the class
    // that has used the smaller fraction of its total weight, ties to the
    // tensor-bound class -- so that every CTA's list mixes both kinds over
    // time and HBM streaming overlaps the tensor work across the SMs.
    std::vector<int32_t>& order = sc.order;
    order.clear();
    {
      int64_t wd = 0, wf = 0;
      for (const Item& it : items) (it.few ? wf : wd) += it.n + kAlpha;
      size_t id = 0, jf = 0;
      int64_t dd = 0, df = 0;
      auto next_of = [&](size_t i, int32_t few) {
        while (i < items.size() && items[i].few != few) ++i;
        return i;
      };
      id = next_of(0, 0);
      jf = next_of(0, 1);
      while (id < items.size() || jf < items.size()) {
        const bool dense = jf >= items.size() || (id < items.size() && dd * wf <= df * wd);
        const size_t k = dense ? id : jf;
        const int64_t w = items[k].n + kAlpha;
        order.push_back(int32_t(k));
        if (dense) {
          dd += w;
          id = next_of(id + 1, 0);
        } else {
          df += w;
          jf = next_of(jf + 1, 1);
        }
      }
    }
    // Time-ordered fill: items go, in that order, to the CTA with the least
    // work so far (ties: lowest index), each CTA capped at ceil(W / C) + 1;
    // an item that does not fit is cut at the cap and continues on the next
    // CTA. (A page weighs the same for one or two live query tiles: the two
    // tiles' softmax warpgroups run side by side, and they set the pace.)
    const int64_t cap = (W + C - 1) / C + kAlpha;
    typedef std::pair<int64_t, int32_t> Slot;
    std::priority_queue<Slot, std::vector<Slot>, std::greater<Slot>> ready;
    for (int32_t c = 0; c < num_ctas; ++c) ready.push(Slot(0, c));
    for (const int32_t k32 : order) {
      const size_t k = size_t(k32);
      const Item& it = items[k];
      int64_t p = 0;
      for (;;) {
        if (ready.empty()) {
          *msg = "attn_plan: internal error (append fill ran out of capacity)";
          return ATTN_ERR_INVALID_ARG;
        }
        const Slot top = ready.top();
        ready.pop();
        const int32_t c = top.second;
        const int64_t avail = cap - top.first;
        const int64_t need = kAlpha + (it.n - p);
        if (need <= avail) {
          emit(it, k, p, it.n, c);
          load[size_t(c)] = top.first + need;
          if (load[size_t(c)] < cap) ready.push(Slot(load[size_t(c)], c));
          break;
        }
        const int64_t take = avail - kAlpha;
        load[size_t(c)] = cap;  // this CTA is full either way
        if (take <= 0) continue;
        emit(it, k, p, p + take, c);
        p += take;
      }
    }
  }

  if (overflow) {
    *msg = "attn_plan: internal error (more units than items + CTAs)";
    return ATTN_ERR_INVALID_ARG;
  }

  // ---- split items, slots in (item, page) order
  std::vector<int32_t>& n_units = sc.n_units;
  std::vector<int32_t>& split_of = sc.split_of;
  std::vector<int32_t>& merge_indptr = sc.merge_indptr;
  std::vector<int4>& merge_items = sc.merge_items;
  n_units.assign(items.size(), 0);
  for (size_t i = 0; i < num_units; ++i) n_units[size_t(gen_item[i])]++;
  split_of.assign(items.size(), -1);
  merge_indptr.assign(1, 0);
  merge_items.clear();
  for (size_t k = 0; k < items.size(); ++k) {
    if (n_units[k] < 2) continue;
    split_of[k] = int32_t(merge_items.size());
    merge_items.push_back(make_int4(items[k].r, items[k].hk, items[k].t, n_units[k]));
    merge_indptr.push_back(merge_indptr.back() + n_units[k]);
  }
  const int32_t slots = merge_indptr.back();
  {
    // units of one item are generated in page order
    std::vector<int32_t>& next = sc.next;
    next.assign(merge_items.size(), 0);
    for (size_t i = 0; i < num_units; ++i) {
      const int32_t sid = split_of[size_t(gen_item[i])];
      if (sid < 0) continue;
      gen[i].split = sid;
      gen[i].slot = merge_indptr[size_t(sid)] + next[size_t(sid)]++;
    }
  }

  // ---- per-CTA lists (generation order within a CTA)
  std::vector<int32_t>& work_indptr = sc.work_indptr;
  work_indptr.assign(size_t(C) + 1, 0);
  for (size_t i = 0; i < num_units; ++i) work_indptr[size_t(gen_cta[i]) + 1]++;
  for (int64_t i = 0; i < C; ++i) work_indptr[i + 1] += work_indptr[i];
  const Unit* unit_table = gen.data();  // decode: the cut emits units in CTA order
  if (decode) {
    // Within a CTA, the units of split items go first (stable): a CTA's
    // list holds at most two of them, the end of the item shared with the
    // previous CTA and the start of the one shared with the next, so both
    // pieces of every shared item run early on their CTAs and the merge
    // (by whichever finishes second) overlaps later units instead of
    // trailing the CTA's last one.
    split_units_first(gen, work_indptr, C, sc.units);
  } else {
    std::vector<Unit>& units = sc.units;
    units.resize(num_units);
    std::vector<int32_t>& at = sc.at;
    at.assign(work_indptr.begin(), work_indptr.end() - 1);
    for (size_t i = 0; i < num_units; ++i) units[size_t(at[size_t(gen_cta[i])]++)] = gen[i];
    unit_table = units.data();
  }
  int64_t max_load = 0;
  for (int64_t i = 0; i < C; ++i) max_load = std::max(max_load, load[size_t(i)]);

  // ---- write tables
  const int64_t S = int64_t(merge_items.size());
  const PlanLayout L = plan_layout(num_ctas, int64_t(num_units), S, slots, rows_per_item,
                                   head_dim);
  if (size_t(L.table_bytes) > host_bytes) {
    *msg = "attn_plan: pinned host workspace too small for the plan tables";
    return ATTN_ERR_WORKSPACE_TOO_SMALL;
  }
  char* hb = static_cast<char*>(host_tables);
  std::memset(hb, 0, size_t(L.table_bytes));
  std::memcpy(hb + L.off_work_indptr, work_indptr.data(), 4 * work_indptr.size());
  if (num_units) std::memcpy(hb + L.off_units, unit_table, sizeof(Unit) * num_units);
  std::memcpy(hb + L.off_merge_indptr, merge_indptr.data(), 4 * merge_indptr.size());
  if (S) std::memcpy(hb + L.off_merge_items, merge_items.data(), 16 * size_t(S));

  attn_plan_t p;
  std::memset(&p, 0, sizeof p);
  p.mode = decode ? ATTN_MODE_DECODE : ATTN_MODE_APPEND;
  p.batch = batch;
  p.page_size = page_size;
  p.num_qo_heads = num_qo_heads;
  p.num_kv_heads = num_kv_heads;
  p.head_dim = head_dim;
  p.causal = decode ? 0 : (causal ? 1 : 0);
  p.num_ctas = num_ctas;
  p.q_tile = q_tile;
  p.rows_per_item = rows_per_item;
  p.num_items = int32_t(items.size());
  p.num_units = int32_t(num_units);
  p.num_split_items = int32_t(S);
  p.num_slots = slots;
  p.total_qo = decode ? batch : (qo_indptr[batch] - qo_indptr[0]);
  p.max_qo_len = int32_t(max_qo_len);
  p.total_weight = W;
  p.max_cta_weight = max_load;
  p.off_work_indptr = L.off_work_indptr;
  p.off_units = L.off_units;
  p.off_merge_indptr = L.off_merge_indptr;
  p.off_merge_items = L.off_merge_items;
  p.off_counters = L.off_counters;
  p.off_partial_o = L.off_partial_o;
  p.off_partial_lse = L.off_partial_lse;
  p.table_bytes = L.table_bytes;
  p.dev_bytes_needed = L.dev_bytes;
  p.fingerprint = plan_fingerprint(qo_indptr, kv_indptr, last_page_len, batch, page_size,
                                   num_qo_heads, num_kv_heads, head_dim, p.causal, num_ctas);
  p.max_kv_len = max_kv_len;
  p.min_kv_minus_qo = min_kv_minus_qo;
  *plan = p;
  return ATTN_OK;
}

uint64_t cascade_fingerprint(const int32_t* qo_indptr, const int32_t* kv_indptr0,
                             const int32_t* last0, int32_t page_size0, const int32_t* kv_indptr1,
                             const int32_t* last1, int32_t page_size1, int32_t prompts,
                             int32_t num_qo_heads, int32_t num_kv_heads, int32_t head_dim,
                             int32_t num_ctas) {
  uint64_t h = plan_fingerprint(qo_indptr, kv_indptr0, last0, prompts, page_size0, num_qo_heads,
                                num_kv_heads, head_dim, 0, num_ctas);
  const int32_t B = prompts > 0 ? qo_indptr[prompts] : 0;
  h = fnv1a(h, kv_indptr1, 4 * (size_t(B) + 1));
  if (B) h = fnv1a(h, last1, 4 * size_t(B));
  return fnv1a(h, &page_size1, sizeof page_size1);
}

// Composable-format (cascade) plan: items are (prompt p, kv head hk); an
// item's segments are the prompt's shared prefix row (prefix table, page
// size P0) and then one suffix row per generation of the prompt (suffix
// table, page size P1). Weights are in tokens: a page weighs its page size,
// a segment adds kCascadeAlpha. The weights are laid end to end and CTA c
// takes the positions [floor(c W / C), floor((c+1) W / C)); a page belongs
// to the CTA that owns its first position, and the pages of a segment owned
// by one CTA form a unit; a segment without pages keeps one zero-page unit,
// owned by the CTA of its overhead position -- kept only when the whole
// item has no page. The units of one item on one CTA form a chain (one row
// state); an item on several CTAs is merged from one partial state per
// chain.
attn_status_t build_cascade_plan(const int32_t* qo_indptr, const int32_t* kv_indptr0,
                                 const int32_t* last0, int32_t page_size0,
                                 const int32_t* kv_indptr1, const int32_t* last1,
                                 int32_t page_size1, int32_t prompts, int32_t num_qo_heads,
                                 int32_t num_kv_heads, int32_t head_dim, int32_t num_ctas,
                                 void* host_tables, size_t host_bytes, attn_plan_t* plan,
                                 const char** msg) {
  *msg = "";
  if (!qo_indptr || !kv_indptr0 || !kv_indptr1 || !plan || !host_tables ||
      (prompts > 0 && !last0)) {
    *msg = "attn_plan_cascade: null pointer argument";
    return ATTN_ERR_INVALID_ARG;
  }
  if (prompts < 0 || page_size0 < 1 || page_size1 < 1 || num_qo_heads < 1 ||
      num_kv_heads < 1 || num_ctas < 1) {
    *msg = "attn_plan_cascade: sizes, page sizes, head counts and num_ctas must be positive";
    return ATTN_ERR_INVALID_ARG;
  }
  if (num_qo_heads % num_kv_heads != 0) {
    *msg = "attn_plan_cascade: num_qo_heads must be a multiple of num_kv_heads";
    return ATTN_ERR_INVALID_ARG;
  }
  if (head_dim != kHeadDim) {
    *msg = "attn_plan_cascade: only head_dim == 128 is implemented";
    return ATTN_ERR_UNSUPPORTED;
  }
  if (qo_indptr[0] != 0) {
    *msg = "attn_plan_cascade: qo_indptr must start at 0";
    return ATTN_ERR_INVALID_ARG;
  }
  const int32_t group = num_qo_heads / num_kv_heads;
  const int32_t B = qo_indptr[prompts];
  if (B > 0 && !last1) {
    *msg = "attn_plan_cascade: null pointer argument";
    return ATTN_ERR_INVALID_ARG;
  }
  int64_t max_n = 0, max_kv = 0, pages = 0;
  auto seg_len = [](const int32_t* indptr, const int32_t* last, int32_t P, int32_t r,
                    int64_t* n_pages, int64_t* kv_len) -> bool {
    const int64_t n = int64_t(indptr[r + 1]) - indptr[r];
    if (n < 0) return false;
    if (n > 0 && (last[r] < 1 || last[r] > P)) return false;
    *n_pages = n;
    *kv_len = n > 0 ? (n - 1) * P + last[r] : 0;
    return *kv_len <= INT32_MAX;
  };
  for (int32_t p = 0; p < prompts; ++p) {
    const int64_t n = int64_t(qo_indptr[p + 1]) - qo_indptr[p];
    if (n < 0) {
      *msg = "attn_plan_cascade: qo_indptr must be non-decreasing";
      return ATTN_ERR_INVALID_ARG;
    }
    max_n = std::max(max_n, n);
  }
  const int32_t rows = few_row_rows(group, int32_t(std::max<int64_t>(max_n, 1)));
  if (rows == 0) {
    *msg = "attn_plan_cascade: num_qo_heads / num_kv_heads x the generations of a prompt must "
           "be at most 16";
    return ATTN_ERR_UNSUPPORTED;
  }
  // segments in order: (item, segment) with their table row geometry
  struct Seg {
    int32_t item, r, kind, j;  // kind 0: prefix row r = p; 1: suffix row r, generation j
    int64_t n, kv_len;
    int32_t page_base;
  };
  std::vector<Seg> segs;
  std::vector<int4> item_of;  // (p, hk, qo_start, n_p)
  segs.reserve(size_t(B + prompts) * num_kv_heads);
  int64_t W = 0;
  for (int32_t p = 0; p < prompts; ++p) {
    const int32_t n_p = qo_indptr[p + 1] - qo_indptr[p];
    int64_t n0, len0;
    if (!seg_len(kv_indptr0, last0, page_size0, p, &n0, &len0)) {
      *msg = "attn_plan_cascade: bad prefix table (kv_indptr decreasing or last_page_len out "
             "of [1, page_size])";
      return ATTN_ERR_INVALID_ARG;
    }
    if (n_p == 0) continue;  // no generations, no rows
    max_kv = std::max(max_kv, len0);
    for (int32_t hk = 0; hk < num_kv_heads; ++hk) {
      const int32_t item = int32_t(item_of.size());
      item_of.push_back(make_int4(p, hk, qo_indptr[p], n_p));
      segs.push_back({item, p, 0, -1, n0, len0, kv_indptr0[p]});
      W += n0 * page_size0 + kCascadeAlpha;
      pages += n0;
      for (int32_t j = 0; j < n_p; ++j) {
        const int32_t b = qo_indptr[p] + j;
        int64_t n1, len1;
        if (!seg_len(kv_indptr1, last1, page_size1, b, &n1, &len1)) {
          *msg = "attn_plan_cascade: bad suffix table (kv_indptr decreasing or last_page_len "
                 "out of [1, page_size])";
          return ATTN_ERR_INVALID_ARG;
        }
        max_kv = std::max(max_kv, len1);
        segs.push_back({item, b, 1, j, n1, len1, kv_indptr1[b]});
        W += n1 * page_size1 + kCascadeAlpha;
        pages += n1;
      }
    }
  }
  const int64_t C = num_ctas;
  // floor(c W / C) without overflow for W < 2^62 / C, computed once
  std::vector<int64_t>& bounds = scratch().bounds;
  bounds.resize(size_t(C) + 1);
  for (int64_t c = 0; c <= C; ++c) bounds[size_t(c)] = (c * (W / C)) + (c * (W % C)) / C;
  auto bound = [&](int64_t c) -> int64_t { return bounds[size_t(c)]; };
  std::vector<int64_t> item_pages(item_of.size(), 0);
  for (const Seg& sg : segs) item_pages[size_t(sg.item)] += sg.n;
  // units in CTA order: the cut walks the segments in order, so the CTA
  // index never decreases
  std::vector<Unit> units;
  std::vector<int32_t> unit_cta, unit_item;
  units.reserve(segs.size() + size_t(C));
  int64_t base = 0;
  int64_t c = 0;
  auto owner = [&](int64_t pos) {
    while (c + 1 < C && bound(c + 1) <= pos) ++c;
    return c;
  };
  for (const Seg& sg : segs) {
    const int4 it = item_of[size_t(sg.item)];
    const int64_t P = sg.kind == 0 ? page_size0 : page_size1;
    auto emit = [&](int64_t p0, int64_t p1, int64_t cta) {
      Unit u;
      u.r = it.x;
      u.hk = it.y;
      u.t = sg.j;  // -1: prefix segment; j: generation j's suffix
      u.p0 = int32_t(p0);
      u.p1 = int32_t(p1);
      u.slot = -1;
      u.split = -1;
      u.page_base = sg.page_base;
      u.kv_len = int32_t(sg.kv_len);
      u.qo_start = it.z;
      u.qo_len = it.w;
      u.pad = sg.kind;
      units.push_back(u);
      unit_cta.push_back(int32_t(cta));
      unit_item.push_back(sg.item);
    };
    if (sg.n == 0) {
      // a segment without pages adds nothing; an item without any page
      // keeps one empty unit (its rows get O = 0, LSE = -inf)
      if (item_pages[size_t(sg.item)] == 0 && sg.kind == 0) emit(0, 0, owner(base));
    } else {
      // the pages of CTA `cur` are those before the first page whose
      // position reaches bound(cur + 1): jump from boundary to boundary
      int64_t k0 = 0;
      int64_t cur = owner(base + kCascadeAlpha);
      while (true) {
        int64_t k1 = sg.n;
        if (cur + 1 < C) {
          const int64_t rel = bound(cur + 1) - base - kCascadeAlpha;  // > k0 P
          k1 = std::min<int64_t>(sg.n, std::max<int64_t>(k0 + 1, (rel + P - 1) / P));
        }
        emit(k0, k1, cur);
        if (k1 >= sg.n) break;
        k0 = k1;
        cur = owner(base + kCascadeAlpha + k0 * P);
      }
    }
    base += sg.n * P + kCascadeAlpha;
  }
  // Chains: consecutive units of one item on one CTA run as one row state
  // (unit.pad bit 1: continues the previous unit, bit 2: continued by the
  // next). An item on several CTAs (one chain on each) is split: each chain
  // writes a partial state to its own slot, numbered in chain order, and
  // the last to finish merges them.
  const int64_t num_items = int64_t(item_of.size());
  const size_t nu = units.size();
  std::vector<int32_t> chain_of(nu), first_chain(static_cast<size_t>(num_items), -1),
      item_chains(static_cast<size_t>(num_items), 0);
  int32_t nchains = 0;
  for (size_t i = 0; i < nu; ++i) {
    const bool cont = i > 0 && unit_item[i] == unit_item[i - 1] && unit_cta[i] == unit_cta[i - 1];
    chain_of[i] = cont ? chain_of[i - 1] : nchains++;
    const size_t it = size_t(unit_item[i]);
    if (!cont) {
      if (first_chain[it] < 0) first_chain[it] = chain_of[i];
      item_chains[it]++;
    }
  }
  std::vector<int32_t> split_of(static_cast<size_t>(num_items), -1);
  std::vector<int32_t> merge_indptr(1, 0);
  std::vector<int4> merge_items;
  for (int64_t k = 0; k < num_items; ++k) {
    if (item_chains[size_t(k)] < 2) continue;
    split_of[size_t(k)] = int32_t(merge_items.size());
    const int4 it = item_of[size_t(k)];
    merge_items.push_back(make_int4(it.x, it.y, 0, item_chains[size_t(k)]));
    merge_indptr.push_back(merge_indptr.back() + item_chains[size_t(k)]);
  }
  for (size_t i = 0; i < nu; ++i) {
    const size_t it = size_t(unit_item[i]);
    const int32_t sid = split_of[it];
    units[i].split = sid;
    units[i].slot = sid < 0 ? -1 : merge_indptr[size_t(sid)] + (chain_of[i] - first_chain[it]);
    const bool cprev = i > 0 && chain_of[i - 1] == chain_of[i];
    const bool cnext = i + 1 < nu && chain_of[i + 1] == chain_of[i];
    units[i].pad |= (cprev ? 2 : 0) | (cnext ? 4 : 0);
  }
  std::vector<int32_t> work_indptr(size_t(C) + 1, 0);
  for (size_t i = 0; i < nu; ++i) work_indptr[size_t(unit_cta[i]) + 1]++;
  for (int64_t i = 0; i < C; ++i) work_indptr[size_t(i) + 1] += work_indptr[size_t(i)];
  // within a CTA, the chains of split items first (stable; chains stay whole)
  split_units_first(units, work_indptr, C, scratch().units);
  int64_t max_load = 0;
  for (int64_t i = 0; i < C; ++i) max_load = std::max(max_load, bound(i + 1) - bound(i));

  const int64_t S = int64_t(merge_items.size());
  const int64_t slots = merge_indptr.back();
  const PlanLayout L = plan_layout(num_ctas, int64_t(units.size()), S, slots, rows, head_dim);
  if (size_t(L.table_bytes) > host_bytes) {
    *msg = "attn_plan_cascade: pinned host workspace too small for the plan tables";
    return ATTN_ERR_WORKSPACE_TOO_SMALL;
  }
  char* hb = static_cast<char*>(host_tables);
  std::memset(hb, 0, size_t(L.table_bytes));
  std::memcpy(hb + L.off_work_indptr, work_indptr.data(), 4 * work_indptr.size());
  if (!units.empty()) std::memcpy(hb + L.off_units, units.data(), sizeof(Unit) * units.size());
  std::memcpy(hb + L.off_merge_indptr, merge_indptr.data(), 4 * merge_indptr.size());
  if (S) std::memcpy(hb + L.off_merge_items, merge_items.data(), 16 * size_t(S));

  attn_plan_t pl;
  std::memset(&pl, 0, sizeof pl);
  pl.mode = ATTN_MODE_CASCADE;
  pl.batch = prompts;
  pl.page_size = page_size0;
  pl.page_size_suffix = page_size1;
  pl.num_qo_heads = num_qo_heads;
  pl.num_kv_heads = num_kv_heads;
  pl.head_dim = head_dim;
  pl.causal = 0;
  pl.num_ctas = num_ctas;
  pl.q_tile = int32_t(max_n);
  pl.rows_per_item = rows;
  pl.num_items = int32_t(num_items);
  pl.num_units = int32_t(units.size());
  pl.num_split_items = int32_t(S);
  pl.num_slots = int32_t(slots);
  pl.total_qo = B;
  pl.max_qo_len = int32_t(max_n);
  pl.total_weight = pages + num_items;
  pl.max_cta_weight = max_load;
  pl.off_work_indptr = L.off_work_indptr;
  pl.off_units = L.off_units;
  pl.off_merge_indptr = L.off_merge_indptr;
  pl.off_merge_items = L.off_merge_items;
  pl.off_counters = L.off_counters;
  pl.off_partial_o = L.off_partial_o;
  pl.off_partial_lse = L.off_partial_lse;
  pl.table_bytes = L.table_bytes;
  pl.dev_bytes_needed = L.dev_bytes;
  pl.fingerprint = cascade_fingerprint(qo_indptr, kv_indptr0, last0, page_size0, kv_indptr1,
                                       last1, page_size1, prompts, num_qo_heads, num_kv_heads,
                                       head_dim, num_ctas);
  pl.max_kv_len = max_kv;
  pl.min_kv_minus_qo = INT64_MAX;
  *plan = pl;
  return ATTN_OK;
}

}  // namespace attn
