"""Reference work partitioner (plan) -- TEST INFRASTRUCTURE ONLY.

Restates, in plain Python, the CPU planning phase of the FlashInfer scheduler
(modb.pro digest, section "动态负载均衡调度": a Stream-K inspired planner that
analyses the length distribution on the CPU and assigns work units to SMs so
that a fixed-grid persistent kernel can follow the plan). The digest gives no
pseudo-code; the exact cut below is the reading used throughout this project:

  items      (request r, kv head hk, query tile t), r-major, then hk, then t;
             decode has one tile per request, append tiles hold
             tq = 256 // group query tokens (group heads x tq tokens = 256 packed
             rows: two 128-row MMA tiles), group must divide 128
  weights    an item costs its pages n plus alpha (its unit's start and end,
             in pages): alpha = 1 in plans of the few-row kernel (decode, and
             appends whose requests all have at most 16 query rows), 16 in
             plans of the append kernel
  decode     the costs w = n + alpha are laid end to end (total W) and CTA c
             takes the positions [floor(c W / C), floor((c+1) W / C)); inside
             an item at base b, position b is its overhead slot and b + alpha
             + k is page k; an intersection without pages is dropped, except
             that an item with n = 0 keeps one zero-page unit, owned by the CTA
             that owns b
  append     the items of requests with at most 16 query rows (group x
             qo_len: "decode-like") and the other items keep their own order
             and are interleaved by weight (next from the class with the
             smaller fraction of its total weight done, ties to the
             non-decode-like class); in that order items go to the CTA with
             the least cost so far (ties: lowest index), each CTA capped at
             ceil(W / C) + alpha; an item that does not fit is cut at the cap
             (the unit takes the cap minus alpha in pages) and its rest
             continues on the next CTA
  slots      items with >= 2 units are split; their units get partial-state
             slots numbered in (item, page) order; merge_indptr lists them.
  order      decode: within each CTA's list the units of split items come
             first, the others after them, each group in cut order.

  cascade    composable formats in one launch: make_cascade_plan below.

It is written independently of the library's C++ planner; the tests require
the two to agree bit for bit.
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import List, Optional, Sequence

ALPHA = 1           # few-row kernel plans: cost of a unit beyond its pages
APPEND_ALPHA = 16   # append-kernel plans (long appends, POD batches)
ITEM_ROWS = 256
FEW_ROWS = 16


@dataclass
class Plan:
    work_indptr: List[int]
    unit_r: List[int] = field(default_factory=list)
    unit_hk: List[int] = field(default_factory=list)
    unit_t: List[int] = field(default_factory=list)
    unit_p0: List[int] = field(default_factory=list)
    unit_p1: List[int] = field(default_factory=list)
    unit_slot: List[int] = field(default_factory=list)
    merge_indptr: List[int] = field(default_factory=lambda: [0])
    merge_r: List[int] = field(default_factory=list)
    merge_hk: List[int] = field(default_factory=list)
    merge_t: List[int] = field(default_factory=list)
    total_weight: int = 0
    num_items: int = 0
    q_tile: int = 1


def kv_length(kv_indptr: Sequence[int], last_page_len: Sequence[int], page_size: int,
              r: int) -> int:
    n = kv_indptr[r + 1] - kv_indptr[r]
    return 0 if n <= 0 else (n - 1) * page_size + last_page_len[r]


def make_plan(kv_indptr: Sequence[int], last_page_len: Sequence[int], page_size: int,
              num_qo_heads: int, num_kv_heads: int, num_ctas: int,
              qo_indptr: Optional[Sequence[int]] = None, causal: bool = False) -> Plan:
    batch = len(kv_indptr) - 1
    group = num_qo_heads // num_kv_heads
    decode = qo_indptr is None
    tq = 1 if decode else ITEM_ROWS // group

    # 1. items, their page counts and their class
    items = []  # (r, hk, t, n)
    few = []    # the request has at most FEW_ROWS query rows
    for r in range(batch):
        kv_len = kv_length(kv_indptr, last_page_len, page_size, r)
        qo_len = 1 if decode else qo_indptr[r + 1] - qo_indptr[r]
        tiles = 1 if decode else -(-qo_len // tq)
        for hk in range(num_kv_heads):
            for t in range(tiles):
                vis = kv_len
                if causal and not decode:
                    last_row = min((t + 1) * tq, qo_len) - 1
                    vis = min(kv_len, max(0, kv_len - qo_len + last_row + 1))
                items.append((r, hk, t, -(-vis // page_size)))
                few.append(group * qo_len <= FEW_ROWS)

    # 2. weights
    alpha = ALPHA if (decode or all(few)) else APPEND_ALPHA  # all(few): the few-row kernel runs it
    weight = [it[3] + alpha for it in items]
    total = sum(weight)
    C = num_ctas
    plan = Plan(work_indptr=[0] * (C + 1), total_weight=total, num_items=len(items),
                q_tile=tq)
    per_cta_units = [[] for _ in range(C)]  # [item index, r, hk, t, p0, p1]

    if decode:
        # 3a. contiguous equal cut of the cost line
        def lo(c):
            return (c * total) // C

        base = 0
        for k, (r, hk, t, n) in enumerate(items):
            w = n + alpha
            for c in range(C):
                a, e = lo(c), lo(c + 1)
                if e <= base or a >= base + w:
                    continue
                if n == 0:
                    if a <= base < e:
                        per_cta_units[c].append([k, r, hk, t, 0, 0])
                    continue
                p0 = max(0, a - base - alpha)
                p1 = min(n, e - base - alpha)
                if p1 > p0:
                    per_cta_units[c].append([k, r, hk, t, p0, p1])
            base += w
    else:
        # 3b. interleave the two classes by weight, then the time-ordered fill
        import heapq
        dense = [k for k in range(len(items)) if not few[k]]
        light = [k for k in range(len(items)) if few[k]]
        wd = sum(weight[k] for k in dense)
        wf = sum(weight[k] for k in light)
        order, i, j, dd, df = [], 0, 0, 0, 0
        while i < len(dense) or j < len(light):
            # class fractions done: dd / wd against df / wf (cross-multiplied)
            if j >= len(light) or (i < len(dense) and dd * wf <= df * wd):
                order.append(dense[i])
                dd += weight[dense[i]]
                i += 1
            else:
                order.append(light[j])
                df += weight[light[j]]
                j += 1
        cap = -(-total // C) + alpha
        ready = [(0, c) for c in range(C)]
        heapq.heapify(ready)
        for k in order:
            r, hk, t, n = items[k]
            p = 0
            while True:
                used, c = heapq.heappop(ready)
                avail = cap - used
                need = alpha + (n - p)
                if need <= avail:
                    per_cta_units[c].append([k, r, hk, t, p, n])
                    if used + need < cap:
                        heapq.heappush(ready, (used + need, c))
                    break
                take = avail - alpha
                if take > 0:
                    per_cta_units[c].append([k, r, hk, t, p, p + take])
                    p += take

    flat = []
    for c in range(C):
        plan.work_indptr[c + 1] = plan.work_indptr[c] + len(per_cta_units[c])
        flat.extend(per_cta_units[c])

    # 4. split items and slot numbering in (item, page) order
    count = {}
    for u in flat:
        count[u[0]] = count.get(u[0], 0) + 1
    order = sorted(range(len(flat)), key=lambda i: (flat[i][0], flat[i][4]))
    slot_of = [-1] * len(flat)
    next_slot = 0
    last_item = None
    for i in order:
        k = flat[i][0]
        if count[k] < 2:
            continue
        if k != last_item:
            plan.merge_r.append(flat[i][1])
            plan.merge_hk.append(flat[i][2])
            plan.merge_t.append(flat[i][3])
            if last_item is not None:
                plan.merge_indptr.append(next_slot)
            last_item = k
        slot_of[i] = next_slot
        next_slot += 1
    if last_item is not None:
        plan.merge_indptr.append(next_slot)

    if decode:
        # split-item units first within each CTA (stable)
        reordered, slot_re = [], []
        for c in range(C):
            idx = list(range(plan.work_indptr[c], plan.work_indptr[c + 1]))
            first = [i for i in idx if slot_of[i] >= 0]
            rest = [i for i in idx if slot_of[i] < 0]
            for i in first + rest:
                reordered.append(flat[i])
                slot_re.append(slot_of[i])
        flat, slot_of = reordered, slot_re

    for i, u in enumerate(flat):
        plan.unit_r.append(u[1])
        plan.unit_hk.append(u[2])
        plan.unit_t.append(u[3])
        plan.unit_p0.append(u[4])
        plan.unit_p1.append(u[5])
        plan.unit_slot.append(slot_of[i])
    return plan


CASCADE_ALPHA = 16  # tokens of overhead per segment


def few_rows(group: int, max_rows: int) -> int:
    """Rows of one few-row item: the smallest power of two >= group x
    max_rows, at most FEW_ROWS (0 if it does not fit)."""
    need = group * max(max_rows, 1)
    r = 1
    while r <= FEW_ROWS:
        if need <= r:
            return r
        r *= 2
    return 0


def make_cascade_plan(qo_indptr: Sequence[int], kv_indptr_prefix: Sequence[int],
                      last_prefix: Sequence[int], page_size_prefix: int,
                      kv_indptr_suffix: Sequence[int], last_suffix: Sequence[int],
                      page_size_suffix: int, num_qo_heads: int, num_kv_heads: int,
                      num_ctas: int) -> Plan:
    """Composable formats in one launch (modb.pro digest, "可组合格式": a shared
    prefix stored once, per-generation suffixes in a second table, partial
    states combined by log-sum-exp). Reading used:

      items      (prompt p, kv head hk) for prompts with generations, p-major
      segments   per item: the prompt's prefix row (t = -1), then the suffix
                 row of each generation j (t = j), in that order
      weight     a segment weighs pages x page size + 16 tokens; laid end to
                 end (total W), CTA c owns positions [floor(c W / C),
                 floor((c+1) W / C)); page k of a segment at base b sits at
                 position b + 16 + k P and belongs to the CTA owning it; the
                 pages of a segment on one CTA form a unit; segments without
                 pages give no unit, except that an item with no page at all
                 keeps one empty prefix unit, on the CTA owning its base
      chains     consecutive units of one item on one CTA; flags: continues
                 the previous unit (2), continued by the next (4), OR-ed
                 into the kind (0 prefix, 1 suffix)
      slots      items with >= 2 chains are split: one slot per chain, in
                 chain order
      order      within a CTA, the units of split items first, each group in
                 cut order

    Extra fields: unit_kind (kind | flags), unit_page_base, unit_kv_len,
    unit_qo_start, unit_qo_len, unit_split; merge_count per split item;
    rows_per_item.
    """
    import bisect
    prompts = len(qo_indptr) - 1
    group = num_qo_heads // num_kv_heads
    C = num_ctas

    def length(indptr, last, P, row):
        n = indptr[row + 1] - indptr[row]
        return n, (0 if n == 0 else (n - 1) * P + last[row])

    segs = []  # (item, p, hk, t, kind, n, kv_len, page_base, P)
    items = []
    max_n = max([qo_indptr[p + 1] - qo_indptr[p] for p in range(prompts)] + [0])
    for p in range(prompts):
        n_p = qo_indptr[p + 1] - qo_indptr[p]
        if n_p == 0:
            continue
        for hk in range(num_kv_heads):
            it = len(items)
            items.append((p, hk))
            n, kv = length(kv_indptr_prefix, last_prefix, page_size_prefix, p)
            segs.append((it, p, hk, -1, 0, n, kv, kv_indptr_prefix[p], page_size_prefix))
            for j in range(n_p):
                b = qo_indptr[p] + j
                n, kv = length(kv_indptr_suffix, last_suffix, page_size_suffix, b)
                segs.append((it, p, hk, j, 1, n, kv, kv_indptr_suffix[b], page_size_suffix))
    item_pages = [0] * len(items)
    for sg in segs:
        item_pages[sg[0]] += sg[5]
    W = sum(s_[5] * s_[8] + CASCADE_ALPHA for s_ in segs)
    bounds = [(c * W) // C for c in range(C)]

    def owner(pos):  # the last CTA whose range starts at or before pos
        return bisect.bisect_right(bounds, pos) - 1

    gen = []  # units in cut order, with their CTA
    base = 0
    for (it, p, hk, t, kind, n, kv, pb, P) in segs:
        rec = dict(item=it, r=p, hk=hk, t=t, kind=kind, kv_len=kv, page_base=pb,
                   qo_start=qo_indptr[p], qo_len=qo_indptr[p + 1] - qo_indptr[p])
        if n == 0:
            if item_pages[it] == 0 and kind == 0:
                gen.append(dict(rec, p0=0, p1=0, cta=owner(base)))
        else:
            owners = [owner(base + CASCADE_ALPHA + k * P) for k in range(n)]
            k0 = 0
            for k in range(1, n + 1):
                if k == n or owners[k] != owners[k0]:
                    gen.append(dict(rec, p0=k0, p1=k, cta=owners[k0]))
                    k0 = k
        base += n * P + CASCADE_ALPHA

    # chains and their slots
    chain = []
    for i, u in enumerate(gen):
        same = i > 0 and gen[i - 1]["item"] == u["item"] and gen[i - 1]["cta"] == u["cta"]
        chain.append(chain[-1] if same else (chain[-1] + 1 if chain else 0))
    chains_of_item = {}
    for i, u in enumerate(gen):
        lst = chains_of_item.setdefault(u["item"], [])
        if chain[i] not in lst:
            lst.append(chain[i])
    plan = Plan(work_indptr=[0] * (C + 1), num_items=len(items), q_tile=max_n)
    plan.merge_indptr = [0]
    plan.merge_count = []
    split_of = {}
    for k in range(len(items)):
        lst = chains_of_item.get(k, [])
        if len(lst) < 2:
            continue
        split_of[k] = len(plan.merge_count)
        plan.merge_r.append(items[k][0])
        plan.merge_hk.append(items[k][1])
        plan.merge_t.append(0)
        plan.merge_count.append(len(lst))
        plan.merge_indptr.append(plan.merge_indptr[-1] + len(lst))
    for i, u in enumerate(gen):
        sid = split_of.get(u["item"], -1)
        u["split"] = sid
        u["slot"] = -1 if sid < 0 else \
            plan.merge_indptr[sid] + chains_of_item[u["item"]].index(chain[i])
        flags = (2 if i > 0 and chain[i - 1] == chain[i] else 0) | \
                (4 if i + 1 < len(gen) and chain[i + 1] == chain[i] else 0)
        u["flags"] = flags

    per_cta = [[] for _ in range(C)]
    for u in gen:
        per_cta[u["cta"]].append(u)
    flat = []
    for c in range(C):
        lst = [u for u in per_cta[c] if u["slot"] >= 0] + [u for u in per_cta[c] if u["slot"] < 0]
        plan.work_indptr[c + 1] = plan.work_indptr[c] + len(lst)
        flat.extend(lst)
    plan.unit_kind, plan.unit_page_base, plan.unit_kv_len = [], [], []
    plan.unit_qo_start, plan.unit_qo_len, plan.unit_split = [], [], []
    for u in flat:
        plan.unit_r.append(u["r"])
        plan.unit_hk.append(u["hk"])
        plan.unit_t.append(u["t"])
        plan.unit_p0.append(u["p0"])
        plan.unit_p1.append(u["p1"])
        plan.unit_slot.append(u["slot"])
        plan.unit_split.append(u["split"])
        plan.unit_kind.append(u["kind"] | u["flags"])
        plan.unit_page_base.append(u["page_base"])
        plan.unit_kv_len.append(u["kv_len"])
        plan.unit_qo_start.append(u["qo_start"])
        plan.unit_qo_len.append(u["qo_len"])
    plan.total_weight = sum(s_[5] for s_ in segs) + len(items)
    plan.rows_per_item = few_rows(group, max_n)
    return plan
