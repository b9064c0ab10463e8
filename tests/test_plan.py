"""The library's C++ planner against the reference partitioner (bit-exact) and
against the properties the balanced cut must have. Host only: no GPU."""
import numpy as np
import pytest

from oracle import plan_ref

C = pytest.importorskip("paged_kv_attention_bsr_gb300._capi")


def _tables(p, buf):
    raw = np.frombuffer(buf.tobytes(), dtype=np.int32)

    def at(off, n):
        return raw[off // 4: off // 4 + n]

    units = at(p.off_units, 12 * p.num_units).reshape(-1, 12)
    return {
        "work_indptr": at(p.off_work_indptr, p.num_ctas + 1).tolist(),
        "units": units,
        "merge_indptr": at(p.off_merge_indptr, p.num_split_items + 1).tolist(),
        "merge_items": at(p.off_merge_items, 4 * p.num_split_items).reshape(-1, 4),
    }


def _lib_plan(kv_indptr, last, P, Hq, Hk, ctas, qo_indptr=None, causal=False):
    B = len(kv_indptr) - 1
    total_qo = int(qo_indptr[-1]) if qo_indptr is not None else B
    _, host = C.workspace_size(max(B, 1), max(total_qo, 1), Hq, Hk, 128, ctas)
    buf = np.zeros(host, np.uint8)
    p = C.plan(qo_indptr, kv_indptr, last, P, Hq, Hk, 128, causal, ctas, buf)
    return p, _tables(p, buf), buf


def _random_case(rng, decode):
    B = int(rng.integers(0, 40))
    P = int(rng.choice([1, 3, 16, 128]))
    Hk = int(rng.choice([1, 2, 8]))
    g = int(rng.choice([1, 2, 4, 8]))
    kv_lens = rng.integers(0, 3000, size=B)
    if B and rng.random() < 0.3:
        kv_lens[rng.integers(0, B)] = 0
    n = (kv_lens + P - 1) // P
    kv_indptr = np.concatenate([[0], np.cumsum(n)]).astype(np.int32)
    last = np.where(n > 0, kv_lens - P * (n - 1), 0).astype(np.int32)
    qo = None
    causal = False
    if not decode:
        causal = bool(rng.random() < 0.6)
        qo_lens = np.minimum(rng.integers(0, 600, size=B), kv_lens) if causal else \
            rng.integers(0, 600, size=B)
        qo = np.concatenate([[0], np.cumsum(qo_lens)]).astype(np.int32)
    ctas = int(rng.choice([1, 2, 7, 152, 304, 5000]))
    return kv_indptr, last, P, Hk * g, Hk, ctas, qo, causal


@pytest.mark.parametrize("decode", [True, False])
def test_plan_bit_exact_vs_reference(decode):
    rng = np.random.default_rng(20260002 if decode else 20260005)
    for _ in range(60):
        kv_indptr, last, P, Hq, Hk, ctas, qo, causal = _random_case(rng, decode)
        p, t, _ = _lib_plan(kv_indptr, last, P, Hq, Hk, ctas, qo, causal)
        ref = plan_ref.make_plan(kv_indptr.tolist(), last.tolist(), P, Hq, Hk, ctas,
                                 qo_indptr=None if qo is None else qo.tolist(), causal=causal)
        assert t["work_indptr"] == ref.work_indptr
        u = t["units"]
        assert u[:, 0].tolist() == ref.unit_r
        assert u[:, 1].tolist() == ref.unit_hk
        assert u[:, 2].tolist() == ref.unit_t
        assert u[:, 3].tolist() == ref.unit_p0
        assert u[:, 4].tolist() == ref.unit_p1
        assert u[:, 5].tolist() == ref.unit_slot
        assert t["merge_indptr"] == ref.merge_indptr
        mi = t["merge_items"]
        assert mi[:, 0].tolist() == ref.merge_r
        assert mi[:, 1].tolist() == ref.merge_hk
        assert mi[:, 2].tolist() == ref.merge_t
        assert p.total_weight == ref.total_weight
        assert p.num_items == ref.num_items
        assert p.q_tile == ref.q_tile
        # the request geometry the planner copies into every unit record
        for row in u:
            r = int(row[0])
            assert row[7] == kv_indptr[r]
            assert row[8] == plan_ref.kv_length(kv_indptr.tolist(), last.tolist(), P, r)
            if qo is None:
                assert (row[9], row[10]) == (r, 1)
            else:
                assert (row[9], row[10]) == (qo[r], qo[r + 1] - qo[r])


def _pages_of_items(kv_indptr, last, P, Hk, g, qo, causal):
    items = {}
    B = len(kv_indptr) - 1
    tq = 1 if qo is None else 256 // g
    for r in range(B):
        kv_len = plan_ref.kv_length(kv_indptr, last, P, r)
        qo_len = 1 if qo is None else qo[r + 1] - qo[r]
        tiles = 1 if qo is None else -(-qo_len // tq)
        for hk in range(Hk):
            for t in range(tiles):
                vis = kv_len
                if causal and qo is not None:
                    vis = min(kv_len, kv_len - qo_len + min((t + 1) * tq, qo_len))
                items[(r, hk, t)] = -(-vis // P)
    return items


@pytest.mark.parametrize("decode", [True, False])
def test_plan_properties(decode):
    rng = np.random.default_rng(7 + decode)
    for _ in range(60):
        kv_indptr, last, P, Hq, Hk, ctas, qo, causal = _random_case(rng, decode)
        p, t, buf = _lib_plan(kv_indptr, last, P, Hq, Hk, ctas, qo, causal)
        items = _pages_of_items(kv_indptr.tolist(), last.tolist(), P, Hk, Hq // Hk,
                                None if qo is None else qo.tolist(), causal)
        u = t["units"]
        # exact coverage: every page of every item exactly once, in order
        covered = {}
        for row in u:
            key = (int(row[0]), int(row[1]), int(row[2]))
            covered.setdefault(key, []).append((int(row[3]), int(row[4])))
        assert set(covered) == set(items)
        for key, n in items.items():
            segs = sorted(covered[key])
            if n == 0:
                assert segs == [(0, 0)]
                continue
            assert segs[0][0] == 0 and segs[-1][1] == n
            for (a0, a1), (b0, b1) in zip(segs, segs[1:]):
                assert a1 == b0 and a0 < a1
        # weights: pages + alpha per item (1 for the few-row kernel's plans:
        # decode and short appends; 16 for the append kernel's)
        alpha = 1 if qo is None or (Hq // Hk) * int(np.diff(qo).max()) <= 16 else 16
        assert p.total_weight == sum(n + alpha for n in items.values())
        # balance: the page share of every CTA is at most ceil(W / C)
        W = p.total_weight
        wi = t["work_indptr"]
        cap = -(-W // ctas)
        for c in range(ctas):
            pages = int((u[wi[c]:wi[c + 1], 4] - u[wi[c]:wi[c + 1], 3]).sum())
            assert pages <= cap
        assert p.max_cta_weight <= cap + (0 if qo is None else alpha)
        # the cut adds at most C - 1 units (decode) / C units (append);
        # split items carry slots in order
        extra = ctas - 1 if qo is None else ctas
        assert p.num_units - p.num_items <= extra
        assert p.num_split_items <= extra
        slots = [int(s) for s in u[:, 5] if s >= 0]
        assert sorted(slots) == list(range(len(slots)))
        if qo is None:  # decode units are already in (item, page) order
            assert slots == list(range(len(slots)))
        by_item = {}
        for row in u:
            if row[5] >= 0:
                by_item.setdefault((int(row[0]), int(row[1]), int(row[2])), []).append(
                    (int(row[3]), int(row[5])))
        for segs in by_item.values():
            segs.sort()
            assert [s for _, s in segs] == list(range(segs[0][1], segs[0][1] + len(segs)))
        assert p.num_slots == len(slots)
        # identical bytes run to run
        p2, _, buf2 = _lib_plan(kv_indptr, last, P, Hq, Hk, ctas, qo, causal)
        assert bytes(buf[:p.table_bytes]) == bytes(buf2[:p2.table_bytes])
        assert p.fingerprint == p2.fingerprint


def test_plan_skewed_workload_balance():
    """The skewed 70B-shaped batch: 4 x 32k + 124 lognormal requests."""
    from paged_kv_attention_bsr_gb300 import synth
    rng = np.random.default_rng(20260003)
    lens = synth.skewed_lengths(rng)
    n = (lens + 15) // 16
    kv_indptr = np.concatenate([[0], np.cumsum(n)]).astype(np.int32)
    last = (lens - 16 * (n - 1)).astype(np.int32)
    p, t, _ = _lib_plan(kv_indptr, last, 16, 64, 8, 304)
    assert p.max_cta_weight - p.total_weight // 304 <= 1
    assert p.num_units <= p.num_items + 303


@pytest.mark.parametrize("bad", ["heads", "lpl_zero", "lpl_big", "indptr", "causal_short",
                                 "head_dim", "group", "pinned"])
def test_plan_rejects_bad_input(bad):
    kv_indptr = np.array([0, 2, 5], np.int32)
    last = np.array([3, 16], np.int32)
    qo = None
    Hq, Hk, D, P, causal = 8, 2, 128, 16, False
    host = 1 << 20
    want = C.ERR_INVALID_ARG
    if bad == "heads":
        Hq = 6
        Hk = 4
    elif bad == "lpl_zero":
        last = np.array([0, 16], np.int32)
    elif bad == "lpl_big":
        last = np.array([17, 16], np.int32)
    elif bad == "indptr":
        kv_indptr = np.array([0, 5, 2], np.int32)
    elif bad == "causal_short":
        qo = np.array([0, 40, 41], np.int32)
        causal = True
    elif bad == "head_dim":
        D = 64
        want = C.ERR_UNSUPPORTED
    elif bad == "group":
        Hq, Hk = 32, 2
        want = C.ERR_UNSUPPORTED
    elif bad == "pinned":
        host = 64
        want = C.ERR_WORKSPACE_TOO_SMALL
    buf = np.zeros(host, np.uint8)
    with pytest.raises(C.AttnError) as ei:
        C.plan(qo, kv_indptr, last, P, Hq, Hk, D, causal, 16, buf)
    assert ei.value.status == want
    assert C.last_error()


@pytest.mark.parametrize("decode", [True, False])
def test_plan_length_summaries(decode):
    """max_kv_len and min_kv_minus_qo (what the RoPE entry points check
    against) follow from the page tables: kv_len = (n - 1) P + last."""
    rng = np.random.default_rng(20260011 if decode else 20260012)
    for _ in range(40):
        kv_indptr, last, P, Hq, Hk, ctas, qo, causal = _random_case(rng, decode)
        p, _, _ = _lib_plan(kv_indptr, last, P, Hq, Hk, ctas, qo, causal)
        n = np.diff(kv_indptr.astype(np.int64))
        kv_len = np.where(n > 0, (n - 1) * P + last, 0)
        qo_len = np.ones_like(kv_len) if qo is None else np.diff(qo.astype(np.int64))
        assert p.max_kv_len == (int(kv_len.max()) if len(kv_len) else 0)
        has_kv = kv_len > 0
        want = int((kv_len - qo_len)[has_kv].min()) if has_kv.any() else np.iinfo(np.int64).max
        assert p.min_kv_minus_qo == want


def test_plan_mixed_prefill_and_decode_batch():
    """A batch of long prefill chunks and single-token decodes in one append
    plan (POD-style): bit-exact against the reference, the decode-like items
    spread through every part of the visiting order, and the two classes'
    weights interleaved so that no CTA list is all of one kind at its start."""
    rng = np.random.default_rng(20260020)
    for ctas in (7, 152):
        qo_lens = np.concatenate([rng.integers(128, 1024, 6), np.ones(40, np.int64)])
        perm = rng.permutation(len(qo_lens))
        qo_lens = qo_lens[perm]
        kv_lens = qo_lens + rng.integers(0, 4000, len(qo_lens))
        n = (kv_lens + 15) // 16
        kv_indptr = np.concatenate([[0], np.cumsum(n)]).astype(np.int32)
        last = (kv_lens - 16 * (n - 1)).astype(np.int32)
        qo = np.concatenate([[0], np.cumsum(qo_lens)]).astype(np.int32)
        p, t, _ = _lib_plan(kv_indptr, last, 16, 32, 8, ctas, qo, True)
        ref = plan_ref.make_plan(kv_indptr.tolist(), last.tolist(), 16, 32, 8, ctas,
                                 qo_indptr=qo.tolist(), causal=True)
        assert t["work_indptr"] == ref.work_indptr
        u = t["units"]
        assert u[:, 0].tolist() == ref.unit_r and u[:, 3].tolist() == ref.unit_p0
        assert u[:, 4].tolist() == ref.unit_p1 and u[:, 5].tolist() == ref.unit_slot
        # decode requests (qo_len 1) are spread over the CTAs and through
        # their lists (interleaved with the prefill tiles, not all at the end)
        decode_r = set(np.nonzero(qo_lens == 1)[0].tolist())
        wi = t["work_indptr"]
        holders, pos = 0, []
        for c in range(ctas):
            rs = [int(x) for x in u[wi[c]:wi[c + 1], 0]]
            at = [i / max(len(rs) - 1, 1) for i, r in enumerate(rs) if r in decode_r]
            holders += bool(at)
            pos.extend(at)
        assert holders >= ctas // 2
        assert 0.3 <= float(np.mean(pos)) <= 0.7


def _random_cascade(rng):
    prompts = int(rng.integers(0, 12))
    Hk = int(rng.choice([1, 2, 8]))
    g = int(rng.choice([1, 2, 4, 8, 16]))
    max_n = 16 // g
    n = rng.integers(0, max_n + 1, size=prompts)
    qo = np.concatenate([[0], np.cumsum(n)]).astype(np.int32)
    B = int(qo[-1])
    P0 = int(rng.choice([16, 64, 128]))
    P1 = int(rng.choice([16, 32]))

    def table(lens, P):
        pages = (lens + P - 1) // P
        ip = np.concatenate([[0], np.cumsum(pages)]).astype(np.int32)
        last = np.where(pages > 0, lens - P * (pages - 1), 0).astype(np.int32)
        return ip, last

    pre_lens = rng.integers(0, 9000, size=prompts)
    if prompts and rng.random() < 0.3:
        pre_lens[rng.integers(0, prompts)] = 0
    suf_lens = rng.integers(0, 1500, size=B)
    if B and rng.random() < 0.3:
        suf_lens[rng.integers(0, B)] = 0
    ip0, l0 = table(pre_lens, P0)
    ip1, l1 = table(suf_lens, P1)
    ctas = int(rng.choice([1, 3, 152, 304, 3000]))
    return qo, ip0, l0, P0, ip1, l1, P1, Hk * g, Hk, ctas


def _lib_cascade(qo, ip0, l0, P0, ip1, l1, P1, Hq, Hk, ctas):
    prompts = len(qo) - 1
    _, host = C.cascade_workspace_size(max(prompts, 1), int(qo[-1]), Hq, Hk, 128, ctas)
    buf = np.zeros(host, np.uint8)
    p = C.plan_cascade(qo, ip0, l0, P0, ip1, l1, P1, Hq, Hk, 128, ctas, buf)
    return p, _tables(p, buf)


def test_cascade_plan_bit_exact_vs_reference():
    rng = np.random.default_rng(20260011)
    for _ in range(80):
        case = _random_cascade(rng)
        qo, ip0, l0, P0, ip1, l1, P1, Hq, Hk, ctas = case
        p, t = _lib_cascade(*case)
        ref = plan_ref.make_cascade_plan(qo.tolist(), ip0.tolist(), l0.tolist(), P0,
                                         ip1.tolist(), l1.tolist(), P1, Hq, Hk, ctas)
        assert p.mode == C.MODE_CASCADE and p.page_size == P0 and p.page_size_suffix == P1
        assert t["work_indptr"] == ref.work_indptr
        u = t["units"]
        cols = (ref.unit_r, ref.unit_hk, ref.unit_t, ref.unit_p0, ref.unit_p1, ref.unit_slot,
                ref.unit_split, ref.unit_page_base, ref.unit_kv_len, ref.unit_qo_start,
                ref.unit_qo_len, ref.unit_kind)
        for k, col in enumerate(cols):
            assert u[:, k].tolist() == col, k
        assert t["merge_indptr"] == ref.merge_indptr
        mi = t["merge_items"]
        assert mi[:, 0].tolist() == ref.merge_r
        assert mi[:, 1].tolist() == ref.merge_hk
        assert mi[:, 3].tolist() == ref.merge_count
        assert p.total_weight == ref.total_weight
        assert p.num_items == ref.num_items
        assert p.num_split_items == len(ref.merge_count)
        assert p.q_tile == ref.q_tile
        assert p.rows_per_item == ref.rows_per_item
        assert p.num_units == len(ref.unit_r)
        assert p.num_slots == ref.merge_indptr[-1]


def test_cascade_plan_covers_every_page_once_and_balances():
    rng = np.random.default_rng(20260012)
    for _ in range(40):
        case = _random_cascade(rng)
        qo, ip0, l0, P0, ip1, l1, P1, Hq, Hk, ctas = case
        p, t = _lib_cascade(*case)
        u = t["units"]
        prompts = len(qo) - 1
        # every page of every segment exactly once, in one unit per CTA visit
        seen = {}
        for row in u:
            r, hk, tt, p0, p1 = (int(x) for x in row[:5])
            key = (r, hk, tt)
            seen.setdefault(key, []).append((p0, p1))
        for pp in range(prompts):
            n_p = int(qo[pp + 1] - qo[pp])
            if n_p == 0:
                assert not any(k[0] == pp for k in seen)
                continue
            for hk in range(Hk):
                for tt in range(-1, n_p):
                    ip = ip0 if tt < 0 else ip1
                    row_i = pp if tt < 0 else int(qo[pp]) + tt
                    n = int(ip[row_i + 1] - ip[row_i])
                    spans = sorted(seen.get((pp, hk, tt), []))
                    if n == 0:
                        assert spans in ([], [(0, 0)])
                        continue
                    assert spans[0][0] == 0 and spans[-1][1] == n
                    for a, b in zip(spans, spans[1:]):
                        assert a[1] == b[0]
        # an item with no page at all has exactly one (empty) unit; the others
        # have none without pages
        for key, spans in seen.items():
            if (0, 0) in spans:
                assert spans == [(0, 0)] and key[2] == -1
        # chains: flags consistent with neighbours, one slot per chain of a
        # split item, split chains first in each CTA
        wi = t["work_indptr"]
        for c in range(ctas):
            rows = u[wi[c]:wi[c + 1]]
            sl = rows[:, 5]
            neg = sl < 0
            assert not (neg[:-1] & ~neg[1:]).any()  # no split unit after an unsplit one
            for k, row in enumerate(rows):
                cprev, cnext = bool(row[11] & 2), bool(row[11] & 4)
                if k == 0:
                    assert not cprev
                if k == len(rows) - 1:
                    assert not cnext
                if cnext:
                    nxt = rows[k + 1]
                    assert nxt[11] & 2 and tuple(nxt[:2]) == tuple(row[:2]) and nxt[5] == row[5]
        # per-CTA token load within one page (+ overhead) of the ideal share
        w = np.zeros(ctas)
        wi = t["work_indptr"]
        for c in range(ctas):
            for row in u[wi[c]:wi[c + 1]]:
                P = P0 if (row[11] & 1) == 0 else P1
                w[c] += (row[4] - row[3]) * P
        total = w.sum()
        assert w.max() <= total / ctas + max(P0, P1) + 16 * (len(u) + 1)


def test_cascade_plan_rejects_bad_input():
    qo = np.array([0, 2], np.int32)
    ip0, l0 = np.array([0, 4], np.int32), np.array([16], np.int32)
    ip1, l1 = np.array([0, 1, 2], np.int32), np.array([3, 17], np.int32)  # 17 > P1
    buf = np.zeros(1 << 20, np.uint8)
    with pytest.raises(C.AttnError) as e:
        C.plan_cascade(qo, ip0, l0, 16, ip1, l1, 16, 8, 2, 128, 4, buf)
    assert e.value.status == 1
    # 8 heads per kv head x 4 generations = 32 rows > 16
    qo4 = np.array([0, 4], np.int32)
    ip1b, l1b = np.array([0, 1, 2, 3, 4], np.int32), np.full(4, 5, np.int32)
    with pytest.raises(C.AttnError) as e:
        C.plan_cascade(qo4, ip0, l0, 16, ip1b, l1b, 16, 16, 2, 128, 4, buf)
    assert e.value.status == 2
