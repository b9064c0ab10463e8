"""Append / prefill (tcgen05 kernel) through the C ABI vs the fp64 oracle,
and the shared-prefix composable path (append + decode + LSE merge)."""
import numpy as np
import pytest
import torch

from paged_kv_attention_bsr_gb300 import synth
from tests.gpu_util import (assert_attn_close, oracle_dtype, oracle_rows_threaded,
                            poison_unused_slots, split_items_of_plan, to_device)

pytestmark = pytest.mark.gpu


def run_append(w, num_ctas=None, layout=0):
    from paged_kv_attention_bsr_gb300.api import PagedAttention
    c = w.cache
    att = PagedAttention(w.num_qo_heads, w.num_kv_heads, w.head_dim, "append",
                         max_batch=max(w.batch, 1), max_total_qo=max(int(w.qo_indptr[-1]), 1),
                         num_ctas=num_ctas)
    att.plan(c.kv_indptr, c.last_page_len, c.page_size, qo_indptr_h=w.qo_indptr,
             causal=w.causal)
    d = to_device(c)
    if layout == 1:  # NHD pools [pages, P, Hk, 128]
        d["k_pool"] = c.k_pool.permute(0, 2, 1, 3).contiguous().cuda()
        d["v_pool"] = c.v_pool.permute(0, 2, 1, 3).contiguous().cuda()
    q = w.q.cuda()
    qo = torch.from_numpy(w.qo_indptr).cuda()
    o = torch.full_like(q, float("nan"))
    lse = torch.full(q.shape[:-1], float("nan"), dtype=torch.float32, device="cuda")
    att.run(q, d["k_pool"], d["v_pool"], d["kv_indptr"], d["kv_indices"], d["last_page_len"],
            w.sm_scale, out=o, lse=lse, qo_indptr=qo, layout=layout, num_pages=c.num_pages)
    torch.cuda.synchronize()
    assert att.status() == 0
    return o, lse, att


def oracle_full(oracle_mod, w):
    c = w.cache
    return oracle_mod.batch_attention(w.q, c.k_pool, c.v_pool, c.kv_indptr, c.kv_indices,
                                      c.last_page_len, c.page_size, w.num_qo_heads,
                                      w.num_kv_heads, w.head_dim, oracle_dtype(oracle_mod, w.dtype),
                                      w.sm_scale, causal=w.causal, qo_indptr=w.qo_indptr)


CASES = [
    # (P, Hq, Hk, dtype, qo_lens, extra kv, causal)
    (16, 32, 8, torch.bfloat16, [1, 31, 32, 33, 100], [0, 5, 200, 17, 300], True),
    (16, 32, 8, torch.bfloat16, [1, 31, 32, 33, 100], [0, 5, 200, 17, 300], False),
    (16, 8, 8, torch.bfloat16, [130, 7, 256], [0, 129, 64], True),
    (32, 16, 8, torch.float16, [64, 3, 90], [10, 300, 0], True),
    (128, 16, 2, torch.bfloat16, [4, 4, 4], [700, 300, 129], False),
    (16, 64, 8, torch.bfloat16, [40, 17], [500, 1000], True),
    (16, 32, 2, torch.bfloat16, [20, 9], [100, 400], True),
]


@pytest.mark.parametrize("case", range(len(CASES)))
@pytest.mark.parametrize("num_ctas", [1, 5, None])
def test_append_small_parity(oracle_mod, case, num_ctas):
    P, Hq, Hk, dtype, qo_lens, extra, causal = CASES[case]
    kv_lens = [q + e for q, e in zip(qo_lens, extra)]
    pool = sum(-(-L // P) for L in kv_lens) + 9
    w = synth.append_workload(f"app{case}", qo_lens, kv_lens, P, pool, Hq, Hk, dtype,
                              seed=500 + case, causal=causal)
    o_ref, lse_ref = oracle_full(oracle_mod, w)
    o, lse, _ = run_append(w, num_ctas)
    assert_attn_close(o, lse, o_ref, lse_ref, f"append case {case} ctas {num_ctas}")


@pytest.mark.parametrize("case", [0, 3])
def test_append_zero_scale(oracle_mod, case):
    """sm_scale = 0 weighs every visible key equally; masked columns (the
    causal diagonal, ragged last tiles) stay out, split items merge."""
    P, Hq, Hk, dtype, qo_lens, extra, causal = CASES[case]
    kv_lens = [q + e for q, e in zip(qo_lens, extra)]
    pool = sum(-(-L // P) for L in kv_lens) + 9
    w = synth.append_workload(f"app_s0_{case}", qo_lens, kv_lens, P, pool, Hq, Hk, dtype,
                              seed=700 + case, causal=causal, sm_scale=0.0)
    o_ref, lse_ref = oracle_full(oracle_mod, w)
    o, lse, _ = run_append(w, 5)
    assert_attn_close(o, lse, o_ref, lse_ref, f"append sm_scale 0 case {case}")


# Short appends (group x longest query count <= 16 packed rows) run on the
# few-row tensor-core kernel: causal and not, groups 1 to 8, empty kv.
SHORT_CASES = [
    # (P, Hq, Hk, dtype, qo_lens, extra kv, causal)
    (16, 32, 8, torch.bfloat16, [1, 2, 4, 3, 4], [0, 5, 200, 17, 3000], True),
    (16, 32, 8, torch.bfloat16, [4, 1, 2], [700, 0, 129], False),
    (16, 16, 8, torch.bfloat16, [8, 5, 1], [100, 1000, 2], True),
    (16, 8, 8, torch.float16, [16, 9], [300, 2000], True),
    (128, 16, 2, torch.bfloat16, [2, 1, 2], [5000, 64, 127], False),
    (32, 16, 2, torch.bfloat16, [2, 2], [-2, 40], False),  # request 0 has no kv
]


@pytest.mark.parametrize("case", range(len(SHORT_CASES)))
@pytest.mark.parametrize("num_ctas", [1, 5, None])
def test_short_append_parity(oracle_mod, case, num_ctas):
    P, Hq, Hk, dtype, qo_lens, extra, causal = SHORT_CASES[case]
    kv_lens = [q + e for q, e in zip(qo_lens, extra)]
    pool = sum(-(-L // P) for L in kv_lens) + 9
    w = synth.append_workload(f"short{case}", qo_lens, kv_lens, P, pool, Hq, Hk, dtype,
                              seed=800 + case, causal=causal)
    o_ref, lse_ref = oracle_full(oracle_mod, w)
    o, lse, _ = run_append(w, num_ctas)
    assert_attn_close(o, lse, o_ref, lse_ref, f"short append case {case} ctas {num_ctas}")


@pytest.mark.parametrize("case", [0, 3, 4])
def test_short_append_stale_pool_slots_are_never_used(oracle_mod, case):
    P, Hq, Hk, dtype, qo_lens, extra, causal = SHORT_CASES[case]
    kv_lens = [q + e for q, e in zip(qo_lens, extra)]
    pool = sum(-(-L // P) for L in kv_lens) + 9
    w = synth.append_workload(f"shortnan{case}", qo_lens, kv_lens, P, pool, Hq, Hk, dtype,
                              seed=850 + case, causal=causal)
    poison_unused_slots(w.cache)
    o_ref, lse_ref = oracle_full(oracle_mod, w)
    for ctas in (1, None):
        o, lse, _ = run_append(w, ctas)
        assert_attn_close(o, lse, o_ref, lse_ref, f"short stale slots case {case} ctas {ctas}")


@pytest.mark.parametrize("case", [0, 2, 4, 6])
def test_append_stale_pool_slots_are_never_used(oracle_mod, case):
    P, Hq, Hk, dtype, qo_lens, extra, causal = CASES[case]
    kv_lens = [q + e for q, e in zip(qo_lens, extra)]
    pool = sum(-(-L // P) for L in kv_lens) + 9
    w = synth.append_workload(f"appnan{case}", qo_lens, kv_lens, P, pool, Hq, Hk, dtype,
                              seed=900 + case, causal=causal)
    poison_unused_slots(w.cache)
    o_ref, lse_ref = oracle_full(oracle_mod, w)
    for ctas in (1, None):
        o, lse, _ = run_append(w, ctas)
        assert_attn_close(o, lse, o_ref, lse_ref, f"append stale slots case {case} ctas {ctas}")


@pytest.mark.parametrize("case", [0, 2, 3, 5])
@pytest.mark.parametrize("num_ctas", [1, None])
def test_append_nhd_layout(oracle_mod, case, num_ctas):
    """NHD pools [pages, P, Hk, 128] in the append kernel (3-D TMA boxes of
    one head's 16 tokens), against the oracle on the same logical cache."""
    P, Hq, Hk, dtype, qo_lens, extra, causal = CASES[case]
    kv_lens = [q + e for q, e in zip(qo_lens, extra)]
    pool = sum(-(-L // P) for L in kv_lens) + 9
    w = synth.append_workload(f"appnhd{case}", qo_lens, kv_lens, P, pool, Hq, Hk, dtype,
                              seed=600 + case, causal=causal)
    poison_unused_slots(w.cache)
    o_ref, lse_ref = oracle_full(oracle_mod, w)
    o, lse, _ = run_append(w, num_ctas, layout=1)
    assert_attn_close(o, lse, o_ref, lse_ref, f"append nhd case {case} ctas {num_ctas}")


@pytest.mark.parametrize("case", [0, 4])
def test_short_append_nhd_layout(oracle_mod, case):
    P, Hq, Hk, dtype, qo_lens, extra, causal = SHORT_CASES[case]
    kv_lens = [q + e for q, e in zip(qo_lens, extra)]
    pool = sum(-(-L // P) for L in kv_lens) + 9
    w = synth.append_workload(f"shortnhd{case}", qo_lens, kv_lens, P, pool, Hq, Hk, dtype,
                              seed=820 + case, causal=causal)
    o_ref, lse_ref = oracle_full(oracle_mod, w)
    o, lse, _ = run_append(w, None, layout=1)
    assert_attn_close(o, lse, o_ref, lse_ref, f"short append nhd case {case}")


def test_append_empty_kv_non_causal(oracle_mod):
    """A request with no KV (non-causal) gives O = 0, LSE = -inf."""
    w = synth.append_workload("emptykv", [5, 3], [0, 40], 16, 10, 8, 2, torch.bfloat16,
                              seed=77, causal=False)
    o_ref, lse_ref = oracle_full(oracle_mod, w)
    o, lse, _ = run_append(w, None)
    assert_attn_close(o, lse, o_ref, lse_ref, "empty kv")


def test_causal_append_full_size(oracle_mod):
    """The full-size causal append in the benchmark's launch configuration:
    every row of every item the plan split across CTAs (the partial-state
    merge path), plus a seeded sample of the other rows, element by element
    against the oracle (rows spread over host threads)."""
    w = synth.causal_append()
    o, lse, att = run_append(w)
    p = att.plan_info
    g = w.num_qo_heads // w.num_kv_heads
    qo = np.diff(w.qo_indptr)
    rows = []
    split = split_items_of_plan(att)
    assert len(split) == p.num_split_items > 0
    for r, hk, t, _ in split:
        for i in range(int(t) * p.q_tile, min((int(t) + 1) * p.q_tile, int(qo[r]))):
            rows.extend((int(r), i, int(hk) * g + hh) for hh in range(g))
    rng = np.random.default_rng(5)
    for _ in range(400):
        r = int(rng.integers(w.batch))
        rows.append((r, int(rng.integers(qo[r])), int(rng.integers(w.num_qo_heads))))
    rows.append((0, 0, 0))
    r_last = int(np.argmax(qo))
    rows.append((r_last, int(qo[r_last]) - 1, w.num_qo_heads - 1))
    o_ref, lse_ref = oracle_rows_threaded(oracle_mod, w, rows, True, qo_indptr=w.qo_indptr)
    idx = torch.tensor([int(w.qo_indptr[r]) + i for r, i, _ in rows])
    hs = torch.tensor([h for _, _, h in rows])
    assert_attn_close(o.cpu()[idx, hs], lse.cpu()[idx, hs], o_ref, lse_ref, w.name)
    assert torch.isfinite(o.float()).all()


def composable_run(w):
    """Prefix pass (append, non-causal, qo_len = n per prompt, P = 128) + suffix
    pass (decode, P = 16) + attn_merge_states."""
    from paged_kv_attention_bsr_gb300 import merge_state
    from paged_kv_attention_bsr_gb300.api import PagedAttention
    pre, suf = w.extra["prefix"], w.cache
    q = w.q.cuda()
    att_p = PagedAttention(w.num_qo_heads, w.num_kv_heads, 128, "append",
                           max_batch=w.extra["prompts"], max_total_qo=w.batch)
    att_p.plan(pre.kv_indptr, pre.last_page_len, pre.page_size,
               qo_indptr_h=w.extra["prefix_qo_indptr"], causal=False)
    dp = to_device(pre)
    o_p, l_p = att_p.run(q, dp["k_pool"], dp["v_pool"], dp["kv_indptr"], dp["kv_indices"],
                         dp["last_page_len"], w.sm_scale,
                         qo_indptr=torch.from_numpy(w.extra["prefix_qo_indptr"]).cuda(),
                         return_lse=True)
    att_s = PagedAttention(w.num_qo_heads, w.num_kv_heads, 128, "decode", max_batch=w.batch)
    att_s.plan(suf.kv_indptr, suf.last_page_len, suf.page_size)
    ds = to_device(suf)
    o_s, l_s = att_s.run(q, ds["k_pool"], ds["v_pool"], ds["kv_indptr"], ds["kv_indices"],
                         ds["last_page_len"], w.sm_scale, return_lse=True)
    o, l = merge_state(o_p, l_p, o_s, l_s)
    torch.cuda.synchronize()
    assert att_p.status() == 0 and att_s.status() == 0
    return o, l


def cascade_run(w):
    """The same composable pass through CascadeAttention's two-pass mode
    (prefix and suffix on two streams, then the merge)."""
    from paged_kv_attention_bsr_gb300.api import CascadeAttention
    pre, suf = w.extra["prefix"], w.cache
    ca = CascadeAttention(w.num_qo_heads, w.num_kv_heads, 128, max_prompts=w.extra["prompts"],
                          max_batch=w.batch, mode="two_pass")
    ca.plan(w.extra["prefix_qo_indptr"], pre.kv_indptr, pre.last_page_len, pre.page_size,
            suf.kv_indptr, suf.last_page_len, suf.page_size)
    o, l = ca.run(w.q.cuda(), to_device(pre), to_device(suf),
                  torch.from_numpy(w.extra["prefix_qo_indptr"]).cuda(), w.sm_scale,
                  return_lse=True)
    torch.cuda.synchronize()
    assert ca.prefix.status() == 0 and ca.suffix.status() == 0
    return o, l


def test_composable_small_vs_flat(oracle_mod):
    w = synth.shared_prefix_decode(seed=99, prompts=3, n=4, prefix_len=512)
    o, l = composable_run(w)
    flat = synth.flat_layout_of_composable(w)
    o_ref, lse_ref = oracle_mod.batch_attention(
        w.q, flat.k_pool, flat.v_pool, flat.kv_indptr, flat.kv_indices, flat.last_page_len, 16,
        32, 8, 128, oracle_mod.BF16, w.sm_scale)
    assert_attn_close(o, l, o_ref, lse_ref, "composable small")
    o2, l2 = cascade_run(w)
    assert_attn_close(o2, l2, o_ref, lse_ref, "composable small, two streams")
    assert torch.equal(o, o2) and torch.equal(l, l2)


def test_composable_full_size(oracle_mod):
    """The full-size shared-prefix workload through CascadeAttention's
    two-pass mode, every row against the oracle on the flat single-format
    layout (host threads)."""
    from tests.gpu_util import oracle_decode_threaded
    w = synth.shared_prefix_decode()
    o, l = cascade_run(w)
    flat = synth.flat_layout_of_composable(w)
    wf = synth.Workload("flat", "decode", w.dtype, 32, 8, 128, w.sm_scale, w.q, flat)
    o_ref, lse_ref = oracle_decode_threaded(oracle_mod, wf)
    assert_attn_close(o, l, o_ref, lse_ref, w.name)
    o3, l3 = composable_run(w)
    assert torch.equal(o, o3) and torch.equal(l, l3)


# ---------------------------------------------------------------- POD-style
# Prefill chunks and single-token decodes in one append plan and one launch.
POD_CASES = [
    # (P, Hq, Hk, qo_lens, extra kv)
    (16, 32, 8, [1, 150, 1, 1, 300, 1, 37, 1], [1000, 200, 0, 77, 50, 2047, 500, 5]),
    (16, 16, 2, [1, 1, 129, 1, 2, 1], [3000, 16, 400, 0, 100, 700]),
    (3, 32, 8, [70, 1, 1, 1, 200], [5, 900, 31, 2, 0]),
]


@pytest.mark.parametrize("case", range(len(POD_CASES)))
@pytest.mark.parametrize("num_ctas", [1, 5, None])
def test_pod_mixed_batch_parity(oracle_mod, case, num_ctas):
    """A batch mixing causal prefill chunks and decode requests (qo_len 1)
    runs as one plan and one launch; every row matches the oracle."""
    P, Hq, Hk, qo_lens, extra = POD_CASES[case]
    kv_lens = [q + e for q, e in zip(qo_lens, extra)]
    pool = sum(-(-L // P) for L in kv_lens) + 9
    w = synth.append_workload(f"pod{case}", qo_lens, kv_lens, P, pool, Hq, Hk, torch.bfloat16,
                              seed=1100 + case, causal=True)
    poison_unused_slots(w.cache)
    o_ref, lse_ref = oracle_full(oracle_mod, w)
    o, lse, att = run_append(w, num_ctas)
    assert att.plan_info.num_items > 0
    assert_attn_close(o, lse, o_ref, lse_ref, f"pod case {case} ctas {num_ctas}")


def test_pod_mixed_batch_full_size(oracle_mod):
    """The benchmark's mixed batch (16 causal prefill chunks + 64 decodes) in
    one launch: every decode row, every row of every split item and a
    seeded sample of the other prefill rows against the oracle."""
    w = synth.pod_mixed_batch()
    o, lse, att = run_append(w)
    p = att.plan_info
    g = w.num_qo_heads // w.num_kv_heads
    qo = np.diff(w.qo_indptr)
    rows = [(int(r), 0, h) for r in w.extra["decode"] for h in range(w.num_qo_heads)]
    for r, hk, t, _ in split_items_of_plan(att):
        for i in range(int(t) * p.q_tile, min((int(t) + 1) * p.q_tile, int(qo[r]))):
            rows.extend((int(r), i, int(hk) * g + hh) for hh in range(g))
    rng = np.random.default_rng(17)
    for _ in range(300):
        r = int(rng.choice(w.extra["prefill"]))
        rows.append((r, int(rng.integers(qo[r])), int(rng.integers(w.num_qo_heads))))
    o_ref, lse_ref = oracle_rows_threaded(oracle_mod, w, rows, True, qo_indptr=w.qo_indptr)
    idx = torch.tensor([int(w.qo_indptr[r]) + i for r, i, _ in rows])
    hs = torch.tensor([h for _, _, h in rows])
    assert_attn_close(o.cpu()[idx, hs], lse.cpu()[idx, hs], o_ref, lse_ref, w.name)
    assert torch.isfinite(o.float()).all()
