"""Append / prefill (tcgen05 kernel) through the C ABI vs the fp64 oracle,
and the shared-prefix composable path (append + decode + LSE merge)."""
import numpy as np
import pytest
import torch

from paged_kv_attention_bsr_gb300 import synth
from tests.gpu_util import assert_attn_close, oracle_dtype, poison_unused_slots, to_device

pytestmark = pytest.mark.gpu


def run_append(w, num_ctas=None):
    from paged_kv_attention_bsr_gb300.api import PagedAttention
    c = w.cache
    att = PagedAttention(w.num_qo_heads, w.num_kv_heads, w.head_dim, "append",
                         max_batch=max(w.batch, 1), max_total_qo=max(int(w.qo_indptr[-1]), 1),
                         num_ctas=num_ctas)
    att.plan(c.kv_indptr, c.last_page_len, c.page_size, qo_indptr_h=w.qo_indptr,
             causal=w.causal)
    d = to_device(c)
    q = w.q.cuda()
    qo = torch.from_numpy(w.qo_indptr).cuda()
    o = torch.full_like(q, float("nan"))
    lse = torch.full(q.shape[:-1], float("nan"), dtype=torch.float32, device="cuda")
    att.run(q, d["k_pool"], d["v_pool"], d["kv_indptr"], d["kv_indices"], d["last_page_len"],
            w.sm_scale, out=o, lse=lse, qo_indptr=qo)
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


def test_append_empty_kv_non_causal(oracle_mod):
    """A request with no KV (non-causal) gives O = 0, LSE = -inf."""
    w = synth.append_workload("emptykv", [5, 3], [0, 40], 16, 10, 8, 2, torch.bfloat16,
                              seed=77, causal=False)
    o_ref, lse_ref = oracle_full(oracle_mod, w)
    o, lse, _ = run_append(w, None)
    assert_attn_close(o, lse, o_ref, lse_ref, "empty kv")


def test_causal_append_full_size_sampled(oracle_mod):
    w = synth.causal_append()
    o, lse, att = run_append(w)
    rng = np.random.default_rng(5)
    c = w.cache
    rows = []
    for _ in range(40):
        r = int(rng.integers(w.batch))
        L = int(w.qo_indptr[r + 1] - w.qo_indptr[r])
        rows.append((r, int(rng.integers(L)), int(rng.integers(w.num_qo_heads))))
    rows.append((0, 0, 0))
    r_last = int(np.argmax(np.diff(w.qo_indptr)))
    rows.append((r_last, int(w.qo_indptr[r_last + 1] - w.qo_indptr[r_last]) - 1, 31))
    o_ref = np.zeros((len(rows), 128))
    lse_ref = np.zeros(len(rows))
    for k, (r, i, h) in enumerate(rows):
        o_ref[k], lse_ref[k] = oracle_mod.attention_row(
            w.q, c.k_pool, c.v_pool, c.kv_indptr, c.kv_indices, c.last_page_len, 16, 32, 8,
            128, oracle_mod.BF16, w.sm_scale, r, i, h, causal=True, qo_indptr=w.qo_indptr)
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


def test_composable_small_vs_flat(oracle_mod):
    w = synth.shared_prefix_decode(seed=99, prompts=3, n=4, prefix_len=512)
    o, l = composable_run(w)
    flat = synth.flat_layout_of_composable(w)
    o_ref, lse_ref = oracle_mod.batch_attention(
        w.q, flat.k_pool, flat.v_pool, flat.kv_indptr, flat.kv_indices, flat.last_page_len, 16,
        32, 8, 128, oracle_mod.BF16, w.sm_scale)
    assert_attn_close(o, l, o_ref, lse_ref, "composable small")


def test_composable_full_size_sampled(oracle_mod):
    w = synth.shared_prefix_decode()
    o, l = composable_run(w)
    flat = synth.flat_layout_of_composable(w)
    rng = np.random.default_rng(44)
    rows = [(int(rng.integers(w.batch)), int(rng.integers(32))) for _ in range(32)]
    o_ref = np.zeros((len(rows), 128))
    lse_ref = np.zeros(len(rows))
    for k, (r, h) in enumerate(rows):
        o_ref[k], lse_ref[k] = oracle_mod.attention_row(
            w.q, flat.k_pool, flat.v_pool, flat.kv_indptr, flat.kv_indices, flat.last_page_len,
            16, 32, 8, 128, oracle_mod.BF16, w.sm_scale, r, 0, h)
    ri = torch.tensor([r for r, _ in rows])
    hi = torch.tensor([h for _, h in rows])
    assert_attn_close(o.cpu()[ri, hi], l.cpu()[ri, hi], o_ref, lse_ref, w.name)
