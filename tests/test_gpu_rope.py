"""Decode and append with rotary position embedding fused into the kernels
(attn_decode_run_rope, attn_append_run_rope) against the fp64 oracle with
the same cos / sin tables (oracle_batch_attention_rope)."""
import numpy as np
import pytest
import torch

from paged_kv_attention_bsr_gb300 import synth
from tests.gpu_util import assert_attn_close, oracle_dtype, poison_unused_slots, to_device

pytestmark = pytest.mark.gpu

CASES = [
    # (page_size, Hq, Hk, dtype, lens)
    (16, 8, 2, torch.bfloat16, [1, 15, 16, 17, 200, 1000, 0, 129]),
    (16, 32, 4, torch.bfloat16, [3000, 64, 511, 2]),
    (48, 8, 4, torch.float16, [47, 48, 49, 1000]),
    (128, 16, 2, torch.bfloat16, [128, 129, 1000, 5]),
]


def run_rope(w, cos, sin, num_ctas=None):
    from paged_kv_attention_bsr_gb300.api import PagedAttention
    c = w.cache
    att = PagedAttention(w.num_qo_heads, w.num_kv_heads, 128, "decode",
                         max_batch=max(w.batch, 1), num_ctas=num_ctas)
    att.plan(c.kv_indptr, c.last_page_len, c.page_size)
    d = to_device(c)
    q = w.q.cuda()
    o = torch.full_like(q, float("nan"))
    lse = torch.full(q.shape[:-1], float("nan"), dtype=torch.float32, device="cuda")
    att.run(q, d["k_pool"], d["v_pool"], d["kv_indptr"], d["kv_indices"], d["last_page_len"],
            w.sm_scale, out=o, lse=lse, rope=(torch.from_numpy(cos).cuda(),
                                             torch.from_numpy(sin).cuda()))
    torch.cuda.synchronize()
    assert att.status() == 0
    return o, lse


def oracle_rope(oracle_mod, w, cos, sin):
    c = w.cache
    return oracle_mod.batch_attention_rope(w.q, c.k_pool, c.v_pool, c.kv_indptr, c.kv_indices,
                                           c.last_page_len, c.page_size, w.num_qo_heads,
                                           w.num_kv_heads, 128, oracle_dtype(oracle_mod, w.dtype),
                                           w.sm_scale, cos, sin)


@pytest.mark.parametrize("case", range(len(CASES)))
@pytest.mark.parametrize("num_ctas", [1, 7, None])
def test_rope_decode_parity(oracle_mod, case, num_ctas):
    P, Hq, Hk, dtype, lens = CASES[case]
    pool = sum(-(-L // P) for L in lens) + 11
    w = synth.decode_workload(f"rope{case}", lens, P, pool, Hq, Hk, dtype, seed=600 + case)
    cos, sin = synth.rope_tables(max(lens) + 3)
    o_ref, lse_ref = oracle_rope(oracle_mod, w, cos, sin)
    o, lse = run_rope(w, cos, sin, num_ctas)
    assert_attn_close(o, lse, o_ref, lse_ref, f"rope case {case} ctas {num_ctas}")


@pytest.mark.parametrize("lens", [[1, 2, 3, 7], [1], [14, 15, 16]])
def test_rope_decode_short_table(oracle_mod, lens):
    """Tables exactly as long as the longest request, shorter than the key
    offset rows a tile derives its angles from."""
    pool = sum(-(-L // 16) for L in lens) + 5
    w = synth.decode_workload("ropeshort", lens, 16, pool, 16, 4, torch.bfloat16, seed=640)
    cos, sin = synth.rope_tables(max(lens))
    o_ref, lse_ref = oracle_rope(oracle_mod, w, cos, sin)
    o, lse = run_rope(w, cos, sin)
    assert_attn_close(o, lse, o_ref, lse_ref, f"rope short table {lens}")


def test_rope_decode_stale_pool_slots(oracle_mod):
    P, Hq, Hk, dtype, lens = CASES[0]
    pool = sum(-(-L // P) for L in lens) + 11
    w = synth.decode_workload("ropenan", lens, P, pool, Hq, Hk, dtype, seed=650)
    poison_unused_slots(w.cache)
    cos, sin = synth.rope_tables(max(lens))
    o_ref, lse_ref = oracle_rope(oracle_mod, w, cos, sin)
    o, lse = run_rope(w, cos, sin)
    assert_attn_close(o, lse, o_ref, lse_ref, "rope stale slots")


def test_rope_identity_table_equals_plain_decode():
    from tests.test_gpu_decode import run_decode
    P, Hq, Hk, dtype, lens = CASES[1]
    pool = sum(-(-L // P) for L in lens) + 11
    w = synth.decode_workload("ropeid", lens, P, pool, Hq, Hk, dtype, seed=660)
    n = max(lens)
    o1, l1 = run_rope(w, np.ones((n, 64), np.float32), np.zeros((n, 64), np.float32))
    o2, l2, _ = run_decode(w)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_rope_decode_full_size_uniform(oracle_mod):
    w = synth.uniform_gqa_decode()
    cos, sin = synth.rope_tables(int(w.cache.kv_lens.max()))
    o, lse = run_rope(w, cos, sin)
    o_ref, lse_ref = oracle_rope(oracle_mod, w, cos, sin)
    assert_attn_close(o, lse, o_ref, lse_ref, "rope uniform full size")


# Short appends (group x the longest query count <= 16) with fused RoPE:
# query row i at position kv_len - qo_len + i, key j at position j.
APPEND_CASES = [
    # (P, Hq, Hk, dtype, qo_lens, extra kv, causal)
    (16, 32, 8, torch.bfloat16, [1, 2, 4, 3, 4], [0, 5, 200, 17, 3000], True),
    (16, 32, 8, torch.bfloat16, [4, 1, 2], [700, 0, 129], False),
    (16, 16, 8, torch.bfloat16, [8, 5, 1], [100, 1000, 2], True),
    (16, 8, 8, torch.float16, [16, 9], [300, 2000], True),
    (128, 16, 2, torch.bfloat16, [2, 1, 2], [5000, 64, 127], False),
    (32, 16, 2, torch.bfloat16, [2, 2], [-2, 40], False),  # request 0 has no kv
]


def run_append_rope(w, cos, sin, num_ctas=None):
    from paged_kv_attention_bsr_gb300.api import PagedAttention
    c = w.cache
    att = PagedAttention(w.num_qo_heads, w.num_kv_heads, 128, "append", max_batch=w.batch,
                         max_total_qo=int(w.qo_indptr[-1]), num_ctas=num_ctas)
    att.plan(c.kv_indptr, c.last_page_len, c.page_size, qo_indptr_h=w.qo_indptr,
             causal=w.causal)
    d = to_device(c)
    q = w.q.cuda()
    o = torch.full_like(q, float("nan"))
    lse = torch.full(q.shape[:-1], float("nan"), dtype=torch.float32, device="cuda")
    att.run(q, d["k_pool"], d["v_pool"], d["kv_indptr"], d["kv_indices"], d["last_page_len"],
            w.sm_scale, out=o, lse=lse, qo_indptr=torch.from_numpy(w.qo_indptr).cuda(),
            rope=(torch.from_numpy(cos).cuda(), torch.from_numpy(sin).cuda()))
    torch.cuda.synchronize()
    assert att.status() == 0
    return o, lse


@pytest.mark.parametrize("case", range(len(APPEND_CASES)))
@pytest.mark.parametrize("num_ctas", [1, None])
def test_rope_short_append_parity(oracle_mod, case, num_ctas):
    P, Hq, Hk, dtype, qo_lens, extra, causal = APPEND_CASES[case]
    kv_lens = [max(q + e, 0) for q, e in zip(qo_lens, extra)]
    pool = sum(-(-L // P) for L in kv_lens) + 9
    w = synth.append_workload(f"ropeapp{case}", qo_lens, kv_lens, P, pool, Hq, Hk, dtype,
                              seed=700 + case, causal=causal)
    poison_unused_slots(w.cache)
    cos, sin = synth.rope_tables(max(kv_lens))
    c = w.cache
    o_ref, lse_ref = oracle_mod.batch_attention_rope(
        w.q, c.k_pool, c.v_pool, c.kv_indptr, c.kv_indices, c.last_page_len, P, Hq, Hk, 128,
        oracle_dtype(oracle_mod, dtype), w.sm_scale, cos, sin, causal=causal,
        qo_indptr=w.qo_indptr)
    o, lse = run_append_rope(w, cos, sin, num_ctas)
    assert_attn_close(o, lse, o_ref, lse_ref, f"rope append case {case} ctas {num_ctas}")


# Appends past 16 packed rows with fused RoPE run on the append kernel, whose
# rope warps turn the query rows and every K tile in shared memory.
LONG_APPEND_CASES = [
    # (P, Hq, Hk, dtype, qo_lens, extra kv, causal)
    (16, 32, 8, torch.bfloat16, [130, 1, 300, 64], [0, 500, 17, 1000], True),
    (16, 16, 2, torch.bfloat16, [40, 100], [300, 7], True),
    (16, 32, 8, torch.bfloat16, [20, 32, 9], [100, 0, 3000], True),   # one query tile
    (16, 8, 8, torch.float16, [200, 129], [0, 300], False),
    (3, 32, 8, torch.bfloat16, [100, 20], [50, 200], True),           # gathered rows
    (128, 16, 1, torch.bfloat16, [17, 3], [900, 10], True),           # group 16
]


@pytest.mark.parametrize("case", range(len(LONG_APPEND_CASES)))
@pytest.mark.parametrize("num_ctas", [1, 5, None])
def test_rope_long_append_parity(oracle_mod, case, num_ctas):
    P, Hq, Hk, dtype, qo_lens, extra, causal = LONG_APPEND_CASES[case]
    kv_lens = [q + e for q, e in zip(qo_lens, extra)]
    pool = sum(-(-L // P) for L in kv_lens) + 9
    w = synth.append_workload(f"ropelong{case}", qo_lens, kv_lens, P, pool, Hq, Hk, dtype,
                              seed=1200 + case, causal=causal)
    poison_unused_slots(w.cache)
    cos, sin = synth.rope_tables(max(kv_lens))
    c = w.cache
    o_ref, lse_ref = oracle_mod.batch_attention_rope(
        w.q, c.k_pool, c.v_pool, c.kv_indptr, c.kv_indices, c.last_page_len, P, Hq, Hk, 128,
        oracle_dtype(oracle_mod, dtype), w.sm_scale, cos, sin, causal=causal,
        qo_indptr=w.qo_indptr)
    o, lse = run_append_rope(w, cos, sin, num_ctas)
    assert_attn_close(o, lse, o_ref, lse_ref, f"rope long append case {case} ctas {num_ctas}")


def test_rope_long_append_identity_table_equals_plain_append():
    from tests.test_gpu_append import run_append
    P, Hq, Hk, dtype, qo_lens, extra, causal = LONG_APPEND_CASES[0]
    kv_lens = [q + e for q, e in zip(qo_lens, extra)]
    pool = sum(-(-L // P) for L in kv_lens) + 9
    w = synth.append_workload("ropelongid", qo_lens, kv_lens, P, pool, Hq, Hk, dtype, seed=1250,
                              causal=causal)
    n = max(kv_lens)
    o1, l1 = run_append_rope(w, np.ones((n, 64), np.float32), np.zeros((n, 64), np.float32))
    o2, l2, _ = run_append(w)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_rope_causal_append_full_size(oracle_mod):
    """The full-size causal append with LLaMA 3.1 RoPE (positions up to ~9k):
    every row of every split item and a seeded sample of the rest against
    the oracle's per-row RoPE attention, on host threads."""
    import concurrent.futures as cf
    from tests.gpu_util import split_items_of_plan
    from paged_kv_attention_bsr_gb300.api import PagedAttention
    w = synth.causal_append()
    c = w.cache
    cos, sin = synth.rope_tables(int(c.kv_lens.max()))
    att = PagedAttention(32, 8, 128, "append", max_batch=w.batch,
                         max_total_qo=int(w.qo_indptr[-1]))
    att.plan(c.kv_indptr, c.last_page_len, 16, qo_indptr_h=w.qo_indptr, causal=True)
    d = to_device(c)
    q = w.q.cuda()
    o, lse = att.run(q, d["k_pool"], d["v_pool"], d["kv_indptr"], d["kv_indices"],
                     d["last_page_len"], w.sm_scale, qo_indptr=torch.from_numpy(w.qo_indptr).cuda(),
                     rope=(torch.from_numpy(cos).cuda(), torch.from_numpy(sin).cuda()),
                     return_lse=True)
    torch.cuda.synchronize()
    assert att.status() == 0
    p = att.plan_info
    qo = np.diff(w.qo_indptr)
    rows = []
    for r, hk, t, _ in split_items_of_plan(att)[:12]:
        for i in range(int(t) * p.q_tile, min((int(t) + 1) * p.q_tile, int(qo[r]))):
            rows.extend((int(r), i, int(hk) * 4 + hh) for hh in range(4))
    rng = np.random.default_rng(23)
    for _ in range(300):
        r = int(rng.integers(w.batch))
        rows.append((r, int(rng.integers(qo[r])), int(rng.integers(32))))
    chunks = [x for x in np.array_split(np.arange(len(rows)), 16) if len(x)]

    def job(idx):
        out = []
        for k in idx:
            r, i, h = rows[k]
            out.append(oracle_mod.attention_row_rope(
                w.q, c.k_pool, c.v_pool, c.kv_indptr, c.kv_indices, c.last_page_len, 16, 32, 8,
                128, oracle_mod.BF16, w.sm_scale, cos, sin, r, i, h, causal=True,
                qo_indptr=w.qo_indptr))
        return out

    with cf.ThreadPoolExecutor(16) as ex:
        res = [x for part in ex.map(job, chunks) for x in part]
    o_ref = np.stack([x[0] for x in res])
    lse_ref = np.array([x[1] for x in res])
    idx = torch.tensor([int(w.qo_indptr[r]) + i for r, i, _ in rows])
    hs = torch.tensor([h for _, _, h in rows])
    assert_attn_close(o.cpu()[idx, hs], lse.cpu()[idx, hs], o_ref, lse_ref, "rope causal append")
