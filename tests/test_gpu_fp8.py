"""Decode over an FP8 (E4M3) KV cache with per-kv-head scales
(attn_decode_run_fp8) against the fp64 oracle that reads the same bytes
(oracle_batch_attention_fp8kv)."""
import concurrent.futures as cf

import numpy as np
import pytest
import torch

from paged_kv_attention_bsr_gb300 import synth
from tests.gpu_util import assert_attn_close, oracle_dtype

pytestmark = pytest.mark.gpu

CASES = [
    # (page_size, Hq, Hk, q dtype, lens)
    (16, 8, 2, torch.bfloat16, [0, 1, 15, 16, 17, 200, 1000]),
    (3, 6, 2, torch.float16, [2, 3, 95, 190]),
    (1, 4, 4, torch.bfloat16, [1, 5, 77, 300]),
    (16, 64, 8, torch.bfloat16, [3000, 17, 512, 1]),
    (128, 16, 2, torch.bfloat16, [128, 129, 1000, 5]),
    (16, 32, 8, torch.float16, [2049, 64, 0, 700]),
]


def _nhd(pool):
    return pool.permute(0, 2, 1, 3).contiguous()


def run_fp8(w, num_ctas=None, layout=0):
    from paged_kv_attention_bsr_gb300.api import PagedAttention
    c = w.cache
    att = PagedAttention(w.num_qo_heads, w.num_kv_heads, 128, "decode",
                         max_batch=max(w.batch, 1), num_ctas=num_ctas)
    att.plan(c.kv_indptr, c.last_page_len, c.page_size)
    kp, vp = (c.k_pool, c.v_pool) if layout == 0 else (_nhd(c.k_pool), _nhd(c.v_pool))
    q = w.q.cuda()
    o = torch.full_like(q, float("nan"))
    lse = torch.full(q.shape[:-1], float("nan"), dtype=torch.float32, device="cuda")
    dev = lambda a: torch.from_numpy(a).cuda()
    att.run(q, kp.cuda(), vp.cuda(), dev(c.kv_indptr), dev(c.kv_indices), dev(c.last_page_len),
            w.sm_scale, out=o, lse=lse, layout=layout, num_pages=c.num_pages,
            kv_scales=(c.k_scale.cuda(), c.v_scale.cuda()))
    torch.cuda.synchronize()
    assert att.status() == 0
    return o, lse, att


def oracle_fp8(oracle_mod, w, rows=None):
    c = w.cache
    return oracle_mod.batch_attention_fp8kv(
        w.q, c.k_pool, c.v_pool, c.kv_indptr, c.kv_indices, c.last_page_len, c.page_size,
        w.num_qo_heads, w.num_kv_heads, 128, oracle_dtype(oracle_mod, w.dtype), w.sm_scale,
        c.k_scale.numpy(), c.v_scale.numpy())


@pytest.mark.parametrize("case", range(len(CASES)))
@pytest.mark.parametrize("num_ctas", [1, 7, None])
def test_fp8_decode_parity(oracle_mod, case, num_ctas):
    P, Hq, Hk, dtype, lens = CASES[case]
    pool = sum(-(-L // P) for L in lens) + 11
    w = synth.fp8_decode_workload(f"f8_{case}", lens, P, pool, Hq, Hk, dtype, seed=1300 + case)
    o_ref, lse_ref = oracle_fp8(oracle_mod, w)
    o, lse, _ = run_fp8(w, num_ctas)
    assert_attn_close(o, lse, o_ref, lse_ref, f"fp8 case {case} ctas {num_ctas}")


@pytest.mark.parametrize("case", [0, 2, 3])
def test_fp8_decode_nhd_and_stale_slots(oracle_mod, case):
    """NHD pools, and every pool slot no request reads set to the E4M3 NaN
    byte (0x7f): nothing past a request's end may reach the arithmetic."""
    P, Hq, Hk, dtype, lens = CASES[case]
    pool = sum(-(-L // P) for L in lens) + 11
    w = synth.fp8_decode_workload(f"f8n_{case}", lens, P, pool, Hq, Hk, dtype, seed=1350 + case)
    c = w.cache
    valid = torch.zeros(c.num_pages, P, dtype=torch.bool)
    for r in range(w.batch):
        pages = c.kv_indices[c.kv_indptr[r]:c.kv_indptr[r + 1]]
        for j, pg in enumerate(pages):
            valid[int(pg), :P if j + 1 < len(pages) else int(c.last_page_len[r])] = True
    for pool_t in (c.k_pool, c.v_pool):
        pool_t.permute(0, 2, 1, 3)[~valid] = 0x7f
    o_ref, lse_ref = oracle_fp8(oracle_mod, w)
    for layout in (0, 1):
        o, lse, _ = run_fp8(w, None, layout)
        assert_attn_close(o, lse, o_ref, lse_ref, f"fp8 case {case} layout {layout}")


def test_fp8_decode_full_size_every_row(oracle_mod):
    """The uniform GQA decode shape over an FP8 cache, default grid, every
    row against the oracle (requests split over host threads)."""
    w = synth.fp8_uniform_gqa_decode()
    o, lse, att = run_fp8(w)
    assert att.plan_info.num_split_items > 0
    c = w.cache
    chunks = [x for x in np.array_split(np.arange(w.batch), 16) if len(x)]

    def job(rs):
        a, b = int(rs[0]), int(rs[-1]) + 1
        return oracle_mod.batch_attention_fp8kv(
            w.q[a:b], c.k_pool, c.v_pool, c.kv_indptr[a:b + 1], c.kv_indices,
            c.last_page_len[a:b], 16, 32, 8, 128, oracle_mod.BF16, w.sm_scale,
            c.k_scale.numpy(), c.v_scale.numpy())

    with cf.ThreadPoolExecutor(16) as ex:
        parts = list(ex.map(job, chunks))
    o_ref = np.concatenate([p[0] for p in parts])
    lse_ref = np.concatenate([p[1] for p in parts])
    assert_attn_close(o, lse, o_ref, lse_ref, w.name)
