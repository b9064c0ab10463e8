"""Batch decode on the GPU through the C ABI vs the fp64 oracle."""
import math

import numpy as np
import pytest
import torch

from paged_kv_attention_bsr_gb300 import synth
from tests.gpu_util import (assert_attn_close, oracle_decode_threaded, oracle_dtype,
                            poison_unused_slots, to_device)

pytestmark = pytest.mark.gpu


def _api():
    from paged_kv_attention_bsr_gb300 import _capi as C
    from paged_kv_attention_bsr_gb300.api import PagedAttention
    return C, PagedAttention


def _nhd(cache):
    return (cache.k_pool.permute(0, 2, 1, 3).contiguous(),
            cache.v_pool.permute(0, 2, 1, 3).contiguous())


def run_decode(w, num_ctas=None, layout=0, graph=False):
    C, PagedAttention = _api()
    c = w.cache
    att = PagedAttention(w.num_qo_heads, w.num_kv_heads, w.head_dim, "decode",
                         max_batch=max(w.batch, 1), num_ctas=num_ctas)
    att.plan(c.kv_indptr, c.last_page_len, c.page_size)
    d = to_device(c)
    if layout == C.LAYOUT_NHD:
        kn, vn = _nhd(c)
        d["k_pool"], d["v_pool"] = kn.cuda(), vn.cuda()
    q = w.q.cuda()
    o = torch.full_like(q, float("nan"))
    lse = torch.full(q.shape[:-1], float("nan"), dtype=torch.float32, device="cuda")
    args = (q, d["k_pool"], d["v_pool"], d["kv_indptr"], d["kv_indices"], d["last_page_len"])
    if graph:
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            att.run(*args, w.sm_scale, out=o, lse=lse, layout=layout, num_pages=c.num_pages,
                    stream=s)
        torch.cuda.current_stream().wait_stream(s)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        o.fill_(float("nan"))
        with torch.cuda.graph(g):
            att.run(*args, w.sm_scale, out=o, lse=lse, layout=layout, num_pages=c.num_pages)
        for _ in range(3):
            g.replay()
    else:
        att.run(*args, w.sm_scale, out=o, lse=lse, layout=layout, num_pages=c.num_pages)
    torch.cuda.synchronize()
    assert att.status() == 0
    return o, lse, att


def oracle_full(oracle_mod, w, layout=0):
    c = w.cache
    return oracle_mod.batch_attention(w.q, c.k_pool, c.v_pool, c.kv_indptr, c.kv_indices,
                                      c.last_page_len, c.page_size, w.num_qo_heads,
                                      w.num_kv_heads, w.head_dim, oracle_dtype(oracle_mod, w.dtype),
                                      w.sm_scale)


SMALL_CASES = [
    # (page_size, Hq, Hk, dtype, lens)
    (16, 8, 2, torch.bfloat16, [0, 1, 15, 16, 17, 63, 64, 65, 200, 1000]),
    (16, 32, 8, torch.bfloat16, [1024, 4096, 37, 129, 0, 2049]),
    (1, 4, 2, torch.bfloat16, [1, 5, 77, 300]),
    (3, 6, 2, torch.float16, [2, 3, 4, 95, 190]),
    (128, 16, 2, torch.bfloat16, [128, 129, 1000, 5]),
    (16, 64, 8, torch.bfloat16, [3000, 17, 512, 1]),
    (16, 4, 4, torch.float16, [2048, 100]),
    (32, 10, 2, torch.bfloat16, [500, 33, 64]),
    (16, 16, 8, torch.bfloat16, [1, 16, 31, 700, 0, 2500]),
    (48, 8, 4, torch.float16, [47, 48, 49, 1000]),
]


@pytest.mark.parametrize("case", range(len(SMALL_CASES)))
@pytest.mark.parametrize("num_ctas", [1, 7, None])
def test_decode_small_parity(oracle_mod, case, num_ctas):
    P, Hq, Hk, dtype, lens = SMALL_CASES[case]
    pool = sum(-(-L // P) for L in lens) + 11
    w = synth.decode_workload(f"small{case}", lens, P, pool, Hq, Hk, dtype, seed=100 + case)
    o_ref, lse_ref = oracle_full(oracle_mod, w)
    o, lse, att = run_decode(w, num_ctas=num_ctas)
    assert_attn_close(o, lse, o_ref, lse_ref, f"case {case} ctas {num_ctas}")


@pytest.mark.parametrize("case", [0, 1, 4, 5, 6, 8, 9])
def test_decode_stale_pool_slots_are_never_used(oracle_mod, case):
    P, Hq, Hk, dtype, lens = SMALL_CASES[case]
    pool = sum(-(-L // P) for L in lens) + 11
    w = synth.decode_workload(f"nan{case}", lens, P, pool, Hq, Hk, dtype, seed=700 + case)
    poison_unused_slots(w.cache)
    o_ref, lse_ref = oracle_full(oracle_mod, w)
    for ctas in (1, None):
        o, lse, _ = run_decode(w, num_ctas=ctas)
        assert_attn_close(o, lse, o_ref, lse_ref, f"stale slots case {case} ctas {ctas}")


@pytest.mark.parametrize("case", [0, 1, 3, 4, 5, 9])
@pytest.mark.parametrize("num_ctas", [1, None])
def test_decode_nhd_layout(oracle_mod, case, num_ctas):
    C, _ = _api()
    P, Hq, Hk, dtype, lens = SMALL_CASES[case]
    pool = sum(-(-L // P) for L in lens) + 11
    w = synth.decode_workload(f"nhd{case}", lens, P, pool, Hq, Hk, dtype, seed=300 + case)
    o_ref, lse_ref = oracle_full(oracle_mod, w)
    o, lse, _ = run_decode(w, num_ctas=num_ctas, layout=C.LAYOUT_NHD)
    assert_attn_close(o, lse, o_ref, lse_ref, f"nhd case {case} ctas {num_ctas}")


def test_decode_graph_replay_and_determinism(oracle_mod):
    P, Hq, Hk, dtype, lens = SMALL_CASES[1]
    w = synth.decode_workload("graph", lens, P, 2000, Hq, Hk, dtype, seed=7)
    o_ref, lse_ref = oracle_full(oracle_mod, w)
    o1, l1, _ = run_decode(w)
    o2, l2, _ = run_decode(w, graph=True)
    assert_attn_close(o2, l2, o_ref, lse_ref, "graph")
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_single_decode_snippet(oracle_mod):
    """q [32,128], k/v [2048,32,128] fp16 -> [32,128] (quick-start snippet)."""
    from paged_kv_attention_bsr_gb300 import single_decode_with_kv_cache
    g = torch.Generator().manual_seed(5)
    q = torch.randn(32, 128, generator=g).half()
    k = torch.randn(2048, 32, 128, generator=g).half()
    v = torch.randn(2048, 32, 128, generator=g).half()
    o, lse = single_decode_with_kv_cache(q.cuda(), k.cuda(), v.cuda(), return_lse=True)
    assert tuple(o.shape) == (32, 128)
    # the oracle sees the same contiguous cache as one NHD page table
    n = 2048 // 16
    o_ref, lse_ref = oracle_mod.batch_attention(
        q.reshape(1, 32, 128), k, v, np.array([0, n], np.int32), np.arange(n, dtype=np.int32),
        np.array([16], np.int32), 16, 32, 32, 128, oracle_mod.F16, 1 / math.sqrt(128),
        layout=oracle_mod.NHD)
    assert_attn_close(o.reshape(1, 32, 128), lse.reshape(1, 32), o_ref, lse_ref, "snippet")


def _sampled_parity(oracle_mod, w, o, lse, n_rows, seed):
    rng = np.random.default_rng(seed)
    c = w.cache
    rows = [(int(rng.integers(w.batch)), int(rng.integers(w.num_qo_heads))) for _ in range(n_rows)]
    # always include the longest request
    rows.append((int(np.argmax(c.kv_lens)), 0))
    o_ref = np.zeros((len(rows), w.head_dim))
    lse_ref = np.zeros(len(rows))
    for i, (r, h) in enumerate(rows):
        o_ref[i], lse_ref[i] = oracle_mod.attention_row(
            w.q, c.k_pool, c.v_pool, c.kv_indptr, c.kv_indices, c.last_page_len, c.page_size,
            w.num_qo_heads, w.num_kv_heads, w.head_dim, oracle_dtype(oracle_mod, w.dtype),
            w.sm_scale, r, 0, h)
    idx_r = torch.tensor([r for r, _ in rows])
    idx_h = torch.tensor([h for _, h in rows])
    return assert_attn_close(o.cpu()[idx_r, idx_h], lse.cpu()[idx_r, idx_h], o_ref, lse_ref,
                             w.name)


@pytest.mark.parametrize("name", ["single_decode", "uniform_decode", "skewed_decode"])
def test_decode_full_size_every_row(oracle_mod, name):
    """The full-size decode workloads, in the launch configuration the
    benchmark times (default grid), compared with the oracle on every output
    row, element by element (the oracle runs over the requests on host
    threads)."""
    w = synth.WORKLOADS[name]()
    o, lse, att = run_decode(w)
    assert att.plan_info.num_split_items > 0  # the split / merge path is exercised
    o_ref, lse_ref = oracle_decode_threaded(oracle_mod, w)
    assert_attn_close(o, lse, o_ref, lse_ref, w.name)
    # every output row is finite and every LSE is finite (no empty requests here)
    assert torch.isfinite(o.float()).all() and torch.isfinite(lse).all()


def test_single_decode_empty_cache():
    """kv_len = 0 through the snippet's call: O = 0 and LSE = -inf, like a
    zero-length request in a batch (no pool pages exist at all)."""
    from paged_kv_attention_bsr_gb300 import single_decode_with_kv_cache
    for hq, hk in ((32, 32), (32, 8)):
        q = torch.randn(hq, 128, dtype=torch.float16, device="cuda")
        k = torch.empty(0, hk, 128, dtype=torch.float16, device="cuda")
        o, lse = single_decode_with_kv_cache(q, k, k.clone(), return_lse=True)
        torch.cuda.synchronize()
        assert torch.equal(o, torch.zeros_like(o))
        assert torch.isneginf(lse).all()


def test_single_decode_strided_inputs(oracle_mod):
    """Strided k / v (slices of one [kv_len, 2, Hk, D] tensor) are read
    correctly: the wrapper makes them dense first."""
    from paged_kv_attention_bsr_gb300 import single_decode_with_kv_cache
    g = torch.Generator().manual_seed(9)
    q = torch.randn(16, 128, generator=g).half()
    kv = torch.randn(300, 2, 4, 128, generator=g).half()
    o, lse = single_decode_with_kv_cache(q.cuda(), kv[:, 0].cuda(), kv[:, 1].cuda(),
                                         return_lse=True)
    k, v = kv[:, 0].contiguous(), kv[:, 1].contiguous()
    o_ref, lse_ref = oracle_mod.batch_attention(
        q.reshape(1, 16, 128), k, v, np.array([0, 75], np.int32), np.arange(75, dtype=np.int32),
        np.array([4], np.int32), 4, 16, 4, 128, oracle_mod.F16, 1 / math.sqrt(128),
        layout=oracle_mod.NHD)
    assert_attn_close(o.reshape(1, 16, 128), lse.reshape(1, 16), o_ref, lse_ref, "strided")


@pytest.mark.parametrize("hq,hk", [(32, 8), (32, 32)])
def test_decode_zero_scale(oracle_mod, hq, hk):
    """sm_scale = 0 weighs every key of a request equally (tensor-core kernel
    at group 4, CUDA-core kernel at group 1), ragged last pages included."""
    w = synth.decode_workload(f"dec_s0_{hq}_{hk}", [1, 17, 300, 1000], 16, 120, hq, hk,
                              torch.bfloat16, seed=811, sm_scale=0.0)
    o_ref, lse_ref = oracle_decode_threaded(oracle_mod, w)
    o, lse, _ = run_decode(w, num_ctas=7)
    assert_attn_close(o, lse, o_ref, lse_ref, f"decode sm_scale 0 group {hq // hk}")
