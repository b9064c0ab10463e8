"""Composable formats in one launch (attn_plan_cascade / attn_cascade_run)
against the fp64 oracle.

Two oracle routes, neither touching the CUDA path: (a) decode over the flat
single-format layout (each generation's prefix pages followed by its own
suffix pages in one table), which is what the composable format must equal;
(b) for ragged shapes the flat layout cannot express (prefix lengths that are
not a whole number of small pages), the oracle's prefix attention
(non-causal, the prompt's generations as query rows) and suffix attention
(decode) merged by the oracle's log-sum-exp merge -- the merge identity is
pinned in the oracle's own tests.
"""
import numpy as np
import pytest
import torch

from paged_kv_attention_bsr_gb300 import synth
from tests.gpu_util import (assert_attn_close, oracle_decode_threaded, oracle_dtype,
                            poison_unused_slots, to_device)

pytestmark = pytest.mark.gpu


def run_one_launch(w, num_ctas=None, poison=False):
    from paged_kv_attention_bsr_gb300.api import CascadeAttention
    pre, suf = w.extra["prefix"], w.cache
    if poison:
        poison_unused_slots(pre)
        poison_unused_slots(suf)
    ca = CascadeAttention(w.num_qo_heads, w.num_kv_heads, 128, max_prompts=max(w.extra["prompts"], 1),
                          max_batch=w.batch, mode="one_launch", num_ctas=num_ctas)
    ca.plan(w.extra["prefix_qo_indptr"], pre.kv_indptr, pre.last_page_len, pre.page_size,
            suf.kv_indptr, suf.last_page_len, suf.page_size)
    assert ca.one_launch
    o, l = ca.run(w.q.cuda(), to_device(pre), to_device(suf),
                  torch.from_numpy(w.extra["prefix_qo_indptr"]).cuda(), w.sm_scale,
                  return_lse=True)
    torch.cuda.synchronize()
    assert ca.status() == 0
    return o, l, ca


def oracle_two_part(oracle_mod, w):
    pre, suf = w.extra["prefix"], w.cache
    dt = oracle_dtype(oracle_mod, w.dtype)
    o_p, l_p = oracle_mod.batch_attention(
        w.q, pre.k_pool, pre.v_pool, pre.kv_indptr, pre.kv_indices, pre.last_page_len,
        pre.page_size, w.num_qo_heads, w.num_kv_heads, 128, dt, w.sm_scale, causal=False,
        qo_indptr=w.extra["prefix_qo_indptr"])
    o_s, l_s = oracle_mod.batch_attention(
        w.q, suf.k_pool, suf.v_pool, suf.kv_indptr, suf.kv_indices, suf.last_page_len,
        suf.page_size, w.num_qo_heads, w.num_kv_heads, 128, dt, w.sm_scale)
    rows = w.batch * w.num_qo_heads
    o, l = oracle_mod.merge_states(np.stack([o_p.reshape(rows, 128), o_s.reshape(rows, 128)]),
                                   np.stack([l_p.reshape(rows), l_s.reshape(rows)]))
    return o.reshape(w.batch, w.num_qo_heads, 128), l.reshape(w.batch, w.num_qo_heads)


def oracle_flat(oracle_mod, w):
    flat = synth.flat_layout_of_composable(w)
    return oracle_mod.batch_attention(
        w.q, flat.k_pool, flat.v_pool, flat.kv_indptr, flat.kv_indices, flat.last_page_len, 16,
        w.num_qo_heads, w.num_kv_heads, 128, oracle_dtype(oracle_mod, w.dtype), w.sm_scale)


@pytest.mark.parametrize("num_ctas", [1, 7, None])
def test_one_launch_small_vs_flat(oracle_mod, num_ctas):
    w = synth.shared_prefix_decode(seed=99, prompts=3, n=4, prefix_len=512)
    o, l, _ = run_one_launch(w, num_ctas)
    o_ref, lse_ref = oracle_flat(oracle_mod, w)
    assert_attn_close(o, l, o_ref, lse_ref, f"one launch, {num_ctas} ctas")


# (gens per prompt, prefix lens, suffix lens or None = random, P0, P1, Hq, Hk, dtype)
RAGGED = [
    # ragged generations, one prompt without generations, prefix tails
    ([3, 0, 1, 2], [1000, 50, 17, 4096], None, 128, 16, 32, 8, torch.bfloat16),
    # empty prefix / empty suffixes
    ([2, 2], [0, 333], [0, 40, 700, 0], 64, 16, 16, 4, torch.float16),
    # group 1 (16 generations), group 16 (one generation)
    ([16, 5], [300, 2000], None, 16, 32, 8, 8, torch.bfloat16),
    ([1, 1, 1], [129, 0, 4000], [5, 0, 900], 32, 16, 32, 2, torch.bfloat16),
    # group 2, 8 generations, long prefix split across many CTAs
    ([8], [20000], None, 128, 16, 16, 8, torch.float16),
    # every row empty
    ([2, 1], [0, 0], [0, 0, 0], 16, 16, 8, 2, torch.bfloat16),
]


@pytest.mark.parametrize("case", range(len(RAGGED)))
@pytest.mark.parametrize("num_ctas", [3, None])
def test_one_launch_ragged_vs_oracle(oracle_mod, case, num_ctas):
    gens, pre_lens, suf_lens, P0, P1, Hq, Hk, dtype = RAGGED[case]
    rng = np.random.default_rng(700 + case)
    B = sum(gens)
    if suf_lens is None:
        suf_lens = rng.integers(0, 1200, size=B).tolist()
    w = synth.cascade_workload(f"ragged{case}", gens, pre_lens, suf_lens, P0, P1, Hq, Hk, dtype,
                               seed=800 + case)
    o, l, _ = run_one_launch(w, num_ctas, poison=True)
    o_ref, lse_ref = oracle_two_part(oracle_mod, w)
    assert_attn_close(o, l, o_ref, lse_ref, f"ragged case {case}")


def test_one_launch_matches_flat_when_flat_exists(oracle_mod):
    """Prefix lengths in whole small pages: the flat-layout oracle and the
    two-part oracle agree, and the kernel matches both."""
    w = synth.cascade_workload("flat-ok", [2, 3, 1], [256, 1024, 32], [10, 0, 300, 17, 1000, 1],
                               128, 16, 32, 8, torch.bfloat16, seed=901)
    o, l, _ = run_one_launch(w)
    o_f, l_f = oracle_flat(oracle_mod, w)
    o_t, l_t = oracle_two_part(oracle_mod, w)
    assert np.abs(o_f - o_t).max() < 1e-12 and np.abs(l_f - l_t).max() < 1e-12
    assert_attn_close(o, l, o_f, l_f, "flat-ok")


def test_one_launch_full_size(oracle_mod):
    """The full-size shared-prefix workload (16 prompts x 4 generations,
    8192-token prefix at P = 128, U[256, 1024] suffixes at P = 16) in the
    launch configuration the benchmark times: every row against the oracle on
    the flat layout (host threads)."""
    w = synth.shared_prefix_decode()
    o, l, ca = run_one_launch(w)
    assert ca.plan_info.num_units > ca.plan_info.num_items
    flat = synth.flat_layout_of_composable(w)
    wf = synth.Workload("flat", "decode", w.dtype, 32, 8, 128, w.sm_scale, w.q, flat)
    o_ref, lse_ref = oracle_decode_threaded(oracle_mod, wf)
    assert_attn_close(o, l, o_ref, lse_ref, w.name)


def test_one_launch_rejects_unsupported_shapes():
    from paged_kv_attention_bsr_gb300 import _capi as C
    from paged_kv_attention_bsr_gb300.api import CascadeAttention
    w = synth.cascade_workload("p8", [2], [100], [10, 20], 8, 16, 8, 2, torch.bfloat16, seed=5)
    pre, suf = w.extra["prefix"], w.cache
    ca = CascadeAttention(8, 2, 128, max_prompts=1, max_batch=2, mode="one_launch")
    with pytest.raises(ValueError):
        ca.plan(w.extra["prefix_qo_indptr"], pre.kv_indptr, pre.last_page_len, pre.page_size,
                suf.kv_indptr, suf.last_page_len, suf.page_size)
    # the C entry point refuses a page size that is not a multiple of 16
    host = torch.zeros(1 << 16, dtype=torch.uint8)
    dev = torch.zeros(1 << 20, dtype=torch.uint8, device="cuda")
    p = C.plan_cascade(w.extra["prefix_qo_indptr"], pre.kv_indptr, pre.last_page_len, 8,
                       suf.kv_indptr, suf.last_page_len, 16, 8, 2, 128, 4, host, dev)
    q = w.q.cuda()
    o = torch.empty_like(q)
    with pytest.raises(C.AttnError) as e:
        C.cascade_run(p, q, torch.from_numpy(w.extra["prefix_qo_indptr"]).cuda(), to_device(pre),
                      to_device(suf), w.sm_scale, o, None, dev)
    assert e.value.status == 2
    torch.cuda.synchronize()
