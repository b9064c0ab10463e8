"""Failure detection on the GPU without a fault.

Every wait in the kernels is bounded: a wait that runs out records a code in
the workspace error word and its kernel returns, the host reads
ATTN_ERR_TIMEOUT, and the context keeps working. attn_wait_selftest runs that
wait on an mbarrier nothing arrives on (a flag that nothing sets), so the
limit is what ends it.
"""
import time

import pytest
import torch

from paged_kv_attention_bsr_gb300 import synth
from tests.gpu_util import assert_attn_close, oracle_dtype, to_device

pytestmark = pytest.mark.gpu


def _decode(att, w, d, q):
    c = w.cache
    att.plan(c.kv_indptr, c.last_page_len, c.page_size)  # also clears the error word
    o, lse = att.run(q, d["k_pool"], d["v_pool"], d["kv_indptr"], d["kv_indices"],
                     d["last_page_len"], w.sm_scale, return_lse=True)
    torch.cuda.synchronize()
    return o, lse


def test_expired_wait_reports_timeout_and_the_context_stays_usable(oracle_mod):
    from paged_kv_attention_bsr_gb300 import _capi as C
    from paged_kv_attention_bsr_gb300.api import PagedAttention
    w = synth.decode_workload("fail", [300, 1000, 17], 16, 200, 32, 8, torch.bfloat16, seed=5)
    c = w.cache
    att = PagedAttention(32, 8, 128, "decode", max_batch=w.batch)
    d, q = to_device(c), w.q.cuda()
    o_ref, lse_ref = oracle_mod.batch_attention(
        w.q, c.k_pool, c.v_pool, c.kv_indptr, c.kv_indices, c.last_page_len, 16, 32, 8, 128,
        oracle_dtype(oracle_mod, w.dtype), w.sm_scale)
    o, lse = _decode(att, w, d, q)
    assert att.status() == 0

    # a 20 ms wait that nothing completes: ends by its limit, reports TIMEOUT
    t0 = time.perf_counter()
    C.wait_selftest(att.dev_ws, 20000)
    code = att.status()
    dt = time.perf_counter() - t0
    assert code == 0x1ff
    assert 0.015 < dt < 2.0, dt
    with pytest.raises(C.AttnError) as ei:
        C._check(C.lib.attn_workspace_status(C._ptr(att.dev_ws), None,
                                            C.ctypes.byref(C.ctypes.c_int32())))
    assert ei.value.status == C.ERR_TIMEOUT

    # with the word already set, a wait gives up at once instead of after 10 s
    t0 = time.perf_counter()
    C.wait_selftest(att.dev_ws, 10_000_000)
    assert att.status() == 0x1ff  # the first code is kept
    assert time.perf_counter() - t0 < 2.0

    # the context is intact: plan clears the word and the next run is correct
    o, lse = _decode(att, w, d, q)
    assert att.status() == 0
    assert_attn_close(o, lse, o_ref, lse_ref, "after a timeout")
