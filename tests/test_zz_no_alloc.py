"""attn_decode_run_noalloc: batch decode for callers that cannot allocate.

Some callers may not allocate device memory when they run attention (an
allocator-free region of a serving engine, a plugin whose host application
owns every allocation, a latency-critical path that must not take allocator
locks). They cannot hand the library the workspaces that attn_plan and
attn_decode_run use, so attn_decode_run_noalloc runs on the library's own
fixed scratch area instead. These tests call it through the C ABI and require
the fp64 oracle's result, and the same result as the workspace path, within
the parity tolerances of the other tests, on consecutive calls that reuse the
shared scratch area; and they check that a bounded wait that runs out on that
scratch area is reported by attn_decode_run_noalloc_status.

This file is named to be collected last.
"""
import numpy as np
import pytest
import torch

from paged_kv_attention_bsr_gb300 import synth
from tests.gpu_util import (LSE_ABS, O_MAX_ABS, O_MEAN_ABS, assert_attn_close, oracle_dtype,
                            to_device)

pytestmark = pytest.mark.gpu


def _workspace_path(w):
    from paged_kv_attention_bsr_gb300.api import PagedAttention
    c = w.cache
    att = PagedAttention(w.num_qo_heads, w.num_kv_heads, 128, "decode", max_batch=w.batch)
    att.plan(c.kv_indptr, c.last_page_len, c.page_size)
    d = to_device(c)
    q = w.q.cuda()
    o, lse = att.run(q, d["k_pool"], d["v_pool"], d["kv_indptr"], d["kv_indices"],
                     d["last_page_len"], w.sm_scale, return_lse=True)
    torch.cuda.synchronize()
    return q, d, o, lse


def _noalloc(w, q, d):
    from paged_kv_attention_bsr_gb300 import _capi as C
    o = torch.full_like(q, float("nan"))
    lse = torch.full(q.shape[:-1], float("nan"), dtype=torch.float32, device="cuda")
    c = w.cache
    C.decode_run_noalloc(c.kv_indptr, c.last_page_len, c.page_size, w.num_qo_heads,
                         w.num_kv_heads, 128, q, d["k_pool"], d["v_pool"], d["kv_indptr"],
                         d["kv_indices"], d["last_page_len"], w.sm_scale, o, lse)
    torch.cuda.synchronize()
    return o, lse


def _assert_same(o, lse, o_ref, lse_ref):
    a = o.float().cpu().numpy().astype(np.float64)
    b = o_ref.float().cpu().numpy().astype(np.float64)
    err = np.abs(a - b)
    assert np.all(np.isfinite(a))
    assert err.max() <= O_MAX_ABS and err.mean() <= O_MEAN_ABS, (err.max(), err.mean())
    la, lb = lse.cpu().numpy(), lse_ref.cpu().numpy()
    fin = np.isfinite(lb)
    assert np.array_equal(np.isneginf(la), np.isneginf(lb))
    assert np.abs(la[fin] - lb[fin]).max() <= LSE_ABS


def _oracle(oracle_mod, w):
    c = w.cache
    return oracle_mod.batch_attention(w.q, c.k_pool, c.v_pool, c.kv_indptr, c.kv_indices,
                                      c.last_page_len, c.page_size, w.num_qo_heads,
                                      w.num_kv_heads, 128, oracle_dtype(oracle_mod, w.dtype),
                                      w.sm_scale)


def test_noalloc_matches_workspace_path_on_consecutive_calls(oracle_mod):
    from paged_kv_attention_bsr_gb300 import _capi as C
    # split-heavy batch (long and short requests, one empty) and a second shape
    w1 = synth.decode_workload("na1", [3000, 50, 2000, 17, 0, 900, 4096], 16, 900, 32, 8,
                               torch.bfloat16, seed=901)
    w2 = synth.decode_workload("na2", [129, 4000, 1, 700], 16, 400, 16, 2, torch.bfloat16,
                               seed=902)
    r1, r2 = _oracle(oracle_mod, w1), _oracle(oracle_mod, w2)
    q1, d1, o1_ref, l1_ref = _workspace_path(w1)
    q2, d2, o2_ref, l2_ref = _workspace_path(w2)
    o, l = _noalloc(w1, q1, d1)
    assert C.decode_run_noalloc_status() == 0
    assert_attn_close(o, l, *r1, "no-alloc, first call")
    _assert_same(o, l, o1_ref, l1_ref)
    o, l = _noalloc(w1, q1, d1)  # same call again: scratch state from the last call
    assert_attn_close(o, l, *r1, "no-alloc, second call")
    _assert_same(o, l, o1_ref, l1_ref)
    o, l = _noalloc(w2, q2, d2)  # another shape on the same scratch area
    assert_attn_close(o, l, *r2, "no-alloc, other shape")
    _assert_same(o, l, o2_ref, l2_ref)


def test_noalloc_status_reports_an_expired_wait(oracle_mod):
    """A wait that nothing completes, run on the no-allocation scratch area,
    ends by its limit; the status call reports TIMEOUT, and the next
    no-allocation call clears the word and still matches the oracle."""
    from paged_kv_attention_bsr_gb300 import _capi as C
    w = synth.decode_workload("na3", [700, 33, 2500], 16, 300, 16, 4, torch.bfloat16, seed=903)
    ref = _oracle(oracle_mod, w)
    q, d = w.q.cuda(), to_device(w.cache)
    o, l = _noalloc(w, q, d)
    assert C.decode_run_noalloc_status() == 0
    C.wait_selftest_noalloc(20000)  # 20 ms
    assert C.decode_run_noalloc_status() == 0x1ff
    with pytest.raises(C.AttnError) as ei:
        C._check(C.lib.attn_decode_run_noalloc_status(None, C.ctypes.byref(C.ctypes.c_int32())))
    assert ei.value.status == C.ERR_TIMEOUT
    o, l = _noalloc(w, q, d)
    assert C.decode_run_noalloc_status() == 0
    assert_attn_close(o, l, *ref, "no-alloc after a timeout")


def test_noalloc_rejects_batches_beyond_its_scratch():
    from paged_kv_attention_bsr_gb300 import _capi as C
    B = 20000  # 160k (request, kv head) items: plan tables alone exceed 4 MiB
    kv_indptr = np.arange(B + 1, dtype=np.int32)
    last = np.ones(B, np.int32)
    dummy = torch.empty(16, dtype=torch.bfloat16, device="cuda")
    p = dummy.data_ptr()
    # straight through the C ABI (the binding's own size checks would reject
    # the dummy tensors first): the library refuses the batch on the host,
    # before any GPU work, so the dummy pointers are never read
    st = C.lib.attn_decode_run_noalloc(
        C._ptr(kv_indptr), C._ptr(last), B, 16, 64, 8, 128, p, p, p, 1, C.LAYOUT_HND, p, p, p,
        C.BF16, C.ctypes.c_float(0.1), p, None, None)
    assert st == C.ERR_WORKSPACE_TOO_SMALL
    assert "4 MiB" in C.last_error()
