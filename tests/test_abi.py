"""The C-ABI library loads and exports every symbol include/attn.h declares;
host-side validation answers with status codes before any CUDA call."""
import ctypes
import os
import re
import subprocess

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    src = open(os.path.join(ROOT, "include", "attn.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(attn_[a-z0-9_]+)\s*\(", src)))


def test_header_declares_the_boundary():
    names = _declared()
    for required in ("attn_plan", "attn_decode_run", "attn_append_run", "attn_merge_states"):
        assert required in names


def test_library_exports_every_declared_symbol():
    C = pytest.importorskip("paged_kv_attention_bsr_gb300._capi")
    lib = ctypes.CDLL(C.LIB_PATH)
    for name in _declared():
        assert hasattr(lib, name), name
    assert set(_declared()) == set(C.EXPORTS)
    out = subprocess.run(["nm", "-D", "--defined-only", C.LIB_PATH], capture_output=True,
                         text=True).stdout
    for name in _declared():
        assert re.search(rf"\bT {name}\b", out), name


def test_workspace_size_and_validation_without_gpu():
    C = pytest.importorskip("paged_kv_attention_bsr_gb300._capi")
    dev, host = C.workspace_size(64, 64, 32, 8, 128, 304)
    assert dev > host > 0 and dev % 256 == 0
    with pytest.raises(C.AttnError) as ei:
        C.workspace_size(0, 1, 32, 8, 128, 304)
    assert ei.value.status == C.ERR_INVALID_ARG
    with pytest.raises(C.AttnError) as ei:
        C.workspace_size(1, 1, 32, 8, 96, 304)
    assert ei.value.status == C.ERR_UNSUPPORTED
    # run calls validate before touching CUDA: wrong mode, null workspace
    buf = np.zeros(host, np.uint8)
    p = C.plan(None, np.array([0, 1], np.int32), np.array([5], np.int32), 16, 32, 8, 128,
               False, 304, buf)
    st = C.lib.attn_append_run(ctypes.byref(p), None, None, None, None, 0, 0, None, None, None,
                               1, 0, ctypes.c_float(1.0), None, None, None, 0, None)
    assert st == C.ERR_INVALID_ARG
    st = C.lib.attn_decode_run(ctypes.byref(p), ctypes.c_void_p(16), ctypes.c_void_p(16),
                               ctypes.c_void_p(16), 1, 0, ctypes.c_void_p(16),
                               ctypes.c_void_p(16), ctypes.c_void_p(16), 1,
                               ctypes.c_float(1.0), ctypes.c_void_p(16), None, None, 0, None)
    assert st == C.ERR_INVALID_ARG and "dev_ws" in C.last_error()
    st = C.lib.attn_decode_run(ctypes.byref(p), ctypes.c_void_p(16), ctypes.c_void_p(16),
                               ctypes.c_void_p(16), 1, 0, ctypes.c_void_p(16),
                               ctypes.c_void_p(16), ctypes.c_void_p(16), 1,
                               ctypes.c_float(1.0), ctypes.c_void_p(16), None,
                               ctypes.c_void_p(256), 16, None)
    assert st == C.ERR_WORKSPACE_TOO_SMALL
    st = C.lib.attn_merge_states(None, None, None, None, None, None, 4, 2, 100, 1, None)
    assert st == C.ERR_UNSUPPORTED
    # fused RoPE decode: tables checked before anything runs
    kvi = np.array([0, 2, 5], np.int32)
    lpl = np.array([3, 16], np.int32)
    buf = np.zeros(1 << 16, np.uint8)
    pr = C.plan(None, kvi, lpl, 16, 8, 2, 128, False, 4, buf)
    assert pr.max_kv_len == 48  # lengths 16+3 and 2*16+16
    fake = ctypes.c_void_p(256)
    args = lambda cos, n, layout: (ctypes.byref(pr), fake, fake, fake, 8, layout, fake, fake,
                                   fake, 1, ctypes.c_float(0.1), cos, cos, n, fake, None, fake,
                                   1 << 30, None)
    assert C.lib.attn_decode_run_rope(*args(None, 100, 0)) == C.ERR_INVALID_ARG
    assert C.lib.attn_decode_run_rope(*args(fake, 47, 0)) == C.ERR_INVALID_ARG
    pr3 = C.plan(None, kvi, lpl, 16, 6, 2, 128, False, 4, buf)  # group 3: CUDA cores only
    assert C.lib.attn_decode_run_rope(ctypes.byref(pr3), fake, fake, fake, 8, 0, fake, fake,
                                      fake, 1, ctypes.c_float(0.1), fake, fake, 48, fake, None,
                                      fake, 1 << 30, None) == C.ERR_UNSUPPORTED
    # fused RoPE append: kv_len >= qo_len
    def append_rope(qo, causal, cos=fake):
        pa = C.plan(np.array(qo, np.int32), kvi, lpl, 16, 8, 2, 128, causal, 4, buf)
        return pa, C.lib.attn_append_run_rope(
            ctypes.byref(pa), fake, fake, fake, fake, 8, 0, fake, fake, fake, 1, int(causal),
            ctypes.c_float(0.1), cos, cos, 48, fake, None, fake, 1 << 30, None)
    pa, st = append_rope([0, 30, 31], False)  # request 0: 19 kv tokens, 30 queries
    assert pa.min_kv_minus_qo == -11 and st == C.ERR_INVALID_ARG
    _, st = append_rope([0, 2, 3], True, ctypes.c_void_p(260))  # misaligned tables
    assert st == C.ERR_INVALID_ARG
    # a pool past 2^31 (page, head, slot) rows: UNSUPPORTED with the reason,
    # found on the host before any CUDA call
    huge = (1 << 31) // (2 * 16) + 1  # pages x Hk (2) x P (16) > 2^31
    st = C.lib.attn_decode_run(ctypes.byref(pr), fake, fake, fake, huge, 0, fake, fake, fake, 1,
                               ctypes.c_float(0.1), fake, None, fake, 1 << 30, None)
    assert st == C.ERR_UNSUPPORTED and "2^31" in C.last_error()
    # the wait self-test validates before it launches anything
    assert C.lib.attn_wait_selftest(None, 1000, None) == C.ERR_INVALID_ARG
    assert C.lib.attn_wait_selftest(ctypes.c_void_p(256), 0, None) == C.ERR_INVALID_ARG
    assert C.lib.attn_wait_selftest(ctypes.c_void_p(256), 10000001, None) == C.ERR_INVALID_ARG


def test_product_path_does_not_import_the_oracle():
    pkg = os.path.join(ROOT, "paged_kv_attention_bsr_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cpp", ".h", ".cuh")):
                text = open(os.path.join(dirpath, f)).read()
                assert "import oracle" not in text and "from oracle" not in text, f
                assert "attn_oracle" not in text, f


def test_rope_table_checks_in_the_binding():
    """The binding rejects malformed cos / sin tables before calling the library."""
    C = pytest.importorskip("paged_kv_attention_bsr_gb300._capi")
    import torch
    good = torch.zeros(10, 64, dtype=torch.float32)
    for cos, sin in [(good.double(), good), (torch.zeros(10, 32), torch.zeros(10, 32)),
                     (good, torch.zeros(11, 64)), (torch.zeros(64, 10).t(), good)]:
        with pytest.raises(ValueError):
            C._check_rope_tables(cos, sin)
    C._check_rope_tables(good, good.clone())


def test_run_size_checks_in_the_binding():
    """Pools, q, out and lse too small for the plan are rejected before the
    library is called (the kernels would read past a smaller pool)."""
    C = pytest.importorskip("paged_kv_attention_bsr_gb300._capi")
    import torch
    _, host = C.workspace_size(4, 4, 8, 2, 128, 4)
    p = C.plan(None, np.array([0, 2, 3], np.int32), np.array([5, 16], np.int32), 16, 8, 2, 128,
               False, 4, np.zeros(host, np.uint8))
    bf = torch.bfloat16
    q = torch.zeros(2, 8, 128, dtype=bf)
    pool = torch.zeros(3, 2, 16, 128, dtype=bf)
    lse = torch.zeros(2, 8)
    C._check_sizes(p, q, pool, pool, q, lse, 3, p.batch)  # consistent: no error
    bad = [
        (q, torch.zeros(3, 1, 16, 128, dtype=bf), pool, q, lse, 3),  # fewer heads
        (q, pool, pool, q, lse, 4),                                   # pool smaller than num_pages
        (q, pool.half(), pool, q, lse, 3),                            # dtype mismatch
        (q[:1], pool, pool, q, lse, 3),                               # too few q rows
        (q, pool, pool, q, lse.double(), 3),                          # lse dtype
        (q, pool, pool, q, lse, 0),                                   # no pages
    ]
    for qq, kp, vp, oo, ll, n in bad:
        with pytest.raises(ValueError):
            C._check_sizes(p, qq, kp, vp, oo, ll, n, p.batch)
    # a plan whose requests hold no kv tokens runs without a pool
    pe = C.plan(None, np.array([0, 0, 0], np.int32), np.array([0, 0], np.int32), 16, 8, 2, 128,
                False, 4, np.zeros(host, np.uint8))
    empty = torch.zeros(0, 2, 16, 128, dtype=bf)
    C._check_sizes(pe, q, empty, empty, q, lse, 0, pe.batch)


def test_strided_views_are_rejected_by_the_binding():
    """The kernels read every tensor as a dense block from its data pointer:
    strided views (a K slice of a [L, 2, H, D] tensor, a transposed q, a
    sliced pool) are rejected instead of being read with the wrong layout."""
    C = pytest.importorskip("paged_kv_attention_bsr_gb300._capi")
    import torch
    _, host = C.workspace_size(4, 4, 8, 2, 128, 4)
    p = C.plan(None, np.array([0, 2, 3], np.int32), np.array([5, 16], np.int32), 16, 8, 2, 128,
               False, 4, np.zeros(host, np.uint8))
    bf = torch.bfloat16
    q = torch.zeros(2, 8, 128, dtype=bf)
    pool = torch.zeros(3, 2, 16, 128, dtype=bf)
    lse = torch.zeros(2, 8)
    kv = torch.zeros(3, 2, 2, 16, 128, dtype=bf)  # [pages, K/V, Hk, P, D]
    q_t = torch.zeros(8, 2, 128, dtype=bf).transpose(0, 1)
    big = torch.zeros(4, 2, 16, 256, dtype=bf)[..., :128]
    for args in [(q, kv[:, 0], pool, q, lse), (q, pool, kv[:, 1], q, lse),
                 (q_t, pool, pool, q, lse), (q, big, big, q, lse),
                 (q, pool, pool, q_t, lse), (q, pool, pool, q, torch.zeros(8, 2).t())]:
        with pytest.raises(ValueError, match="contiguous"):
            C._check_sizes(p, *args, 3, p.batch)
    o = torch.zeros(4, 2, 128, dtype=bf)
    l = torch.zeros(4, 2)
    with pytest.raises(ValueError, match="contiguous"):
        C.merge_states(o, l, torch.zeros(2, 4, 128, dtype=bf).transpose(0, 1), l, o, l)
    with pytest.raises(ValueError, match="contiguous"):
        C.merge_states(o, torch.zeros(2, 4).t(), o, l, o, l)


def test_noalloc_binding_checks_sizes():
    """decode_run_noalloc checks its tensors against the explicit shapes
    before the library is called (the C side only sees raw pointers)."""
    C = pytest.importorskip("paged_kv_attention_bsr_gb300._capi")
    import torch
    bf = torch.bfloat16
    kvi = np.array([0, 2, 3], np.int32)
    lpl = np.array([5, 16], np.int32)
    q = torch.zeros(2, 8, 128, dtype=bf)
    pool = torch.zeros(3, 2, 16, 128, dtype=bf)
    lse = torch.zeros(2, 8)
    d32 = torch.zeros(3, dtype=torch.int32)
    for qq, kp, vp, oo, ll in [(q, pool[:, :1].contiguous(), pool, q, lse),
                               (q[:1], pool, pool, q, lse), (q, pool, pool, q[:1], lse),
                               (q, pool, pool, q, lse[:1]), (q, pool.half(), pool, q, lse),
                               (q, pool[:2], pool, q, lse)]:
        with pytest.raises(ValueError):
            C.decode_run_noalloc(kvi, lpl, 16, 8, 2, 128, qq, kp, vp, d32, d32, d32, 0.1, oo,
                                 ll, num_pages=3)


def test_merge_shape_checks_in_the_binding():
    C = pytest.importorskip("paged_kv_attention_bsr_gb300._capi")
    import torch
    o = torch.zeros(4, 2, 128, dtype=torch.bfloat16)
    l = torch.zeros(4, 2)
    for args in [(o, l, o[:3], l, o, l), (o, l, o, l[:3], o, l), (o, l, o, l, o.half(), l),
                 (o, l, o, l.double(), o, l)]:
        with pytest.raises(ValueError):
            C.merge_states(*args)


def test_cascade_entry_points_validate_without_gpu():
    C = pytest.importorskip("paged_kv_attention_bsr_gb300._capi")
    dev, host = C.cascade_workspace_size(4, 8, 32, 8, 128, 152)
    assert dev > host > 0
    with pytest.raises(C.AttnError) as ei:
        C.cascade_workspace_size(0, 8, 32, 8, 128, 152)
    assert ei.value.status == C.ERR_INVALID_ARG
    qo = np.array([0, 2, 3], np.int32)
    ip0, l0 = np.array([0, 4, 5], np.int32), np.array([16, 3], np.int32)
    ip1, l1 = np.array([0, 1, 3, 3], np.int32), np.array([5, 8, 0], np.int32)
    buf = np.zeros(host, np.uint8)
    p = C.plan_cascade(qo, ip0, l0, 16, ip1, l1, 8, 32, 8, 128, 152, buf)
    assert p.mode == C.MODE_CASCADE and p.total_qo == 3 and p.page_size_suffix == 8
    fake = ctypes.c_void_p(256)

    def run(plan, dev_ws=fake, dev_bytes=1 << 30, suffix_pool=fake, layout=0, pages=8):
        return C.lib.attn_cascade_run(ctypes.byref(plan), fake, fake, fake, fake, pages, fake,
                                      fake, fake, suffix_pool, suffix_pool, pages, fake, fake,
                                      fake, layout, 1, ctypes.c_float(0.1), fake, None, dev_ws,
                                      dev_bytes, None)
    assert run(p, dev_ws=None) == C.ERR_INVALID_ARG and "dev_ws" in C.last_error()
    assert run(p, dev_bytes=16) == C.ERR_WORKSPACE_TOO_SMALL
    assert run(p, suffix_pool=None) == C.ERR_INVALID_ARG and "suffix" in C.last_error()
    assert run(p, layout=7) == C.ERR_INVALID_ARG
    # a decode plan is not a cascade plan
    pd = C.plan(None, np.array([0, 1], np.int32), np.array([5], np.int32), 16, 32, 8, 128,
                False, 152, np.zeros(1 << 20, np.uint8))
    assert run(pd) == C.ERR_INVALID_ARG and "mode" in C.last_error()
    # gathered rows (suffix page size 8): 32-bit row indices, checked on the host
    huge = (1 << 31) // (8 * 8) + 1
    assert run(p, pages=huge) == C.ERR_UNSUPPORTED and "2^31" in C.last_error()


@pytest.mark.parametrize("bad", [-0.125, float("nan"), float("inf")])
def test_run_entry_points_reject_bad_sm_scale_without_gpu(bad):
    """Every run entry point checks sm_scale first (finite, >= 0): a bad scale
    returns INVALID_ARG naming sm_scale before anything touches a device."""
    C = pytest.importorskip("paged_kv_attention_bsr_gb300._capi")
    plan = C.Plan()
    fake = ctypes.c_void_p(256)
    names = ["attn_decode_run", "attn_decode_run_rope", "attn_decode_run_fp8",
             "attn_append_run", "attn_append_run_rope", "attn_cascade_run",
             "attn_decode_run_noalloc"]
    for name in names:
        fn = getattr(C.lib, name)
        args = []
        for t in fn.argtypes:
            if t is ctypes.c_float:
                args.append(ctypes.c_float(bad))
            elif t is ctypes.c_void_p:
                args.append(fake)
            elif t in (ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t):
                args.append(t(1))
            else:  # the plan
                args.append(ctypes.byref(plan))
        assert fn(*args) == C.ERR_INVALID_ARG, name
        assert "sm_scale" in C.last_error(), (name, C.last_error())
