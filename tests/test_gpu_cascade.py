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


@pytest.mark.parametrize("num_ctas", [1, 7, None, 304])
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
@pytest.mark.parametrize("num_ctas", [3, None, 304])
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


def _nhd(cache):
    """The same pool in the NHD layout [pages, P, Hk, D]."""
    return (cache.k_pool.permute(0, 2, 1, 3).contiguous(),
            cache.v_pool.permute(0, 2, 1, 3).contiguous())


# (gens, prefix lens, suffix lens, P0, P1, Hq, Hk, dtype, layout): page sizes
# that are not multiples of 16 and NHD pools copy rows one by one
ANY_PAGE = [
    ([2, 3], [100, 37], [5, 0, 70, 16, 200], 8, 16, 16, 4, torch.bfloat16, 0),
    ([4, 1], [1000, 0], [33, 1, 0, 90, 256], 128, 3, 32, 8, torch.float16, 0),
    ([3, 2], [512, 80], [16, 17, 0, 300, 40], 16, 16, 32, 8, torch.bfloat16, 1),
    ([2, 2], [45, 9], [1, 30, 7, 0], 1, 1, 16, 4, torch.bfloat16, 1),
    ([5], [333], [24, 48, 5, 0, 99], 24, 5, 6, 2, torch.float16, 1),
]


@pytest.mark.parametrize("case", range(len(ANY_PAGE)))
@pytest.mark.parametrize("num_ctas", [3, None, 304])
def test_one_launch_any_page_size_and_layout(oracle_mod, case, num_ctas):
    from paged_kv_attention_bsr_gb300.api import CascadeAttention
    gens, pre_lens, suf_lens, P0, P1, Hq, Hk, dtype, layout = ANY_PAGE[case]
    w = synth.cascade_workload(f"anyp{case}", gens, pre_lens, suf_lens, P0, P1, Hq, Hk, dtype,
                               seed=950 + case)
    pre, suf = w.extra["prefix"], w.cache
    poison_unused_slots(pre)
    poison_unused_slots(suf)
    o_ref, lse_ref = oracle_two_part(oracle_mod, w)  # on the HND pools: same logical cache
    dp, ds = to_device(pre), to_device(suf)
    if layout == 1:
        for d, c in ((dp, pre), (ds, suf)):
            kn, vn = _nhd(c)
            d["k_pool"], d["v_pool"] = kn.cuda(), vn.cuda()
    ca = CascadeAttention(Hq, Hk, 128, max_prompts=len(gens), max_batch=w.batch,
                          mode="one_launch", num_ctas=num_ctas)
    ca.plan(w.extra["prefix_qo_indptr"], pre.kv_indptr, pre.last_page_len, P0, suf.kv_indptr,
            suf.last_page_len, P1)
    o, l = ca.run(w.q.cuda(), dp, ds, torch.from_numpy(w.extra["prefix_qo_indptr"]).cuda(),
                  w.sm_scale, return_lse=True, layout=layout)
    torch.cuda.synchronize()
    assert ca.status() == 0
    assert_attn_close(o, l, o_ref, lse_ref, f"any page size case {case}")


def test_one_launch_rejects_more_than_16_rows():
    from paged_kv_attention_bsr_gb300 import _capi as C
    from paged_kv_attention_bsr_gb300.api import CascadeAttention
    # 8 query heads per kv head x 3 generations = 24 packed rows
    w = synth.cascade_workload("rows24", [3], [100], [10, 20, 30], 16, 16, 16, 2,
                               torch.bfloat16, seed=5)
    pre, suf = w.extra["prefix"], w.cache
    ca = CascadeAttention(16, 2, 128, max_prompts=1, max_batch=3, mode="one_launch")
    with pytest.raises(ValueError):
        ca.plan(w.extra["prefix_qo_indptr"], pre.kv_indptr, pre.last_page_len, 16,
                suf.kv_indptr, suf.last_page_len, 16)
    host = torch.zeros(1 << 16, dtype=torch.uint8)
    with pytest.raises(C.AttnError) as e:
        C.plan_cascade(w.extra["prefix_qo_indptr"], pre.kv_indptr, pre.last_page_len, 16,
                       suf.kv_indptr, suf.last_page_len, 16, 16, 2, 128, 4, host)
    assert e.value.status == 2
    # "auto" falls back to the two passes and still matches the flat result
    ca2 = CascadeAttention(16, 2, 128, max_prompts=1, max_batch=3, mode="auto")
    ca2.plan(w.extra["prefix_qo_indptr"], pre.kv_indptr, pre.last_page_len, 16,
             suf.kv_indptr, suf.last_page_len, 16)
    assert not ca2.one_launch


def test_one_launch_graph_replay_is_bit_identical(oracle_mod):
    """attn_cascade_run captured in a CUDA graph and replayed three times
    (the arrival counters reset inside the kernel) gives the eager result
    bit for bit."""
    w = synth.cascade_workload("graph", [3, 2, 4], [700, 2000, 130], [50, 0, 300, 17, 900, 64,
                                                                     1, 640, 260],
                               128, 16, 32, 8, torch.bfloat16, seed=905)
    o0, l0, ca = run_one_launch(w, num_ctas=5)
    pre, suf = w.extra["prefix"], w.cache
    q = w.q.cuda()
    dp, ds = to_device(pre), to_device(suf)
    qo = torch.from_numpy(w.extra["prefix_qo_indptr"]).cuda()
    o = torch.full_like(q, float("nan"))
    lse = torch.full(q.shape[:-1], float("nan"), dtype=torch.float32, device="cuda")
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):  # warm-up off the default stream, as capture requires
        ca.run(q, dp, ds, qo, w.sm_scale, out=o, lse=lse)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    o.fill_(float("nan"))
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        ca.run(q, dp, ds, qo, w.sm_scale, out=o, lse=lse)
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    assert ca.status() == 0
    assert torch.equal(o, o0) and torch.equal(lse, l0)


DEBUG_SCRIPT = """
import sys
import torch
sys.path.insert(0, {root!r})
from paged_kv_attention_bsr_gb300 import _capi as C, synth
from paged_kv_attention_bsr_gb300.api import CascadeAttention
from tests.gpu_util import to_device
w = synth.cascade_workload("dbg", [2, 1], [300, 40], [20, 0, 90], 16, 16, 16, 4,
                           torch.bfloat16, seed=907)
pre, suf = w.extra["prefix"], w.cache
ca = CascadeAttention(16, 4, 128, max_prompts=2, max_batch=3, mode="one_launch")
ca.plan(w.extra["prefix_qo_indptr"], pre.kv_indptr, pre.last_page_len, 16, suf.kv_indptr,
        suf.last_page_len, 16)
q = w.q.cuda()
qo = torch.from_numpy(w.extra["prefix_qo_indptr"]).cuda()
dp, ds = to_device(pre), to_device(suf)
used_p = int(pre.kv_indices.max()) + 1
used_s = int(suf.kv_indices.max()) + 1
dp["num_pages"], ds["num_pages"] = used_p, used_s
ca.run(q, dp, ds, qo, w.sm_scale)  # consistent tables: passes the checks
torch.cuda.synchronize()
out = []
bad = dict(ds)
bad["kv_indices"] = ds["kv_indices"].clone()
bad["kv_indices"][1] = used_s  # one past the declared suffix pages (inside the pool)
try:
    ca.run(q, dp, bad, qo, w.sm_scale)
    out.append("suffix index: accepted")
except C.AttnError as e:
    out.append(f"suffix index: {{e.status}} {{C.last_error()}}")
qo2 = qo.clone()
qo2[1] = 1  # a device qo_indptr that is not the plan's
try:
    ca.run(q, dp, ds, qo2, w.sm_scale)
    out.append("qo: accepted")
except C.AttnError as e:
    out.append(f"qo: {{e.status}} {{C.last_error()}}")
torch.cuda.synchronize()
assert ca.status() == 0
print("|".join(out))
"""


def test_one_launch_debug_checks_reject_bad_tables():
    """ATTN_DEBUG_CHECKS=1: an out-of-range suffix index and a device qo_indptr
    that differs from the plan's are rejected on the host before any launch
    (child process: the variable is read once per process)."""
    import os
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    env = dict(os.environ, ATTN_DEBUG_CHECKS="1")
    r = subprocess.run([sys.executable, "-c", DEBUG_SCRIPT.format(root=root)],
                       capture_output=True, text=True, env=env, cwd=root, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    idx, qo = r.stdout.strip().splitlines()[-1].split("|")
    assert idx.startswith("suffix index: 1 ") and "suffix kv_indices" in idx, idx
    assert qo.startswith("qo: 1 ") and "differ from the plan" in qo, qo
