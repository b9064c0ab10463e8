"""ATTN_DEBUG_CHECKS=1: the run calls read the device page table back and
check it on the host before any launch.

The variable is read once per process, so each check runs in a child
process. The bad inputs stay inside the memory the tensors own (an index past
the num_pages the call declares but inside the real pool), so nothing would
read outside an allocation even if a check were missing.
"""
import os
import subprocess
import sys
import textwrap

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

SCRIPT = textwrap.dedent("""
    import sys
    import numpy as np
    import torch
    sys.path.insert(0, {root!r})
    from paged_kv_attention_bsr_gb300 import _capi as C, synth
    from paged_kv_attention_bsr_gb300.api import PagedAttention
    from tests.gpu_util import to_device

    w = synth.decode_workload("dbg", [300, 40, 0, 129], 16, 64, 16, 4, torch.bfloat16, seed=3)
    c = w.cache
    att = PagedAttention(16, 4, 128, "decode", max_batch=4)
    att.plan(c.kv_indptr, c.last_page_len, 16)
    d = to_device(c)
    q = w.q.cuda()
    args = (q, d["k_pool"], d["v_pool"], d["kv_indptr"], d["kv_indices"], d["last_page_len"],
            w.sm_scale)
    used = int(c.kv_indices.max()) + 1
    att.run(*args, num_pages=used)  # consistent table: passes the checks
    torch.cuda.synchronize()
    out = []
    # one index past the declared num_pages (still inside the real pool)
    bad = d["kv_indices"].clone()
    bad[3] = used
    try:
        att.run(q, d["k_pool"], d["v_pool"], d["kv_indptr"], bad, d["last_page_len"],
                w.sm_scale, num_pages=used)
        out.append("index: accepted")
    except C.AttnError as e:
        out.append(f"index: {{e.status}} {{C.last_error()}}")
    # a device last_page_len that is not the plan's
    lpl = d["last_page_len"].clone()
    lpl[0] = 1
    try:
        att.run(q, d["k_pool"], d["v_pool"], d["kv_indptr"], d["kv_indices"], lpl, w.sm_scale,
                num_pages=used)
        out.append("table: accepted")
    except C.AttnError as e:
        out.append(f"table: {{e.status}} {{C.last_error()}}")
    torch.cuda.synchronize()
    assert att.status() == 0
    print("|".join(out))
""")


def _run(env_value):
    env = dict(os.environ)
    env["ATTN_DEBUG_CHECKS"] = env_value
    r = subprocess.run([sys.executable, "-c", SCRIPT.format(root=ROOT)], capture_output=True,
                       text=True, env=env, cwd=ROOT, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    return r.stdout.strip().splitlines()[-1]


def test_debug_checks_reject_bad_tables_before_launch():
    line = _run("1")
    index, table = line.split("|")
    assert index.startswith("index: 1 ") and "outside [0, num_pages" in index, index
    assert table.startswith("table: 1 ") and "differ from the plan" in table, table
