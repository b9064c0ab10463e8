#!/usr/bin/env python
"""Benchmark of the BSR paged-KV attention path on GB300.

Headline (one JSON line): paged batch decode, Llama-3.1-8B attention shape
(B = 64, Hq = 32, Hk = 8, D = 128, bf16, page_size 16, kv_len ~ U[1024, 4096],
pages drawn from a shuffled 20000-page pool). One step = plan() on the host
(table upload included) + one persistent decode launch (split units merged
in-kernel). `value` is algorithmic HBM bytes per step / step time (GB/s).

The line also carries, for the other workloads of the pages (single-request
decode, skewed 70B-shaped decode, shared-prefix composable decode, causal
append), their own time and roofline fraction under "workloads".

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

N > 1 runs independent replicas (one per GPU, launched by torchrun); the only
collectives are the timing barrier and a max over ranks.
"""
from __future__ import annotations

import argparse
import concurrent.futures as cf
import hashlib
import json
import math
import os
import re
import subprocess
import sys
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "paged decode attention HBM GB/s (% of ~8 TB/s); causal append TFLOP/s (% peak)"
L2_FLUSH_BYTES = 512 << 20  # > 2 x the 126 MB L2
L2_SCRUB_BYTES = 256 << 20
HOST_COVER_CYCLES = 2_000_000  # ~1 ms of GPU sleep before each timed step


# ------------------------------------------------------------------ helpers
def max_over_ranks(times, device):
    """Element-wise max of per-rank times over the process group (the job
    takes as long as its slowest replica)."""
    t = torch.tensor(times, device=device, dtype=torch.float64)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return [float(x) for x in t]


def whole_job_gbs(bytes_per_step, world, step_s):
    """Whole-job throughput: every replica moves bytes_per_step per step and
    the step time is the slowest replica's."""
    return bytes_per_step * world / step_s / 1e9


class L2Flush:
    """Between timed steps: write 512 MB (evicts every line of the previous
    step), then read 256 MB of another buffer, so that the dirty lines of the
    write are written back to HBM here and not during the next timed step
    (which then starts with an L2 holding only clean, unrelated lines)."""

    def __init__(self):
        self.buf = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device="cuda")
        self.scrub = torch.ones(L2_SCRUB_BYTES // 4, dtype=torch.int32, device="cuda")

    def __call__(self):
        self.buf.zero_()
        self.scrub.max()


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), float(p["bf16_tflops"]), "measured"
    except Exception:
        return 6800.0, 1900.0, "fallback"


def source_hash(*names):
    h = hashlib.sha256()
    for n in names:
        with open(os.path.join(ROOT, "paged_kv_attention_bsr_gb300", "csrc", n), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


# ncu summaries under profiles/ per workload, with the sources whose hash
# they record (the kernel's own files and the planner, whose cut sets the
# split items' partial-state traffic)
_TC = ["decode_tc.cu", "tc.cuh", "ptx.cuh", "plan.cpp", "internal.h"]
PROFILES = {
    "uniform_decode": ("decode_tc_kernel_uniform_gqa_b64.md", _TC),
    "skewed_decode": ("decode_tc_kernel_skewed_b128.md", _TC),
    "shared_prefix": ("decode_tc_kernel_cascade_16x4.md", _TC),
    "sparse_decode": ("decode_tc_kernel_sparse_p1_b64.md", _TC),
    "rope_decode": ("decode_tc_kernel_rope_uniform_gqa_b64.md", _TC),
    "fp8_decode": ("decode_tc_kernel_fp8_uniform_gqa_b64.md", _TC),
    "single_decode": ("decode_kernel_single_h32_kv2048.md",
                      ["decode.cu", "ptx.cuh", "plan.cpp", "internal.h"]),
    "causal_append": ("append_kernel_causal_b16.md",
                      ["append.cu", "tc.cuh", "ptx.cuh", "plan.cpp", "internal.h"]),
}


def profile_traffic(profile_name, kernel_sources):
    """DRAM bytes per launch recorded by an ncu capture, if the kernel source
    has not changed since (profiles/<name> lists the source hash)."""
    path = os.path.join(ROOT, "profiles", profile_name)
    if not os.path.exists(path):
        return None
    text = open(path).read()
    m = re.search(r"source_hash:\s*([0-9a-f]+)", text)
    t = re.search(r"traffic_bytes_per_launch:\s*([0-9.eE+]+)", text)
    if not m or not t or m.group(1) != source_hash(*kernel_sources):
        return None
    return float(t.group(1))


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled during the timed region."""
    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.idx = gpu_index
        self.proc = None
        self.out = None

    def start(self):
        try:
            self.out = open(f"/tmp/bench_clocks_{os.getpid()}.csv", "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.idx), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"], stdout=self.out,
                stderr=subprocess.DEVNULL)
            time.sleep(1.0)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.out.close()
        rows = []
        for line in open(self.out.name):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 10:
                rows.append(parts)
        os.remove(self.out.name)
        return rows


def summarise_clocks(rows, t0, t1):
    if not rows:
        return None
    sel = []
    for r in rows:
        try:
            ts = time.mktime(time.strptime(r[0].split(".")[0], "%Y/%m/%d %H:%M:%S"))
        except Exception:
            ts = None
        if ts is None or (t0 - 1.0 <= ts <= t1 + 1.0):
            sel.append(r)
    sel = sel or rows
    sm = [float(r[2]) for r in sel if r[2].replace(".", "").isdigit()]
    mx = [float(r[3]) for r in sel if r[3].replace(".", "").isdigit()]
    reasons = set()
    names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
    for r in sel:
        for k, name in enumerate(names):
            if "Active" in r[6 + k] and "Not" not in r[6 + k]:
                reasons.add(name)
    return {"sm_mhz": float(np.median(sm)) if sm else None,
            "sm_max_mhz": max(mx) if mx else None, "reasons": sorted(reasons),
            "samples": len(sel)}


def decode_bytes(w):
    c = w.cache
    elt = 2
    kv = int(c.kv_lens.sum()) * 2 * w.num_kv_heads * w.head_dim * elt
    qo = 2 * w.batch * w.num_qo_heads * w.head_dim * elt + 4 * w.batch * w.num_qo_heads
    idx = 4 * len(c.kv_indices) + 4 * (w.batch + 1) + 4 * w.batch
    return kv + qo + idx


def append_flops(w):
    qo = np.diff(w.qo_indptr).astype(np.float64)
    E = w.cache.kv_lens.astype(np.float64) - qo
    return float(np.sum(w.num_qo_heads * 4.0 * w.head_dim * (qo * E + qo * (qo + 1) / 2)))


def dev_cache(cache):
    return dict(k_pool=cache.k_pool.cuda(), v_pool=cache.v_pool.cuda(),
                kv_indptr=torch.from_numpy(cache.kv_indptr).cuda(),
                kv_indices=torch.from_numpy(cache.kv_indices).cuda(),
                last_page_len=torch.from_numpy(cache.last_page_len).cuda())


# --------------------------------------------------------------- our path
class DecodeStep:
    """plan + run of one decode batch through the public API."""

    def __init__(self, w, rope=None):
        from paged_kv_attention_bsr_gb300.api import PagedAttention
        self.w = w
        self.rope = rope
        c = w.cache
        self.att = PagedAttention(w.num_qo_heads, w.num_kv_heads, w.head_dim, "decode",
                                  max_batch=w.batch)
        self.d = dev_cache(c)
        self.q = w.q.cuda()
        self.o = torch.empty_like(self.q)
        self.lse = torch.empty(self.q.shape[:-1], dtype=torch.float32, device="cuda")

    def plan(self):
        c = self.w.cache
        self.att.plan(c.kv_indptr, c.last_page_len, c.page_size)

    def run(self):
        d = self.d
        self.att.run(self.q, d["k_pool"], d["v_pool"], d["kv_indptr"], d["kv_indices"],
                     d["last_page_len"], self.w.sm_scale, out=self.o, lse=self.lse,
                     rope=self.rope)


def time_steps(step_fns, steps, warmup, flush, kernel_split=1):
    """Per-step CUDA events on the current stream. step_fns: list of callables
    run in order; events are recorded before fn[0], before fn[kernel_split]
    and after the last, so `kernel` times fns[kernel_split:]."""
    for _ in range(warmup):
        flush()
        for f in step_fns:
            f()
    torch.cuda.synchronize()
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(steps)]
    for k in range(steps):
        flush()
        # keep the GPU busy while the host enqueues the step, so that the
        # events time the step's device work, not the host's enqueue latency
        torch.cuda._sleep(HOST_COVER_CYCLES)
        evs[k][0].record()
        for i, f in enumerate(step_fns):
            if i == kernel_split:
                evs[k][1].record()
            f()
        if kernel_split >= len(step_fns):
            evs[k][1].record()
        evs[k][2].record()
    torch.cuda.synchronize()
    step_ms = np.array([e[0].elapsed_time(e[2]) for e in evs])
    kern_ms = np.array([e[1].elapsed_time(e[2]) for e in evs])
    return step_ms, kern_ms


def bench_decode_workload(key, hbm_peak, bf16_peak, flush, steps, warmup):
    from paged_kv_attention_bsr_gb300 import synth
    w = synth.WORKLOADS[key]()
    st = DecodeStep(w)
    step_ms, kern_ms = time_steps([st.plan, st.run], steps, warmup, flush)
    b = decode_bytes(w)
    k_s = float(np.median(kern_ms)) * 1e-3
    res = {"kind": "decode", "bytes": b, "kernel_us": k_s * 1e6,
           "step_us": float(np.median(step_ms)) * 1e3,
           "GB/s": b / k_s / 1e9, "roofline_frac_hbm": b / k_s / 1e9 / hbm_peak,
           "units": st.att.plan_info.num_units,
           "split_items": st.att.plan_info.num_split_items}
    assert st.att.status() == 0
    del st
    torch.cuda.empty_cache()
    return w.name, res


def bench_causal_append(hbm_peak, bf16_peak, flush, steps, warmup):
    from paged_kv_attention_bsr_gb300 import synth
    from paged_kv_attention_bsr_gb300.api import PagedAttention
    w = synth.causal_append()
    c = w.cache
    att = PagedAttention(w.num_qo_heads, w.num_kv_heads, 128, "append", max_batch=w.batch,
                         max_total_qo=int(w.qo_indptr[-1]))
    d = dev_cache(c)
    q = w.q.cuda()
    qo = torch.from_numpy(w.qo_indptr).cuda()
    o = torch.empty_like(q)
    lse = torch.empty(q.shape[:-1], dtype=torch.float32, device="cuda")

    def plan_a():
        att.plan(c.kv_indptr, c.last_page_len, 16, qo_indptr_h=w.qo_indptr, causal=True)

    def run_a():
        att.run(q, d["k_pool"], d["v_pool"], d["kv_indptr"], d["kv_indices"], d["last_page_len"],
                w.sm_scale, out=o, lse=lse, qo_indptr=qo)

    step_ms, kern_ms = time_steps([plan_a, run_a], steps, warmup, flush)
    fl = append_flops(w)
    k_s = float(np.median(kern_ms)) * 1e-3
    res = {"kind": "append", "flops": fl, "kernel_us": k_s * 1e6,
           "step_us": float(np.median(step_ms)) * 1e3, "TFLOP/s": fl / k_s / 1e12,
           "roofline_frac_bf16": fl / k_s / 1e12 / bf16_peak,
           "units": att.plan_info.num_units, "split_items": att.plan_info.num_split_items,
           "launches_per_step": 1 + (att.plan_info.num_split_items > 0)}
    assert att.status() == 0
    del d, att
    torch.cuda.empty_cache()
    return w.name, res


def bench_shared_prefix(hbm_peak, bf16_peak, flush, steps, warmup):
    """Composable formats in one launch (CascadeAttention: prefix pages at
    P = 128 read once per prompt and suffix pages at P = 16 balanced together
    by attn_plan_cascade, merged inside the kernel), beside the two-pass
    variant (prefix append and suffix decode on two streams + LSE merge) and
    the same logical KV as one flat P = 16 decode."""
    from paged_kv_attention_bsr_gb300 import synth
    from paged_kv_attention_bsr_gb300.synth import Workload
    w = synth.shared_prefix_decode()
    pre, suf = w.extra["prefix"], w.cache
    q = w.q.cuda()
    dp, ds = dev_cache(pre), dev_cache(suf)
    pqo_h = w.extra["prefix_qo_indptr"]
    pqo = torch.from_numpy(pqo_h).cuda()
    from paged_kv_attention_bsr_gb300.api import CascadeAttention
    o_m = torch.empty_like(q)
    l_m = torch.empty(q.shape[:-1], dtype=torch.float32, device="cuda")
    kvb = 2 * 8 * 128 * 2
    b_pre = int(pre.kv_lens.sum()) * kvb
    b_suf = int(suf.kv_lens.sum()) * kvb
    b_flat = int(pre.kv_lens.sum()) * w.extra["n"] * kvb + b_suf

    def timed(mode):
        ca = CascadeAttention(32, 8, 128, max_prompts=w.extra["prompts"], max_batch=w.batch,
                              mode=mode)

        def plans():
            ca.plan(pqo_h, pre.kv_indptr, pre.last_page_len, pre.page_size, suf.kv_indptr,
                    suf.last_page_len, suf.page_size)

        def runs():
            ca.run(q, dp, ds, pqo, w.sm_scale, out=o_m, lse=l_m)

        step_ms, kern_ms = time_steps([plans, runs], steps, warmup, flush)
        assert ca.status() == 0
        return ca, float(np.median(step_ms)) * 1e3, float(np.median(kern_ms)) * 1e-3

    ca, step_us, k_s = timed("one_launch")
    # host planning time of attn_plan_cascade alone (tables into host memory)
    from paged_kv_attention_bsr_gb300 import _capi as C
    _, host_bytes = C.cascade_workspace_size(w.extra["prompts"], w.batch, 32, 8, 128,
                                             ca.num_ctas)
    hbuf = np.zeros(host_bytes, np.uint8)
    pts = []
    for _ in range(200):
        t0 = time.perf_counter()
        C.plan_cascade(pqo_h, pre.kv_indptr, pre.last_page_len, pre.page_size, suf.kv_indptr,
                       suf.last_page_len, suf.page_size, 32, 8, 128, ca.num_ctas, hbuf)
        pts.append(time.perf_counter() - t0)
    res_plan_us = float(np.median(pts)) * 1e6
    res = {"kind": "composable", "bytes": b_pre + b_suf, "flat_layout_bytes": b_flat,
           "plan_us_host": res_plan_us,
           "kernel_us": k_s * 1e6, "step_us": step_us,
           "GB/s": (b_pre + b_suf) / k_s / 1e9,
           "roofline_frac_hbm": (b_pre + b_suf) / k_s / 1e9 / hbm_peak,
           "launches_per_step": 1,
           "path": "one launch: prefix and suffix units of every (prompt, kv head) in one "
                   "persistent few-row kernel, merged in the kernel",
           "plan_units": ca.plan_info.num_units}
    ca2, step2_us, k2_s = timed("two_pass")
    res["two_pass"] = {"kernel_us": k2_s * 1e6, "step_us": step2_us,
                       "GB/s": (b_pre + b_suf) / k2_s / 1e9,
                       "roofline_frac_hbm": (b_pre + b_suf) / k2_s / 1e9 / hbm_peak,
                       "launches_per_step": 3 + (ca2.prefix.plan_info.num_split_items > 0),
                       "streams": "prefix pass and suffix pass on two streams, merge after "
                                  "the join"}
    del dp, ds, ca, ca2
    flat = synth.flat_layout_of_composable(w)
    wf = Workload("flat", "decode", torch.bfloat16, 32, 8, 128, w.sm_scale, w.q, flat)
    st = DecodeStep(wf)
    _, kern_ms = time_steps([st.plan, st.run], steps, warmup, flush)
    res["flat_layout_kernel_us"] = float(np.median(kern_ms)) * 1e3
    del st
    torch.cuda.empty_cache()
    return w.name, res


def bench_rope_decode(hbm_peak, bf16_peak, flush, steps, warmup):
    """The uniform GQA decode batch with LLaMA 3.1 RoPE fused into the kernel
    (keys cached un-rotated, turned in shared memory), beside the same batch
    without RoPE."""
    from paged_kv_attention_bsr_gb300 import synth
    w = synth.uniform_gqa_decode()
    max_pos = int(w.cache.kv_lens.max())
    cos, sin = synth.rope_tables(max_pos)
    rope = (torch.from_numpy(cos).cuda(), torch.from_numpy(sin).cuda())
    st = DecodeStep(w, rope=rope)
    step_ms, kern_ms = time_steps([st.plan, st.run], steps, warmup, flush)
    b = decode_bytes(w) + 2 * max_pos * 64 * 4  # + the cos / sin rows
    k_s = float(np.median(kern_ms)) * 1e-3
    res = {"kind": "decode+rope", "bytes": b, "kernel_us": k_s * 1e6,
           "step_us": float(np.median(step_ms)) * 1e3,
           "GB/s": b / k_s / 1e9, "roofline_frac_hbm": b / k_s / 1e9 / hbm_peak}
    assert st.att.status() == 0
    plain = DecodeStep(w)
    _, kern_plain = time_steps([plain.plan, plain.run], steps, warmup, flush)
    res["without_rope_kernel_us"] = float(np.median(kern_plain)) * 1e3
    del st, plain
    torch.cuda.empty_cache()
    return w.name + "_rope", res


def bench_fp8_decode(hbm_peak, bf16_peak, flush, steps, warmup):
    """The uniform GQA decode shape over an FP8 E4M3 KV cache (per-head
    scales), beside the bf16 cache's time for the same lengths."""
    from paged_kv_attention_bsr_gb300 import synth
    from paged_kv_attention_bsr_gb300.api import PagedAttention
    w = synth.fp8_uniform_gqa_decode()
    c = w.cache
    att = PagedAttention(w.num_qo_heads, w.num_kv_heads, 128, "decode", max_batch=w.batch)
    d = dev_cache(c)
    scales = (c.k_scale.cuda(), c.v_scale.cuda())
    q = w.q.cuda()
    o = torch.empty_like(q)
    lse = torch.empty(q.shape[:-1], dtype=torch.float32, device="cuda")

    def plan_f():
        att.plan(c.kv_indptr, c.last_page_len, 16)

    def run_f():
        att.run(q, d["k_pool"], d["v_pool"], d["kv_indptr"], d["kv_indices"], d["last_page_len"],
                w.sm_scale, out=o, lse=lse, kv_scales=scales)

    step_ms, kern_ms = time_steps([plan_f, run_f], steps, warmup, flush)
    assert att.status() == 0
    kv = int(c.kv_lens.sum()) * 2 * w.num_kv_heads * w.head_dim  # one byte per element
    qo = 2 * w.batch * w.num_qo_heads * w.head_dim * 2 + 4 * w.batch * w.num_qo_heads
    idx = 4 * len(c.kv_indices) + 8 * w.batch + 4 + 8 * w.num_kv_heads
    b = kv + qo + idx
    k_s = float(np.median(kern_ms)) * 1e-3
    res = {"kind": "decode_fp8kv", "bytes": b, "kernel_us": k_s * 1e6,
           "step_us": float(np.median(step_ms)) * 1e3, "GB/s": b / k_s / 1e9,
           "roofline_frac_hbm": b / k_s / 1e9 / hbm_peak,
           "kernel": "decode_tc_kernel<bf16 q, 4 rows, decode, FP8 K/V> (tensor cores; E4M3 tiles staged by TMA and widened to f16 in shared memory)"}
    del d, att
    torch.cuda.empty_cache()
    return w.name, res


def bench_rope_append(hbm_peak, bf16_peak, flush, steps, warmup):
    """The causal append with LLaMA 3.1 RoPE fused into the append kernel
    (keys cached un-rotated, turned in shared memory by the rope warps),
    beside the same batch without RoPE."""
    from paged_kv_attention_bsr_gb300 import synth
    from paged_kv_attention_bsr_gb300.api import PagedAttention
    w = synth.causal_append()
    c = w.cache
    cos, sin = synth.rope_tables(int(c.kv_lens.max()))
    rope = (torch.from_numpy(cos).cuda(), torch.from_numpy(sin).cuda())
    att = PagedAttention(w.num_qo_heads, w.num_kv_heads, 128, "append", max_batch=w.batch,
                         max_total_qo=int(w.qo_indptr[-1]))
    d = dev_cache(c)
    q = w.q.cuda()
    qo = torch.from_numpy(w.qo_indptr).cuda()
    o = torch.empty_like(q)
    lse = torch.empty(q.shape[:-1], dtype=torch.float32, device="cuda")

    def plan_a():
        att.plan(c.kv_indptr, c.last_page_len, 16, qo_indptr_h=w.qo_indptr, causal=True)

    def run_rope():
        att.run(q, d["k_pool"], d["v_pool"], d["kv_indptr"], d["kv_indices"], d["last_page_len"],
                w.sm_scale, out=o, lse=lse, qo_indptr=qo, rope=rope)

    def run_plain():
        att.run(q, d["k_pool"], d["v_pool"], d["kv_indptr"], d["kv_indices"], d["last_page_len"],
                w.sm_scale, out=o, lse=lse, qo_indptr=qo)

    step_ms, kern_ms = time_steps([plan_a, run_rope], steps, warmup, flush)
    assert att.status() == 0
    _, kern_plain = time_steps([plan_a, run_plain], steps, warmup, flush)
    fl = append_flops(w)
    k_s = float(np.median(kern_ms)) * 1e-3
    res = {"kind": "append+rope", "flops": fl, "kernel_us": k_s * 1e6,
           "step_us": float(np.median(step_ms)) * 1e3, "TFLOP/s": fl / k_s / 1e12,
           "roofline_frac_bf16": fl / k_s / 1e12 / bf16_peak,
           "without_rope_kernel_us": float(np.median(kern_plain)) * 1e3}
    del d, att
    torch.cuda.empty_cache()
    return w.name + "_rope", res


def bench_pod_mixed(hbm_peak, bf16_peak, flush, steps, warmup):
    """POD-style: one batch of 16 causal prefill chunks and 64 decodes, run
    as one plan and one persistent launch, beside the same batch run as two
    launches (the prefill requests on the append kernel, the decode requests
    on the decode kernel)."""
    from paged_kv_attention_bsr_gb300 import synth
    from paged_kv_attention_bsr_gb300.api import PagedAttention
    w = synth.pod_mixed_batch()
    c = w.cache
    d = dev_cache(c)
    q = w.q.cuda()
    qo = torch.from_numpy(w.qo_indptr).cuda()
    o = torch.empty_like(q)
    lse = torch.empty(q.shape[:-1], dtype=torch.float32, device="cuda")
    att = PagedAttention(32, 8, 128, "append", max_batch=w.batch,
                         max_total_qo=int(w.qo_indptr[-1]))

    def plan_f():
        att.plan(c.kv_indptr, c.last_page_len, 16, qo_indptr_h=w.qo_indptr, causal=True)

    def run_f():
        att.run(q, d["k_pool"], d["v_pool"], d["kv_indptr"], d["kv_indices"], d["last_page_len"],
                w.sm_scale, out=o, lse=lse, qo_indptr=qo)

    step_ms, kern_ms = time_steps([plan_f, run_f], steps, warmup, flush)
    assert att.status() == 0
    fused_us = float(np.median(kern_ms)) * 1e3
    # the same requests as two batches: prefill (append kernel), decode (decode kernel)
    wa = synth.sub_batch(w, w.extra["prefill"])
    wd = synth.sub_batch(w, w.extra["decode"], as_decode=True)
    da = {k: torch.from_numpy(getattr(wa.cache, k)).cuda()
          for k in ("kv_indptr", "kv_indices", "last_page_len")}
    dd = {k: torch.from_numpy(getattr(wd.cache, k)).cuda()
          for k in ("kv_indptr", "kv_indices", "last_page_len")}
    qa, qd = wa.q.cuda(), wd.q.cuda()
    qoa = torch.from_numpy(wa.qo_indptr).cuda()
    oa, od = torch.empty_like(qa), torch.empty_like(qd)
    la = torch.empty(qa.shape[:-1], dtype=torch.float32, device="cuda")
    ld = torch.empty(qd.shape[:-1], dtype=torch.float32, device="cuda")
    att_a = PagedAttention(32, 8, 128, "append", max_batch=wa.batch,
                           max_total_qo=int(wa.qo_indptr[-1]))
    att_d = PagedAttention(32, 8, 128, "decode", max_batch=wd.batch)

    def plans():
        att_a.plan(wa.cache.kv_indptr, wa.cache.last_page_len, 16, qo_indptr_h=wa.qo_indptr,
                   causal=True)
        att_d.plan(wd.cache.kv_indptr, wd.cache.last_page_len, 16)

    def runs():
        att_a.run(qa, d["k_pool"], d["v_pool"], da["kv_indptr"], da["kv_indices"],
                  da["last_page_len"], w.sm_scale, out=oa, lse=la, qo_indptr=qoa)
        att_d.run(qd, d["k_pool"], d["v_pool"], dd["kv_indptr"], dd["kv_indices"],
                  dd["last_page_len"], w.sm_scale, out=od, lse=ld)

    _, kern_sep = time_steps([plans, runs], steps, warmup, flush)
    assert att_a.status() == 0 and att_d.status() == 0
    sep_us = float(np.median(kern_sep)) * 1e3
    fl = append_flops(wa)
    kv_dec = int(wd.cache.kv_lens.sum()) * 2 * 8 * 128 * 2
    res = {"kind": "pod", "prefill_flops": fl, "decode_kv_bytes": kv_dec,
           "kernel_us": fused_us, "step_us": float(np.median(step_ms)) * 1e3,
           "separate_two_launches_kernel_us": sep_us, "fused_speedup": sep_us / fused_us,
           "launches_per_step": 1 + (att.plan_info.num_split_items > 0),
           "units": att.plan_info.num_units, "split_items": att.plan_info.num_split_items}
    del d, att, att_a, att_d
    torch.cuda.empty_cache()
    return w.name, res


WORKLOAD_BENCH = {
    "single_decode": lambda *a: bench_decode_workload("single_decode", *a),
    "skewed_decode": lambda *a: bench_decode_workload("skewed_decode", *a),
    "uniform_decode": lambda *a: bench_decode_workload("uniform_decode", *a),
    "causal_append": bench_causal_append,
    "shared_prefix": bench_shared_prefix,
    "rope_decode": bench_rope_decode,
    "sparse_decode": lambda *a: bench_decode_workload("sparse_decode", *a),
    "pod_mixed": bench_pod_mixed,
    "rope_append": bench_rope_append,
    "fp8_decode": bench_fp8_decode,
}


def extra_workloads(hbm_peak, bf16_peak, flush, steps=30, warmup=3):
    """Every other workload of the pages; per workload the median over
    `steps` CUDA-event-timed steps (kernel_us: the run's launches only)."""
    out = {}
    for key in ("single_decode", "skewed_decode", "causal_append", "shared_prefix",
                "rope_decode", "rope_append", "sparse_decode", "pod_mixed", "fp8_decode"):
        name, res = WORKLOAD_BENCH[key](hbm_peak, bf16_peak, flush, steps, warmup)
        if key in PROFILES:  # DRAM bytes per launch from the ncu capture at this source
            t = profile_traffic(*PROFILES[key])
            res["traffic_bytes_per_launch"] = t
            if t is not None and "bytes" in res:
                res["traffic_over_algorithmic"] = t / res["bytes"]
        out[name] = res
    return out


def cpu_oracle_baseline(w, threads):
    """The fp64 C oracle over the whole batch, requests split across threads
    (ctypes releases the GIL, so threads run on separate cores)."""
    import oracle
    c = w.cache
    B = w.batch
    chunks = np.array_split(np.arange(B), threads)
    odt = oracle.BF16 if w.dtype == torch.bfloat16 else oracle.F16

    def job(rs):
        if len(rs) == 0:
            return
        a, b = int(rs[0]), int(rs[-1]) + 1
        oracle.batch_attention(w.q[a:b], c.k_pool, c.v_pool, c.kv_indptr[a:b + 1],
                               c.kv_indices, c.last_page_len[a:b], c.page_size,
                               w.num_qo_heads, w.num_kv_heads, w.head_dim, odt, w.sm_scale)

    oracle.build()
    passes = 0
    t0 = time.perf_counter()
    with cf.ThreadPoolExecutor(threads) as ex:
        while True:  # whole passes over the batch, ~10+ s of CPU work in total
            list(ex.map(job, chunks))
            passes += 1
            if (time.perf_counter() - t0) * threads >= 10.0 or passes >= 64:
                break
    return (time.perf_counter() - t0) / passes, passes


def _decode_oracle_job(w, odt):
    """A callable that runs the fp64 oracle over requests [a, b) of a decode
    workload."""
    import oracle
    c = w.cache

    def job(rs):
        if len(rs) == 0:
            return
        a, b = int(rs[0]), int(rs[-1]) + 1
        oracle.batch_attention(w.q[a:b], c.k_pool, c.v_pool, c.kv_indptr[a:b + 1],
                               c.kv_indices, c.last_page_len[a:b], c.page_size,
                               w.num_qo_heads, w.num_kv_heads, w.head_dim, odt, w.sm_scale)
    return job


def _timed_pass(job, units, threads):
    """Seconds for one pass of `job` over `units` split into `threads` chunks."""
    chunks = np.array_split(np.asarray(units), threads)
    t0 = time.perf_counter()
    if threads == 1:
        job(chunks[0])
    else:
        with cf.ThreadPoolExecutor(threads) as ex:
            list(ex.map(job, chunks))
    return time.perf_counter() - t0


def cpu_oracle_per_workload(threads):
    """The fp64 oracle as it stands on the host cores, per workload of the
    pages: single-threaded and on `threads` threads (requests split across
    threads). Workloads 1-4 run in full; the causal append runs on a fixed
    seeded subset of (request, query head) pairs and is extrapolated by
    unmasked FLOPs, and labelled so."""
    import oracle
    from paged_kv_attention_bsr_gb300 import synth
    oracle.build()
    out = {}
    for key in ("single_decode", "uniform_decode", "skewed_decode"):
        w = synth.WORKLOADS[key]()
        odt = oracle.BF16 if w.dtype == torch.bfloat16 else oracle.F16
        b = decode_bytes(w)
        if w.batch >= threads:  # requests split across threads
            job = _decode_oracle_job(w, odt)
            units = np.arange(w.batch)
        else:  # fewer requests than threads: (request, head) rows split across threads
            c = w.cache
            units = np.arange(w.batch * w.num_qo_heads)

            def job(idx, w=w, c=c, odt=odt):
                for u in idx:
                    r, h = divmod(int(u), w.num_qo_heads)
                    oracle.attention_row(w.q, c.k_pool, c.v_pool, c.kv_indptr, c.kv_indices,
                                         c.last_page_len, c.page_size, w.num_qo_heads,
                                         w.num_kv_heads, w.head_dim, odt, w.sm_scale, r, 0, h)
        t1 = _timed_pass(job, units, 1)
        tn = _timed_pass(job, units, threads)
        out[w.name] = {"unit": "GB/s", "threads_1": b / t1 / 1e9, f"threads_{threads}": b / tn / 1e9,
                       "sample": "whole workload, one pass"}
    # shared prefix: prefix pass (qo_len = n per prompt, non-causal) + suffix
    # decode + LSE merge, over the bytes the composable layout reads
    w = synth.shared_prefix_decode()
    pre, suf = w.extra["prefix"], w.cache
    n = w.extra["n"]
    pqo = w.extra["prefix_qo_indptr"]

    def comp_job(ps):
        for p_ in ps:
            p_ = int(p_)
            rs = slice(p_ * n, (p_ + 1) * n)
            op, lp = oracle.batch_attention(
                w.q[rs], pre.k_pool, pre.v_pool, pre.kv_indptr[p_:p_ + 2], pre.kv_indices,
                pre.last_page_len[p_:p_ + 1], pre.page_size, 32, 8, 128, oracle.BF16, w.sm_scale,
                qo_indptr=pqo[p_:p_ + 2] - pqo[p_])
            os_, ls = oracle.batch_attention(
                w.q[rs], suf.k_pool, suf.v_pool, suf.kv_indptr[p_ * n:(p_ + 1) * n + 1],
                suf.kv_indices, suf.last_page_len[rs], suf.page_size, 32, 8, 128, oracle.BF16,
                w.sm_scale)
            oracle.merge_states(np.stack([op.reshape(-1, 128), os_.reshape(-1, 128)]),
                                np.stack([lp.reshape(-1), ls.reshape(-1)]))

    kvb = 2 * 8 * 128 * 2
    b = (int(pre.kv_lens.sum()) + int(suf.kv_lens.sum())) * kvb
    t1 = _timed_pass(comp_job, np.arange(w.extra["prompts"]), 1)
    tn = _timed_pass(comp_job, np.arange(w.extra["prompts"]), threads)
    out[w.name] = {"unit": "GB/s", "threads_1": b / t1 / 1e9, f"threads_{threads}": b / tn / 1e9,
                   "sample": "whole workload, one pass (prefix + suffix + merge)"}
    # causal append: a seeded subset of (request, head) pairs, every query row
    w = synth.causal_append()
    c = w.cache
    qo = np.diff(w.qo_indptr)
    E = c.kv_lens - qo
    rng = np.random.default_rng(20260005)
    pairs = [(int(rng.integers(w.batch)), int(rng.integers(w.num_qo_heads)))
             for _ in range(threads)]

    def pair_flops(r):
        L = float(qo[r])
        return 4.0 * w.head_dim * (L * E[r] + L * (L + 1) / 2)

    def app_job(idx):
        for k in idx:
            r, h = pairs[int(k)]
            for i in range(int(qo[r])):
                oracle.attention_row(w.q, c.k_pool, c.v_pool, c.kv_indptr, c.kv_indices,
                                     c.last_page_len, 16, 32, 8, 128, oracle.BF16, w.sm_scale,
                                     r, i, h, causal=True, qo_indptr=w.qo_indptr)

    f1 = pair_flops(pairs[0][0])
    t1 = _timed_pass(app_job, [0], 1)
    fn = sum(pair_flops(r) for r, _ in pairs)
    tn = _timed_pass(app_job, np.arange(len(pairs)), threads)
    total = append_flops(w)
    out[w.name] = {"unit": "TFLOP/s", "threads_1": f1 / t1 / 1e12,
                   f"threads_{threads}": fn / tn / 1e12,
                   "sample": f"subset: 1 (request, head) pair single-threaded, {len(pairs)} pairs "
                             f"on {threads} threads (seeded), every query row of each pair; "
                             f"extrapolated to the whole workload ({total / 1e12:.3f} TFLOP) by "
                             f"unmasked FLOPs",
                   "extrapolated_whole_workload_s": {"threads_1": total / (f1 / t1),
                                                     f"threads_{threads}": total / (fn / tn)}}
    return out


def plan_times(w, num_ctas):
    """Host planning time of the headline batch: attn_plan through the C ABI
    with no device workspace (the planner alone), and the public API's plan()
    (planner + table upload enqueue), median over repeated calls."""
    from paged_kv_attention_bsr_gb300 import _capi as C
    from paged_kv_attention_bsr_gb300.api import PagedAttention
    c = w.cache
    _, host = C.workspace_size(w.batch, w.batch, w.num_qo_heads, w.num_kv_heads, 128, num_ctas)
    buf = np.zeros(host, np.uint8)
    kvi = np.ascontiguousarray(c.kv_indptr, np.int32)
    lpl = np.ascontiguousarray(c.last_page_len, np.int32)
    t = []
    for _ in range(300):
        t0 = time.perf_counter()
        C.plan(None, kvi, lpl, c.page_size, w.num_qo_heads, w.num_kv_heads, 128, False,
               num_ctas, buf)
        t.append(time.perf_counter() - t0)
    att = PagedAttention(w.num_qo_heads, w.num_kv_heads, 128, "decode", max_batch=w.batch,
                         num_ctas=num_ctas)
    t2 = []
    for _ in range(300):
        t0 = time.perf_counter()
        att.plan(kvi, lpl, c.page_size)
        t2.append(time.perf_counter() - t0)
    torch.cuda.synchronize()
    return {"c_abi_host_only_us": float(np.median(t)) * 1e6,
            "api_plan_with_upload_us": float(np.median(t2)) * 1e6,
            "note": "median of 300 calls on the host (ctypes call included); the upload is an "
                    "asynchronous copy enqueued on the stream"}


def run_ours(args, rank, world):
    from paged_kv_attention_bsr_gb300 import synth
    hbm_peak, bf16_peak, peak_src = peaks()
    torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", 0)))
    w = synth.uniform_gqa_decode()
    st = DecodeStep(w)
    flush = L2Flush()
    b = decode_bytes(w)

    sampler = ClockSampler(torch.cuda.current_device()) if rank == 0 else None
    if sampler:
        sampler.start()
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    t_wall0 = time.time()
    step_ms, kern_ms = time_steps([st.plan, st.run], args.steps, args.warmup, flush)
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    t_wall1 = time.time()
    clocks = summarise_clocks(sampler.stop(), t_wall0, t_wall1) if sampler else None
    assert st.att.status() == 0, "a kernel reported a timeout"

    step_s = float(np.mean(step_ms)) * 1e-3
    kern_s = float(np.mean(kern_ms)) * 1e-3
    if world > 1:
        step_s, kern_s = max_over_ranks([step_s, kern_s], "cuda")
    value = whole_job_gbs(b, world, step_s)

    # end to end through the public API with host buffers
    e2e = None
    if rank == 0:
        from paged_kv_attention_bsr_gb300.api import PagedAttention
        c = w.cache
        att = st.att
        # The step's inputs (q and the page table) live in one pinned host
        # buffer and its outputs (o and LSE) in another, so each direction is
        # one copy; the device tensors are views of matching device buffers.
        def packed(parts):
            offs, at = [], 0
            for t in parts:
                offs.append(at)
                at = (at + t.numel() * t.element_size() + 255) // 256 * 256
            return offs, at

        in_parts = [w.q, torch.from_numpy(c.kv_indptr), torch.from_numpy(c.kv_indices),
                    torch.from_numpy(c.last_page_len)]
        in_offs, in_bytes = packed(in_parts)
        in_h = torch.zeros(in_bytes, dtype=torch.uint8).pin_memory()
        in_d = torch.empty(in_bytes, dtype=torch.uint8, device="cuda")

        def view(buf, off, t):
            n = t.numel() * t.element_size()
            return buf[off:off + n].view(t.dtype).view(t.shape)

        for t, off in zip(in_parts, in_offs):
            view(in_h, off, t).copy_(t)
        q_d, kvi_d, kvx_d, lpl_d = (view(in_d, off, t) for t, off in zip(in_parts, in_offs))
        out_parts = [torch.empty_like(w.q), torch.empty(w.q.shape[:-1], dtype=torch.float32)]
        out_offs, out_bytes = packed(out_parts)
        out_h = torch.empty(out_bytes, dtype=torch.uint8).pin_memory()
        out_d = torch.empty(out_bytes, dtype=torch.uint8, device="cuda")
        o_d, lse_d = (view(out_d, off, t) for t, off in zip(out_parts, out_offs))
        n_e2e = max(3, min(args.steps, 200))
        h2d = in_bytes + (att.plan_info.table_bytes if att.plan_info is not None else 0)
        d2h = out_bytes

        def e2e_step():
            in_d.copy_(in_h, non_blocking=True)
            att.plan(c.kv_indptr, c.last_page_len, c.page_size)
            att.run(q_d, st.d["k_pool"], st.d["v_pool"], kvi_d, kvx_d, lpl_d, w.sm_scale,
                    out=o_d, lse=lse_d)
            out_h.copy_(out_d, non_blocking=True)
            torch.cuda.current_stream().synchronize()

        for _ in range(3):
            flush()
            e2e_step()
        tot = 0.0
        for _ in range(n_e2e):
            flush()
            torch.cuda.synchronize()
            t0 = time.perf_counter()
            e2e_step()
            tot += time.perf_counter() - t0
        serial = b / (tot / n_e2e) / 1e9

        # The same steps as a serving loop issues them: step k + 1's input
        # copy, planning and launch are enqueued while step k runs, and the
        # host reads step k's output (from one of two pinned buffers) once
        # step k + 1 is enqueued. Every step still copies its inputs in and
        # its output out; one stream orders copies and kernels.
        out_hs = [out_h, torch.empty(out_bytes, dtype=torch.uint8).pin_memory()]
        done = [torch.cuda.Event(), torch.cuda.Event()]
        lse_off = out_offs[1]

        def enqueue(k):
            in_d.copy_(in_h, non_blocking=True)
            att.plan(c.kv_indptr, c.last_page_len, c.page_size)
            att.run(q_d, st.d["k_pool"], st.d["v_pool"], kvi_d, kvx_d, lpl_d, w.sm_scale,
                    out=o_d, lse=lse_d)
            out_hs[k % 2].copy_(out_d, non_blocking=True)
            done[k % 2].record()

        def consume(k):
            done[k % 2].synchronize()
            return float(out_hs[k % 2][lse_off:lse_off + 4].view(torch.float32)[0])

        for k in range(4):
            enqueue(k)
        consume(3)
        flush()
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        for k in range(n_e2e):
            enqueue(k)
            if k > 0:
                consume(k - 1)
        last = consume(n_e2e - 1)
        tot_p = time.perf_counter() - t0
        assert math.isfinite(last)
        e2e = {"value": b * n_e2e / tot_p / 1e9, "unit": "GB/s", "h2d_bytes_per_step": int(h2d),
               "d2h_bytes_per_step": int(d2h), "steps": n_e2e,
               "serialized_value": serial,
               "note": "KV pool stays resident in HBM (it is the cache); per-step inputs "
                       "(q and the page table, packed in one pinned buffer, plus the plan "
                       "tables attn_plan uploads) and outputs (o and lse, one buffer) cross "
                       "the host link every step. value: steps pipelined as a serving loop "
                       "issues them (step k + 1 enqueued while step k runs, step k's output "
                       "read after that), wall clock over all steps; serialized_value: each "
                       "step enqueued, run and read back before the next starts"}

    if rank != 0:
        return None
    traffic = profile_traffic(*PROFILES["uniform_decode"])
    achieved = b / kern_s / 1e9
    line = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": step_s * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": w.name, "batch": w.batch, "num_qo_heads": 32, "num_kv_heads": 8,
                   "head_dim": 128, "page_size": 16, "kv_len": "U[1024,4096]",
                   "pool_pages": 20000, "total_kv_tokens": int(w.cache.kv_lens.sum()),
                   "num_ctas": st.att.num_ctas, "step": "attn_plan + attn_decode_run",
                   "l2": "flushed between steps outside the timed events (512 MB write, then "
                         "a 256 MB read so the write-back happens there); "
                         "each step also reads 677 MB of KV, > 126 MB L2",
                   "timing": "CUDA events around each step; a GPU sleep before the step's "
                             "start event covers the host enqueue (outside the events)",
                   "parallelism": f"replicas x{world}"},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": hbm_peak, "unit": "GB/s",
                     "frac": achieved / hbm_peak, "traffic": traffic,
                     "peak_source": f"{peak_src} hbm_gbs (MEASURED_PEAKS.json)",
                     "kernel": "decode_tc_kernel<bf16, group 4> (one launch per run; "
                               "split items merged inside it)",
                     "kernel_us": kern_s * 1e6, "algorithmic_bytes_per_launch": b},
        # per timed step: attn_plan's table upload (copy_tables_kernel) and
        # the decode kernel
        "gpu_launches": 2 * args.steps,
        "clocks": clocks,
        "e2e": e2e,
    }
    if rank == 0:
        line["plan_us"] = plan_times(w, st.att.num_ctas)
    if world == 1 and not args.skip_cpu:
        threads = max(1, min(os.cpu_count() or 1, 16))
        secs, passes = cpu_oracle_baseline(w, threads)
        line["cpu_baseline"] = {"value": b / secs / 1e9, "unit": "GB/s", "cores": threads,
                                "kind": "oracle",
                                "sample": f"{passes} whole passes over the workload (64 "
                                          f"requests x 32 heads), fp64 C oracle on {threads} "
                                          f"threads, {secs:.2f} s per pass",
                                "per_workload": cpu_oracle_per_workload(threads)}
    if world == 1 and not args.headline_only:
        del st
        torch.cuda.empty_cache()
        line["workloads"] = extra_workloads(hbm_peak, bf16_peak, flush)
    return line


# ---------------------------------------------------------- reference arm
def run_reference(args):
    """The fp64 oracle as it stands, timed on the host cores on the same
    workload, metric and unit; each step is a bounded sample of (request,
    kv head) items so that the whole run stays within a few minutes."""
    import oracle
    from paged_kv_attention_bsr_gb300 import synth
    w = synth.uniform_gqa_decode()
    c = w.cache
    threads = max(1, min(os.cpu_count() or 1, 16))
    oracle.build()
    budget_s = 90.0 / max(1, args.steps + args.warmup)
    # one item (r, hk) ~ kv_len x g x D x 3 fp64 ops; calibrate with one item
    g = w.num_qo_heads // w.num_kv_heads

    def item_job(r, hk):
        for hh in range(g):
            oracle.attention_row(w.q, c.k_pool, c.v_pool, c.kv_indptr, c.kv_indices,
                                 c.last_page_len, 16, 32, 8, 128, oracle.BF16, w.sm_scale, r, 0,
                                 hk * g + hh)

    t0 = time.perf_counter()
    item_job(0, 0)
    per_item = max(1e-4, time.perf_counter() - t0)
    n_items = max(1, int(budget_s * threads / per_item))
    items = [(r, hk) for r in range(w.batch) for hk in range(w.num_kv_heads)]
    kvb = 2 * 128 * 2
    total_b = 0
    total_t = 0.0
    pos = 0
    with cf.ThreadPoolExecutor(threads) as ex:
        for k in range(args.steps + args.warmup):
            sel = [items[(pos + i) % len(items)] for i in range(n_items)]
            pos += n_items
            t0 = time.perf_counter()
            list(ex.map(lambda rh: item_job(*rh), sel))
            dt = time.perf_counter() - t0
            if k == 0 and args.warmup > 0:
                # re-size the sample from a whole parallel step (threads share
                # the host's memory bandwidth, so one item alone is optimistic)
                n_items = max(1, int(n_items * budget_s / max(dt, 1e-6)))
            if k >= args.warmup:
                total_t += dt
                total_b += sum(int(c.kv_lens[r]) * kvb + 2 * g * 256 for r, _ in sel)
    value = total_b / total_t / 1e9
    sample = (f"{n_items} (request, kv head) items per step of the uniform GQA decode "
              f"workload, fp64 C oracle on {threads} threads")
    return {"impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s",
            "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": total_t / args.steps * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": w.name, "batch": w.batch},
            "cpu_baseline": {"value": value, "unit": "GB/s", "cores": threads, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=4000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--headline-only", action="store_true",
                    help="skip the other workloads (single, skewed, shared-prefix, append)")
    ap.add_argument("--skip-cpu", action="store_true", help="skip the CPU oracle baseline")
    ap.add_argument("--workload", choices=sorted(WORKLOAD_BENCH),
                    help="time one workload alone and print only its result")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if args.gpus > 1 and world == 1:
        sys.exit("for --gpus > 1 launch with torch.distributed.run (one rank per GPU)")
    if args.workload:
        # one workload alone (used for profiling captures); prints its own line
        hbm_peak, bf16_peak, _ = peaks()
        flush = L2Flush()
        name, res = WORKLOAD_BENCH[args.workload](hbm_peak, bf16_peak, flush, args.steps,
                                                  args.warmup)
        print(json.dumps({"workload": name, **res}), flush=True)
        return
    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args)), flush=True)
        return
    if world > 1:
        torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", 0)))
        torch.distributed.init_process_group("nccl")
    line = run_ours(args, rank, world)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
