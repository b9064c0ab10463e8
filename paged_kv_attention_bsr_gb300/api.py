"""Torch-facing conveniences over the C ABI: workspace ownership and call order.

PyTorch supplies device memory, pinned host memory and streams; every step of
the attention itself runs in libattn.so's kernels.
"""
from __future__ import annotations

import math
from typing import Optional

import numpy as np
import torch

from . import _capi as C


class PagedAttention:
    """Owns the workspaces of one attention call site and runs plan() / run().

    mode "decode": one query row per request (attn_decode_run).
    mode "append": ragged query rows per request (attn_append_run).
    The plan tables go through a ring of pinned staging buffers; a buffer is
    reused only after its previous upload has executed.
    """

    RING = 4

    def __init__(self, num_qo_heads: int, num_kv_heads: int, head_dim: int = 128,
                 mode: str = "decode", max_batch: int = 256, max_total_qo: Optional[int] = None,
                 num_ctas: Optional[int] = None, device=None):
        if mode not in ("decode", "append"):
            raise ValueError("mode must be 'decode' or 'append'")
        self.mode = mode
        self.num_qo_heads, self.num_kv_heads, self.head_dim = num_qo_heads, num_kv_heads, head_dim
        self.device = torch.device(device if device is not None else "cuda")
        dev_index = self.device.index if self.device.index is not None else torch.cuda.current_device()
        cmode = C.MODE_DECODE if mode == "decode" else C.MODE_APPEND
        self.num_ctas = num_ctas or C.default_num_ctas(dev_index, cmode)
        self.max_batch = max_batch
        self.max_total_qo = max_total_qo if max_total_qo is not None else max_batch
        dev_bytes, host_bytes = C.workspace_size(max_batch, self.max_total_qo, num_qo_heads,
                                                 num_kv_heads, head_dim, self.num_ctas)
        self.dev_ws = torch.empty(dev_bytes, dtype=torch.uint8, device=self.device)
        self._pinned = [torch.empty(host_bytes, dtype=torch.uint8).pin_memory()
                        for _ in range(self.RING)]
        self._events = [None] * self.RING  # created on first use, then re-recorded
        self._turn = 0
        self.plan_info: Optional[C.Plan] = None

    def plan(self, kv_indptr_h, last_page_len_h, page_size: int, qo_indptr_h=None,
             causal: bool = False, stream=None) -> C.Plan:
        if (self.mode == "decode") != (qo_indptr_h is None):
            raise ValueError("decode plans take no qo_indptr; append plans need one")
        i = self._turn
        self._turn = (self._turn + 1) % self.RING
        ev = self._events[i]
        if ev is None:
            ev = self._events[i] = torch.cuda.Event()
        else:
            ev.synchronize()  # the previous upload from this staging buffer has run
        if stream is None:
            stream = torch.cuda.current_stream()
        self.plan_info = C.plan(qo_indptr_h, kv_indptr_h, last_page_len_h, page_size,
                                self.num_qo_heads, self.num_kv_heads, self.head_dim, causal,
                                self.num_ctas, self._pinned[i], self.dev_ws, stream)
        ev.record(stream)
        self._causal = bool(causal)
        return self.plan_info

    def run(self, q, k_pool, v_pool, kv_indptr, kv_indices, last_page_len, sm_scale=None,
            out=None, lse=None, qo_indptr=None, layout: int = C.LAYOUT_HND, num_pages=None,
            return_lse: bool = False, stream=None, rope=None, kv_scales=None):
        """rope: optional (cos, sin) device float32 tables [max_pos, head_dim / 2]
        of the angles pos * theta_d: rotary position embedding fused into the
        kernels (decode and append).
        kv_scales: optional (k_scale, v_scale) device float32 [num_kv_heads]:
        the pools hold FP8 E4M3 bytes with these per-head scales (decode)."""
        if self.plan_info is None:
            raise RuntimeError("run() before plan()")
        if sm_scale is None:
            sm_scale = 1.0 / math.sqrt(self.head_dim)
        if out is None:
            out = torch.empty_like(q)
        if lse is None and return_lse:
            lse = torch.empty(q.shape[:-1], dtype=torch.float32, device=q.device)
        if kv_scales is not None:
            if self.mode != "decode" or rope is not None:
                raise ValueError("FP8 K/V pools are supported by decode without RoPE")
            C.decode_run_fp8(self.plan_info, q, k_pool, v_pool, kv_indptr, kv_indices,
                             last_page_len, kv_scales[0], kv_scales[1], sm_scale, out, lse,
                             self.dev_ws, layout, num_pages, stream)
        elif self.mode == "decode" and rope is not None:
            C.decode_run_rope(self.plan_info, q, k_pool, v_pool, kv_indptr, kv_indices,
                              last_page_len, sm_scale, rope[0], rope[1], out, lse,
                              self.dev_ws, layout, num_pages, stream)
        elif rope is not None:
            C.append_run_rope(self.plan_info, q, qo_indptr, k_pool, v_pool, kv_indptr,
                              kv_indices, last_page_len, self._causal, sm_scale, rope[0],
                              rope[1], out, lse, self.dev_ws, layout, num_pages, stream)
        elif self.mode == "decode":
            C.decode_run(self.plan_info, q, k_pool, v_pool, kv_indptr, kv_indices,
                         last_page_len, sm_scale, out, lse, self.dev_ws, layout, num_pages,
                         stream)
        else:
            C.append_run(self.plan_info, q, qo_indptr, k_pool, v_pool, kv_indptr, kv_indices,
                         last_page_len, self._causal, sm_scale, out, lse, self.dev_ws, layout,
                         num_pages, stream)
        return (out, lse) if return_lse else out

    def status(self, stream=None) -> int:
        """Synchronise and return the workspace error word (0 = no kernel timed out)."""
        return C.workspace_status(self.dev_ws, stream)


class CascadeAttention:
    """Composable formats (shared prefix + unique suffix) for decode.

    The prompt's common prefix is stored once in a pool with large pages and
    read once for its n generations; each generation's own suffix lives in a
    second pool (small pages). Two ways to run it:

    * one launch (attn_plan_cascade / attn_cascade_run), taken when
      group x n <= 16 (any page sizes, either layout): one persistent
      few-row kernel balances the prefix and suffix pages of every (prompt,
      kv head) together and merges the partial states inside the kernel;
    * otherwise two passes: a non-causal append for the prefix (the n
      generations' rows per prompt) and a decode for the suffixes, enqueued
      on two streams (the suffix on a side stream forked from and joined back
      into the caller's stream), then attn_merge_states.

    mode: "auto" (one launch when the shapes allow it), "one_launch" (raise
    if they do not) or "two_pass".
    """

    RING = 4

    def __init__(self, num_qo_heads: int, num_kv_heads: int, head_dim: int = 128,
                 max_prompts: int = 64, max_batch: int = 256, device=None, mode: str = "auto",
                 num_ctas: Optional[int] = None):
        if mode not in ("auto", "one_launch", "two_pass"):
            raise ValueError("mode must be 'auto', 'one_launch' or 'two_pass'")
        self.mode = mode
        self.num_qo_heads, self.num_kv_heads, self.head_dim = num_qo_heads, num_kv_heads, head_dim
        self.prefix = PagedAttention(num_qo_heads, num_kv_heads, head_dim, "append",
                                     max_batch=max_prompts, max_total_qo=max_batch,
                                     device=device)
        self.suffix = PagedAttention(num_qo_heads, num_kv_heads, head_dim, "decode",
                                     max_batch=max_batch, device=device)
        self.device = self.prefix.device
        self.side = torch.cuda.Stream(device=self.device)
        self._fork = torch.cuda.Event()
        self._join = torch.cuda.Event()
        self._bufs = None
        self.one_launch = False
        self.plan_info: Optional[C.Plan] = None
        if mode != "two_pass":
            dev_index = self.device.index if self.device.index is not None else \
                torch.cuda.current_device()
            self.num_ctas = num_ctas or C.default_num_ctas(dev_index, C.MODE_CASCADE)
            dev_bytes, host_bytes = C.cascade_workspace_size(max_prompts, max_batch,
                                                             num_qo_heads, num_kv_heads,
                                                             head_dim, self.num_ctas)
            self.dev_ws = torch.empty(dev_bytes, dtype=torch.uint8, device=self.device)
            self._pinned = [torch.empty(host_bytes, dtype=torch.uint8).pin_memory()
                            for _ in range(self.RING)]
            self._events = [None] * self.RING
            self._turn = 0

    def _fits_one_launch(self, qo_indptr_h) -> bool:
        qo = np.asarray(qo_indptr_h)
        max_n = int(np.diff(qo).max()) if len(qo) > 1 else 0
        group = self.num_qo_heads // self.num_kv_heads
        return group * max(max_n, 1) <= 16

    def plan(self, qo_indptr_prefix_h, kv_indptr_prefix_h, last_page_len_prefix_h,
             page_size_prefix: int, kv_indptr_suffix_h, last_page_len_suffix_h,
             page_size_suffix: int, stream=None):
        """Plans the run; the tables are uploaded on `stream`."""
        fits = self._fits_one_launch(qo_indptr_prefix_h)
        if self.mode == "one_launch" and not fits:
            raise ValueError("one launch needs num_qo_heads / num_kv_heads x the generations "
                             "of a prompt <= 16")
        self.one_launch = self.mode != "two_pass" and fits
        if self.one_launch:
            i = self._turn
            self._turn = (self._turn + 1) % self.RING
            ev = self._events[i]
            if ev is None:
                ev = self._events[i] = torch.cuda.Event()
            else:
                ev.synchronize()  # the previous upload from this staging buffer has run
            if stream is None:
                stream = torch.cuda.current_stream()
            self.plan_info = C.plan_cascade(
                qo_indptr_prefix_h, kv_indptr_prefix_h, last_page_len_prefix_h,
                page_size_prefix, kv_indptr_suffix_h, last_page_len_suffix_h, page_size_suffix,
                self.num_qo_heads, self.num_kv_heads, self.head_dim, self.num_ctas,
                self._pinned[i], self.dev_ws, stream)
            ev.record(stream)
            return self.plan_info
        self.prefix.plan(kv_indptr_prefix_h, last_page_len_prefix_h, page_size_prefix,
                         qo_indptr_h=qo_indptr_prefix_h, causal=False, stream=stream)
        self.suffix.plan(kv_indptr_suffix_h, last_page_len_suffix_h, page_size_suffix,
                         stream=stream)
        self.plan_info = None
        return None

    def run(self, q, prefix, suffix, qo_indptr_prefix, sm_scale=None, out=None, lse=None,
            return_lse: bool = False, layout: int = C.LAYOUT_HND):
        """q [batch, Hq, D] (one row per generation, grouped by prompt);
        prefix / suffix: dicts with k_pool, v_pool, kv_indptr, kv_indices,
        last_page_len device tensors (both pools in `layout`). Returns o
        (and lse)."""
        if sm_scale is None:
            sm_scale = 1.0 / math.sqrt(self.head_dim)
        stream = torch.cuda.current_stream()
        if out is None:
            out = torch.empty_like(q)
        if lse is None and return_lse:
            lse = torch.empty(q.shape[:-1], dtype=torch.float32, device=q.device)
        if self.one_launch:
            C.cascade_run(self.plan_info, q, qo_indptr_prefix, prefix, suffix, sm_scale, out,
                          lse, self.dev_ws, layout, stream)
            return (out, lse) if return_lse else out
        if self._bufs is None or self._bufs[0].shape != q.shape or \
                self._bufs[0].dtype != q.dtype:
            mk = lambda: torch.empty(q.shape[:-1], dtype=torch.float32, device=q.device)
            self._bufs = (torch.empty_like(q), mk(), torch.empty_like(q), mk())
        o_p, l_p, o_s, l_s = self._bufs
        self._fork.record(stream)
        self.side.wait_event(self._fork)
        with torch.cuda.stream(self.side):
            self.suffix.run(q, suffix["k_pool"], suffix["v_pool"], suffix["kv_indptr"],
                            suffix["kv_indices"], suffix["last_page_len"], sm_scale, out=o_s,
                            lse=l_s, layout=layout, stream=self.side)
            self._join.record(self.side)
        self.prefix.run(q, prefix["k_pool"], prefix["v_pool"], prefix["kv_indptr"],
                        prefix["kv_indices"], prefix["last_page_len"], sm_scale, out=o_p,
                        lse=l_p, qo_indptr=qo_indptr_prefix, layout=layout, stream=stream)
        stream.wait_event(self._join)
        if lse is None:
            lse = torch.empty(q.shape[:-1], dtype=torch.float32, device=q.device)
        C.merge_states(o_p, l_p, o_s, l_s, out, lse, stream=stream)
        return (out, lse) if return_lse else out

    def status(self, stream=None) -> int:
        """Synchronise and return the one-launch workspace's error word (0 = none)."""
        if self.mode == "two_pass":
            return max(self.prefix.status(stream), self.suffix.status(stream))
        return C.workspace_status(self.dev_ws, stream)


_single_cache = {}


def single_decode_with_kv_cache(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor,
                                sm_scale: Optional[float] = None, return_lse: bool = False):
    """Decode attention of one request over contiguous K/V.

    q [num_qo_heads, head_dim], k / v [kv_len, num_kv_heads, head_dim] (the
    quick-start snippet's shapes); returns [num_qo_heads, head_dim]. The
    contiguous cache is read in place as a BSR row of pages in the NHD layout
    (pages 0..n-1 in order), so the balanced plan can split it across SMs.
    The page size is the largest power of two up to 16 that divides kv_len,
    so the pages cover exactly the caller's tensors. Strided k / v / q are
    copied to dense tensors first. kv_len = 0 gives O = 0 and LSE = -inf.
    """
    k, v, q = k.contiguous(), v.contiguous(), q.contiguous()  # read in place as dense pages
    kv_len, Hk, D = k.shape
    Hq = q.shape[0]
    P = 16
    while P > 1 and kv_len % P:
        P //= 2
    n_pages = (kv_len + P - 1) // P
    key = (q.device, Hq, Hk, D)
    att = _single_cache.get(key)
    if att is None:
        att = PagedAttention(Hq, Hk, D, "decode", max_batch=1, device=q.device)
        _single_cache[key] = att
    kv_indptr_h = np.array([0, n_pages], np.int32)
    last_h = np.array([kv_len - P * (n_pages - 1) if n_pages else 0], np.int32)
    att.plan(kv_indptr_h, last_h, P)
    kv_indptr = torch.from_numpy(kv_indptr_h).to(q.device, non_blocking=True)
    last = torch.from_numpy(last_h).to(q.device, non_blocking=True)
    kv_indices = torch.arange(n_pages, dtype=torch.int32, device=q.device)
    res = att.run(q.reshape(1, Hq, D), k, v, kv_indptr, kv_indices, last, sm_scale,
                  layout=C.LAYOUT_NHD, num_pages=n_pages, return_lse=return_lse)
    if return_lse:
        o, lse = res
        return o.reshape(Hq, D), lse.reshape(Hq)
    return res.reshape(Hq, D)


def merge_state(o_a, lse_a, o_b, lse_b, out=None, lse_out=None):
    """LSE merge of two attention states [n, H, D] (+ [n, H] fp32 LSE)."""
    if out is None:
        out = torch.empty_like(o_a)
    if lse_out is None:
        lse_out = torch.empty_like(lse_a)
    C.merge_states(o_a, lse_a, o_b, lse_b, out, lse_out)
    return out, lse_out
