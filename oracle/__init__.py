"""fp64 CPU oracle for BSR paged-KV attention -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline / reference
legs of ``bench.py`` may import this package. The library path
(``paged_kv_attention_bsr_gb300``) never does, and the two share no code.

Contents:
  * ``attn_oracle.c``  -- plain single-threaded C, double precision: BSR gather,
    softmax attention with optional end-aligned causal mask and optional
    rotary position embedding of q and k, LSE merge.
  * ``plan_ref.py``    -- restatement of the work partition spec (plan()).
  * this module        -- builds ``liboracle.so`` with gcc and wraps it with
    ctypes over numpy arrays.

What is computed follows the FlashInfer paper digest (modb.pro page, sections
"统一的 KV 缓存存储格式" and "动态负载均衡调度") and the yeyulingfeng.com page
("FlashAttention 的遗产"); the readings of silent points are listed in the
header comment of attn_oracle.h.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "attn_oracle.c")
_HDR = os.path.join(_HERE, "attn_oracle.h")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

F16, BF16 = 0, 1
HND, NHD = 0, 1


def build(force: bool = False) -> str:
    """Compile liboracle.so with gcc (portable flags: runs on x86_64 and aarch64)."""
    newest = max(os.path.getmtime(_SRC), os.path.getmtime(_HDR))
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < newest:
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(
            ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fno-fast-math",
             "-ffp-contract=off", _SRC, "-o", tmp, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            i32, i64, dbl = ctypes.c_int32, ctypes.c_int64, ctypes.c_double
            vp = ctypes.c_void_p
            lib.oracle_widen.restype = dbl
            lib.oracle_widen.argtypes = [ctypes.c_uint16, i32]
            lib.oracle_attention_row.restype = i32
            lib.oracle_attention_row.argtypes = [
                vp, vp, vp, vp, i64, i32, vp, vp, vp, i32, i32, i32, i32, i32,
                i32, i32, dbl, i32, i32, i32, vp, vp]
            lib.oracle_batch_attention.restype = i32
            lib.oracle_batch_attention.argtypes = [
                vp, vp, vp, vp, i64, i32, vp, vp, vp, i32, i32, i32, i32, i32,
                i32, i32, dbl, vp, vp, vp, vp]
            lib.oracle_batch_attention_rope.restype = i32
            lib.oracle_batch_attention_rope.argtypes = [
                vp, vp, vp, vp, i64, i32, vp, vp, vp, i32, i32, i32, i32, i32,
                i32, i32, dbl, vp, vp, i64, vp, vp]
            lib.oracle_attention_row_rope.restype = i32
            lib.oracle_attention_row_rope.argtypes = [
                vp, vp, vp, vp, i64, i32, vp, vp, vp, i32, i32, i32, i32, i32,
                i32, i32, dbl, vp, vp, i64, i32, i32, i32, vp, vp]
            lib.oracle_widen_e4m3.restype = dbl
            lib.oracle_widen_e4m3.argtypes = [ctypes.c_uint8]
            lib.oracle_batch_attention_fp8kv.restype = i32
            lib.oracle_batch_attention_fp8kv.argtypes = [
                vp, vp, vp, vp, i64, i32, vp, vp, vp, i32, i32, i32, i32, i32,
                i32, i32, dbl, vp, vp, vp, vp]
            lib.oracle_round.restype = dbl
            lib.oracle_round.argtypes = [dbl, i32]
            lib.oracle_merge_states.restype = None
            lib.oracle_merge_states.argtypes = [vp, vp, i32, i64, i32, vp, vp]
            _lib = lib
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _u16(a) -> np.ndarray:
    """Raw 16-bit storage words of a numpy float16 / uint16 / torch tensor."""
    if hasattr(a, "detach"):  # torch tensor (bf16 / fp16) on CPU
        import torch
        a = a.detach().contiguous().cpu().view(torch.int16).numpy()
    a = np.ascontiguousarray(a)
    return a.view(np.uint16)


def _i32(a):
    if a is None:
        return None
    if hasattr(a, "detach"):
        a = a.detach().cpu().numpy()
    return np.ascontiguousarray(a, dtype=np.int32)


def widen(bits: int, dtype: int) -> float:
    return _load().oracle_widen(int(bits) & 0xFFFF, dtype)


def batch_attention(q, k_pool, v_pool, kv_indptr, kv_indices, last_page_len,
                    page_size, num_qo_heads, num_kv_heads, head_dim, dtype,
                    sm_scale, causal=False, qo_indptr=None, layout=HND,
                    kv_begin=None, kv_end=None):
    """All rows. Returns (o float64 [total_qo, Hq, D], lse float64 [total_qo, Hq])."""
    lib = _load()
    q16, k16, v16 = _u16(q), _u16(k_pool), _u16(v_pool)
    kv_indptr, kv_indices = _i32(kv_indptr), _i32(kv_indices)
    last_page_len, qo_indptr = _i32(last_page_len), _i32(qo_indptr)
    kv_begin, kv_end = _i32(kv_begin), _i32(kv_end)
    batch = len(kv_indptr) - 1
    total_qo = int(qo_indptr[-1]) if qo_indptr is not None else batch
    num_pages = k16.size // (page_size * num_kv_heads * head_dim)
    o = np.zeros((total_qo, num_qo_heads, head_dim), np.float64)
    lse = np.zeros((total_qo, num_qo_heads), np.float64)
    rc = lib.oracle_batch_attention(
        _ptr(q16), _ptr(qo_indptr), _ptr(k16), _ptr(v16), num_pages, layout,
        _ptr(kv_indptr), _ptr(kv_indices), _ptr(last_page_len), batch, page_size,
        num_qo_heads, num_kv_heads, head_dim, dtype, int(bool(causal)),
        float(sm_scale), _ptr(kv_begin), _ptr(kv_end), _ptr(o), _ptr(lse))
    if rc != 0:
        raise ValueError(f"oracle_batch_attention rejected its arguments (code {rc})")
    return o, lse


def batch_attention_rope(q, k_pool, v_pool, kv_indptr, kv_indices, last_page_len,
                         page_size, num_qo_heads, num_kv_heads, head_dim, dtype,
                         sm_scale, rope_cos, rope_sin, causal=False, qo_indptr=None,
                         layout=HND):
    """All rows with rotary position embedding (tables float32 [max_pos, D/2])."""
    lib = _load()
    q16, k16, v16 = _u16(q), _u16(k_pool), _u16(v_pool)
    kv_indptr, kv_indices = _i32(kv_indptr), _i32(kv_indices)
    last_page_len, qo_indptr = _i32(last_page_len), _i32(qo_indptr)
    cos = np.ascontiguousarray(rope_cos, np.float32)
    sin = np.ascontiguousarray(rope_sin, np.float32)
    assert cos.shape == sin.shape and cos.shape[1] == head_dim // 2
    batch = len(kv_indptr) - 1
    total_qo = int(qo_indptr[-1]) if qo_indptr is not None else batch
    num_pages = k16.size // (page_size * num_kv_heads * head_dim)
    o = np.zeros((total_qo, num_qo_heads, head_dim), np.float64)
    lse = np.zeros((total_qo, num_qo_heads), np.float64)
    rc = lib.oracle_batch_attention_rope(
        _ptr(q16), _ptr(qo_indptr), _ptr(k16), _ptr(v16), num_pages, layout,
        _ptr(kv_indptr), _ptr(kv_indices), _ptr(last_page_len), batch, page_size,
        num_qo_heads, num_kv_heads, head_dim, dtype, int(bool(causal)),
        float(sm_scale), _ptr(cos), _ptr(sin), cos.shape[0], _ptr(o), _ptr(lse))
    if rc != 0:
        raise ValueError(f"oracle_batch_attention_rope rejected its arguments (code {rc})")
    return o, lse


def widen_e4m3(bits: int) -> float:
    return _load().oracle_widen_e4m3(int(bits) & 0xFF)


def _u8(a) -> np.ndarray:
    """Raw bytes of an FP8 tensor (torch float8 / uint8) or a uint8 array."""
    if hasattr(a, "detach"):
        import torch
        a = a.detach().contiguous().cpu().view(torch.uint8).numpy()
    return np.ascontiguousarray(a).view(np.uint8)


def batch_attention_fp8kv(q, k_pool, v_pool, kv_indptr, kv_indices, last_page_len,
                          page_size, num_qo_heads, num_kv_heads, head_dim, q_dtype, sm_scale,
                          k_scale, v_scale, causal=False, qo_indptr=None, layout=HND):
    """All rows with an FP8 E4M3 K/V cache (bytes) and per-kv-head float
    scales. Returns (o float64 [total_qo, Hq, D], lse float64 [total_qo, Hq])."""
    lib = _load()
    q16, k8, v8 = _u16(q), _u8(k_pool), _u8(v_pool)
    kv_indptr, kv_indices = _i32(kv_indptr), _i32(kv_indices)
    last_page_len, qo_indptr = _i32(last_page_len), _i32(qo_indptr)
    ks = np.ascontiguousarray(k_scale, np.float32)
    vs = np.ascontiguousarray(v_scale, np.float32)
    assert ks.shape == (num_kv_heads,) and vs.shape == (num_kv_heads,)
    batch = len(kv_indptr) - 1
    total_qo = int(qo_indptr[-1]) if qo_indptr is not None else batch
    num_pages = k8.size // (page_size * num_kv_heads * head_dim)
    o = np.zeros((total_qo, num_qo_heads, head_dim), np.float64)
    lse = np.zeros((total_qo, num_qo_heads), np.float64)
    rc = lib.oracle_batch_attention_fp8kv(
        _ptr(q16), _ptr(qo_indptr), _ptr(k8), _ptr(v8), num_pages, layout, _ptr(kv_indptr),
        _ptr(kv_indices), _ptr(last_page_len), batch, page_size, num_qo_heads, num_kv_heads,
        head_dim, q_dtype, int(bool(causal)), float(sm_scale), _ptr(ks), _ptr(vs), _ptr(o),
        _ptr(lse))
    if rc != 0:
        raise ValueError(f"oracle_batch_attention_fp8kv rejected its arguments (code {rc})")
    return o, lse


def round_to(v: float, dtype: int) -> float:
    """A double rounded to the 16-bit storage type (ties to even)."""
    return _load().oracle_round(float(v), dtype)


def attention_row(q, k_pool, v_pool, kv_indptr, kv_indices, last_page_len,
                  page_size, num_qo_heads, num_kv_heads, head_dim, dtype,
                  sm_scale, r, i, h, causal=False, qo_indptr=None, layout=HND,
                  ):
    """One (request, query row, query head). Returns (o float64 [D], lse float)."""
    lib = _load()
    q16, k16, v16 = _u16(q), _u16(k_pool), _u16(v_pool)
    kv_indptr, kv_indices = _i32(kv_indptr), _i32(kv_indices)
    last_page_len, qo_indptr = _i32(last_page_len), _i32(qo_indptr)
    batch = len(kv_indptr) - 1
    num_pages = k16.size // (page_size * num_kv_heads * head_dim)
    o = np.zeros(head_dim, np.float64)
    lse = np.zeros(1, np.float64)
    rc = lib.oracle_attention_row(
        _ptr(q16), _ptr(qo_indptr), _ptr(k16), _ptr(v16), num_pages, layout,
        _ptr(kv_indptr), _ptr(kv_indices), _ptr(last_page_len), batch, page_size,
        num_qo_heads, num_kv_heads, head_dim, dtype, int(bool(causal)),
        float(sm_scale), int(r), int(i), int(h), _ptr(o), _ptr(lse))
    if rc != 0:
        raise ValueError(f"oracle_attention_row rejected its arguments (code {rc})")
    return o, float(lse[0])


def attention_row_rope(q, k_pool, v_pool, kv_indptr, kv_indices, last_page_len,
                       page_size, num_qo_heads, num_kv_heads, head_dim, dtype,
                       sm_scale, rope_cos, rope_sin, r, i, h, causal=False, qo_indptr=None,
                       layout=HND):
    """One row of batch_attention_rope. Returns (o float64 [D], lse float)."""
    lib = _load()
    q16, k16, v16 = _u16(q), _u16(k_pool), _u16(v_pool)
    kv_indptr, kv_indices = _i32(kv_indptr), _i32(kv_indices)
    last_page_len, qo_indptr = _i32(last_page_len), _i32(qo_indptr)
    cos = np.ascontiguousarray(rope_cos, np.float32)
    sin = np.ascontiguousarray(rope_sin, np.float32)
    batch = len(kv_indptr) - 1
    num_pages = k16.size // (page_size * num_kv_heads * head_dim)
    o = np.zeros(head_dim, np.float64)
    lse = np.zeros(1, np.float64)
    rc = lib.oracle_attention_row_rope(
        _ptr(q16), _ptr(qo_indptr), _ptr(k16), _ptr(v16), num_pages, layout,
        _ptr(kv_indptr), _ptr(kv_indices), _ptr(last_page_len), batch, page_size,
        num_qo_heads, num_kv_heads, head_dim, dtype, int(bool(causal)),
        float(sm_scale), _ptr(cos), _ptr(sin), cos.shape[0], int(r), int(i), int(h),
        _ptr(o), _ptr(lse))
    if rc != 0:
        raise ValueError(f"oracle_attention_row_rope rejected its arguments (code {rc})")
    return o, float(lse[0])


def merge_states(o_states, lse_states):
    """LSE merge. o_states [n, rows, D], lse_states [n, rows] -> (o [rows, D], lse [rows])."""
    lib = _load()
    o_in = np.ascontiguousarray(o_states, np.float64)
    lse_in = np.ascontiguousarray(lse_states, np.float64)
    n, rows, d = o_in.shape
    o = np.zeros((rows, d), np.float64)
    lse = np.zeros(rows, np.float64)
    lib.oracle_merge_states(_ptr(o_in), _ptr(lse_in), n, rows, d, _ptr(o), _ptr(lse))
    return o, lse
