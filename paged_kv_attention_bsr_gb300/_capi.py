"""ctypes binding of libattn.so (include/attn.h): argument marshalling only.

Every function here has the name of a C entry point without the ``attn_``
prefix and does nothing but turn torch tensors / numpy arrays into pointers,
call the library, and raise ``AttnError`` on a non-OK status. All attention
work runs in the library's CUDA kernels; there is no fallback path.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np
import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libattn.so")

OK, ERR_INVALID_ARG, ERR_UNSUPPORTED, ERR_WORKSPACE_TOO_SMALL, ERR_CUDA, ERR_TIMEOUT = range(6)
F16, BF16 = 0, 1
LAYOUT_HND, LAYOUT_NHD = 0, 1
MODE_DECODE, MODE_APPEND, MODE_CASCADE = 0, 1, 2

STATUS_NAMES = {0: "OK", 1: "INVALID_ARG", 2: "UNSUPPORTED", 3: "WORKSPACE_TOO_SMALL",
                4: "CUDA", 5: "TIMEOUT"}

# Every symbol include/attn.h declares (checked by the tests).
EXPORTS = ("attn_workspace_size", "attn_default_num_ctas", "attn_plan", "attn_decode_run",
           "attn_append_run", "attn_merge_states", "attn_workspace_status", "attn_last_error",
           "attn_decode_run_noalloc", "attn_wait_selftest", "attn_decode_run_rope",
           "attn_append_run_rope", "attn_decode_run_noalloc_status",
           "attn_wait_selftest_noalloc", "attn_decode_run_fp8", "attn_cascade_workspace_size",
           "attn_plan_cascade", "attn_cascade_run")


class AttnError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{STATUS_NAMES.get(status, status)}: {message}")
        self.status = status


class Plan(ctypes.Structure):
    """Mirror of attn_plan_t."""
    _fields_ = [(n, ctypes.c_int32) for n in (
        "mode", "batch", "page_size", "num_qo_heads", "num_kv_heads", "head_dim", "causal",
        "num_ctas", "q_tile", "rows_per_item", "num_items", "num_units", "num_split_items",
        "num_slots", "total_qo", "max_qo_len")] + [(n, ctypes.c_int64) for n in (
        "total_weight", "max_cta_weight", "off_work_indptr", "off_units", "off_merge_indptr",
        "off_merge_items", "off_counters", "off_partial_o", "off_partial_lse", "table_bytes",
        "dev_bytes_needed")] + [("fingerprint", ctypes.c_uint64), ("max_kv_len", ctypes.c_int64),
                              ("min_kv_minus_qo", ctypes.c_int64),
                              ("page_size_suffix", ctypes.c_int32), ("reserved", ctypes.c_int32)]


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(
            f"{LIB_PATH} is missing: build the CUDA library first "
            "(python -c 'import __graft_entry__ as g; g.build()')")
    lib = ctypes.CDLL(LIB_PATH)
    i32, i64, sz, f32 = ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t, ctypes.c_float
    vp = ctypes.c_void_p
    P = ctypes.POINTER
    sig = {
        "attn_workspace_size": [i32, i32, i32, i32, i32, i32, P(sz), P(sz)],
        "attn_default_num_ctas": [i32, i32, P(i32)],
        "attn_plan": [vp, vp, vp, i32, i32, i32, i32, i32, i32, i32, vp, sz, vp, sz, vp,
                      P(Plan)],
        "attn_decode_run": [P(Plan), vp, vp, vp, i64, i32, vp, vp, vp, i32, f32, vp, vp, vp,
                            sz, vp],
        "attn_append_run": [P(Plan), vp, vp, vp, vp, i64, i32, vp, vp, vp, i32, i32, f32, vp,
                            vp, vp, sz, vp],
        "attn_merge_states": [vp, vp, vp, vp, vp, vp, i32, i32, i32, i32, vp],
        "attn_workspace_status": [vp, vp, P(i32)],
        "attn_wait_selftest": [vp, i32, vp],
        "attn_decode_run_rope": [P(Plan), vp, vp, vp, i64, i32, vp, vp, vp, i32, f32, vp, vp,
                                 i64, vp, vp, vp, sz, vp],
        "attn_append_run_rope": [P(Plan), vp, vp, vp, vp, i64, i32, vp, vp, vp, i32, i32, f32,
                                 vp, vp, i64, vp, vp, vp, sz, vp],
        "attn_decode_run_noalloc": [vp, vp, i32, i32, i32, i32, i32, vp, vp, vp, i64, i32, vp,
                                    vp, vp, i32, f32, vp, vp, vp],
        "attn_decode_run_noalloc_status": [vp, P(i32)],
        "attn_decode_run_fp8": [P(Plan), vp, vp, vp, i64, i32, vp, vp, vp, i32, vp, vp, f32, vp,
                                vp, vp, sz, vp],
        "attn_wait_selftest_noalloc": [i32, vp],
        "attn_cascade_workspace_size": [i32, i32, i32, i32, i32, i32, P(sz), P(sz)],
        "attn_plan_cascade": [vp, vp, vp, i32, vp, vp, i32, i32, i32, i32, i32, i32, vp, sz, vp,
                              sz, vp, P(Plan)],
        "attn_cascade_run": [P(Plan), vp, vp, vp, vp, i64, vp, vp, vp, vp, vp, i64, vp, vp, vp,
                             i32, i32, f32, vp, vp, vp, sz, vp],
    }
    for name, args in sig.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = ctypes.c_int
    lib.attn_last_error.argtypes = []
    lib.attn_last_error.restype = ctypes.c_char_p
    return lib


lib = _load()


def last_error() -> str:
    return lib.attn_last_error().decode()


def _check(status: int):
    if status != OK:
        raise AttnError(status, last_error())


def _ptr(x):
    """Device/host address of a tensor or numpy array as an int (None -> NULL);
    the c_void_p argtypes take ints as they are."""
    if x is None:
        return None
    if isinstance(x, torch.Tensor):
        return x.data_ptr()
    if isinstance(x, np.ndarray):
        return x.ctypes.data
    if isinstance(x, int):
        return x
    raise TypeError(f"cannot take the address of {type(x)}")


def _host_i32(x):
    if x is None:
        return None
    if isinstance(x, np.ndarray) and x.dtype == np.int32 and x.flags.c_contiguous:
        return x
    if isinstance(x, torch.Tensor):
        x = x.detach().cpu().numpy()
    return np.ascontiguousarray(x, dtype=np.int32)


def dtype_code(t: torch.dtype) -> int:
    if t == torch.bfloat16:
        return BF16
    if t == torch.float16:
        return F16
    raise TypeError(f"unsupported dtype {t}; use torch.float16 or torch.bfloat16")


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def workspace_size(max_batch, max_total_qo, num_qo_heads, num_kv_heads, head_dim, num_ctas):
    dev = ctypes.c_size_t()
    host = ctypes.c_size_t()
    _check(lib.attn_workspace_size(max_batch, max_total_qo, num_qo_heads, num_kv_heads,
                                   head_dim, num_ctas, ctypes.byref(dev), ctypes.byref(host)))
    return dev.value, host.value


def default_num_ctas(device: int = 0, mode: int = MODE_DECODE) -> int:
    n = ctypes.c_int32()
    _check(lib.attn_default_num_ctas(device, mode, ctypes.byref(n)))
    return n.value


def plan(qo_indptr_h, kv_indptr_h, last_page_len_h, page_size, num_qo_heads, num_kv_heads,
         head_dim, causal, num_ctas, pinned_ws, dev_ws=None, stream=None) -> Plan:
    """attn_plan. Host arrays; pinned_ws: host tensor / array; dev_ws: CUDA tensor or None."""
    kv_indptr_h = _host_i32(kv_indptr_h)
    last_page_len_h = _host_i32(last_page_len_h)
    qo_indptr_h = _host_i32(qo_indptr_h)
    batch = len(kv_indptr_h) - 1
    host_bytes = pinned_ws.numel() * pinned_ws.element_size() if isinstance(
        pinned_ws, torch.Tensor) else pinned_ws.nbytes
    dev_bytes = 0 if dev_ws is None else dev_ws.numel() * dev_ws.element_size()
    p = Plan()
    _check(lib.attn_plan(_ptr(qo_indptr_h), _ptr(kv_indptr_h), _ptr(last_page_len_h), batch,
                         page_size, num_qo_heads, num_kv_heads, head_dim, int(bool(causal)),
                         num_ctas, _ptr(pinned_ws), host_bytes, _ptr(dev_ws), dev_bytes,
                         _stream(stream) if dev_ws is not None else None, ctypes.byref(p)))
    return p


def cascade_workspace_size(max_prompts, max_batch, num_qo_heads, num_kv_heads, head_dim,
                           num_ctas):
    dev = ctypes.c_size_t()
    host = ctypes.c_size_t()
    _check(lib.attn_cascade_workspace_size(max_prompts, max_batch, num_qo_heads, num_kv_heads,
                                           head_dim, num_ctas, ctypes.byref(dev),
                                           ctypes.byref(host)))
    return dev.value, host.value


def plan_cascade(qo_indptr_h, kv_indptr_prefix_h, last_prefix_h, page_size_prefix,
                 kv_indptr_suffix_h, last_suffix_h, page_size_suffix, num_qo_heads, num_kv_heads,
                 head_dim, num_ctas, pinned_ws, dev_ws=None, stream=None) -> Plan:
    """attn_plan_cascade. Host arrays; dev_ws None plans on the host only."""
    qo_indptr_h = _host_i32(qo_indptr_h)
    kv_indptr_prefix_h, last_prefix_h = _host_i32(kv_indptr_prefix_h), _host_i32(last_prefix_h)
    kv_indptr_suffix_h, last_suffix_h = _host_i32(kv_indptr_suffix_h), _host_i32(last_suffix_h)
    prompts = len(qo_indptr_h) - 1
    if len(kv_indptr_prefix_h) != prompts + 1 or len(last_prefix_h) < prompts:
        raise ValueError("the prefix table needs one row per prompt")
    batch = int(qo_indptr_h[-1]) if prompts > 0 else 0
    if len(kv_indptr_suffix_h) != batch + 1 or len(last_suffix_h) < batch:
        raise ValueError("the suffix table needs one row per generation (qo_indptr[-1])")
    host_bytes = pinned_ws.numel() * pinned_ws.element_size() if isinstance(
        pinned_ws, torch.Tensor) else pinned_ws.nbytes
    dev_bytes = 0 if dev_ws is None else dev_ws.numel() * dev_ws.element_size()
    p = Plan()
    _check(lib.attn_plan_cascade(_ptr(qo_indptr_h), _ptr(kv_indptr_prefix_h), _ptr(last_prefix_h),
                                 page_size_prefix, _ptr(kv_indptr_suffix_h), _ptr(last_suffix_h),
                                 page_size_suffix, prompts, num_qo_heads, num_kv_heads, head_dim,
                                 num_ctas, _ptr(pinned_ws), host_bytes, _ptr(dev_ws), dev_bytes,
                                 _stream(stream) if dev_ws is not None else None,
                                 ctypes.byref(p)))
    return p


def cascade_run(p: Plan, q, qo_indptr, prefix, suffix, sm_scale, o, lse, dev_ws,
                layout=LAYOUT_HND, stream=None):
    """attn_cascade_run. prefix / suffix: dicts of device tensors k_pool,
    v_pool (both in `layout`), kv_indptr, kv_indices, last_page_len and
    optionally num_pages (default: the pool's first dimension)."""
    n0 = int(prefix.get("num_pages", prefix["k_pool"].shape[0]))
    n1 = int(suffix.get("num_pages", suffix["k_pool"].shape[0]))
    has_kv = p.total_weight > p.num_items
    _check_shapes(p.num_qo_heads, p.num_kv_heads, p.page_size, p.head_dim, has_kv, q,
                  prefix["k_pool"], prefix["v_pool"], o, lse, n0, p.total_qo)
    _check_shapes(p.num_qo_heads, p.num_kv_heads, p.page_size_suffix, p.head_dim, has_kv, q,
                  suffix["k_pool"], suffix["v_pool"], o, lse, n1, p.total_qo)
    _check(lib.attn_cascade_run(
        ctypes.byref(p), _ptr(q), _ptr(qo_indptr), _ptr(prefix["k_pool"]),
        _ptr(prefix["v_pool"]), n0, _ptr(prefix["kv_indptr"]), _ptr(prefix["kv_indices"]),
        _ptr(prefix["last_page_len"]), _ptr(suffix["k_pool"]), _ptr(suffix["v_pool"]), n1,
        _ptr(suffix["kv_indptr"]), _ptr(suffix["kv_indices"]), _ptr(suffix["last_page_len"]),
        int(layout), dtype_code(q.dtype), float(sm_scale), _ptr(o), _ptr(lse), _ptr(dev_ws),
        dev_ws.numel() * dev_ws.element_size(), _stream(stream)))


def _check_dense(**tensors):
    """The kernels address every tensor as a dense row-major block starting at
    its data pointer, so a strided view (a slice of a larger KV tensor, a
    transpose) would be read with the wrong layout."""
    for name, t in tensors.items():
        if t is not None and not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous (dense row-major); "
                             f"call .contiguous() on it first")


def _check_shapes(num_qo_heads, num_kv_heads, page_size, head_dim, needs_pool, q, k_pool,
                  v_pool, o, lse, num_pages, rows):
    """Tensor sizes, dtypes and layout against the shapes the kernels will
    use, before the library is called: the kernels address the pools with
    those heads and page size, so a smaller pool would be read past its end."""
    _check_dense(q=q, k_pool=k_pool, v_pool=v_pool, out=o, lse=lse)
    per_row = num_qo_heads * head_dim
    need_kv = int(num_pages) * num_kv_heads * page_size * head_dim
    if (needs_pool and num_pages < 1) or k_pool.numel() < need_kv or v_pool.numel() < need_kv:
        raise ValueError(f"k_pool / v_pool hold fewer than num_pages ({num_pages}) x "
                         f"{num_kv_heads} heads x {page_size} slots x {head_dim} elements")
    if k_pool.dtype != q.dtype or v_pool.dtype != q.dtype or o.dtype != q.dtype:
        raise ValueError("q, k_pool, v_pool and out must share one dtype")
    if q.numel() < rows * per_row or o.numel() < rows * per_row:
        raise ValueError(f"q / out need {rows} rows x {num_qo_heads} heads x {head_dim}")
    if lse is not None and (lse.dtype != torch.float32 or lse.numel() < rows * num_qo_heads):
        raise ValueError(f"lse must be float32 with {rows} x {num_qo_heads} elements")


def _check_sizes(p: Plan, q, k_pool, v_pool, o, lse, num_pages, rows):
    """_check_shapes with the plan's shapes; the pool may be empty only when
    the plan's requests hold no kv tokens at all."""
    _check_shapes(p.num_qo_heads, p.num_kv_heads, p.page_size, p.head_dim,
                  p.total_weight > p.num_items, q, k_pool, v_pool, o, lse, num_pages, rows)


def decode_run(p: Plan, q, k_pool, v_pool, kv_indptr, kv_indices, last_page_len, sm_scale, o,
               lse, dev_ws, layout=LAYOUT_HND, num_pages=None, stream=None):
    if num_pages is None:
        num_pages = k_pool.shape[0]
    _check_sizes(p, q, k_pool, v_pool, o, lse, num_pages, p.batch)
    _check(lib.attn_decode_run(ctypes.byref(p), _ptr(q), _ptr(k_pool), _ptr(v_pool),
                               int(num_pages), layout, _ptr(kv_indptr), _ptr(kv_indices),
                               _ptr(last_page_len), dtype_code(q.dtype), float(sm_scale),
                               _ptr(o), _ptr(lse), _ptr(dev_ws),
                               dev_ws.numel() * dev_ws.element_size(), _stream(stream)))


def decode_run_fp8(p: Plan, q, k_pool, v_pool, kv_indptr, kv_indices, last_page_len, k_scale,
                   v_scale, sm_scale, o, lse, dev_ws, layout=LAYOUT_HND, num_pages=None,
                   stream=None):
    """attn_decode_run_fp8: k_pool / v_pool hold FP8 E4M3 bytes (uint8 or
    torch.float8_e4m3fn tensors), k_scale / v_scale device float32
    [num_kv_heads]."""
    if num_pages is None:
        num_pages = k_pool.shape[0]
    _check_dense(q=q, k_pool=k_pool, v_pool=v_pool, out=o, lse=lse, k_scale=k_scale,
                 v_scale=v_scale)
    for t in (k_pool, v_pool):
        if t.element_size() != 1:
            raise ValueError("FP8 pools must be 1-byte tensors (uint8 or float8_e4m3fn)")
    need_kv = int(num_pages) * p.num_kv_heads * p.page_size * p.head_dim
    if ((p.total_weight > p.num_items and num_pages < 1) or k_pool.numel() < need_kv or
            v_pool.numel() < need_kv):
        raise ValueError(f"k_pool / v_pool hold fewer than num_pages ({num_pages}) x "
                         f"{p.num_kv_heads} heads x {p.page_size} slots x {p.head_dim} bytes")
    for t in (k_scale, v_scale):
        if t.dtype != torch.float32 or t.numel() < p.num_kv_heads:
            raise ValueError("k_scale / v_scale must be float32 with num_kv_heads elements")
    per_row = p.num_qo_heads * p.head_dim
    if o.dtype != q.dtype or q.numel() < p.batch * per_row or o.numel() < p.batch * per_row:
        raise ValueError(f"q / out need {p.batch} rows x {p.num_qo_heads} heads x {p.head_dim}"
                         " of one dtype")
    if lse is not None and (lse.dtype != torch.float32 or lse.numel() < p.batch * p.num_qo_heads):
        raise ValueError(f"lse must be float32 with {p.batch} x {p.num_qo_heads} elements")
    _check(lib.attn_decode_run_fp8(ctypes.byref(p), _ptr(q), _ptr(k_pool), _ptr(v_pool),
                                   int(num_pages), layout, _ptr(kv_indptr), _ptr(kv_indices),
                                   _ptr(last_page_len), dtype_code(q.dtype), _ptr(k_scale),
                                   _ptr(v_scale), float(sm_scale), _ptr(o), _ptr(lse),
                                   _ptr(dev_ws), dev_ws.numel() * dev_ws.element_size(),
                                   _stream(stream)))


def _check_rope_tables(rope_cos, rope_sin):
    for t in (rope_cos, rope_sin):
        if t.dtype != torch.float32 or t.dim() != 2 or t.shape[1] != 64 or not t.is_contiguous():
            raise ValueError("rope tables must be contiguous float32 [max_pos, 64]")
    if rope_sin.shape != rope_cos.shape:
        raise ValueError("rope_cos and rope_sin differ in shape")


def decode_run_rope(p: Plan, q, k_pool, v_pool, kv_indptr, kv_indices, last_page_len, sm_scale,
                    rope_cos, rope_sin, o, lse, dev_ws, layout=LAYOUT_HND, num_pages=None,
                    stream=None):
    """attn_decode_run_rope: rope_cos / rope_sin device float32 [max_pos, 64]."""
    _check_rope_tables(rope_cos, rope_sin)
    if num_pages is None:
        num_pages = k_pool.shape[0]
    _check_sizes(p, q, k_pool, v_pool, o, lse, num_pages, p.batch)
    _check(lib.attn_decode_run_rope(ctypes.byref(p), _ptr(q), _ptr(k_pool), _ptr(v_pool),
                                    int(num_pages), layout, _ptr(kv_indptr), _ptr(kv_indices),
                                    _ptr(last_page_len), dtype_code(q.dtype), float(sm_scale),
                                    _ptr(rope_cos), _ptr(rope_sin), int(rope_cos.shape[0]),
                                    _ptr(o), _ptr(lse), _ptr(dev_ws),
                                    dev_ws.numel() * dev_ws.element_size(), _stream(stream)))


def append_run(p: Plan, q, qo_indptr, k_pool, v_pool, kv_indptr, kv_indices, last_page_len,
               causal, sm_scale, o, lse, dev_ws, layout=LAYOUT_HND, num_pages=None,
               stream=None):
    if num_pages is None:
        num_pages = k_pool.shape[0]
    _check_sizes(p, q, k_pool, v_pool, o, lse, num_pages, p.total_qo)
    _check(lib.attn_append_run(ctypes.byref(p), _ptr(q), _ptr(qo_indptr), _ptr(k_pool),
                               _ptr(v_pool), int(num_pages), layout, _ptr(kv_indptr),
                               _ptr(kv_indices), _ptr(last_page_len), dtype_code(q.dtype),
                               int(bool(causal)), float(sm_scale), _ptr(o), _ptr(lse),
                               _ptr(dev_ws), dev_ws.numel() * dev_ws.element_size(),
                               _stream(stream)))


def append_run_rope(p: Plan, q, qo_indptr, k_pool, v_pool, kv_indptr, kv_indices,
                    last_page_len, causal, sm_scale, rope_cos, rope_sin, o, lse, dev_ws,
                    layout=LAYOUT_HND, num_pages=None, stream=None):
    """attn_append_run_rope: rope_cos / rope_sin device float32 [max_pos, 64]."""
    _check_rope_tables(rope_cos, rope_sin)
    if num_pages is None:
        num_pages = k_pool.shape[0]
    _check_sizes(p, q, k_pool, v_pool, o, lse, num_pages, p.total_qo)
    _check(lib.attn_append_run_rope(ctypes.byref(p), _ptr(q), _ptr(qo_indptr), _ptr(k_pool),
                                    _ptr(v_pool), int(num_pages), layout, _ptr(kv_indptr),
                                    _ptr(kv_indices), _ptr(last_page_len), dtype_code(q.dtype),
                                    int(bool(causal)), float(sm_scale), _ptr(rope_cos),
                                    _ptr(rope_sin), int(rope_cos.shape[0]), _ptr(o), _ptr(lse),
                                    _ptr(dev_ws), dev_ws.numel() * dev_ws.element_size(),
                                    _stream(stream)))


def merge_states(o_a, lse_a, o_b, lse_b, o_out, lse_out, stream=None):
    _check_dense(o_a=o_a, lse_a=lse_a, o_b=o_b, lse_b=lse_b, o_out=o_out, lse_out=lse_out)
    n, h, d = o_a.shape
    for t in (o_b, o_out):
        if t.shape != o_a.shape or t.dtype != o_a.dtype:
            raise ValueError("o_a, o_b and o_out must share shape [n, H, D] and dtype")
    for t in (lse_a, lse_b, lse_out):
        if tuple(t.shape) != (n, h) or t.dtype != torch.float32:
            raise ValueError("lse_a, lse_b and lse_out must be float32 [n, H]")
    _check(lib.attn_merge_states(_ptr(o_a), _ptr(lse_a), _ptr(o_b), _ptr(lse_b), _ptr(o_out),
                                 _ptr(lse_out), n, h, d, dtype_code(o_a.dtype), _stream(stream)))


def wait_selftest(dev_ws, limit_us, stream=None):
    """attn_wait_selftest: one bounded wait that nothing completes."""
    _check(lib.attn_wait_selftest(_ptr(dev_ws), int(limit_us), _stream(stream)))


def workspace_status(dev_ws, stream=None) -> int:
    code = ctypes.c_int32()
    st = lib.attn_workspace_status(_ptr(dev_ws), _stream(stream), ctypes.byref(code))
    if st not in (OK, ERR_TIMEOUT):
        _check(st)
    return code.value


def decode_run_noalloc(kv_indptr_h, last_page_len_h, page_size, num_qo_heads, num_kv_heads,
                       head_dim, q, k_pool, v_pool, kv_indptr, kv_indices, last_page_len,
                       sm_scale, o, lse, layout=LAYOUT_HND, num_pages=None, stream=None):
    """attn_decode_run_noalloc: plan + decode in one call, no caller workspace."""
    kv_indptr_h = _host_i32(kv_indptr_h)
    last_page_len_h = _host_i32(last_page_len_h)
    if num_pages is None:
        num_pages = k_pool.shape[0]
    batch = len(kv_indptr_h) - 1
    has_pages = batch > 0 and int(kv_indptr_h[-1]) > int(kv_indptr_h[0])
    _check_shapes(num_qo_heads, num_kv_heads, page_size, head_dim, has_pages, q, k_pool, v_pool,
                  o, lse, num_pages, batch)
    _check(lib.attn_decode_run_noalloc(
        _ptr(kv_indptr_h), _ptr(last_page_len_h), len(kv_indptr_h) - 1, page_size,
        num_qo_heads, num_kv_heads, head_dim, _ptr(q), _ptr(k_pool), _ptr(v_pool),
        int(num_pages), layout, _ptr(kv_indptr), _ptr(kv_indices), _ptr(last_page_len),
        dtype_code(q.dtype), float(sm_scale), _ptr(o), _ptr(lse), _stream(stream)))


def decode_run_noalloc_status(stream=None) -> int:
    """attn_decode_run_noalloc_status: synchronise, then the no-allocation
    scratch area's error word on the current device (0 = no kernel gave up)."""
    code = ctypes.c_int32()
    st = lib.attn_decode_run_noalloc_status(_stream(stream), ctypes.byref(code))
    if st not in (OK, ERR_TIMEOUT):
        _check(st)
    return code.value


def wait_selftest_noalloc(limit_us, stream=None):
    """attn_wait_selftest_noalloc: one bounded wait that nothing completes,
    reporting into the no-allocation scratch area's error word."""
    _check(lib.attn_wait_selftest_noalloc(int(limit_us), _stream(stream)))
