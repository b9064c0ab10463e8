"""Helpers shared by the GPU parity tests (CUDA path vs fp64 oracle)."""
from __future__ import annotations

import numpy as np
import torch

# Tolerances of the parity bar (outputs are bf16/fp16, compared with the
# unrounded fp64 oracle): max |err| <= 2e-2, mean |err| <= 2e-3 on O,
# |err| <= 1e-3 on the natural-log LSE.
O_MAX_ABS = 2e-2
O_MEAN_ABS = 2e-3
LSE_ABS = 1e-3


def oracle_dtype(oracle_mod, dtype):
    return oracle_mod.BF16 if dtype == torch.bfloat16 else oracle_mod.F16


def to_device(cache, device="cuda"):
    return dict(
        k_pool=cache.k_pool.to(device), v_pool=cache.v_pool.to(device),
        kv_indptr=torch.from_numpy(cache.kv_indptr).to(device),
        kv_indices=torch.from_numpy(cache.kv_indices).to(device),
        last_page_len=torch.from_numpy(cache.last_page_len).to(device))


def assert_attn_close(o_gpu, lse_gpu, o_ref, lse_ref, what=""):
    o = o_gpu.detach().float().cpu().numpy().astype(np.float64).reshape(o_ref.shape)
    lse = lse_gpu.detach().float().cpu().numpy().astype(np.float64).reshape(lse_ref.shape)
    assert np.all(np.isfinite(o)), f"{what}: non-finite output"
    err = np.abs(o - o_ref)
    assert err.max() <= O_MAX_ABS, f"{what}: max |dO| = {err.max():.3e}"
    assert err.mean() <= O_MEAN_ABS, f"{what}: mean |dO| = {err.mean():.3e}"
    empty = ~np.isfinite(lse_ref)
    assert np.all(np.isneginf(lse[empty])), f"{what}: empty rows must give LSE = -inf"
    assert np.all(o[empty] == 0), f"{what}: empty rows must give O = 0"
    if np.any(~empty):
        d = np.abs(lse[~empty] - lse_ref[~empty])
        assert d.max() <= LSE_ABS, f"{what}: max |dLSE| = {d.max():.3e}"
    return float(err.max()), float(err.mean())


def poison_unused_slots(cache):
    """Fill every pool slot no request reads with NaN: a kernel that lets a
    stale row reach its arithmetic (even multiplied by a zero probability)
    then produces NaN instead of a plausible number."""
    P = cache.page_size
    valid = torch.zeros(cache.num_pages, P, dtype=torch.bool)
    for r in range(len(cache.kv_indptr) - 1):
        pages = cache.kv_indices[cache.kv_indptr[r]:cache.kv_indptr[r + 1]]
        for j, pg in enumerate(pages):
            n = P if j + 1 < len(pages) else int(cache.last_page_len[r])
            valid[int(pg), :n] = True
    bad = ~valid  # [pages, P] -> HND pools [pages, Hk, P, D]
    for pool in (cache.k_pool, cache.v_pool):
        pool.permute(0, 2, 1, 3)[bad] = float("nan")


def oracle_decode_threaded(oracle_mod, w, threads=16):
    """The fp64 oracle over every row of a decode batch, requests split across
    host threads (the C oracle releases the GIL). Returns (o, lse) like
    oracle_mod.batch_attention."""
    import concurrent.futures as cf
    c = w.cache
    dt = oracle_dtype(oracle_mod, w.dtype)
    chunks = [x for x in np.array_split(np.arange(w.batch), threads) if len(x)]

    def job(rs):
        a, b = int(rs[0]), int(rs[-1]) + 1
        return oracle_mod.batch_attention(w.q[a:b], c.k_pool, c.v_pool, c.kv_indptr[a:b + 1],
                                          c.kv_indices, c.last_page_len[a:b], c.page_size,
                                          w.num_qo_heads, w.num_kv_heads, w.head_dim, dt,
                                          w.sm_scale)

    with cf.ThreadPoolExecutor(threads) as ex:
        parts = list(ex.map(job, chunks))
    return np.concatenate([p[0] for p in parts]), np.concatenate([p[1] for p in parts])


def oracle_rows_threaded(oracle_mod, w, rows, causal, qo_indptr=None, threads=16):
    """The fp64 oracle on selected (request, query index, query head) rows,
    across host threads. Returns (o [n, D], lse [n])."""
    import concurrent.futures as cf
    c = w.cache
    dt = oracle_dtype(oracle_mod, w.dtype)
    chunks = [x for x in np.array_split(np.arange(len(rows)), threads) if len(x)]

    def job(idx):
        out_o = np.zeros((len(idx), w.head_dim))
        out_l = np.zeros(len(idx))
        for j, k in enumerate(idx):
            r, i, h = rows[k]
            out_o[j], out_l[j] = oracle_mod.attention_row(
                w.q, c.k_pool, c.v_pool, c.kv_indptr, c.kv_indices, c.last_page_len,
                c.page_size, w.num_qo_heads, w.num_kv_heads, w.head_dim, dt, w.sm_scale, r, i,
                h, causal=causal, qo_indptr=qo_indptr)
        return out_o, out_l

    with cf.ThreadPoolExecutor(threads) as ex:
        parts = list(ex.map(job, chunks))
    return np.concatenate([p[0] for p in parts]), np.concatenate([p[1] for p in parts])


def split_items_of_plan(att):
    """(r, hk, t, n_units) of every split item of the plan `att` (a
    PagedAttention) last made, read from its pinned host copy of the tables."""
    p = att.plan_info
    buf = att._pinned[(att._turn - 1) % att.RING].numpy()
    raw = buf[p.off_merge_items:p.off_merge_items + 16 * p.num_split_items]
    return raw.view(np.int32).reshape(-1, 4).copy()
