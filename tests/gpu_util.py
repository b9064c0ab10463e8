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
