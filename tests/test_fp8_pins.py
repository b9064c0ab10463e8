"""Pins of the FP8 (E4M3) KV-cache oracle (oracle_batch_attention_fp8kv).
No GPU.

The stored byte b of kv head hk stands for widen_e4m3(b) * scale[hk]. The
pins: the widening agrees with torch's float8_e4m3fn conversion on all 256
patterns; attention over an FP8 cache equals torch float64 SDPA over keys and
values that the test dequantizes itself (torch's conversion, times the
scale) and gathers with numpy, for decode and causal append; scaling the key
scales is a scaling of sm_scale and scaling the value scales scales O.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from paged_kv_attention_bsr_gb300 import synth


def test_e4m3_widening_matches_torch_on_every_pattern():
    bits = torch.arange(256, dtype=torch.int64).to(torch.uint8)
    ref = bits.view(torch.float8_e4m3fn).double().numpy()
    got = np.array([oracle.widen_e4m3(b) for b in range(256)])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan) and nan.sum() == 2  # 0x7f and 0xff
    assert np.array_equal(got[~nan], ref[~nan])
    assert got[0x7e] == 448.0 and got[0x01] == 2.0 ** -9 and got[0x80] == 0.0


def _dequant(pool_u8, scale):
    return pool_u8.view(torch.float8_e4m3fn).double() * scale.double()[None, :, None, None]


def _reference(w, causal):
    """numpy gather of dequantized K / V + torch float64 SDPA, per request."""
    c = w.cache
    k = _dequant(c.k_pool, c.k_scale).numpy()
    v = _dequant(c.v_pool, c.v_scale).numpy()
    q = w.q.double().numpy()
    qo = w.qo_indptr if w.qo_indptr is not None else np.arange(w.batch + 1)
    g = w.num_qo_heads // w.num_kv_heads
    P = c.page_size
    outs, lses = [], []
    for r in range(w.batch):
        L = int(c.kv_lens[r])
        rows = q[qo[r]:qo[r + 1]]
        n = rows.shape[0]
        if L == 0:
            outs.append(np.zeros_like(rows))
            lses.append(np.full(rows.shape[:2], -np.inf))
            continue
        pages = c.kv_indices[c.kv_indptr[r]:c.kv_indptr[r + 1]]
        kk = np.stack([k[pages[t // P], :, t % P] for t in range(L)], axis=1)  # [Hk, L, D]
        vv = np.stack([v[pages[t // P], :, t % P] for t in range(L)], axis=1)
        qt = torch.from_numpy(rows).permute(1, 0, 2)
        kt = torch.from_numpy(kk).repeat_interleave(g, 0)
        vt = torch.from_numpy(vv).repeat_interleave(g, 0)
        mask = None
        if causal:
            qpos = L - n + np.arange(n)
            mask = torch.from_numpy(np.arange(L)[None, :] <= qpos[:, None])
        o = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, attn_mask=mask,
                                                             scale=w.sm_scale)
        logits = (qt @ kt.transpose(1, 2)) * w.sm_scale
        if mask is not None:
            logits = logits.masked_fill(~mask, -math.inf)
        outs.append(o.permute(1, 0, 2).numpy())
        lses.append(torch.logsumexp(logits, -1).permute(1, 0).numpy())
    return np.concatenate(outs), np.concatenate(lses)


def _run(w, causal=False, k_scale=None, v_scale=None, sm_scale=None):
    c = w.cache
    return oracle.batch_attention_fp8kv(
        w.q, c.k_pool, c.v_pool, c.kv_indptr, c.kv_indices, c.last_page_len, c.page_size,
        w.num_qo_heads, w.num_kv_heads, 128,
        oracle.BF16 if w.dtype == torch.bfloat16 else oracle.F16,
        w.sm_scale if sm_scale is None else sm_scale,
        c.k_scale.numpy() if k_scale is None else k_scale,
        c.v_scale.numpy() if v_scale is None else v_scale, causal=causal,
        qo_indptr=w.qo_indptr)


@pytest.mark.parametrize("P,Hq,Hk,dt", [(16, 8, 2, torch.bfloat16), (3, 16, 4, torch.float16),
                                        (1, 4, 4, torch.bfloat16)])
def test_fp8_decode_matches_sdpa_on_dequantized_kv(P, Hq, Hk, dt):
    lens = [1, 37, 300, 0, 129]
    pool = sum(-(-L // P) for L in lens) + 5
    w = synth.fp8_decode_workload("f8", lens, P, pool, Hq, Hk, dt, seed=31)
    o, l = _run(w)
    o_ref, l_ref = _reference(w, False)
    fin = np.isfinite(l_ref)
    assert np.abs(o - o_ref).max() < 1e-12
    assert np.abs(l[fin] - l_ref[fin]).max() < 1e-12 and np.all(np.isneginf(l[~fin]))


def test_fp8_causal_append_matches_sdpa_on_dequantized_kv():
    P = 16
    qo, ex = [1, 7, 30], [0, 200, 900]
    kv = [a + b for a, b in zip(qo, ex)]
    pool = sum(-(-L // P) for L in kv) + 3
    cache = synth.make_fp8_cache(kv, P, pool, 2, seed=41)
    qo_indptr = np.concatenate([[0], np.cumsum(qo)]).astype(np.int32)
    q = synth.normal_values((int(qo_indptr[-1]), 8, 128), torch.bfloat16, 42)
    w = synth.Workload("f8a", "append", torch.bfloat16, 8, 2, 128, 1 / math.sqrt(128), q, cache,
                       qo_indptr=qo_indptr, causal=True)
    o, l = _run(w, causal=True)
    o_ref, l_ref = _reference(w, True)
    assert np.abs(o - o_ref).max() < 1e-12 and np.abs(l - l_ref).max() < 1e-12


def test_fp8_scales_act_as_multipliers():
    lens = [50, 700]
    w = synth.fp8_decode_workload("f8s", lens, 16, 60, 8, 2, torch.bfloat16, seed=51)
    ks, vs = w.cache.k_scale.numpy(), w.cache.v_scale.numpy()
    o, l = _run(w)
    # doubling every key scale is doubling sm_scale
    o2, l2 = _run(w, k_scale=2 * ks)
    o3, l3 = _run(w, sm_scale=2 * w.sm_scale)
    assert np.abs(o2 - o3).max() < 1e-12 and np.abs(l2 - l3).max() < 1e-12
    assert np.abs(o2 - o).max() > 1e-3  # and it changes the result
    # doubling every value scale doubles O and leaves the LSE alone
    o4, l4 = _run(w, v_scale=2 * vs)
    assert np.abs(o4 - 2 * o).max() < 1e-12 and np.array_equal(l4, l)
