"""Pins of the rotary-position-embedding oracle (oracle_batch_attention_rope)
and of the RoPE table builder. No GPU.

The oracle rotates q (position kv_len - qo_len + i) and k (position j) in
pairs (d, d + D/2), rounds them to the storage type and then computes exact
attention. The pins: an identity table reproduces the plain oracle bit for
bit; quarter-turn tables (exact rotations) and general LLaMA 3.1 tables
match torch's float64 scaled_dot_product_attention on q / k rotated here
with numpy (rounded by this file's own routine); the rounding routine agrees
with torch's conversions.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from paged_kv_attention_bsr_gb300 import synth


def _round_np(x, dtype):
    """float64 -> nearest bf16 / fp16 value (ties to even), numpy only."""
    bits = 8 if dtype == oracle.BF16 else 11
    emin = -126 if dtype == oracle.BF16 else -14
    m, e = np.frexp(x)
    q = np.maximum(e - bits, emin - bits + 1)
    return np.where(x == 0, 0.0, np.ldexp(np.rint(np.ldexp(x, -q)), q))


def _rotate(x, pos, cos, sin):
    """rotate-half RoPE of rows x [..., D] at integer positions pos [...]."""
    h = x.shape[-1] // 2
    c, s = cos[pos].astype(np.float64), sin[pos].astype(np.float64)
    a, b = x[..., :h], x[..., h:]
    return np.concatenate([a * c - b * s, b * c + a * s], axis=-1)


def _gather(pool, kv_indptr, kv_indices, P, r, n):
    pages = kv_indices[kv_indptr[r]:kv_indptr[r + 1]]
    rows = [pool[pages[t // P], :, t % P, :] for t in range(n)]  # HND
    return np.stack(rows, axis=1) if rows else np.zeros((pool.shape[1], 0, pool.shape[3]))


def _reference(w, cos, sin, dtype, causal):
    """RoPE (numpy) + rounding (numpy) + torch float64 SDPA, per request."""
    c = w.cache
    q = w.q.float().numpy().astype(np.float64)
    k = c.k_pool.float().numpy().astype(np.float64)
    v = c.v_pool.float().numpy().astype(np.float64)
    qo = w.qo_indptr if w.qo_indptr is not None else np.arange(w.batch + 1)
    g = w.num_qo_heads // w.num_kv_heads
    outs, lses = [], []
    for r in range(w.batch):
        L = int(c.kv_lens[r])
        rows = q[qo[r]:qo[r + 1]]  # [n, Hq, D]
        n = rows.shape[0]
        if L == 0:
            outs.append(np.zeros_like(rows))
            lses.append(np.full(rows.shape[:2], -np.inf))
            continue
        qpos = L - n + np.arange(n)
        qr = _round_np(_rotate(rows, qpos[:, None].repeat(rows.shape[1], 1), cos, sin), dtype)
        kk = _gather(k, c.kv_indptr, c.kv_indices, c.page_size, r, L)  # [Hk, L, D]
        vv = _gather(v, c.kv_indptr, c.kv_indices, c.page_size, r, L)
        kr = _round_np(_rotate(kk, np.arange(L)[None, :].repeat(kk.shape[0], 0), cos, sin), dtype)
        qt = torch.from_numpy(qr).permute(1, 0, 2)  # [Hq, n, D]
        kt = torch.from_numpy(kr).repeat_interleave(g, 0)
        vt = torch.from_numpy(vv).repeat_interleave(g, 0)
        mask = None
        if causal:
            mask = torch.from_numpy(np.arange(L)[None, :] <= qpos[:, None])
        o = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, attn_mask=mask,
                                                             scale=w.sm_scale)
        logits = (qt @ kt.transpose(1, 2)) * w.sm_scale
        if mask is not None:
            logits = logits.masked_fill(~mask, -math.inf)
        outs.append(o.permute(1, 0, 2).numpy())
        lses.append(torch.logsumexp(logits, -1).permute(1, 0).numpy())
    return np.concatenate(outs), np.concatenate(lses)


def _run(w, cos, sin, dtype, causal):
    c = w.cache
    return oracle.batch_attention_rope(w.q, c.k_pool, c.v_pool, c.kv_indptr, c.kv_indices,
                                       c.last_page_len, c.page_size, w.num_qo_heads,
                                       w.num_kv_heads, 128, dtype, w.sm_scale, cos, sin,
                                       causal=causal, qo_indptr=w.qo_indptr)


def _decode(lens, P=16, Hq=8, Hk=2, dt=torch.bfloat16, seed=1):
    pool = sum(-(-L // P) for L in lens) + 5
    return synth.decode_workload("r", lens, P, pool, Hq, Hk, dt, seed=seed)


def test_identity_table_reproduces_the_plain_oracle_bit_for_bit():
    w = _decode([1, 37, 300, 0, 129])
    c = w.cache
    cos = np.ones((400, 64), np.float32)
    sin = np.zeros((400, 64), np.float32)
    o1, l1 = _run(w, cos, sin, oracle.BF16, False)
    o2, l2 = oracle.batch_attention(w.q, c.k_pool, c.v_pool, c.kv_indptr, c.kv_indices,
                                    c.last_page_len, 16, 8, 2, 128, oracle.BF16, w.sm_scale)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


def test_quarter_turns_match_sdpa_on_numpy_rotated_inputs():
    # cos, sin in {0, +-1}: rotations are exact (swaps / sign flips)
    rng = np.random.default_rng(4)
    turns = rng.integers(0, 4, size=(600, 64))
    cos = np.array([1, 0, -1, 0], np.float32)[turns]
    sin = np.array([0, 1, 0, -1], np.float32)[turns]
    for dt, od in ((torch.bfloat16, oracle.BF16), (torch.float16, oracle.F16)):
        w = _decode([5, 300, 17, 520], P=16, Hq=16, Hk=4, dt=dt, seed=2)
        o, l = _run(w, cos, sin, od, False)
        o_ref, l_ref = _reference(w, cos, sin, od, False)
        assert np.abs(o - o_ref).max() < 1e-12 and np.abs(l - l_ref).max() < 1e-12


@pytest.mark.parametrize("causal", [False, True])
def test_llama31_tables_match_sdpa_on_numpy_rotated_inputs(causal):
    cos, sin = synth.rope_tables(2000)
    P = 16
    qo, ex = [1, 7, 30], [0, 200, 900]
    kv = [a + b for a, b in zip(qo, ex)]
    pool = sum(-(-L // P) for L in kv) + 3
    w = synth.append_workload("ra", qo, kv, P, pool, 8, 2, torch.bfloat16, seed=9,
                              causal=causal)
    o, l = _run(w, cos, sin, oracle.BF16, causal)
    o_ref, l_ref = _reference(w, cos, sin, oracle.BF16, causal)
    assert np.abs(o - o_ref).max() < 1e-12 and np.abs(l - l_ref).max() < 1e-12
    # and RoPE changed the result (the pin is not vacuous)
    c = w.cache
    o0, _ = oracle.batch_attention(w.q, c.k_pool, c.v_pool, c.kv_indptr, c.kv_indices,
                                   c.last_page_len, P, 8, 2, 128, oracle.BF16, w.sm_scale,
                                   causal=causal, qo_indptr=w.qo_indptr)
    assert np.abs(o - o0).max() > 1e-2


@pytest.mark.parametrize("causal", [False, True])
def test_row_rope_matches_sdpa_on_numpy_rotated_inputs(causal):
    """oracle_attention_row_rope (one row at a time) against the numpy
    rotation + torch float64 SDPA reference, on every row of a small ragged
    batch (and a few rows sit at positions near the end of the table)."""
    cos, sin = synth.rope_tables(1200)
    P = 3
    qo, ex = [1, 9, 20], [0, 500, 1171]
    kv = [a + b for a, b in zip(qo, ex)]
    pool = sum(-(-L // P) for L in kv) + 3
    w = synth.append_workload("rr", qo, kv, P, pool, 16, 4, torch.bfloat16, seed=13,
                              causal=causal)
    o_ref, l_ref = _reference(w, cos, sin, oracle.BF16, causal)
    c = w.cache
    for r in range(w.batch):
        for i in range(qo[r]):
            for h in (0, 5, 15):
                o, l = oracle.attention_row_rope(
                    w.q, c.k_pool, c.v_pool, c.kv_indptr, c.kv_indices, c.last_page_len, P,
                    16, 4, 128, oracle.BF16, w.sm_scale, cos, sin, r, i, h, causal=causal,
                    qo_indptr=w.qo_indptr)
                row = int(w.qo_indptr[r]) + i
                assert np.abs(o - o_ref[row, h]).max() < 1e-12
                assert abs(l - l_ref[row, h]) < 1e-12


def test_rounding_matches_torch_conversions():
    rng = np.random.default_rng(5)
    vals = np.concatenate([rng.normal(0, 10, 2000), rng.normal(0, 1e-6, 200),
                           np.array([0.0, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, 65519.0, 65520.0])])
    vals = vals.astype(np.float32).astype(np.float64)  # exact in fp32, so torch rounds once
    for od, tdt in ((oracle.BF16, torch.bfloat16), (oracle.F16, torch.float16)):
        ref = torch.from_numpy(vals.astype(np.float32)).to(tdt).double().numpy()
        got = np.array([oracle.round_to(v, od) for v in vals])
        assert np.array_equal(got, ref)
        assert np.array_equal(_round_np(vals[np.isfinite(ref)], od), ref[np.isfinite(ref)])


def test_rope_table_properties():
    cos, sin = synth.rope_tables(9000)
    assert cos.dtype == np.float32 and cos.shape == (9000, 64)
    assert np.all(cos[0] == 1) and np.all(sin[0] == 0)
    assert np.abs(cos.astype(np.float64) ** 2 + sin.astype(np.float64) ** 2 - 1).max() < 1e-6
    # angle addition: row p+q is row p turned by row q (angles are linear in pos)
    p, q = 1234, 4321
    c = cos[p].astype(np.float64) * cos[q] - sin[p].astype(np.float64) * sin[q]
    s = sin[p].astype(np.float64) * cos[q] + cos[p].astype(np.float64) * sin[q]
    assert np.abs(c - cos[p + q]).max() < 1e-3 and np.abs(s - sin[p + q]).max() < 1e-3
    # LLaMA 3.1 rescaling: the fastest pair keeps f = 1, the slowest is divided
    # by the factor, and frequencies stay ordered
    plain_c, plain_s = synth.rope_tables(2, llama31=False)
    f_plain = np.arctan2(plain_s[1], plain_c[1])
    f_31 = np.arctan2(sin[1], cos[1])
    assert abs(f_31[0] - 1.0) < 1e-6 and abs(f_plain[0] - 1.0) < 1e-6
    assert abs(f_31[-1] * 8.0 / f_plain[-1] - 1.0) < 1e-4
    assert np.all(np.diff(f_31) < 0)
