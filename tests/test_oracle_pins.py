"""Pins for the fp64 oracle against things other than itself.

* a library routine: torch scaled_dot_product_attention in float64 on CPU,
  with torch's own end-aligned causal bias (causal_lower_right), on K/V that
  the test gathers from the page table with numpy fancy indexing;
* scipy.special.logsumexp of numpy-computed logits for the LSE;
* exact widening of every 16-bit pattern against numpy / torch conversions;
* closed forms (kv_len = 1, q = 0, equal keys, one dominant logit, causal
  first row);
* the invariants the pages imply: the result does not depend on page size,
  physical page order or pool layout (bit-identical); split + LSE merge equals
  the unsplit result; shared prefix + suffix + merge equals one flat layout.
"""
import math

import numpy as np
import pytest
import torch
from scipy.special import logsumexp

from paged_kv_attention_bsr_gb300 import synth

D = 128


def _bf16(shape, seed, scale=1.0):
    g = torch.Generator().manual_seed(seed)
    return (torch.randn(shape, generator=g, dtype=torch.float32) * scale).to(torch.bfloat16)


def _gather_dense(cache, r, hk):
    """Logical K, V of request r / kv head hk via numpy fancy indexing (HND pool)."""
    pages = cache.kv_indices[cache.kv_indptr[r]:cache.kv_indptr[r + 1]]
    n = len(pages)
    kv_len = 0 if n == 0 else (n - 1) * cache.page_size + int(cache.last_page_len[r])
    k = cache.k_pool[torch.as_tensor(pages, dtype=torch.long), hk].reshape(-1, cache.head_dim)
    v = cache.v_pool[torch.as_tensor(pages, dtype=torch.long), hk].reshape(-1, cache.head_dim)
    return k[:kv_len].double(), v[:kv_len].double()


def _sdpa_rows(q_rows, k, v, sm_scale, causal):
    """q_rows [L, D] against k, v [N, D] -> o [L, D] via torch SDPA (float64)."""
    from torch.nn.attention.bias import causal_lower_right
    L, N = q_rows.shape[0], k.shape[0]
    qq, kk, vv = q_rows[None, None], k[None, None], v[None, None]
    if causal:
        mask = causal_lower_right(L, N)
        return torch.nn.functional.scaled_dot_product_attention(
            qq, kk, vv, attn_mask=mask, scale=sm_scale)[0, 0]
    return torch.nn.functional.scaled_dot_product_attention(qq, kk, vv, scale=sm_scale)[0, 0]


def _lse_rows(q_rows, k, sm_scale, causal):
    x = sm_scale * (q_rows.numpy() @ k.numpy().T)
    L, N = x.shape
    if causal:
        for i in range(L):
            x[i, N - L + i + 1:] = -np.inf
    return logsumexp(x, axis=1)


def test_widen_every_pattern(oracle_mod):
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref16 = bits.view(np.float16).astype(np.float64)
    refb = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).double().numpy()
    got16 = np.array([oracle_mod.widen(b, oracle_mod.F16) for b in bits])
    gotb = np.array([oracle_mod.widen(b, oracle_mod.BF16) for b in bits])
    np.testing.assert_array_equal(np.isnan(got16), np.isnan(ref16))
    np.testing.assert_array_equal(np.isnan(gotb), np.isnan(refb))
    np.testing.assert_array_equal(np.nan_to_num(got16, nan=7.0), np.nan_to_num(ref16, nan=7.0))
    np.testing.assert_array_equal(np.nan_to_num(gotb, nan=7.0), np.nan_to_num(refb, nan=7.0))


@pytest.mark.parametrize("page_size", [1, 3, 16])
@pytest.mark.parametrize("group", [1, 2, 4, 8])
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16])
def test_decode_matches_sdpa(oracle_mod, page_size, group, dtype):
    Hk = 2
    Hq = Hk * group
    rng = np.random.default_rng(1000 + page_size * 10 + group)
    kv_lens = rng.integers(0, 70, size=4)
    kv_lens[1] = 1
    w = synth.decode_workload("t", kv_lens, page_size, 200, Hq, Hk, dtype,
                              seed=int(rng.integers(1 << 30)), head_dim=D)
    c = w.cache
    odt = oracle_mod.BF16 if dtype == torch.bfloat16 else oracle_mod.F16
    o, lse = oracle_mod.batch_attention(w.q, c.k_pool, c.v_pool, c.kv_indptr, c.kv_indices,
                                        c.last_page_len, page_size, Hq, Hk, D, odt, w.sm_scale)
    for r in range(w.batch):
        for hk in range(Hk):
            k, v = _gather_dense(c, r, hk)
            q_rows = w.q[r, hk * group:(hk + 1) * group].double()
            if k.shape[0] == 0:
                assert np.all(o[r, hk * group:(hk + 1) * group] == 0)
                assert np.all(np.isneginf(lse[r, hk * group:(hk + 1) * group]))
                continue
            ref = _sdpa_rows(q_rows, k, v, w.sm_scale, False).numpy()
            np.testing.assert_allclose(o[r, hk * group:(hk + 1) * group], ref, rtol=0, atol=1e-12)
            ref_lse = _lse_rows(q_rows, k, w.sm_scale, False)
            np.testing.assert_allclose(lse[r, hk * group:(hk + 1) * group], ref_lse, rtol=0, atol=1e-12)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("page_size", [2, 16])
def test_append_matches_sdpa(oracle_mod, causal, page_size):
    Hk, group = 2, 4
    Hq = Hk * group
    rng = np.random.default_rng(77 + page_size + 5 * causal)
    qo_lens = rng.integers(1, 20, size=3)
    kv_lens = qo_lens + rng.integers(0, 40, size=3)
    qo_lens[2] = kv_lens[2]  # fully causal-square request
    w = synth.append_workload("t", qo_lens, kv_lens, page_size, 100, Hq, Hk, torch.bfloat16,
                              seed=int(rng.integers(1 << 30)), causal=causal, head_dim=D)
    c = w.cache
    o, lse = oracle_mod.batch_attention(w.q, c.k_pool, c.v_pool, c.kv_indptr, c.kv_indices,
                                        c.last_page_len, page_size, Hq, Hk, D, oracle_mod.BF16,
                                        w.sm_scale, causal=causal, qo_indptr=w.qo_indptr)
    for r in range(w.batch):
        a, b = w.qo_indptr[r], w.qo_indptr[r + 1]
        for h in range(Hq):
            k, v = _gather_dense(c, r, h // group)
            q_rows = w.q[a:b, h].double()
            ref = _sdpa_rows(q_rows, k, v, w.sm_scale, causal).numpy()
            np.testing.assert_allclose(o[a:b, h], ref, rtol=0, atol=1e-12)
            np.testing.assert_allclose(lse[a:b, h], _lse_rows(q_rows, k, w.sm_scale, causal),
                                       rtol=0, atol=1e-12)


def _one_request(oracle_mod, q, k_rows, v_rows, sm_scale, causal=False, qo_len=1):
    """Helper: single request, contiguous pages of 16, bf16 storage."""
    n = k_rows.shape[0]
    P = 16
    pages = max(1, -(-n // P))
    kp = torch.zeros((pages, 1, P, D), dtype=torch.bfloat16)
    vp = torch.zeros((pages, 1, P, D), dtype=torch.bfloat16)
    kp.view(-1, D)[:n] = k_rows
    vp.view(-1, D)[:n] = v_rows
    indptr = np.array([0, pages if n else 0], np.int32)
    last = np.array([n - P * (pages - 1) if n else 0], np.int32)
    qo_indptr = None if qo_len == 1 and not causal else np.array([0, qo_len], np.int32)
    return oracle_mod.batch_attention(q.reshape(-1, 1, D), kp, vp, indptr,
                                      np.arange(pages, dtype=np.int32), last, P, 1, 1, D,
                                      oracle_mod.BF16, sm_scale, causal=causal,
                                      qo_indptr=qo_indptr)


def test_closed_forms(oracle_mod):
    s = 1.0 / math.sqrt(D)
    q = _bf16((1, D), 1)
    k = _bf16((40, D), 2)
    v = _bf16((40, D), 3)
    # kv_len = 1: O = v0 exactly, LSE = s <q, k0>
    o, lse = _one_request(oracle_mod, q, k[:1], v[:1], s)
    np.testing.assert_array_equal(o[0, 0], v[0].double().numpy())
    assert lse[0, 0] == pytest.approx(s * float((q[0].double() * k[0].double()).sum()), abs=1e-13)
    # q = 0: O = mean of V, LSE = ln N
    o, lse = _one_request(oracle_mod, torch.zeros((1, D), dtype=torch.bfloat16), k, v, s)
    np.testing.assert_allclose(o[0, 0], v.double().mean(0).numpy(), atol=1e-14, rtol=0)
    assert lse[0, 0] == pytest.approx(math.log(40), abs=1e-14)
    # all keys equal: O = mean of V, LSE = x + ln N
    keq = k[:1].repeat(40, 1)
    o, lse = _one_request(oracle_mod, q, keq, v, s)
    x = s * float((q[0].double() * k[0].double()).sum())
    np.testing.assert_allclose(o[0, 0], v.double().mean(0).numpy(), atol=1e-14, rtol=0)
    assert lse[0, 0] == pytest.approx(x + math.log(40), abs=1e-13)
    # one logit ~40 above the rest: O = v_j to within 1e-15 relative to |v|
    qh = torch.zeros((1, D), dtype=torch.bfloat16)
    qh[0, 5] = 1.0
    kd = torch.zeros((40, D), dtype=torch.bfloat16)
    kd[:, 7] = _bf16((40,), 9)
    kd[23, 5] = 452.0  # s * 452 = 39.96
    o, lse = _one_request(oracle_mod, qh, kd, v, s)
    np.testing.assert_allclose(o[0, 0], v[23].double().numpy(), atol=1e-15 * 40, rtol=0)
    # causal with qo_len = kv_len: row 0 sees only j = 0, row i sees j <= i
    qs = _bf16((6, D), 4)
    o, lse = _one_request(oracle_mod, qs, k[:6], v[:6], s, causal=True, qo_len=6)
    np.testing.assert_array_equal(o[0, 0], v[0].double().numpy())
    o_last = _sdpa_rows(qs[5:6].double(), k[:6].double(), v[:6].double(), s, False).numpy()
    np.testing.assert_allclose(o[5, 0], o_last[0], atol=1e-13, rtol=0)


def _repage(cache, new_page, rng, layout_nhd=False):
    """Same logical KV re-stored with another page size, in a permuted pool."""
    B = len(cache.kv_indptr) - 1
    Hk = cache.num_kv_heads
    lens = []
    ks, vs = [], []
    for r in range(B):
        kr = [_gather_dense(cache, r, hk)[0] for hk in range(Hk)]
        vr = [_gather_dense(cache, r, hk)[1] for hk in range(Hk)]
        lens.append(kr[0].shape[0])
        ks.append(torch.stack(kr, 0))
        vs.append(torch.stack(vr, 0))
    npages = [-(-L // new_page) for L in lens]
    total = sum(npages)
    pool = total + 7
    perm = rng.permutation(pool)[:total]
    shape = (pool, Hk, new_page, D)
    kp = torch.full(shape, 3.0, dtype=torch.float64)
    vp = torch.full(shape, -5.0, dtype=torch.float64)
    indptr = [0]
    indices = []
    last = []
    at = 0
    for r in range(B):
        for j in range(npages[r]):
            pg = perm[at]
            at += 1
            indices.append(pg)
            seg_k = ks[r][:, j * new_page:(j + 1) * new_page]
            seg_v = vs[r][:, j * new_page:(j + 1) * new_page]
            kp[pg, :, :seg_k.shape[1]] = seg_k
            vp[pg, :, :seg_v.shape[1]] = seg_v
        indptr.append(len(indices))
        last.append(lens[r] - new_page * (npages[r] - 1) if npages[r] else 0)
    kp, vp = kp.to(torch.bfloat16), vp.to(torch.bfloat16)
    if layout_nhd:
        kp = kp.permute(0, 2, 1, 3).contiguous()
        vp = vp.permute(0, 2, 1, 3).contiguous()
    return kp, vp, np.array(indptr, np.int32), np.array(indices, np.int32), np.array(last, np.int32)


@pytest.mark.parametrize("causal", [False, True])
def test_repaging_and_layout_bit_identical(oracle_mod, causal):
    Hk, group = 2, 2
    Hq = Hk * group
    rng = np.random.default_rng(5)
    qo_lens = np.array([3, 1, 5])
    kv_lens = np.array([37, 16, 50])
    w = synth.append_workload("t", qo_lens, kv_lens, 16, 20, Hq, Hk, torch.bfloat16, seed=99,
                              causal=causal, head_dim=D)
    c = w.cache
    base = oracle_mod.batch_attention(w.q, c.k_pool, c.v_pool, c.kv_indptr, c.kv_indices,
                                      c.last_page_len, 16, Hq, Hk, D, oracle_mod.BF16,
                                      w.sm_scale, causal=causal, qo_indptr=w.qo_indptr)
    for P in [1, 2, 3, 16, 128, 50]:
        for nhd in (False, True):
            kp, vp, ip, ix, last = _repage(c, P, rng, layout_nhd=nhd)
            got = oracle_mod.batch_attention(
                w.q, kp, vp, ip, ix, last, P, Hq, Hk, D, oracle_mod.BF16, w.sm_scale,
                causal=causal, qo_indptr=w.qo_indptr,
                layout=oracle_mod.NHD if nhd else oracle_mod.HND)
            np.testing.assert_array_equal(got[0], base[0])
            np.testing.assert_array_equal(got[1], base[1])


def test_split_merge_equals_unsplit(oracle_mod):
    Hk, group = 2, 4
    Hq = Hk * group
    rng = np.random.default_rng(11)
    kv_lens = rng.integers(1, 200, size=5)
    w = synth.decode_workload("t", kv_lens, 16, 100, Hq, Hk, torch.bfloat16, seed=3, head_dim=D)
    c = w.cache
    args = (w.q, c.k_pool, c.v_pool, c.kv_indptr, c.kv_indices, c.last_page_len, 16, Hq, Hk,
            D, oracle_mod.BF16, w.sm_scale)
    full = oracle_mod.batch_attention(*args)
    # 3-way split at arbitrary (page-unaligned) points, including empty pieces
    cuts = [np.sort(rng.integers(0, L + 1, size=2)) for L in kv_lens]
    b0 = np.zeros(5, np.int32)
    b1 = np.array([x[0] for x in cuts], np.int32)
    b2 = np.array([x[1] for x in cuts], np.int32)
    b3 = np.asarray(kv_lens, np.int32)
    parts = [oracle_mod.batch_attention(*args, kv_begin=lo, kv_end=hi)
             for lo, hi in ((b0, b1), (b1, b2), (b2, b3))]
    o_states = np.stack([p[0].reshape(-1, D) for p in parts])
    lse_states = np.stack([p[1].reshape(-1) for p in parts])
    o, lse = oracle_mod.merge_states(o_states, lse_states)
    np.testing.assert_allclose(o, full[0].reshape(-1, D), atol=1e-12, rtol=0)
    np.testing.assert_allclose(lse, full[1].reshape(-1), atol=1e-12, rtol=0)


def test_merge_special_cases(oracle_mod):
    rng = np.random.default_rng(2)
    o1 = rng.standard_normal((3, 4, D))
    l1 = rng.standard_normal((3, 4))
    # merging with an empty state (lse = -inf) is the identity
    o, l = oracle_mod.merge_states(np.stack([o1[0], np.zeros((4, D))]),
                                   np.stack([l1[0], np.full(4, -np.inf)]))
    np.testing.assert_allclose(o, o1[0], atol=1e-15, rtol=0)
    np.testing.assert_allclose(l, l1[0], atol=1e-15, rtol=0)
    # two identical states: same o, lse + ln 2
    o, l = oracle_mod.merge_states(np.stack([o1[0], o1[0]]), np.stack([l1[0], l1[0]]))
    np.testing.assert_allclose(o, o1[0], atol=1e-14, rtol=0)
    np.testing.assert_allclose(l, l1[0] + math.log(2), atol=1e-14, rtol=0)
    # both empty: o = 0, lse = -inf, no NaN
    o, l = oracle_mod.merge_states(np.zeros((2, 4, D)), np.full((2, 4), -np.inf))
    assert np.all(o == 0) and np.all(np.isneginf(l))
    # weights from scipy's logsumexp
    o, l = oracle_mod.merge_states(o1, l1)
    ref_l = logsumexp(l1, axis=0)
    np.testing.assert_allclose(l, ref_l, atol=1e-14, rtol=0)
    ref_o = np.einsum("sr,srd->rd", np.exp(l1 - ref_l[None]), o1)
    np.testing.assert_allclose(o, ref_o, atol=1e-14, rtol=0)


def test_prefix_suffix_equals_flat(oracle_mod):
    """Composable formats: prefix (P=128, shared, one pass with qo_len = n) +
    suffix (P=16) + LSE merge == one flat P=16 layout (small instance)."""
    w = synth.shared_prefix_decode(seed=4242, prompts=3, n=4, prefix_len=256)
    pre = w.extra["prefix"]
    suf = w.cache
    Hq, Hk = w.num_qo_heads, w.num_kv_heads
    op, lp = oracle_mod.batch_attention(w.q, pre.k_pool, pre.v_pool, pre.kv_indptr,
                                        pre.kv_indices, pre.last_page_len, pre.page_size, Hq,
                                        Hk, D, oracle_mod.BF16, w.sm_scale, causal=False,
                                        qo_indptr=w.extra["prefix_qo_indptr"])
    os_, ls = oracle_mod.batch_attention(w.q, suf.k_pool, suf.v_pool, suf.kv_indptr,
                                         suf.kv_indices, suf.last_page_len, suf.page_size, Hq,
                                         Hk, D, oracle_mod.BF16, w.sm_scale)
    o, l = oracle_mod.merge_states(np.stack([op.reshape(-1, D), os_.reshape(-1, D)]),
                                   np.stack([lp.reshape(-1), ls.reshape(-1)]))
    flat = synth.flat_layout_of_composable(w)
    of, lf = oracle_mod.batch_attention(w.q, flat.k_pool, flat.v_pool, flat.kv_indptr,
                                        flat.kv_indices, flat.last_page_len, 16, Hq, Hk, D,
                                        oracle_mod.BF16, w.sm_scale)
    np.testing.assert_allclose(o, of.reshape(-1, D), atol=1e-12, rtol=0)
    np.testing.assert_allclose(l, lf.reshape(-1), atol=1e-12, rtol=0)


def test_snippet_shape_golden(oracle_mod):
    """The quick-start snippet fixes the single-decode shapes (tests/golden)."""
    import json, os
    g = json.load(open(os.path.join(os.path.dirname(__file__), "golden",
                                    "single_decode_snippet_shapes.json")))
    w = synth.single_request_decode()
    assert list(w.q.shape[1:]) == g["q"]
    assert w.cache.kv_lens[0] == g["k"][0] and w.num_kv_heads == g["k"][1]
    # the oracle returns [num_qo_heads, head_dim] per request
    o, lse = oracle_mod.batch_attention(w.q, w.cache.k_pool, w.cache.v_pool, w.cache.kv_indptr,
                                        w.cache.kv_indices, w.cache.last_page_len, 16, 32, 32,
                                        D, oracle_mod.F16, w.sm_scale)
    assert list(o.shape[1:]) == g["out"]
    assert np.all(np.isfinite(o)) and np.all(np.isfinite(lse))
