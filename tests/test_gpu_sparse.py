"""Page sizes that are not a multiple of 16, down to one token per page
(vector-level sparsity). The few-row tensor-core kernel copies K / V rows
through the page table with cp.async (decode: four copy warps, a quarter of
each tile's rows each; short appends and RoPE decode: one warp); the long
append kernel gathers rows four at a time (TMA tile::gather4). Parity
against the fp64 oracle."""
import numpy as np
import pytest
import torch

from paged_kv_attention_bsr_gb300 import synth
from tests.gpu_util import assert_attn_close, oracle_dtype, poison_unused_slots
from tests.test_gpu_decode import oracle_full, run_decode

pytestmark = pytest.mark.gpu

CASES = [
    # (page_size, Hq, Hk, dtype, lens)
    (1, 16, 4, torch.bfloat16, [1, 2, 3, 4, 5, 127, 128, 129, 700]),
    (1, 64, 8, torch.bfloat16, [2000, 33, 0, 130]),
    (2, 8, 4, torch.float16, [1, 2, 3, 255, 256, 257]),
    (3, 32, 8, torch.bfloat16, [3, 4, 95, 190, 1000]),
    (5, 16, 2, torch.bfloat16, [5, 6, 641, 9]),
    (24, 16, 4, torch.float16, [23, 24, 25, 500, 1531]),
    (100, 16, 8, torch.bfloat16, [99, 100, 101, 3000]),
    # group 8 in fp16, last tiles of 1..31 rows: copy warps with no rows
    (1, 16, 2, torch.float16, [1, 31, 32, 33, 95, 97, 160, 250]),
    (7, 32, 16, torch.bfloat16, [1, 7, 8, 64, 65, 383]),
]


@pytest.mark.parametrize("case", range(len(CASES)))
@pytest.mark.parametrize("num_ctas", [1, 7, None])
def test_sparse_decode_parity(oracle_mod, case, num_ctas):
    P, Hq, Hk, dtype, lens = CASES[case]
    pool = sum(-(-L // P) for L in lens) + 13
    w = synth.decode_workload(f"sparse{case}", lens, P, pool, Hq, Hk, dtype, seed=900 + case)
    o_ref, lse_ref = oracle_full(oracle_mod, w)
    o, lse, _ = run_decode(w, num_ctas)
    assert_attn_close(o, lse, o_ref, lse_ref, f"sparse case {case} ctas {num_ctas}")


@pytest.mark.parametrize("case", [0, 3, 5])
def test_sparse_decode_stale_pool_slots_are_never_used(oracle_mod, case):
    P, Hq, Hk, dtype, lens = CASES[case]
    pool = sum(-(-L // P) for L in lens) + 13
    w = synth.decode_workload(f"sparsenan{case}", lens, P, pool, Hq, Hk, dtype, seed=950 + case)
    poison_unused_slots(w.cache)
    o_ref, lse_ref = oracle_full(oracle_mod, w)
    o, lse, _ = run_decode(w)
    assert_attn_close(o, lse, o_ref, lse_ref, f"sparse stale slots case {case}")


def test_sparse_decode_matches_the_same_cache_at_page_size_16():
    """The same logical KV at P = 1 and at P = 16 gives the same attention."""
    lens = [1, 17, 300, 1024, 2049]
    w16 = synth.decode_workload("dense16", lens, 16, sum(-(-L // 16) for L in lens) + 3,
                                32, 8, torch.bfloat16, seed=990)
    c = w16.cache
    # re-page: token t of request r -> its own one-token page (fresh order)
    rng = np.random.default_rng(991)
    total = int(sum(lens))
    order = rng.permutation(total + 5)
    k1 = torch.zeros((total + 5, 8, 1, 128), dtype=torch.bfloat16)
    v1 = torch.zeros_like(k1)
    kv_indices, kv_indptr, n = [], [0], 0
    for r, L in enumerate(lens):
        pages = c.kv_indices[c.kv_indptr[r]:c.kv_indptr[r + 1]]
        for t in range(L):
            src = int(pages[t // 16])
            k1[order[n], :, 0] = c.k_pool[src, :, t % 16]
            v1[order[n], :, 0] = c.v_pool[src, :, t % 16]
            kv_indices.append(int(order[n]))
            n += 1
        kv_indptr.append(n)
    cache1 = synth.BSRCache(1, 8, 128, k1, v1, np.array(kv_indptr, np.int32),
                            np.array(kv_indices, np.int32),
                            np.array([1 if L else 0 for L in lens], np.int32),
                            np.asarray(lens, np.int64))
    w1 = synth.Workload("sparse1", "decode", torch.bfloat16, 32, 8, 128, w16.sm_scale, w16.q,
                        cache1)
    o16, l16, _ = run_decode(w16)
    o1, l1, _ = run_decode(w1)
    d = (o16.float() - o1.float()).abs().max().item()
    assert d <= 2e-2 and (l16 - l1).abs().max().item() <= 1e-3


def test_sparse_decode_full_size(oracle_mod):
    """The full-size P = 1 batch in the benchmark's launch configuration,
    every row against the oracle (rows spread over host threads)."""
    from tests.gpu_util import oracle_decode_threaded
    w = synth.WORKLOADS["sparse_decode"]()
    o, lse, _ = run_decode(w)
    o_ref, lse_ref = oracle_decode_threaded(oracle_mod, w)
    assert_attn_close(o, lse, o_ref, lse_ref, w.name)


APPEND_CASES = [
    # (P, Hq, Hk, dtype, qo_lens, extra kv, causal)
    (1, 32, 8, torch.bfloat16, [1, 2, 4, 3], [0, 5, 200, 1000], True),
    (3, 16, 8, torch.bfloat16, [8, 5, 1], [100, 700, 2], True),
    (7, 8, 8, torch.float16, [16, 9], [300, 20], False),
]


@pytest.mark.parametrize("case", range(len(APPEND_CASES)))
@pytest.mark.parametrize("num_ctas", [1, None])
def test_sparse_short_append_parity(oracle_mod, case, num_ctas):
    from tests.test_gpu_append import oracle_full as append_oracle, run_append
    P, Hq, Hk, dtype, qo_lens, extra, causal = APPEND_CASES[case]
    kv_lens = [q + e for q, e in zip(qo_lens, extra)]
    pool = sum(-(-L // P) for L in kv_lens) + 9
    w = synth.append_workload(f"sparseapp{case}", qo_lens, kv_lens, P, pool, Hq, Hk, dtype,
                              seed=960 + case, causal=causal)
    poison_unused_slots(w.cache)
    o_ref, lse_ref = append_oracle(oracle_mod, w)
    o, lse, _ = run_append(w, num_ctas)
    assert_attn_close(o, lse, o_ref, lse_ref, f"sparse short append {case} ctas {num_ctas}")


LONG_APPEND_CASES = [
    # (P, Hq, Hk, dtype, qo_lens, extra kv, causal, layout): past 16 packed
    # rows, so the append kernel gathers rows four at a time
    (1, 32, 8, torch.bfloat16, [40, 130, 1, 257], [0, 300, 1000, 17], True, 0),
    (3, 32, 8, torch.bfloat16, [100, 33, 7], [100, 700, 2], True, 0),
    (3, 16, 4, torch.float16, [64, 200], [500, 3], False, 0),
    (5, 32, 8, torch.bfloat16, [90, 20], [77, 400], True, 1),
    (1, 16, 2, torch.bfloat16, [300], [129], True, 1),
]


@pytest.mark.parametrize("case", range(len(LONG_APPEND_CASES)))
@pytest.mark.parametrize("num_ctas", [1, 5, None])
def test_sparse_long_append_parity(oracle_mod, case, num_ctas):
    """Causal and non-causal appends past 16 packed rows at page sizes 1, 3
    and 5 (HND and NHD), stale pool slots set to NaN."""
    from tests.test_gpu_append import oracle_full as append_oracle, run_append
    P, Hq, Hk, dtype, qo_lens, extra, causal, layout = LONG_APPEND_CASES[case]
    kv_lens = [q + e for q, e in zip(qo_lens, extra)]
    pool = sum(-(-L // P) for L in kv_lens) + 9
    w = synth.append_workload(f"sparselong{case}", qo_lens, kv_lens, P, pool, Hq, Hk, dtype,
                              seed=970 + case, causal=causal)
    poison_unused_slots(w.cache)
    o_ref, lse_ref = append_oracle(oracle_mod, w)
    o, lse, _ = run_append(w, num_ctas, layout=layout)
    assert_attn_close(o, lse, o_ref, lse_ref, f"sparse long append {case} ctas {num_ctas}")


@pytest.mark.parametrize("P", [1, 5])
def test_sparse_rope_decode_parity(oracle_mod, P):
    from tests.test_gpu_rope import oracle_rope, run_rope
    lens = [1, 2, 130, 1000, 0, 77]
    pool = sum(-(-L // P) for L in lens) + 11
    w = synth.decode_workload(f"sparserope{P}", lens, P, pool, 32, 8, torch.bfloat16,
                              seed=980 + P)
    poison_unused_slots(w.cache)
    cos, sin = synth.rope_tables(max(lens))
    o_ref, lse_ref = oracle_rope(oracle_mod, w, cos, sin)
    o, lse = run_rope(w, cos, sin)
    assert_attn_close(o, lse, o_ref, lse_ref, f"sparse rope P {P}")


@pytest.mark.parametrize("case", [0, 3, 5])
def test_sparse_decode_nhd_layout(oracle_mod, case):
    """Gathered rows from an NHD pool [pages, P, Hk, 128]."""
    from paged_kv_attention_bsr_gb300 import _capi as C
    P, Hq, Hk, dtype, lens = CASES[case]
    pool = sum(-(-L // P) for L in lens) + 13
    w = synth.decode_workload(f"sparsenhd{case}", lens, P, pool, Hq, Hk, dtype, seed=930 + case)
    o_ref, lse_ref = oracle_full(oracle_mod, w)
    o, lse, _ = run_decode(w, layout=C.LAYOUT_NHD)
    assert_attn_close(o, lse, o_ref, lse_ref, f"sparse nhd case {case}")
