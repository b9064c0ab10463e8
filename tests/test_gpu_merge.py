"""Public LSE merge kernel (attn_merge_states) vs the oracle's merge."""
import numpy as np
import pytest
import torch

from tests.gpu_util import LSE_ABS, O_MAX_ABS, O_MEAN_ABS

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16])
@pytest.mark.parametrize("shape", [(1, 1, 128), (64, 32, 128), (37, 8, 64), (5, 3, 8)])
def test_merge_states_parity(oracle_mod, dtype, shape):
    from paged_kv_attention_bsr_gb300 import merge_state
    n, h, d = shape
    g = torch.Generator().manual_seed(n * 131 + h)
    o_a = torch.randn(shape, generator=g).to(dtype)
    o_b = torch.randn(shape, generator=g).to(dtype)
    l_a = (torch.randn(n, h, generator=g) * 4).float()
    l_b = (torch.randn(n, h, generator=g) * 4).float()
    # special rows: one side empty, both empty, equal lse
    l_a[0, 0] = -float("inf")
    if n > 1:
        l_a[1, 0] = l_b[1, 0] = -float("inf")
    if n > 2:
        l_b[2, 0] = l_a[2, 0]
    o, lse = merge_state(o_a.cuda(), l_a.cuda(), o_b.cuda(), l_b.cuda())
    torch.cuda.synchronize()
    o_ref, lse_ref = oracle_mod.merge_states(
        np.stack([o_a.double().numpy().reshape(-1, d), o_b.double().numpy().reshape(-1, d)]),
        np.stack([l_a.double().numpy().reshape(-1), l_b.double().numpy().reshape(-1)]))
    got = o.float().cpu().numpy().reshape(-1, d)
    err = np.abs(got - o_ref)
    assert err.max() <= O_MAX_ABS and err.mean() <= O_MEAN_ABS
    gl = lse.cpu().numpy().reshape(-1).astype(np.float64)
    fin = np.isfinite(lse_ref)
    assert np.all(np.isneginf(gl[~fin]))
    assert np.abs(gl[fin] - lse_ref[fin]).max() <= LSE_ABS


def test_merge_states_in_place():
    from paged_kv_attention_bsr_gb300 import merge_state
    o_a = torch.randn(8, 4, 128, device="cuda").bfloat16()
    o_b = torch.randn(8, 4, 128, device="cuda").bfloat16()
    l_a = torch.randn(8, 4, device="cuda")
    l_b = torch.randn(8, 4, device="cuda")
    ref, ref_l = merge_state(o_a, l_a, o_b, l_b)
    out, out_l = merge_state(o_a, l_a, o_b, l_b, out=o_a)
    torch.cuda.synchronize()
    assert torch.equal(ref, out) and torch.equal(ref_l, out_l)
