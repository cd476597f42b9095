"""LSE merge kernel against the oracle's merge (through the C ABI)."""

import numpy as np
import pytest
import torch

import oracle
import synth
from parity import check_lse, check_o, gpu_or_skip

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("n,s,d", [(1, 1, 128), (37, 5, 128), (300, 16, 128), (64, 3, 64), (9, 40, 1024), (5, 2, 4),
                                   (200, 17, 128), (70, 19, 128), (33, 32, 128), (33, 33, 128), (21, 19, 64)])
def test_merge_fp32_matches_oracle(n, s, d):
    """Rows of up to 16 and of 17-32 splits (D <= 128) take the one-round-trip
    paths; more splits, or wider rows, the batched one."""
    dev = gpu_or_skip()
    import causal_gqa_flashattention_attn_gb300 as attn
    o_part, lse_part = synth.merge_inputs(n, s, d, seed=n * 7 + s)
    o, lse = attn.attn_lse_merge(o_part.to(dev), lse_part.to(dev), o_dtype=torch.float32)
    torch.cuda.synchronize()
    o_ref, lse_ref = oracle.lse_merge(o_part.double().numpy(), lse_part.double().numpy())
    np.testing.assert_allclose(o.cpu().double().numpy(), o_ref, rtol=1e-5, atol=1e-5)
    check_lse(lse, lse_ref, fp32=True)
    # the all-empty first row
    assert np.all(o[0].cpu().numpy() == 0) and lse[0].item() == float("-inf")


def test_merge_bf16_output():
    dev = gpu_or_skip()
    import causal_gqa_flashattention_attn_gb300 as attn
    o_part, lse_part = synth.merge_inputs(128, 8, 128, seed=3)
    o, lse = attn.attn_lse_merge(o_part.to(dev), lse_part.to(dev), o_dtype=torch.bfloat16)
    torch.cuda.synchronize()
    o_ref, lse_ref = oracle.lse_merge(o_part.double().numpy(), lse_part.double().numpy())
    check_o(o, o_ref)
    check_lse(lse, lse_ref)


# the short-row kernel takes up to 16 splits with D <= 128; (2048, 16, 128) is
# the bf16 decode's partial shape, a whole wave of it; 17 splits or D = 132
# go to the general kernel
@pytest.mark.parametrize("n,s,d", [(1, 1, 128), (37, 5, 128), (300, 16, 128), (2048, 16, 128), (9, 40, 1024),
                                   (5, 2, 4), (64, 17, 128), (33, 16, 132)])
def test_merge_bwd_matches_oracle(n, s, d):
    """Gradient of the merge ("splitk_kernels.py", _splitK_reduce_varargs_backward)."""
    dev = gpu_or_skip()
    import causal_gqa_flashattention_attn_gb300 as attn
    o_part, lse_part = synth.merge_inputs(n, s, d, seed=n + 3 * s)
    g = torch.Generator().manual_seed(n * 11 + d)
    d_o = torch.randn(n, d, generator=g)
    d_lse = torch.randn(n, generator=g)
    go, gl = attn.attn_lse_merge_bwd(o_part.to(dev), lse_part.to(dev), d_o.to(dev), d_lse.to(dev))
    torch.cuda.synchronize()
    ro, rl = oracle.lse_merge_bwd(o_part.double().numpy(), lse_part.double().numpy(), d_o.double().numpy(),
                                  d_lse.double().numpy())
    np.testing.assert_allclose(go.cpu().double().numpy(), ro, rtol=1e-5, atol=1e-5)
    np.testing.assert_allclose(gl.cpu().double().numpy(), rl, rtol=1e-5, atol=1e-4)
    # the all-empty first row gets zero gradients
    assert torch.all(go[0] == 0) and torch.all(gl[0] == 0)
    # without d_lse
    go2, gl2 = attn.attn_lse_merge_bwd(o_part.to(dev), lse_part.to(dev), d_o.to(dev), None)
    torch.cuda.synchronize()
    ro2, rl2 = oracle.lse_merge_bwd(o_part.double().numpy(), lse_part.double().numpy(), d_o.double().numpy())
    np.testing.assert_allclose(gl2.cpu().double().numpy(), rl2, rtol=1e-5, atol=1e-4)
