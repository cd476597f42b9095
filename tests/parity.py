"""Helpers shared by the GPU parity tests: tolerances and comparisons.

Tolerances (fixed by the method's problem statement):
  * bf16 outputs O: max-abs error <= 2e-2 and mean-abs error <= 2e-3;
  * fp32 LSE: <= 1e-3 absolute (and -inf exactly where the oracle has -inf);
  * fp32-input workloads: <= 1e-4 absolute on O and LSE;
  * indexing: bit-exact.
"""

import numpy as np
import pytest
import torch

BF16_MAX, BF16_MEAN = 2e-2, 2e-3
LSE_TOL = 1e-3
FP32_TOL = 1e-4


def gpu_or_skip():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    import __graft_entry__
    __graft_entry__.build()
    import causal_gqa_flashattention_attn_gb300 as attn
    attn.lib()
    return torch.device("cuda:0")


def np64(t):
    return t.detach().float().cpu().double().numpy() if t.dtype != torch.float64 else t.cpu().numpy()


def check_o(o_gpu, o_ref, fp32=False, what="O"):
    o = np64(o_gpu)
    assert o.shape == o_ref.shape, (o.shape, o_ref.shape)
    assert np.all(np.isfinite(o)), f"{what}: non-finite values"
    err = np.abs(o - o_ref)
    if fp32:
        assert err.max() <= FP32_TOL, f"{what}: max err {err.max():.3e} > {FP32_TOL}"
    else:
        assert err.max() <= BF16_MAX, f"{what}: max err {err.max():.3e} > {BF16_MAX}"
        assert err.mean() <= BF16_MEAN, f"{what}: mean err {err.mean():.3e} > {BF16_MEAN}"
    return err.max(), err.mean()


def check_lse(lse_gpu, lse_ref, fp32=False, what="LSE"):
    lse = np64(lse_gpu)
    assert lse.shape == lse_ref.shape
    dead = np.isneginf(lse_ref)
    assert np.array_equal(np.isneginf(lse), dead), f"{what}: -inf pattern differs"
    live = ~dead
    tol = FP32_TOL if fp32 else LSE_TOL
    if live.any():
        err = np.abs(lse[live] - lse_ref[live]).max()
        assert err <= tol, f"{what}: max err {err:.3e} > {tol}"
        return err
    return 0.0
