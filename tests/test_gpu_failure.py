"""A pipeline wait that is never satisfied ends with a status word, not a
hang: the bounded mbarrier wait every kernel uses gives up, records
ATTN_DEV_WAIT_TIMEOUT and returns, and the CUDA context stays usable."""

import time

import pytest
import torch

import oracle
import synth
from parity import check_o, gpu_or_skip

pytestmark = pytest.mark.gpu


def test_unsatisfied_wait_reports_timeout_and_context_survives():
    dev = gpu_or_skip()
    import causal_gqa_flashattention_attn_gb300 as attn
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    t0 = time.perf_counter()
    attn.attn_selftest_wait_timeout(status, limit_us=20000)
    torch.cuda.synchronize()
    elapsed = time.perf_counter() - t0
    assert status.item() == attn.ATTN_DEV_WAIT_TIMEOUT
    assert elapsed < 5.0
    # the context still runs kernels correctly afterwards
    shape = synth.TINY_PREFILL_FP32
    q, k, v = synth.prefill_inputs(shape, seed=1)
    o, _ = attn.attn_prefill_fwd(q.to(dev), k.to(dev), v.to(dev))
    torch.cuda.synchronize()
    o_ref, _ = oracle.prefill(q.double().numpy(), k.double().numpy(), v.double().numpy())
    check_o(o, o_ref)
