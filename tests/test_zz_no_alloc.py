"""attn_decode_paged_splitk_static, the decode entry point that allocates
nothing, checked against attn_decode_paged_splitk through the C ABI.

It exists for callers that cannot allocate device memory while they run
(plugin or callback interfaces that receive only input and output buffers,
serving loops that forbid cudaMalloc after start-up); its split partials live
in a fixed array inside the library instead of a caller-provided workspace.
This file is collected last on purpose, so a run that stops at the first
failure has already run every other test.
"""

from dataclasses import replace

import numpy as np
import pytest
import torch

import synth
from parity import check_lse, check_o, gpu_or_skip

pytestmark = pytest.mark.gpu


def _inputs(dev, shape, seed, lens):
    inp = synth.decode_inputs(shape, seed=seed, lens=lens)
    return {k: v.to(dev) for k, v in inp.items() if torch.is_tensor(v)}


def _both(attn, t, shape, max_len):
    status = torch.zeros(1, dtype=torch.int32, device=t["q"].device)
    o_ref, lse_ref, _ = attn.attn_decode_paged_splitk(t["q"], t["k_cache"], t["v_cache"], t["block_table"],
                                                      t["seq_lens"], shape.split_tokens, max_len,
                                                      n_groups=shape.n_groups)
    o, lse = attn.attn_decode_paged_splitk_static(t["q"], t["k_cache"], t["v_cache"], t["block_table"],
                                                  t["seq_lens"], shape.split_tokens, max_len,
                                                  n_groups=shape.n_groups, dev_status=status)
    torch.cuda.synchronize()
    assert status.item() == 0
    return o, lse, o_ref, lse_ref


def _compare(o, lse, o_ref, lse_ref):
    check_o(o, o_ref.float().cpu().double().numpy(), what="static O")
    check_lse(lse, lse_ref.cpu().double().numpy(), what="static LSE")


def test_static_entry_matches_workspace_entry_on_two_calls_in_a_row():
    dev = gpu_or_skip()
    import causal_gqa_flashattention_attn_gb300 as attn
    # first call: a long bf16 batch (many splits); second call: a short int4
    # batch, so stale partials of the first call would show up if read
    s1 = replace(synth.PAGED_DECODE_BF16, B=6)
    lens1 = [5000, 1, 2048, 2049, 333, 7000]
    t1 = _inputs(dev, s1, 3, lens1)
    o, lse, o_ref, lse_ref = _both(attn, t1, s1, max(lens1))
    _compare(o, lse, o_ref, lse_ref)

    s2 = replace(synth.PAGED_DECODE_INT4, B=3)
    lens2 = [700, 64, 1]
    t2 = _inputs(dev, s2, 4, lens2)
    o, lse, o_ref, lse_ref = _both(attn, t2, s2, max(lens2))
    _compare(o, lse, o_ref, lse_ref)


def test_static_entry_rejects_sizes_beyond_its_maximum():
    gpu_or_skip()
    import causal_gqa_flashattention_attn_gb300 as attn
    # B=64, Hq=32, 2^17 tokens at split 2048 -> 64 splits -> 64 MiB of partials
    need = attn.attn_decode_workspace_bytes(64, 32, 1 << 17, 2048, 128)
    assert need > attn.ATTN_DECODE_STATIC_SCRATCH_BYTES
    fake = torch.zeros(16, dtype=torch.int32, device="cuda")
    L = attn.lib()
    p = fake.data_ptr()
    st = L.attn_decode_paged_splitk_static(p, p, p, p, 512, p, attn.ATTN_BF16, 1, 64, 32, 8, 128, 1, 256, 2048,
                                           1 << 17, 0.1, p, None, None, None)
    assert st == -3, attn.attn_status_string(st)


def test_static_entry_allocates_nothing_on_a_warm_call():
    """With its outputs given, a call after the first on the device leaves
    both torch's allocator and the device's free memory unchanged."""
    dev = gpu_or_skip()
    import causal_gqa_flashattention_attn_gb300 as attn
    shape = replace(synth.PAGED_DECODE_BF16, B=4)
    lens = [3000, 17, 2048, 900]
    t = _inputs(dev, shape, 5, lens)
    o = torch.empty(shape.B, shape.Hq, shape.D, dtype=torch.bfloat16, device=dev)
    lse = torch.empty(shape.B, shape.Hq, dtype=torch.float32, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)

    def call():
        attn.attn_decode_paged_splitk_static(t["q"], t["k_cache"], t["v_cache"], t["block_table"], t["seq_lens"],
                                             shape.split_tokens, max(lens), o=o, lse=lse, dev_status=status)
        torch.cuda.synchronize()

    call()                      # first call: address lookup, kernels loaded
    first_o, first_lse = o.clone(), lse.clone()
    torch.cuda.synchronize()
    alloc0 = torch.cuda.memory_allocated(dev)
    free0 = torch.cuda.mem_get_info(dev)[0]
    call()
    assert torch.cuda.memory_allocated(dev) == alloc0
    assert torch.cuda.mem_get_info(dev)[0] == free0
    assert status.item() == 0
    assert torch.equal(o, first_o) and torch.equal(lse, first_lse)
