"""fp8 (e4m3) row-wise paged decode ("splitk_kernels.py", FP8_QUANTIZED)
against the oracle, through the C ABI."""

from dataclasses import replace

import numpy as np
import pytest
import torch

import oracle
import synth
from parity import check_lse, check_o, gpu_or_skip

pytestmark = pytest.mark.gpu

CASES = [
    # (Hq, Hkv, q_len, page, split, lens)
    (32, 8, 1, 256, 2048, [700, 1, 2049, 3000]),
    (32, 8, 1, 64, 128, [0, 65, 64, 63, 1000]),
    (8, 8, 1, 256, 256, [513, 7]),        # G = 1
    (32, 4, 1, 256, 512, [1100, 3]),      # G = 8
    (32, 4, 1, 256, 1024, [900, 40]),     # Hkv = 4 (coefficient box at offset 0 only)
    (32, 8, 4, 256, 2048, [700, 4, 2100]),   # multi-query, 16 rows
    (32, 8, 9, 256, 512, [900, 30]),         # multi-query, 36 rows in 3 groups
    (16, 8, 1, 128, 256, [600, 129]),        # G = 2, page 128
    (64, 4, 1, 256, 1024, [1500, 99]),       # G = 16
    # the persistent kernel (Hkv a multiple of 8, at most 8 rows): 32-token
    # split steps, two queries of 4 heads (8 rows), two groups of 8 KV heads
    (32, 8, 1, 64, 96, [0, 65, 200, 31, 97]),
    (32, 8, 2, 256, 512, [700, 3, 2]),
    (64, 16, 1, 256, 512, [900, 40]),
]


@pytest.mark.parametrize("hq,hkv,nq,ps,split,lens", CASES)
def test_fp8_decode_matches_oracle(hq, hkv, nq, ps, split, lens):
    dev = gpu_or_skip()
    import causal_gqa_flashattention_attn_gb300 as attn
    shape = replace(synth.PAGED_DECODE_FP8, B=len(lens), Hq=hq, Hkv=hkv, page_size=ps, split_tokens=split)
    inp = synth.decode_inputs(shape, seed=len(lens) + nq, lens=lens)
    t = {k: v.to(dev) for k, v in inp.items() if torch.is_tensor(v)}
    if nq == 1:
        q = inp["q"]
    else:
        g = torch.Generator().manual_seed(7 + nq)
        q = torch.randn(len(lens), hq, nq, 128, generator=g).to(torch.bfloat16)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    o, lse, _ = attn.attn_decode_paged_splitk_fp8(q.to(dev), t["k_cache"], t["v_cache"], t["k_scale_shift"],
                                                  t["v_scale_shift"], t["block_table"], t["seq_lens"], split,
                                                  max(lens), dev_status=status)
    torch.cuda.synchronize()
    assert status.item() == 0
    q4 = q.double().numpy() if nq > 1 else q.double().numpy()[:, :, None, :]
    o_ref, lse_ref = oracle.decode_mq(q4, inp["k_cache"].numpy(), inp["v_cache"].numpy(), inp["block_table"].numpy(),
                                      lens, ps, split, kv_format="fp8", max_kv_len=max(lens),
                                      k_scale_shift=inp["k_scale_shift"].numpy(),
                                      v_scale_shift=inp["v_scale_shift"].numpy())
    if nq == 1:
        o_ref, lse_ref = o_ref[:, :, 0], lse_ref[:, :, 0]
    check_o(o, o_ref)
    check_lse(lse, lse_ref)


def test_fp8_full_size_sampled():
    """The int4 workload's shape (B16, 16384 tokens) with an fp8 cache; the
    oracle checks three sequences."""
    dev = gpu_or_skip()
    import causal_gqa_flashattention_attn_gb300 as attn
    shape = synth.PAGED_DECODE_FP8
    # the split the benchmark takes: the one that fills the GPU
    split = attn.attn_decode_split_tokens("fp8", shape.B, shape.Hq, shape.Hkv, shape.len_hi)
    assert split > 0
    shape = replace(shape, split_tokens=split)
    inp = synth.decode_inputs(shape, seed=0)
    t = {k: v.to(dev) for k, v in inp.items() if torch.is_tensor(v)}
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    o, lse, _ = attn.attn_decode_paged_splitk_fp8(t["q"], t["k_cache"], t["v_cache"], t["k_scale_shift"],
                                                  t["v_scale_shift"], t["block_table"], t["seq_lens"],
                                                  shape.split_tokens, shape.len_hi, dev_status=status)
    torch.cuda.synchronize()
    assert status.item() == 0
    picks = [0, 7, 15]
    o_ref, lse_ref = oracle.decode(inp["q"].double().numpy(), inp["k_cache"].numpy(), inp["v_cache"].numpy(),
                                   inp["block_table"].numpy(), inp["lens"], shape.page_size, shape.split_tokens,
                                   kv_format="fp8", max_kv_len=shape.len_hi, batches=picks,
                                   k_scale_shift=inp["k_scale_shift"].numpy(),
                                   v_scale_shift=inp["v_scale_shift"].numpy())
    check_o(o[picks], o_ref[picks])
    check_lse(lse[picks], lse_ref[picks])


def test_fp8_split_partials_match_oracle():
    """With no output pointer the workspace holds the per-split partials."""
    dev = gpu_or_skip()
    import causal_gqa_flashattention_attn_gb300 as attn
    lens = [1000, 64, 3]
    split = 256
    shape = replace(synth.PAGED_DECODE_FP8, B=3, split_tokens=split)
    inp = synth.decode_inputs(shape, seed=15, lens=lens)
    t = {k: v.to(dev) for k, v in inp.items() if torch.is_tensor(v)}
    o, lse, ws = attn.attn_decode_paged_splitk_fp8(t["q"], t["k_cache"], t["v_cache"], t["k_scale_shift"],
                                                   t["v_scale_shift"], t["block_table"], t["seq_lens"], split, 1300,
                                                   write_output=False)
    torch.cuda.synchronize()
    assert o is None and lse is None
    o_part, lse_part = attn.decode_partials_view(ws, 3, shape.Hq, 1300, split, 128)
    op_ref, lp_ref = oracle.decode_split_partials(inp["q"].double().numpy(), inp["k_cache"].numpy(),
                                                  inp["v_cache"].numpy(), inp["block_table"].numpy(), lens,
                                                  shape.page_size, split, kv_format="fp8", max_kv_len=1300,
                                                  k_scale_shift=inp["k_scale_shift"].numpy(),
                                                  v_scale_shift=inp["v_scale_shift"].numpy())
    check_o(o_part, op_ref, what="O_s")
    check_lse(lse_part, lp_ref, what="LSE_s")


def test_fp8_bad_page_is_flagged_and_left_out():
    """A block-table entry outside the pool sets ATTN_DEV_PAGE_OUT_OF_RANGE and
    its page's tokens are left out: the result is the oracle's decode of the
    sequence with that page removed from its page list."""
    dev = gpu_or_skip()
    import causal_gqa_flashattention_attn_gb300 as attn
    lens = [600, 300]
    shape = replace(synth.PAGED_DECODE_FP8, B=2)
    inp = synth.decode_inputs(shape, seed=3, lens=lens)
    t = {k: v.to(dev) for k, v in inp.items() if torch.is_tensor(v)}
    bad = t["block_table"].clone()
    bad[0, 1] = -7
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    o, lse, _ = attn.attn_decode_paged_splitk_fp8(t["q"], t["k_cache"], t["v_cache"], t["k_scale_shift"],
                                                  t["v_scale_shift"], bad, t["seq_lens"], 2048, 600,
                                                  dev_status=status)
    torch.cuda.synchronize()
    assert status.item() & attn.ATTN_DEV_PAGE_OUT_OF_RANGE
    table = inp["block_table"].numpy().copy()
    table[0, 1:-1] = table[0, 2:]
    table[0, -1] = -1
    o_ref, lse_ref = oracle.decode(inp["q"].double().numpy(), inp["k_cache"].numpy(), inp["v_cache"].numpy(), table,
                                   [600 - 256, 300], 256, 2048, kv_format="fp8", max_kv_len=600,
                                   k_scale_shift=inp["k_scale_shift"].numpy(),
                                   v_scale_shift=inp["v_scale_shift"].numpy())
    check_o(o, o_ref)
    check_lse(lse, lse_ref)
