"""Causal multi-query split-K decode ("splitk_kernels.py", NUM_QUERIES_CAUSAL)
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
    # (kv format, n_groups, Hq, Hkv, q_len, split, lens)
    ("dense", 1, 32, 8, 4, 2048, [700, 4, 2049, 3000]),     # 16 rows per CTA
    ("dense", 1, 32, 8, 16, 512, [1200, 16, 300]),          # 64 rows: four row groups
    ("dense", 1, 32, 8, 3, 256, [513, 2, 256, 257]),        # 12 rows; lengths shorter than q_len
    ("dense", 1, 8, 8, 7, 192, [600, 64]),                  # G = 1
    ("dense", 1, 32, 2, 2, 1024, [1500, 100]),              # G = 16, two row groups
    ("int4", 4, 32, 8, 4, 2048, [700, 4, 2100]),
    ("int4", 4, 32, 8, 9, 512, [900, 30]),
    ("int4", 2, 32, 4, 2, 256, [300, 77]),                  # G = 8, 16 rows
    ("int4", 8, 16, 8, 5, 1024, [1100, 9]),                 # G = 2
]


@pytest.mark.parametrize("fmt,ng,hq,hkv,nq,split,lens", CASES)
def test_multi_query_decode_matches_oracle(fmt, ng, hq, hkv, nq, split, lens):
    dev = gpu_or_skip()
    import causal_gqa_flashattention_attn_gb300 as attn
    base = synth.PAGED_DECODE_BF16 if fmt == "dense" else synth.PAGED_DECODE_INT4
    shape = replace(base, B=len(lens), Hq=hq, Hkv=hkv, n_groups=ng, split_tokens=split)
    inp = synth.decode_inputs(shape, seed=nq + len(lens), lens=lens)
    g = torch.Generator().manual_seed(100 + nq)
    q = torch.randn(len(lens), hq, nq, 128, generator=g).to(torch.bfloat16)
    t = {k: v.to(dev) for k, v in inp.items() if torch.is_tensor(v)}
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    o, lse, _ = attn.attn_decode_paged_splitk_mq(q.to(dev), t["k_cache"], t["v_cache"], t["block_table"],
                                                 t["seq_lens"], split, max(lens), n_groups=ng, dev_status=status)
    torch.cuda.synchronize()
    assert status.item() == 0
    kc, vc = (inp["k_cache"].double().numpy(), inp["v_cache"].double().numpy()) if fmt == "dense" else \
        (inp["k_cache"].numpy(), inp["v_cache"].numpy())
    o_ref, lse_ref = oracle.decode_mq(q.double().numpy(), kc, vc, inp["block_table"].numpy(), lens, 256, split,
                                      kv_format=fmt, n_groups=ng, max_kv_len=max(lens))
    check_o(o, o_ref)
    check_lse(lse, lse_ref)


def test_multi_query_with_one_query_equals_single_query_entry():
    dev = gpu_or_skip()
    import causal_gqa_flashattention_attn_gb300 as attn
    lens = [900, 31]
    shape = replace(synth.PAGED_DECODE_BF16, B=2)
    inp = synth.decode_inputs(shape, seed=5, lens=lens)
    t = {k: v.to(dev) for k, v in inp.items() if torch.is_tensor(v)}
    o1, l1, _ = attn.attn_decode_paged_splitk(t["q"], t["k_cache"], t["v_cache"], t["block_table"], t["seq_lens"],
                                              2048, 900)
    o2, l2, _ = attn.attn_decode_paged_splitk_mq(t["q"][:, :, None, :].contiguous(), t["k_cache"], t["v_cache"],
                                                 t["block_table"], t["seq_lens"], 2048, 900)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2[:, :, 0]) and torch.equal(l1, l2[:, :, 0])
