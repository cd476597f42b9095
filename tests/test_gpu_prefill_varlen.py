"""Ragged (varlen) causal GQA prefill over a paged KV cache ("gpt-o3 /
triton6fd1ef", run) against the oracle, through the C ABI."""

import numpy as np
import pytest
import torch

import oracle
import synth
from parity import check_lse, check_o, gpu_or_skip

pytestmark = pytest.mark.gpu

CASES = [
    # (Hq, Hkv, page_size, q_lens, kv_lens)
    (32, 4, 1, [300, 1, 129, 64], [700, 1, 129, 1000]),     # G = 8, the page's head layout
    (32, 4, 1, [200, 77], [200, 77]),                        # no cached prefix
    (16, 4, 16, [150, 33, 300], [400, 40, 300]),             # G = 4, page size 16, partial last pages
    (8, 8, 1, [260, 5], [300, 5]),                           # G = 1
    (32, 2, 256, [100, 500], [1000, 700]),                   # G = 16, large pages
    (32, 4, 1, [90, 10], [40, 10]),                          # q_len > kv_len: early rows see nothing
    (28, 4, 16, [300, 19, 40], [500, 19, 300]),              # G = 7: 18 positions x 7 heads per tile
    (12, 4, 1, [100, 43], [260, 43]),                        # G = 3: 42 x 3 rows
]


def _entry(attn, ws):
    """The in-kernel gather, or the entry that copies the pages into a
    contiguous workspace first (sized to exactly the listed rows)."""
    if not ws:
        return attn.attn_prefill_paged_varlen

    def run(q, k, v, qo, kvp, kvi, last, **kw):
        rows = int(kvp[-1].item()) * k.shape[1]
        return attn.attn_prefill_paged_varlen_ws(q, k, v, qo, kvp, kvi, last, max_kv_rows=max(rows, 1), **kw)
    return run


@pytest.mark.parametrize("ws", [False, True], ids=["gather", "workspace"])
@pytest.mark.parametrize("hq,hkv,ps,q_lens,kv_lens", CASES)
def test_varlen_paged_prefill_matches_oracle(hq, hkv, ps, q_lens, kv_lens, ws):
    dev = gpu_or_skip()
    import causal_gqa_flashattention_attn_gb300 as attn
    shape = synth.VarlenShape("t", len(q_lens), hq, hkv, 128, 1, 1, 0, 0, page_size=ps)
    inp = synth.varlen_inputs(shape, seed=len(q_lens) + ps, q_lens=q_lens, kv_lens=kv_lens)
    t = {k: v.to(dev) for k, v in inp.items() if torch.is_tensor(v)}
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    o, lse = _entry(attn, ws)(t["q"], t["k_cache"], t["v_cache"], t["qo_indptr"], t["kv_indptr"],
                              t["kv_indices"], t["kv_last_page_len"], dev_status=status)
    torch.cuda.synchronize()
    assert status.item() == 0
    o_ref, lse_ref = oracle.prefill_paged_varlen(inp["q"].double().numpy(), inp["k_cache"].double().numpy(),
                                                 inp["v_cache"].double().numpy(), inp["qo_indptr"].numpy(),
                                                 inp["kv_indptr"].numpy(), inp["kv_indices"].numpy(), ps,
                                                 inp["kv_last_page_len"].numpy())
    check_o(o, o_ref)
    check_lse(lse, lse_ref)


@pytest.mark.parametrize("ws", [False, True], ids=["gather", "workspace"])
def test_varlen_bench_workload_sampled(ws):
    """The benchmark's ragged batch (8 sequences, page size 1); the oracle
    checks two whole sequences."""
    dev = gpu_or_skip()
    import causal_gqa_flashattention_attn_gb300 as attn
    shape = synth.VARLEN_PAGED_PREFILL
    inp = synth.varlen_inputs(shape, seed=0)
    t = {k: v.to(dev) for k, v in inp.items() if torch.is_tensor(v)}
    o, lse = _entry(attn, ws)(t["q"], t["k_cache"], t["v_cache"], t["qo_indptr"], t["kv_indptr"],
                              t["kv_indices"], t["kv_last_page_len"])
    torch.cuda.synchronize()
    qo = inp["qo_indptr"].tolist()
    for b in (0, shape.B - 1):
        sub_qo = np.array([0, qo[b + 1] - qo[b]])
        kvp = inp["kv_indptr"].tolist()
        sub_kvp = np.array([0, kvp[b + 1] - kvp[b]])
        sub_idx = inp["kv_indices"][kvp[b]:kvp[b + 1]].numpy()
        o_ref, lse_ref = oracle.prefill_paged_varlen(inp["q"][qo[b]:qo[b + 1]].double().numpy(),
                                                     inp["k_cache"].double().numpy(),
                                                     inp["v_cache"].double().numpy(), sub_qo, sub_kvp, sub_idx, 1)
        check_o(o[qo[b]:qo[b + 1]], o_ref, what=f"O seq {b}")
        check_lse(lse[qo[b]:qo[b + 1]], lse_ref, what=f"LSE seq {b}")


def _run(attn, inp, dev, ws=False):
    t = {k: v.to(dev) for k, v in inp.items() if torch.is_tensor(v)}
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    o, lse = _entry(attn, ws)(t["q"], t["k_cache"], t["v_cache"], t["qo_indptr"], t["kv_indptr"],
                              t["kv_indices"], t["kv_last_page_len"], dev_status=status)
    torch.cuda.synchronize()
    assert status.item() == 0
    return o, lse


def _check_seq(inp, o, lse, b, ps, pools):
    qo = inp["qo_indptr"].tolist()
    kvp = inp["kv_indptr"].tolist()
    o_ref, lse_ref = oracle.prefill_paged_varlen(
        inp["q"][qo[b]:qo[b + 1]].double().numpy(), pools[0], pools[1], np.array([0, qo[b + 1] - qo[b]]),
        np.array([0, kvp[b + 1] - kvp[b]]), inp["kv_indices"][kvp[b]:kvp[b + 1]].numpy(), ps,
        inp["kv_last_page_len"][b:b + 1].numpy())
    check_o(o[qo[b]:qo[b + 1]], o_ref, what=f"O seq {b}")
    check_lse(lse[qo[b]:qo[b + 1]], lse_ref, what=f"LSE seq {b}")


@pytest.mark.parametrize("ws", [False, True], ids=["gather", "workspace"])
def test_varlen_many_short_sequences(ws):
    """300 sequences of mixed short lengths: many work items share a KV tile
    count, so the longest-first order has long runs of ties; every sequence
    is checked."""
    dev = gpu_or_skip()
    import causal_gqa_flashattention_attn_gb300 as attn
    g = torch.Generator().manual_seed(11)
    q_lens = torch.randint(1, 100, (300,), generator=g).tolist()
    kv_lens = [q + int(x) for q, x in zip(q_lens, torch.randint(0, 300, (300,), generator=g))]
    shape = synth.VarlenShape("t", len(q_lens), 16, 2, 128, 1, 1, 0, 0, page_size=16)
    inp = synth.varlen_inputs(shape, seed=5, q_lens=q_lens, kv_lens=kv_lens)
    o, lse = _run(attn, inp, dev, ws)
    pools = (inp["k_cache"].double().numpy(), inp["v_cache"].double().numpy())
    for b in range(len(q_lens)):
        _check_seq(inp, o, lse, b, 16, pools)


def test_varlen_over_the_sorted_list_capacity():
    """2048 sequences of 65 new tokens (3 query blocks each at G = 8: 6144
    pairs, more than the 4096 the sorted work list holds), so the kernel walks
    the items in sequence order; sampled sequences are checked."""
    dev = gpu_or_skip()
    import causal_gqa_flashattention_attn_gb300 as attn
    B = 2048
    q_lens = [65] * B
    kv_lens = [65 + (b * 7) % 40 for b in range(B)]
    shape = synth.VarlenShape("t", B, 8, 1, 128, 1, 1, 0, 0, page_size=1)
    inp = synth.varlen_inputs(shape, seed=6, q_lens=q_lens, kv_lens=kv_lens)
    o, lse = _run(attn, inp, dev)
    pools = (inp["k_cache"].double().numpy(), inp["v_cache"].double().numpy())
    for b in list(range(0, B, 97)) + [B - 1]:
        _check_seq(inp, o, lse, b, 1, pools)


def test_varlen_workspace_too_small_is_flagged():
    """A page list longer than the workspace's rows sets
    ATTN_DEV_SEQ_TOO_LONG (the copy is cut, nothing is written out of it)."""
    dev = gpu_or_skip()
    import causal_gqa_flashattention_attn_gb300 as attn
    shape = synth.VarlenShape("t", 2, 32, 4, 128, 1, 1, 0, 0, page_size=1)
    inp = synth.varlen_inputs(shape, seed=9, q_lens=[40, 20], kv_lens=[300, 100])
    t = {k: v.to(dev) for k, v in inp.items() if torch.is_tensor(v)}
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    attn.attn_prefill_paged_varlen_ws(t["q"], t["k_cache"], t["v_cache"], t["qo_indptr"], t["kv_indptr"],
                                      t["kv_indices"], t["kv_last_page_len"], max_kv_rows=256, dev_status=status)
    torch.cuda.synchronize()
    assert status.item() & attn.ATTN_DEV_SEQ_TOO_LONG
