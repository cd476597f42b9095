"""The C-ABI calls allocate and synchronise nothing, so a sequence of them
can be captured into a CUDA graph and replayed: the replay must give the
same results as the eager calls."""

import pytest
import torch
from dataclasses import replace

import synth
from parity import gpu_or_skip

pytestmark = pytest.mark.gpu


def test_prefill_decode_and_ragged_prefill_replay_from_a_cuda_graph():
    dev = gpu_or_skip()
    import causal_gqa_flashattention_attn_gb300 as attn
    # dense prefill
    pshape = replace(synth.LLAMA_GQA_PREFILL, B=1, Hq=8, Hkv=2, q_len=300, kv_len=900)
    q, k, v = (t.to(dev) for t in synth.prefill_inputs(pshape, seed=1))
    po, plse = torch.empty_like(q), torch.empty(1, 8, 300, dtype=torch.float32, device=dev)
    # the same through the split schedule: its counters must come back to zero
    # after every replay, as nothing re-zeroes them inside the graph
    assert attn.attn_prefill_plan(torch.bfloat16, 1, 8, 2, 300, 900, 128)[0] == 1
    pws = torch.zeros(attn.attn_prefill_workspace_bytes(torch.bfloat16, 1, 8, 2, 300, 900, 128), dtype=torch.uint8,
                      device=dev)
    so, slse = torch.empty_like(q), torch.empty(1, 8, 300, dtype=torch.float32, device=dev)
    # paged decode (int4) with its merge
    dshape = replace(synth.PAGED_DECODE_INT4, B=3, len_lo=1, len_hi=900)
    dinp = synth.decode_inputs(dshape, seed=2, lens=[900, 64, 5])
    dt = {k_: v_.to(dev) for k_, v_ in dinp.items() if torch.is_tensor(v_)}
    ws = torch.empty(attn.attn_decode_workspace_bytes(3, dshape.Hq, 900, 256, 128), dtype=torch.uint8, device=dev)
    do_ = torch.empty(3, dshape.Hq, 128, dtype=torch.bfloat16, device=dev)
    dl = torch.empty(3, dshape.Hq, dtype=torch.float32, device=dev)
    # ragged prefill through the page copy
    vs = synth.VarlenShape("g", 2, 8, 2, 128, 1, 1, 0, 0, page_size=1)
    vinp = synth.varlen_inputs(vs, seed=3, q_lens=[100, 37], kv_lens=[300, 37])
    vt = {k_: v_.to(dev) for k_, v_ in vinp.items() if torch.is_tensor(v_)}
    rows = vt["k_cache"].shape[0]
    vws = torch.empty(attn.attn_prefill_varlen_workspace_bytes(rows, 2, 128), dtype=torch.uint8, device=dev)
    vo = torch.empty_like(vt["q"])
    vl = torch.empty(vt["q"].shape[0], 8, dtype=torch.float32, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)

    def calls(stream):
        attn.attn_prefill_fwd(q, k, v, o=po, lse=plse, dev_status=status, stream=stream)
        attn.attn_prefill_fwd_ws(q, k, v, workspace=pws, o=so, lse=slse, dev_status=status, stream=stream)
        attn.attn_decode_paged_splitk(dt["q"], dt["k_cache"], dt["v_cache"], dt["block_table"], dt["seq_lens"], 256,
                                      900, n_groups=dshape.n_groups, workspace=ws, o=do_, lse=dl,
                                      dev_status=status, stream=stream)
        attn.attn_prefill_paged_varlen_ws(vt["q"], vt["k_cache"], vt["v_cache"], vt["qo_indptr"], vt["kv_indptr"],
                                          vt["kv_indices"], vt["kv_last_page_len"], max_kv_rows=rows, workspace=vws,
                                          o=vo, lse=vl, dev_status=status, stream=stream)

    side = torch.cuda.Stream(dev)
    with torch.cuda.stream(side):
        calls(side)   # eager, also warms up the library (device queries, kernel attributes)
    side.synchronize()
    outs = (po, plse, so, slse, do_, dl, vo, vl)
    eager = [t.clone() for t in outs]
    for t in outs:
        t.zero_()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=side):
        calls(side)
    for t in outs:
        t.zero_()
    for _ in range(2):
        graph.replay()
    torch.cuda.synchronize()
    assert status.item() == 0
    assert int(pws[:16 * 2 * 5].count_nonzero()) == 0   # counters of the 10 work items (Hkv 2 x 5 blocks)
    for got, ref in zip(outs, eager):
        assert torch.equal(got, ref)
