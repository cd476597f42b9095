"""The paged decode with the LSE merge inside the same launch
(attn_decode_paged_fused: the last split of each (sequence, KV head) to
finish merges its partials, or, in the persistent int4 and fp8 kernels'
cooperative launch, the whole grid merges after one grid barrier;
"splitk_kernels.py" _splitK_reduce) against the oracle, through the C ABI;
and its workspace contract (arrival counters and barrier words that start at
zero and are left at zero)."""

from dataclasses import replace

import numpy as np
import pytest
import torch

import oracle
import synth
from parity import check_lse, check_o, gpu_or_skip

pytestmark = pytest.mark.gpu

CASES = [
    # (format, n_groups, Hq, Hkv, q_len, split, lens)
    ("dense", 1, 32, 8, 1, 2048, [700, 1, 333, 2048, 2049, 5000, 0]),
    ("dense", 1, 32, 2, 1, 512, [1500, 999]),           # G = 16
    ("dense", 1, 8, 8, 1, 256, [513, 7]),               # G = 1
    ("dense", 1, 32, 8, 4, 2048, [700, 4, 2049, 3000]),  # multi-query, 16 rows per CTA
    ("dense", 1, 32, 8, 16, 512, [1200, 16, 300]),      # multi-query, four row groups
    ("int4", 4, 32, 8, 1, 2048, [700, 1, 2100, 64, 0]),  # the persistent kernel (8 KV heads a CTA)
    ("int4", 4, 32, 8, 1, 896, [16384, 5000, 31]),      # many splits per sequence
    ("int4", 4, 32, 8, 1, 864, [16384, 2000, 865, 33]),  # a 32-token split step
    ("int4", 4, 32, 8, 2, 512, [900, 30]),              # multi-query on the persistent kernel
    ("int4", 2, 32, 8, 1, 256, [300, 0, 129]),          # the general int4 kernel
    ("int4", 4, 32, 4, 1, 2048, [900, 2]),              # G = 8, Hkv 4: the general kernel
    ("int4", 4, 32, 8, 9, 512, [900, 30]),              # 36 rows: the general kernel, row groups
    ("fp8", 1, 32, 8, 1, 2048, [700, 1, 2049, 3000]),
    ("fp8", 1, 32, 8, 4, 2048, [700, 4, 2100]),
    # the persistent kernels' cooperative merge: about 7 units per CTA (64-token
    # splits), and two groups of 8 KV heads with an empty sequence
    ("int4", 4, 32, 8, 1, 64, [16384, 16384, 16000, 16383]),
    ("fp8", 1, 64, 16, 1, 256, [3000, 700, 5, 0]),
]


def _inputs(fmt, ng, hq, hkv, nq, split, lens, seed):
    base = {"dense": synth.PAGED_DECODE_BF16, "int4": synth.PAGED_DECODE_INT4, "fp8": synth.PAGED_DECODE_FP8}[fmt]
    shape = replace(base, B=len(lens), Hq=hq, Hkv=hkv, n_groups=ng, split_tokens=split)
    inp = synth.decode_inputs(shape, seed=seed, lens=lens)
    q = inp["q"]
    if nq > 1:
        g = torch.Generator().manual_seed(200 + seed)
        q = torch.randn(len(lens), hq, nq, 128, generator=g).to(torch.bfloat16)
    return shape, inp, q


def _fused(attn, dev, shape, inp, q, split, max_len, workspace=None, status=None):
    t = {k: v.to(dev) for k, v in inp.items() if torch.is_tensor(v)}
    extra = {}
    if shape.kv_format == "fp8":
        extra = dict(k_scale_shift=t["k_scale_shift"], v_scale_shift=t["v_scale_shift"])
    return attn.attn_decode_paged_fused(q.to(dev), t["k_cache"], t["v_cache"], t["block_table"], t["seq_lens"], split,
                                        max_len, n_groups=shape.n_groups, workspace=workspace, dev_status=status,
                                        **extra)


def _oracle(shape, inp, q, split, max_len):
    fmt = shape.kv_format
    kc, vc = (inp["k_cache"].double().numpy(), inp["v_cache"].double().numpy()) if fmt == "dense" else \
        (inp["k_cache"].numpy(), inp["v_cache"].numpy())
    extra = {}
    if fmt == "fp8":
        extra = dict(k_scale_shift=inp["k_scale_shift"].numpy(), v_scale_shift=inp["v_scale_shift"].numpy())
    q4 = q.double().numpy() if q.dim() == 4 else q.double().numpy()[:, :, None, :]
    o, lse = oracle.decode_mq(q4, kc, vc, inp["block_table"].numpy(), inp["lens"], shape.page_size, split,
                              kv_format=fmt, n_groups=shape.n_groups, max_kv_len=max_len, **extra)
    if q.dim() == 3:
        o, lse = o[:, :, 0], lse[:, :, 0]
    return o, lse


@pytest.mark.parametrize("fmt,ng,hq,hkv,nq,split,lens", CASES)
def test_fused_decode_matches_oracle_and_leaves_counters_zero(fmt, ng, hq, hkv, nq, split, lens):
    dev = gpu_or_skip()
    import causal_gqa_flashattention_attn_gb300 as attn
    shape, inp, q = _inputs(fmt, ng, hq, hkv, nq, split, lens, seed=len(lens) + nq + ng)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    max_len = max(max(lens), 1)
    o, lse, ws = _fused(attn, dev, shape, inp, q, split, max_len, status=status)
    torch.cuda.synchronize()
    assert status.item() == 0, status.item()
    o_ref, lse_ref = _oracle(shape, inp, q, split, max_len)
    check_o(o, o_ref)
    check_lse(lse, lse_ref)
    partial = attn.attn_decode_workspace_bytes(len(lens), hq * nq, max_len, split, 128)
    assert int(ws[partial:].count_nonzero()) == 0          # every counter back at zero
    # a second call on the same workspace gives the same bits
    o2, lse2, _ = _fused(attn, dev, shape, inp, q, split, max_len, workspace=ws, status=status)
    torch.cuda.synchronize()
    assert status.item() == 0
    assert torch.equal(o, o2) and torch.equal(lse, lse2)


@pytest.mark.parametrize("fmt,ng", [("int4", 4), ("fp8", 1)])
def test_cooperative_and_last_arrival_merges_agree(fmt, ng):
    """The persistent kernels' fused modes: with cooperative launches (the grid
    merges after a grid barrier) and without (attn_decode_cooperative(False):
    the last split to arrive merges), both against the oracle, with the same
    bits, and both leave the workspace's counters and barrier words zero."""
    dev = gpu_or_skip()
    import causal_gqa_flashattention_attn_gb300 as attn
    lens = [3000, 700, 64, 0, 1]
    shape, inp, q = _inputs(fmt, ng, 32, 8, 1, 256, lens, seed=61)
    partial = attn.attn_decode_workspace_bytes(len(lens), 32, 3000, 256, 128)
    assert attn.attn_decode_cooperative() is True           # the default
    outs = []
    try:
        for coop in (True, False):
            attn.attn_decode_cooperative(coop)
            status = torch.zeros(1, dtype=torch.int32, device=dev)
            o, lse, ws = _fused(attn, dev, shape, inp, q, 256, 3000, status=status)
            torch.cuda.synchronize()
            assert status.item() == 0, (coop, status.item())
            assert int(ws[partial:].count_nonzero()) == 0, coop
            outs.append((o, lse))
    finally:
        attn.attn_decode_cooperative(True)
    o_ref, lse_ref = _oracle(shape, inp, q, 256, 3000)
    for o, lse in outs:
        check_o(o, o_ref)
        check_lse(lse, lse_ref)
    assert torch.equal(outs[0][0], outs[1][0]) and torch.equal(outs[0][1], outs[1][1])


@pytest.mark.parametrize("fmt", ["dense", "int4"])
def test_fused_decode_equals_decode_then_merge(fmt):
    """The merge inside the launch adds the splits in the same order and with
    the same weights as attn_lse_merge: identical bits."""
    dev = gpu_or_skip()
    import causal_gqa_flashattention_attn_gb300 as attn
    lens = [5000, 700, 64, 1]
    ng = 4 if fmt == "int4" else 1
    shape, inp, q = _inputs(fmt, ng, 32, 8, 1, 512, lens, seed=31)
    o, lse, _ = _fused(attn, dev, shape, inp, q, 512, 5000)
    t = {k: v.to(dev) for k, v in inp.items() if torch.is_tensor(v)}
    o2, lse2, _ = attn.attn_decode_paged_splitk(t["q"], t["k_cache"], t["v_cache"], t["block_table"], t["seq_lens"],
                                                512, 5000, n_groups=ng)
    torch.cuda.synchronize()
    assert torch.equal(o, o2) and torch.equal(lse, lse2)


def test_fused_workspace_not_zeroed_is_flagged():
    """Counters that do not start at zero (every byte 0x7F) are reported as
    ATTN_DEV_WORKSPACE_STATE; zeroed again, the same workspace gives correct
    results."""
    dev = gpu_or_skip()
    import causal_gqa_flashattention_attn_gb300 as attn
    lens = [900, 64]
    shape, inp, q = _inputs("int4", 4, 32, 8, 1, 256, lens, seed=41)
    ws = torch.full((attn.attn_decode_fused_workspace_bytes(2, 32, 8, 900, 256, 128),), 0x7F, dtype=torch.uint8,
                    device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    _fused(attn, dev, shape, inp, q, 256, 900, workspace=ws, status=status)
    torch.cuda.synchronize()
    assert status.item() & attn.ATTN_DEV_WORKSPACE_STATE
    ws.zero_()
    status.zero_()
    o, lse, _ = _fused(attn, dev, shape, inp, q, 256, 900, workspace=ws, status=status)
    torch.cuda.synchronize()
    assert status.item() == 0
    o_ref, lse_ref = _oracle(shape, inp, q, 256, 900)
    check_o(o, o_ref)
    check_lse(lse, lse_ref)


def test_fused_decode_replays_from_a_cuda_graph():
    """Nothing re-zeroes the counters inside a graph: every replay must leave
    them at zero and give the eager call's bits."""
    dev = gpu_or_skip()
    import causal_gqa_flashattention_attn_gb300 as attn
    lens = [3000, 900, 17]
    shapes = [_inputs(f, ng, 32, 8, 1, 512, lens, seed=50 + i)
              for i, (f, ng) in enumerate([("dense", 1), ("int4", 4), ("fp8", 1)])]
    ts = [{k: v.to(dev) for k, v in inp.items() if torch.is_tensor(v)} for _, inp, _ in shapes]
    wss = [torch.zeros(attn.attn_decode_fused_workspace_bytes(3, 32, 8, 3000, 512, 128), dtype=torch.uint8,
                       device=dev) for _ in shapes]
    outs = [(torch.empty(3, 32, 128, dtype=torch.bfloat16, device=dev), torch.empty(3, 32, device=dev))
            for _ in shapes]
    status = torch.zeros(1, dtype=torch.int32, device=dev)

    def calls(stream):
        for (shape, _, q), t, ws, (o, lse) in zip(shapes, ts, wss, outs):
            extra = {}
            if shape.kv_format == "fp8":
                extra = dict(k_scale_shift=t["k_scale_shift"], v_scale_shift=t["v_scale_shift"])
            attn.attn_decode_paged_fused(t["q"], t["k_cache"], t["v_cache"], t["block_table"], t["seq_lens"], 512,
                                         3000, n_groups=shape.n_groups, workspace=ws, o=o, lse=lse,
                                         dev_status=status, stream=stream, **extra)

    side = torch.cuda.Stream(dev)
    with torch.cuda.stream(side):
        calls(side)
    side.synchronize()
    eager = [(o.clone(), lse.clone()) for o, lse in outs]
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=side):
        calls(side)
    for o, lse in outs:
        o.zero_()
        lse.zero_()
    for _ in range(3):
        graph.replay()
    torch.cuda.synchronize()
    assert status.item() == 0
    partial = attn.attn_decode_workspace_bytes(3, 32, 3000, 512, 128)
    for ws in wss:
        assert int(ws[partial:].count_nonzero()) == 0
    for (o, lse), (eo, el) in zip(outs, eager):
        assert torch.equal(o, eo) and torch.equal(lse, el)
