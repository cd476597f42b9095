"""Causal GQA prefill (tensor-core and CUDA-core paths) against the oracle,
through the C ABI."""

from dataclasses import replace

import numpy as np
import pytest
import torch

import oracle
import synth
from parity import check_lse, check_o, gpu_or_skip

pytestmark = pytest.mark.gpu


def _run(shape, seed=0, entry="plain"):
    """One prefill through attn_prefill_fwd ("plain": whole work items) or
    attn_prefill_fwd_ws ("ws": with split-schedule scratch, zeroed)."""
    dev = gpu_or_skip()
    import causal_gqa_flashattention_attn_gb300 as attn
    q, k, v = synth.prefill_inputs(shape, seed=seed)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    if entry == "ws":
        o, lse = attn.attn_prefill_fwd_ws(q.to(dev), k.to(dev), v.to(dev), dev_status=status)
    else:
        o, lse = attn.attn_prefill_fwd(q.to(dev), k.to(dev), v.to(dev), dev_status=status)
    torch.cuda.synchronize()
    assert status.item() == 0, status.item()
    return (q, k, v), o, lse


def _np(t):
    return t.double().numpy()


def test_tiny_fp32_workload_matches_oracle_to_1e4():
    """The fp32 workload: B=1, Hq=4, Hkv=2, q_len=kv_len=128, D=64."""
    (q, k, v), o, lse = _run(synth.TINY_PREFILL_FP32)
    o_ref, lse_ref = oracle.prefill(_np(q), _np(k), _np(v))
    check_o(o, o_ref, fp32=True)
    check_lse(lse, lse_ref, fp32=True)


@pytest.mark.parametrize("hq,hkv,lq,lk", [(8, 4, 100, 100), (6, 3, 70, 200), (2, 2, 300, 40)])
def test_fp32_other_shapes(hq, hkv, lq, lk):
    shape = replace(synth.TINY_PREFILL_FP32, B=2, Hq=hq, Hkv=hkv, q_len=lq, kv_len=lk)
    (q, k, v), o, lse = _run(shape, seed=lq)
    o_ref, lse_ref = oracle.prefill(_np(q), _np(k), _np(v))
    check_o(o, o_ref, fp32=True)
    check_lse(lse, lse_ref, fp32=True)


BF16_CASES = [
    # (B, Hq, Hkv, q_len, kv_len): several tiles and a ragged tail each
    (2, 8, 1, 200, 328),    # G = 8, delta = 128
    (1, 8, 2, 300, 300),    # G = 4, square
    (1, 4, 4, 257, 400),    # G = 1 (plain multi-head)
    (2, 4, 2, 130, 130),    # G = 2
    (1, 16, 1, 100, 612),   # G = 16
    (1, 32, 1, 40, 1000),   # G = 32
    (1, 8, 1, 1, 333),      # a single query row
    (1, 8, 2, 260, 120),    # q_len > kv_len: the first rows see no key
    (3, 8, 8, 64, 64),      # G = 1, short
    (1, 28, 4, 300, 500),   # G = 7: 18 positions x 7 heads = 126 of the 128 tile rows
    (2, 12, 4, 200, 200),   # G = 3: 42 x 3 = 126 rows
    (1, 20, 4, 150, 350),   # G = 5: 25 x 5 = 125 rows
    (1, 24, 4, 140, 100),   # G = 6, q_len > kv_len
    (1, 100, 1, 5, 300),    # G = 100: one position per tile, 28 rows unused
]


@pytest.mark.parametrize("entry", ["plain", "ws"])
@pytest.mark.parametrize("bsz,hq,hkv,lq,lk", BF16_CASES)
def test_bf16_tensor_core_path_matches_oracle(bsz, hq, hkv, lq, lk, entry):
    """Both entries; with its workspace, most of these small cases (too few
    work items to fill the GPU) take the split schedule."""
    shape = replace(synth.LLAMA_GQA_PREFILL, B=bsz, Hq=hq, Hkv=hkv, q_len=lq, kv_len=lk)
    (q, k, v), o, lse = _run(shape, seed=lq + lk, entry=entry)
    o_ref, lse_ref = oracle.prefill(_np(q), _np(k), _np(v))
    check_o(o, o_ref)
    check_lse(lse, lse_ref)


def test_bf16_sharp_softmax_k_scaled():
    """K x 2 (as in the batched workload) sharpens the softmax and exercises the
    lazy rescaling of the running max."""
    shape = replace(synth.BATCHED_SQUARE_PREFILL, B=1, Hq=8, Hkv=2, q_len=520, kv_len=520)
    (q, k, v), o, lse = _run(shape, seed=4)
    o_ref, lse_ref = oracle.prefill(_np(q), _np(k), _np(v))
    check_o(o, o_ref)
    check_lse(lse, lse_ref)


D64_CASES = [
    # (B, Hq, Hkv, q_len, kv_len) at D = 64: the tiles' second halves stay zero
    (1, 4, 2, 150, 200),    # G = 2
    (2, 32, 4, 300, 500),   # G = 8, several blocks and a ragged tail
    (1, 8, 8, 129, 129),    # G = 1
    (1, 28, 4, 100, 60),    # G = 7, q_len > kv_len
    (1, 16, 1, 40, 700),    # G = 16, long KV
]


@pytest.mark.parametrize("entry", ["plain", "ws"])
@pytest.mark.parametrize("bsz,hq,hkv,lq,lk", D64_CASES)
def test_bf16_head_dim_64_tensor_core_path(bsz, hq, hkv, lq, lk, entry):
    shape = replace(synth.LLAMA_GQA_PREFILL, B=bsz, Hq=hq, Hkv=hkv, q_len=lq, kv_len=lk, D=64)
    (q, k, v), o, lse = _run(shape, seed=lq + 3, entry=entry)
    o_ref, lse_ref = oracle.prefill(_np(q), _np(k), _np(v))
    check_o(o, o_ref)
    check_lse(lse, lse_ref)


def test_bf16_group_over_128_cuda_core_path():
    """More than 128 query heads per KV head do not fit a tile's rows: the
    CUDA-core path."""
    shape = replace(synth.LLAMA_GQA_PREFILL, B=1, Hq=256, Hkv=1, q_len=20, kv_len=50)
    (q, k, v), o, lse = _run(shape, seed=2)
    o_ref, lse_ref = oracle.prefill(_np(q), _np(k), _np(v))
    check_o(o, o_ref)
    check_lse(lse, lse_ref)


def _sampled_rows(shape, n_heads, rows_per_head, seed, entry="ws"):
    """Full-size workload in the benchmark's launch configuration (the
    workspace entry); the oracle computes sampled rows (first, last, around
    multiples of the tile sizes and random ones) of sampled heads one by one."""
    (q, k, v), o, lse = _run(shape, seed=0, entry=entry)
    rng = np.random.default_rng(seed)
    o_np = o.float().cpu().double().numpy()
    lse_np = lse.cpu().double().numpy()
    assert np.isfinite(o_np).all() and np.isfinite(lse_np).all()
    fixed = [0, 1, 15, 16, 31, 32, 127, 128, 255, shape.q_len - 1]
    for _ in range(n_heads):
        b = int(rng.integers(shape.B))
        h = int(rng.integers(shape.Hq))
        rows = sorted(set(fixed + rng.integers(0, shape.q_len, rows_per_head).tolist()))
        o_ref, lse_ref = oracle.prefill_rows(_np(q[b:b + 1]), _np(k[b:b + 1]), _np(v[b:b + 1]), 0, h, rows)
        check_o(torch.from_numpy(o_np[b, h, rows]), o_ref, what=f"O[b={b},h={h}]")
        check_lse(torch.from_numpy(lse_np[b, h, rows]), lse_ref, what=f"LSE[b={b},h={h}]")


def test_schedule_choice():
    """The split schedule is taken where whole items leave most SMs idle (a
    512-token chunk against a 64K cache: 16 items of 512 KV tiles); the
    benchmark workloads (256 and 4096 items) keep whole items, since a cut
    costs about as much as the tail it removes."""
    gpu_or_skip()
    import causal_gqa_flashattention_attn_gb300 as attn
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    long_kv = replace(synth.LLAMA_GQA_PREFILL, Hq=8, Hkv=1, q_len=512, kv_len=65536)
    for shape, want in ((synth.LLAMA_GQA_PREFILL, 0), (synth.BATCHED_SQUARE_PREFILL, 0), (long_kv, 1)):
        sched, grid = attn.attn_prefill_plan(torch.bfloat16, shape.B, shape.Hq, shape.Hkv, shape.q_len,
                                             shape.kv_len, shape.D)
        assert sched == want and grid == sms


@pytest.mark.parametrize("entry", ["ws", "plain"])
def test_full_size_llama_gqa_prefill_sampled(entry):
    _sampled_rows(synth.LLAMA_GQA_PREFILL, n_heads=6, rows_per_head=24, seed=1, entry=entry)


def test_full_size_batched_square_prefill_sampled():
    _sampled_rows(synth.BATCHED_SQUARE_PREFILL, n_heads=4, rows_per_head=16, seed=2)


@pytest.mark.parametrize("bsz,hq,hkv,lq,lk", [
    (2, 16, 4, 33, 4000),     # 8 items of 32 KV tiles over 152 CTAs: up to 19 pieces per item
    (1, 8, 2, 900, 500),      # q_len > kv_len: the first 6 query blocks see no key at all
    (1, 8, 2, 160, 1100),     # G = 4
    (1, 8, 1, 640, 600),      # G = 8
    (1, 4, 4, 600, 500),      # G = 1
    (1, 32, 1, 40, 1000),     # G = 32
])
def test_split_schedule_matches_oracle(bsz, hq, hkv, lq, lk):
    gpu_or_skip()
    import causal_gqa_flashattention_attn_gb300 as attn
    assert attn.attn_prefill_plan(torch.bfloat16, bsz, hq, hkv, lq, lk, 128)[0] == 1
    shape = replace(synth.LLAMA_GQA_PREFILL, B=bsz, Hq=hq, Hkv=hkv, q_len=lq, kv_len=lk)
    (q, k, v), o, lse = _run(shape, seed=lq, entry="ws")
    o_ref, lse_ref = oracle.prefill(_np(q), _np(k), _np(v))
    check_o(o, o_ref)
    check_lse(lse, lse_ref)


def test_split_workspace_reused_and_left_zero():
    """Consecutive calls share one workspace: each leaves its counters zero,
    and the merge adds the pieces in a fixed order, so the results are
    bit-identical from call to call."""
    dev = gpu_or_skip()
    import causal_gqa_flashattention_attn_gb300 as attn
    shape = replace(synth.LLAMA_GQA_PREFILL, B=1, Hq=32, Hkv=4, q_len=512, kv_len=4096)
    q, k, v = (t.to(dev) for t in synth.prefill_inputs(shape, seed=8))
    assert attn.attn_prefill_plan(torch.bfloat16, 1, 32, 4, 512, 4096, 128)[0] == 1
    ws = torch.zeros(attn.attn_prefill_workspace_bytes(torch.bfloat16, 1, 32, 4, 512, 4096, 128),
                     dtype=torch.uint8, device=dev)
    n_items = 4 * ((512 + 31) // 32)            # G = 8: 16 positions per tile, 32 per item
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    first = None
    for _ in range(3):
        o, lse = attn.attn_prefill_fwd_ws(q, k, v, workspace=ws, dev_status=status)
        torch.cuda.synchronize()
        assert status.item() == 0
        assert int(ws[:n_items * 16].count_nonzero()) == 0
        if first is None:
            first = (o.clone(), lse.clone())
        else:
            assert torch.equal(o, first[0]) and torch.equal(lse, first[1])
    o_ref, lse_ref = oracle.prefill(_np(q.cpu()), _np(k.cpu()), _np(v.cpu()))
    check_o(o, o_ref)
    check_lse(lse, lse_ref)


def test_long_kv_prefill_sampled():
    """512 new queries against a 64K-token cache (G = 8): 512 KV tiles per
    work item; the oracle checks sampled rows of sampled heads."""
    shape = replace(synth.LLAMA_GQA_PREFILL, B=1, Hq=8, Hkv=1, q_len=512, kv_len=65536)
    _sampled_rows(shape, n_heads=3, rows_per_head=8, seed=3)


def test_host_buffer_entry_matches_device_entry():
    """attn_prefill_fwd_host (host tensors in and out, copies enqueued on the
    stream) gives exactly the O and LSE of the device entry with a workspace
    (the same schedule)."""
    dev = gpu_or_skip()
    import causal_gqa_flashattention_attn_gb300 as attn
    shape = replace(synth.LLAMA_GQA_PREFILL, B=2, Hq=8, Hkv=2, q_len=300, kv_len=700)
    q, k, v = synth.prefill_inputs(shape, seed=4)
    o_d, lse_d = attn.attn_prefill_fwd_ws(q.to(dev), k.to(dev), v.to(dev))
    hq, hk, hv = (t.pin_memory() for t in (q, k, v))
    ho = torch.empty(q.shape, dtype=q.dtype).pin_memory()
    hl = torch.empty(shape.B, shape.Hq, shape.q_len, dtype=torch.float32).pin_memory()
    stream = torch.cuda.current_stream()
    attn.attn_prefill_fwd_host(hq, hk, hv, ho, hl, stream=stream)
    stream.synchronize()
    assert torch.equal(ho, o_d.cpu())
    assert torch.equal(hl, lse_d.cpu())


def test_split_workspace_not_zeroed_is_flagged():
    """A workspace whose counters do not start at zero (here every byte 0x7F)
    is reported as ATTN_DEV_WORKSPACE_STATE; zeroed again, it gives correct
    results.  Every wait in the split epilogue is bounded, and with these
    counters they end at once."""
    dev = gpu_or_skip()
    import causal_gqa_flashattention_attn_gb300 as attn
    shape = replace(synth.LLAMA_GQA_PREFILL, B=1, Hq=8, Hkv=2, q_len=160, kv_len=1100)
    q, k, v = (t.to(dev) for t in synth.prefill_inputs(shape, seed=12))
    assert attn.attn_prefill_plan(torch.bfloat16, 1, 8, 2, 160, 1100, 128)[0] == 1
    ws = torch.full((attn.attn_prefill_workspace_bytes(torch.bfloat16, 1, 8, 2, 160, 1100, 128),), 0x7F,
                    dtype=torch.uint8, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    attn.attn_prefill_fwd_ws(q, k, v, workspace=ws, dev_status=status)
    torch.cuda.synchronize()
    assert status.item() & attn.ATTN_DEV_WORKSPACE_STATE
    ws.zero_()
    status.zero_()
    o, lse = attn.attn_prefill_fwd_ws(q, k, v, workspace=ws, dev_status=status)
    torch.cuda.synchronize()
    assert status.item() == 0
    o_ref, lse_ref = oracle.prefill(_np(q.cpu()), _np(k.cpu()), _np(v.cpu()))
    check_o(o, o_ref)
    check_lse(lse, lse_ref)
