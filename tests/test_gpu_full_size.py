"""Every output of the four full-size workloads against the oracle, through the
C ABI, in the launch configuration the benchmark times:

* the Llama-style prefill (B1 Hq32 Hkv4 q2048 kv4096 D128 bf16) and the batched
  square prefill (B8 Hq32 Hkv8 q=kv=4096, K x2) through attn_prefill_fwd_ws
  with a zeroed workspace;
* the bf16 paged decode (B64, lengths U[512, 32768], split 2048) and the int4
  paged decode (B16, 16384 tokens, N_GROUPS 4, the split attn_decode_split_tokens
  picks) through attn_decode_paged_splitk writing partials only, then
  attn_lse_merge; the int4 one also through attn_decode_paged_fused (the merge
  inside the launch);
* the fp8 decode on the int4 workload's shape, the same way.

Each compares O element by element (maximum and mean absolute error over the
whole output) and LSE (absolute error, -inf pattern) at the stated
tolerances: bf16 O max 2e-2 / mean 2e-3, LSE 1e-3.  The prefill oracle runs
per (batch, KV head) in a spawn process pool (oracle_pool); the decode oracle
runs in this process, one sequence after another.
"""

from dataclasses import replace

import numpy as np
import pytest
import torch

import oracle
import oracle_pool
import synth
from parity import BF16_MAX, BF16_MEAN, LSE_TOL, gpu_or_skip

pytestmark = pytest.mark.gpu


def _assert_within(chk, what):
    assert chk.o_max <= BF16_MAX, f"{what}: O max err {chk.o_max:.3e} > {BF16_MAX}"
    assert chk.o_mean <= BF16_MEAN, f"{what}: O mean err {chk.o_mean:.3e} > {BF16_MEAN}"
    assert chk.lse_max <= LSE_TOL, f"{what}: LSE max err {chk.lse_max:.3e} > {LSE_TOL}"


def _prefill_whole(shape):
    dev = gpu_or_skip()
    import causal_gqa_flashattention_attn_gb300 as attn
    q, k, v = synth.prefill_inputs(shape, seed=0)
    ws = torch.zeros(attn.attn_prefill_workspace_bytes(q.dtype, shape.B, shape.Hq, shape.Hkv, shape.q_len,
                                                       shape.kv_len, shape.D), dtype=torch.uint8, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    o, lse = attn.attn_prefill_fwd_ws(q.to(dev), k.to(dev), v.to(dev), workspace=ws, dev_status=status)
    torch.cuda.synchronize()
    assert status.item() == 0, status.item()
    o_np = o.float().cpu().numpy()
    lse_np = lse.cpu().numpy()
    del o, lse
    g = shape.Hq // shape.Hkv
    chk = oracle_pool.WholeOutputCheck()
    seen = set()
    for b, kvh, o_ref, lse_ref in oracle_pool.prefill_by_group(q.float().numpy(), k.float().numpy(),
                                                               v.float().numpy()):
        heads = slice(kvh * g, (kvh + 1) * g)
        chk.add(o_np[b:b + 1, heads], o_ref, lse_np[b:b + 1, heads], lse_ref)
        seen.add((b, kvh))
    assert len(seen) == shape.B * shape.Hkv
    assert chk.rows == shape.B * shape.Hq * shape.q_len
    _assert_within(chk, shape.name)
    return chk


def test_llama_gqa_prefill_every_output():
    _prefill_whole(synth.LLAMA_GQA_PREFILL)


def test_batched_square_prefill_every_output():
    _prefill_whole(synth.BATCHED_SQUARE_PREFILL)


def _decode_whole(shape, fused=False):
    """Partials-only decode then the merge, as the benchmark's hot path launches
    them (fused: attn_decode_paged_fused, the merge inside the launch); the
    oracle decodes every sequence (all heads, all splits, merged)."""
    dev = gpu_or_skip()
    import causal_gqa_flashattention_attn_gb300 as attn
    if shape.kv_format in ("int4", "fp8"):
        split = attn.attn_decode_split_tokens(shape.kv_format, shape.B, shape.Hq, shape.Hkv, shape.len_hi,
                                              n_groups=shape.n_groups, D=shape.D)
        assert split > 0 and split % (32 if shape.kv_format in ("int4", "fp8") else 64) == 0
        shape = replace(shape, split_tokens=split)
    inp = synth.decode_inputs(shape, seed=0)
    lens = inp["lens"]
    t = {k: x.to(dev) for k, x in inp.items() if torch.is_tensor(x)}
    max_len = shape.len_hi
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    extra = {}
    if shape.kv_format == "fp8":
        extra = dict(k_scale_shift=t["k_scale_shift"], v_scale_shift=t["v_scale_shift"])
    if fused:
        ws = torch.zeros(attn.attn_decode_fused_workspace_bytes(shape.B, shape.Hq, shape.Hkv, max_len,
                                                                shape.split_tokens, shape.D),
                         dtype=torch.uint8, device=dev)
        o, lse, _ = attn.attn_decode_paged_fused(t["q"], t["k_cache"], t["v_cache"], t["block_table"],
                                                 t["seq_lens"], shape.split_tokens, max_len, n_groups=shape.n_groups,
                                                 workspace=ws, dev_status=status, **extra)
    else:
        ws = torch.empty(attn.attn_decode_workspace_bytes(shape.B, shape.Hq, max_len, shape.split_tokens, shape.D),
                         dtype=torch.uint8, device=dev)
        if shape.kv_format == "fp8":
            attn.attn_decode_paged_splitk_fp8(t["q"], t["k_cache"], t["v_cache"], t["k_scale_shift"],
                                              t["v_scale_shift"], t["block_table"], t["seq_lens"],
                                              shape.split_tokens, max_len, workspace=ws, dev_status=status,
                                              write_output=False)
        else:
            attn.attn_decode_paged_splitk(t["q"], t["k_cache"], t["v_cache"], t["block_table"], t["seq_lens"],
                                          shape.split_tokens, max_len, n_groups=shape.n_groups, workspace=ws,
                                          dev_status=status, write_output=False)
        o_part, lse_part = attn.decode_partials_view(ws, shape.B, shape.Hq, max_len, shape.split_tokens, shape.D)
        o = torch.empty(shape.B * shape.Hq, shape.D, dtype=torch.bfloat16, device=dev)
        lse = torch.empty(shape.B * shape.Hq, dtype=torch.float32, device=dev)
        attn.attn_lse_merge(o_part.reshape(shape.B * shape.Hq, -1, shape.D),
                            lse_part.reshape(shape.B * shape.Hq, -1), o=o, lse=lse)
    torch.cuda.synchronize()
    assert status.item() == 0, status.item()
    o_np = o.float().cpu().numpy().reshape(shape.B, shape.Hq, shape.D)
    lse_np = lse.cpu().numpy().reshape(shape.B, shape.Hq)
    del t, ws
    if shape.kv_format == "dense":
        kc, vc = inp["k_cache"].float().numpy(), inp["v_cache"].float().numpy()
    else:
        kc, vc = inp["k_cache"].numpy(), inp["v_cache"].numpy()
    extra = {}
    if shape.kv_format == "fp8":
        extra = dict(k_scale_shift=inp["k_scale_shift"].numpy(), v_scale_shift=inp["v_scale_shift"].numpy())
    qn = inp["q"].double().numpy()
    table = inp["block_table"].numpy()
    chk = oracle_pool.WholeOutputCheck()
    for b in range(shape.B):
        o_ref, lse_ref = oracle.decode(qn, kc, vc, table, lens, shape.page_size, shape.split_tokens,
                                       kv_format=shape.kv_format, n_groups=shape.n_groups, max_kv_len=max_len,
                                       batches=[b], **extra)
        chk.add(o_np[b], o_ref[b], lse_np[b], lse_ref[b])
    assert chk.rows == shape.B * shape.Hq
    _assert_within(chk, shape.name)
    return chk


def test_paged_decode_bf16_every_output():
    _decode_whole(synth.PAGED_DECODE_BF16)


def test_paged_decode_int4_every_output():
    _decode_whole(synth.PAGED_DECODE_INT4)


def test_paged_decode_int4_fused_every_output():
    _decode_whole(synth.PAGED_DECODE_INT4, fused=True)


def test_paged_decode_fp8_every_output():
    _decode_whole(synth.PAGED_DECODE_FP8)
