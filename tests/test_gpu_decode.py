"""Paged split-K decode (bf16 and int4 caches) against the oracle, through the C ABI."""

from dataclasses import replace

import numpy as np
import pytest
import torch

import oracle
import synth
from parity import check_lse, check_o, gpu_or_skip

pytestmark = pytest.mark.gpu


def _run(shape, lens, split, seed=0, max_kv_len=None, write_output=True):
    dev = gpu_or_skip()
    import causal_gqa_flashattention_attn_gb300 as attn
    inp = synth.decode_inputs(shape, seed=seed, lens=lens)
    t = {k: v.to(dev) for k, v in inp.items() if torch.is_tensor(v)}
    max_kv_len = max(lens) if max_kv_len is None else max_kv_len
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    o, lse, ws = attn.attn_decode_paged_splitk(t["q"], t["k_cache"], t["v_cache"], t["block_table"], t["seq_lens"],
                                               split, max_kv_len, n_groups=shape.n_groups, dev_status=status,
                                               write_output=write_output)
    torch.cuda.synchronize()
    assert status.item() == 0
    return inp, o, lse, ws


def _oracle_inputs(shape, inp):
    if shape.kv_format == "dense":
        return inp["k_cache"].double().numpy(), inp["v_cache"].double().numpy()
    return inp["k_cache"].numpy(), inp["v_cache"].numpy()


def _oracle(shape, inp, split, max_kv_len, batches=None):
    kc, vc = _oracle_inputs(shape, inp)
    return oracle.decode(inp["q"].double().numpy(), kc, vc, inp["block_table"].numpy(), inp["lens"],
                         shape.page_size, split, kv_format=shape.kv_format, n_groups=shape.n_groups,
                         max_kv_len=max_kv_len, batches=batches)


BF16_CASES = [
    # (Hq, Hkv, page_size, split, lens)
    (32, 8, 256, 2048, [700, 1, 333, 2048, 2049, 5000]),
    (32, 8, 64, 128, [0, 65, 64, 63, 1000]),
    (8, 8, 256, 256, [513, 7]),          # G = 1
    (16, 8, 128, 192, [400, 191, 192]),  # G = 2, split not a power of two
    (32, 4, 256, 512, [1100, 3]),        # G = 8
    (32, 2, 256, 1024, [1500, 999]),     # G = 16
]


@pytest.mark.parametrize("hq,hkv,ps,split,lens", BF16_CASES)
def test_decode_bf16_matches_oracle(hq, hkv, ps, split, lens):
    shape = replace(synth.PAGED_DECODE_BF16, B=len(lens), Hq=hq, Hkv=hkv, page_size=ps, split_tokens=split)
    inp, o, lse, _ = _run(shape, lens, split, seed=len(lens) + hq)
    o_ref, lse_ref = _oracle(shape, inp, split, max(lens))
    check_o(o, o_ref)
    check_lse(lse, lse_ref)
    for b, n in enumerate(lens):
        if n == 0:
            assert torch.all(o[b] == 0) and torch.all(lse[b] == float("-inf"))


INT4_CASES = [
    (32, 8, 4, 256, 2048, [700, 1, 2100, 64]),
    (32, 8, 1, 256, 512, [600, 65]),
    (32, 8, 2, 64, 256, [300, 0, 129]),
    (32, 8, 8, 256, 1024, [1500, 17]),
    (32, 4, 4, 256, 2048, [900, 2]),   # G = 8
    (32, 2, 4, 256, 2048, [900, 33]),  # G = 16
    (8, 8, 4, 256, 2048, [333]),       # G = 1
]


@pytest.mark.parametrize("hq,hkv,ng,ps,split,lens", INT4_CASES)
def test_decode_int4_matches_oracle(hq, hkv, ng, ps, split, lens):
    shape = replace(synth.PAGED_DECODE_INT4, B=len(lens), Hq=hq, Hkv=hkv, n_groups=ng, page_size=ps,
                    split_tokens=split)
    inp, o, lse, _ = _run(shape, lens, split, seed=ng + len(lens))
    o_ref, lse_ref = _oracle(shape, inp, split, max(lens))
    check_o(o, o_ref)
    check_lse(lse, lse_ref)


@pytest.mark.parametrize("fmt", ["dense", "int4"])
def test_split_partials_match_oracle(fmt):
    """With no output pointer the workspace holds the per-split partials
    (O_s divided by its own l, natural LSE_s; O_s = 0 / LSE_s = -inf when empty)."""
    import causal_gqa_flashattention_attn_gb300 as attn
    base = synth.PAGED_DECODE_BF16 if fmt == "dense" else synth.PAGED_DECODE_INT4
    lens = [1000, 64, 3]
    split = 256
    shape = replace(base, B=3, split_tokens=split)
    inp, o, lse, ws = _run(shape, lens, split, seed=5, max_kv_len=1300, write_output=False)
    assert o is None and lse is None
    o_part, lse_part = attn.decode_partials_view(ws, 3, shape.Hq, 1300, split, 128)
    kc, vc = _oracle_inputs(shape, inp)
    op_ref, lp_ref = oracle.decode_split_partials(inp["q"].double().numpy(), kc, vc, inp["block_table"].numpy(),
                                                  lens, shape.page_size, split, kv_format=fmt,
                                                  n_groups=shape.n_groups, max_kv_len=1300)
    assert o_part.shape == op_ref.shape
    check_o(o_part, op_ref, what="O_s")
    check_lse(lse_part, lp_ref, what="LSE_s")


def test_block_table_indexing_is_exact():
    """q = 0 makes every weight equal, so each split's O_s is the plain mean of
    the V rows it gathered.  V rows hold small integers that encode their
    physical (page, slot, head), so the fp32 partial means are exact and any
    wrong row would move them by at least 1/split_tokens."""
    dev = gpu_or_skip()
    import causal_gqa_flashattention_attn_gb300 as attn
    lens = [1999, 256, 1, 777]
    split = 512
    shape = replace(synth.PAGED_DECODE_BF16, B=4, split_tokens=split)
    inp = synth.decode_inputs(shape, seed=9, lens=lens)
    n_pages = inp["n_pages"]
    page = torch.arange(n_pages).view(-1, 1, 1, 1)
    slot = torch.arange(256).view(1, -1, 1, 1)
    head = torch.arange(8).view(1, 1, -1, 1)
    dim = torch.arange(128).view(1, 1, 1, -1)
    v = ((page * 7 + slot * 3 + head * 5 + dim) % 16).to(torch.bfloat16)     # exact small integers
    q = torch.zeros_like(inp["q"])
    t = {k: x.to(dev) for k, x in inp.items() if torch.is_tensor(x)}
    o, lse, ws = attn.attn_decode_paged_splitk(q.to(dev), t["k_cache"], v.to(dev), t["block_table"],
                                               t["seq_lens"], split, max(lens), write_output=False)
    torch.cuda.synchronize()
    o_part, lse_part = attn.decode_partials_view(ws, 4, 32, max(lens), split, 128)
    op_ref, lp_ref = oracle.decode_split_partials(q.double().numpy(), inp["k_cache"].double().numpy(),
                                                  v.double().numpy(), inp["block_table"].numpy(), lens, 256, split,
                                                  max_kv_len=max(lens))
    got = o_part.cpu().double().numpy()
    # means of at most 512 integers in 0..15 with fp32 accumulation: exact to ~1e-6
    assert np.abs(got - op_ref).max() < 1e-5
    live = np.isfinite(lp_ref)
    # LSE of all-zero scores is log(count): checks the length bookkeeping exactly
    np.testing.assert_allclose(lse_part.cpu().double().numpy()[live], lp_ref[live], rtol=0, atol=1e-5)
    assert np.array_equal(np.isneginf(lse_part.cpu().numpy()), ~live)


@pytest.mark.parametrize("fmt,len0", [("dense", 600), ("int4", 600), ("int4", 1024)])
def test_device_status_flags_bad_page_and_length(fmt, len0):
    """A block-table entry outside the pool is reported in the device status
    word and its page's tokens are left out of the split, so the result is the
    decode of the sequence without that page (finite, checked against the
    oracle on the table with the page removed); a length past max_kv_len is
    reported too."""
    dev = gpu_or_skip()
    import causal_gqa_flashattention_attn_gb300 as attn
    lens = [len0, 300]    # 1024: the int4 kernel's split is whole stages (its pipelined loop)
    base = synth.PAGED_DECODE_BF16 if fmt == "dense" else synth.PAGED_DECODE_INT4
    shape = replace(base, B=2)
    inp = synth.decode_inputs(shape, seed=2, lens=lens)
    t = {k: x.to(dev) for k, x in inp.items() if torch.is_tensor(x)}
    bad = t["block_table"].clone()
    bad[0, 1] = inp["n_pages"] + 5
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    o, lse, _ = attn.attn_decode_paged_splitk(t["q"], t["k_cache"], t["v_cache"], bad, t["seq_lens"], 2048, len0,
                                              n_groups=shape.n_groups, dev_status=status)
    torch.cuda.synchronize()
    assert status.item() & attn.ATTN_DEV_PAGE_OUT_OF_RANGE
    assert torch.isfinite(o.float()).all() and torch.isfinite(lse).all()
    # the same sequences with the bad page taken out of the first one's page list
    table = inp["block_table"].numpy().copy()
    table[0, 1:-1] = table[0, 2:]
    table[0, -1] = -1
    kc, vc = _oracle_inputs(shape, inp)
    o_ref, lse_ref = oracle.decode(inp["q"].double().numpy(), kc, vc, table, [len0 - 256, 300], 256, 2048,
                                   kv_format=fmt, n_groups=shape.n_groups, max_kv_len=len0)
    check_o(o, o_ref)
    check_lse(lse, lse_ref)
    status.zero_()
    attn.attn_decode_paged_splitk(t["q"], t["k_cache"], t["v_cache"], t["block_table"], t["seq_lens"], 2048,
                                  len0 - 200, n_groups=shape.n_groups, dev_status=status)
    torch.cuda.synchronize()
    assert status.item() & attn.ATTN_DEV_SEQ_TOO_LONG


def _full_size(shape, sample):
    """The full workload in the benchmark's launch configuration (for int4 the
    split from attn_decode_split_tokens, as the benchmark takes it); the
    oracle checks a sample of sequences (every head of each)."""
    dev = gpu_or_skip()
    import causal_gqa_flashattention_attn_gb300 as attn
    if shape.kv_format == "int4":
        split = attn.attn_decode_split_tokens("int4", shape.B, shape.Hq, shape.Hkv, shape.len_hi,
                                              n_groups=shape.n_groups)
        assert split > 0 and split % 32 == 0
        shape = replace(shape, split_tokens=split)
    inp = synth.decode_inputs(shape, seed=0)
    lens = inp["lens"]
    t = {k: x.to(dev) for k, x in inp.items() if torch.is_tensor(x)}
    max_len = shape.len_hi
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    o, lse, _ = attn.attn_decode_paged_splitk(t["q"], t["k_cache"], t["v_cache"], t["block_table"], t["seq_lens"],
                                              shape.split_tokens, max_len, n_groups=shape.n_groups,
                                              dev_status=status)
    torch.cuda.synchronize()
    assert status.item() == 0
    assert torch.isfinite(o.float()).all() and torch.isfinite(lse).all()
    picks = sorted(set(sample(lens)))
    o_ref, lse_ref = _oracle(shape, inp, shape.split_tokens, max_len, batches=picks)
    check_o(o[picks], o_ref[picks])
    check_lse(lse[picks], lse_ref[picks])


def test_full_size_paged_decode_bf16_sampled():
    _full_size(synth.PAGED_DECODE_BF16,
               lambda lens: [int(np.argmax(lens)), int(np.argmin(lens)), 0, len(lens) - 1, 17])


def test_full_size_paged_decode_int4_sampled():
    _full_size(synth.PAGED_DECODE_INT4, lambda lens: [0, 5, 15])


def test_split_tokens_fills_the_gpu():
    """attn_decode_split_tokens on the int4 and fp8 workloads (16 sequences x
    8 KV heads, 16384 tokens): a multiple of 64 (32 for the persistent int4
    and fp8 kernels) whose CTA count is not the 2.25 waves of 2048-token
    splits, and never more pieces than tiles."""
    gpu_or_skip()
    import causal_gqa_flashattention_attn_gb300 as attn
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    for fmt in ("int4", "fp8", "bf16"):
        split = attn.attn_decode_split_tokens(fmt, 16, 32, 8, 16384, n_groups=4)
        assert split > 0 and split % (32 if fmt in ("int4", "fp8") else 64) == 0 and split <= 16384
        ctas = 16 * 8 * -(-16384 // split)
        assert ctas >= sms
    assert attn.attn_decode_split_tokens("int4", 16, 32, 8, 16384, n_groups=3) == 0
    assert attn.attn_decode_split_tokens("bf16", 16, 32, 8, 16384, q_len=17) == 0


@pytest.mark.parametrize("fmt", ["dense", "int4"])
def test_long_context_decode(fmt):
    """A 128K-token sequence (64 splits of 2048 tokens, all merged) beside a
    short one: the largest split count the tests reach."""
    base = synth.PAGED_DECODE_BF16 if fmt == "dense" else synth.PAGED_DECODE_INT4
    shape = replace(base, B=2, Hq=4, Hkv=1)
    lens = [131072, 300]
    inp, o, lse, _ = _run(shape, lens, 2048, seed=21)
    o_ref, lse_ref = _oracle(shape, inp, 2048, max(lens))
    check_o(o, o_ref)
    check_lse(lse, lse_ref)
