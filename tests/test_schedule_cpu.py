"""Host-side schedule choices, for a described device (no GPU needed):
the prefill's whole-item / split schedule and the decode's split size."""

import math

import pytest
import torch


@pytest.fixture(scope="module")
def attn():
    import causal_gqa_flashattention_attn_gb300 as a
    a.lib()
    return a


BF16 = torch.bfloat16


def test_prefill_schedule_of_the_benchmark_workloads(attn):
    """On 152 SMs: the Llama-style and batched workloads keep whole items
    (256 and 4096 of them); a 512-token chunk against a 64K cache (16 items of
    512 KV tiles) is split; so is a small batch with fewer KV tile steps than
    SMs, on as many CTAs as steps."""
    assert attn.attn_prefill_plan_sms(BF16, 1, 32, 4, 2048, 4096, 128, 152) == (0, 152)
    assert attn.attn_prefill_plan_sms(BF16, 8, 32, 8, 4096, 4096, 128, 152) == (0, 152)
    assert attn.attn_prefill_plan_sms(BF16, 1, 8, 1, 512, 65536, 128, 152) == (1, 152)
    # 2 KV heads x 3 query blocks of 8, 9 and 9 KV tiles: 52 steps
    assert attn.attn_prefill_plan_sms(BF16, 1, 8, 2, 160, 1100, 128, 152) == (1, 52)


@pytest.mark.parametrize("sms", [1, 7, 152])
@pytest.mark.parametrize("b,hq,hkv,lq,lk", [
    (1, 32, 4, 2048, 4096), (8, 32, 8, 4096, 4096), (1, 8, 1, 512, 65536), (1, 8, 2, 160, 1100),
    (2, 16, 4, 33, 4000), (1, 8, 2, 900, 500), (3, 8, 8, 64, 64), (1, 128, 1, 777, 1500), (1, 4, 4, 1, 1),
    (1, 28, 4, 2048, 4096), (2, 24, 8, 300, 300), (1, 100, 1, 90, 700),   # groups of 7, 3, 100
])
def test_prefill_schedule_bounds(attn, sms, b, hq, hkv, lq, lk):
    """Whatever the choice, the grid is at least one CTA and at most one per
    SM, and no more than there are whole items (whole-item schedule)."""
    sched, grid = attn.attn_prefill_plan_sms(BF16, b, hq, hkv, lq, lk, 128, sms)
    assert sched in (0, 1)
    assert 1 <= grid <= sms
    g = hq // hkv
    items = b * hkv * math.ceil(lq / (2 * (128 // g)))
    if sched == 0:
        assert grid == min(items, sms)


def test_prefill_schedule_refusals(attn):
    assert attn.attn_prefill_plan_sms(BF16, 1, 32, 4, 2048, 4096, 128, 0) == (-1, 0)      # no SMs
    assert attn.attn_prefill_plan_sms(BF16, 1, 32, 5, 2048, 4096, 128, 152) == (-1, 0)    # Hq % Hkv
    assert attn.attn_prefill_plan_sms(BF16, 0, 32, 4, 2048, 4096, 128, 152) == (-1, 0)
    assert attn.attn_prefill_plan_sms(torch.float32, 1, 4, 2, 128, 128, 64, 152) == (0, 0)  # CUDA-core path
    assert attn.attn_prefill_plan_sms(BF16, 1, 256, 1, 128, 128, 128, 152) == (0, 0)        # G = 256: CUDA cores
    assert attn.attn_prefill_plan_sms(BF16, 1, 4, 2, 128, 128, 64, 152) == (0, 2)           # D = 64: tensor cores, 2 items
    # a group of 3 heads takes the tensor cores: P = 42 positions per tile, 2 blocks of 84
    kind, grid = attn.attn_prefill_plan_sms(BF16, 1, 6, 2, 128, 128, 128, 152)
    assert kind in (0, 1) and grid > 0


def _waves(units, n, slots):
    w = units * n / slots
    return w, w / math.ceil(w)


@pytest.mark.parametrize("sms,occ", [(152, 3), (152, 2), (132, 2), (8, 1)])
@pytest.mark.parametrize("b,hq,hkv,qlen,length", [
    (16, 32, 8, 1, 16384), (64, 32, 8, 1, 32768), (1, 32, 8, 1, 1000), (3, 16, 2, 4, 70000),
    (128, 32, 8, 1, 512), (7, 64, 4, 1, 4097), (16, 8, 8, 16, 2048),
])
def test_decode_split_fills_whole_waves(attn, sms, occ, b, hq, hkv, qlen, length):
    """The split is a multiple of 64 tokens; the pieces per sequence are the
    fewest whose CTAs make at least one wave with the last wave at least 90 %
    full, when any number of pieces does (checked by trying every count);
    otherwise no piece count fills the last wave better."""
    split = attn.attn_decode_split_tokens_for(sms, occ, b, hq, hkv, length, q_len=qlen)
    assert split > 0 and split % 64 == 0 and split <= 64 * math.ceil(length / 64)
    g = hq // hkv
    rows = g * qlen
    r = 1
    while r < rows and r < 16:
        r *= 2
    units = b * hkv * math.ceil(rows / r)
    slots = sms * occ
    n = math.ceil(length / split)
    # every piece count that 64-token splits can give
    counts = sorted({math.ceil(length / (64 * t)) for t in range(1, math.ceil(length / 64) + 1)})
    good = [k for k in counts if _waves(units, k, slots)[0] >= 1 and _waves(units, k, slots)[1] >= 0.9]
    if good:
        assert n == good[0]
    else:
        assert _waves(units, n, slots)[1] >= max(_waves(units, k, slots)[1] for k in counts) - 1e-12


def test_decode_split_on_the_int4_workload(attn):
    """16 sequences x 8 KV heads x 16384 tokens on 152 SMs x 3 CTAs: 2048-token
    pieces would make 1024 CTAs (2.25 waves); the choice is 7 pieces of 2368
    tokens, 896 CTAs (1.96 waves)."""
    assert attn.attn_decode_split_tokens_for(152, 3, 16, 32, 8, 16384) == 2368


def test_decode_split_refusals(attn):
    assert attn.attn_decode_split_tokens_for(0, 3, 16, 32, 8, 16384) == 0
    assert attn.attn_decode_split_tokens_for(152, 0, 16, 32, 8, 16384) == 0
    assert attn.attn_decode_split_tokens_for(152, 3, 16, 24, 8, 16384) == 0    # G = 3
    assert attn.attn_decode_split_tokens_for(152, 3, 16, 32, 8, 16384, q_len=17) == 0
    assert attn.attn_decode_split_tokens_for(152, 3, 16, 32, 8, 0) == 0


def _balanced_cost(split, B, groups, L, sms, unit_cost=64):
    """Largest per-CTA token sum when `sms` CTAs walk the units (group, chunk,
    sequence) round-robin, written out unit by unit."""
    S = -(-L // split)
    units = B * groups * S
    grid = min(units, sms)
    load = [0] * grid
    for u in range(units):
        s = (u % (B * S)) // B
        load[u % grid] += min(split, L - s * split) + unit_cost
    return max(load)


@pytest.mark.parametrize("tile", [32, 64])
@pytest.mark.parametrize("sms,B,groups,L", [
    (152, 16, 1, 16384), (152, 64, 1, 32768), (152, 2, 1, 131372), (148, 7, 2, 5000), (1, 3, 1, 700),
    (7, 1, 3, 64), (152, 40, 1, 1),
])
def test_balanced_decode_split_minimises_the_busiest_cta(attn, sms, B, groups, L, tile):
    """The persistent int4 decode's split: the multiple of `tile` whose
    round-robin walk gives the smallest busiest-CTA sum (64 tokens per unit for
    its fixed cost), the larger split on ties; checked against every candidate."""
    got = attn.attn_decode_split_tokens_balanced_for(sms, B, groups, L, tile)
    top = tile * -(-L // tile)
    assert got % tile == 0 and tile <= got <= top
    costs = {sp: _balanced_cost(sp, B, groups, L, sms) for sp in range(tile, top + 1, tile)}
    best = min(costs.values())
    assert costs[got] == best and got == max(sp for sp, c in costs.items() if c == best)


def test_balanced_decode_split_of_the_int4_workload(attn):
    """16 sequences of 16384 tokens, one group of 8 KV heads, 152 SMs: in
    32-token steps, 19 chunks of 864 tokens (304 units, two per CTA, busiest
    CTA 1728 tokens); in 64-token steps 1856 (9 chunks, one unit per CTA) ties
    with 896 and the larger is taken.  Bad sizes give 0."""
    assert attn.attn_decode_split_tokens_balanced_for(152, 16, 1, 16384, 32) == 864
    assert attn.attn_decode_split_tokens_balanced_for(152, 16, 1, 16384, 64) == 1856
    assert attn.attn_decode_split_tokens_balanced_for(0, 16, 1, 16384, 32) == 0
    assert attn.attn_decode_split_tokens_balanced_for(152, 16, 0, 16384, 32) == 0
    assert attn.attn_decode_split_tokens_balanced_for(152, 16, 1, 16384, 48) == 0
