"""Seeded synthetic inputs shared by the tests, the benchmark and the smoke check.

This package holds shapes and random draws only; it contains none of the
attention arithmetic, so the oracle and the CUDA path can both be fed from it
without sharing any of the method.

Every generator draws from a CPU ``torch.Generator`` seeded explicitly, in the
order given in its docstring, so a (workload, seed) pair names one input set
on any machine.  Tensors are built on the CPU; callers move them to a device.
"""

from dataclasses import dataclass, field

import torch


@dataclass(frozen=True)
class PrefillShape:
    name: str
    B: int
    Hq: int
    Hkv: int
    q_len: int
    kv_len: int
    D: int
    dtype: torch.dtype
    k_scale: float = 1.0


@dataclass(frozen=True)
class DecodeShape:
    name: str
    B: int
    Hq: int
    Hkv: int
    D: int
    len_lo: int
    len_hi: int
    page_size: int
    split_tokens: int
    kv_format: str = "dense"        # "dense" (bf16), "int4" or "fp8"
    n_groups: int = 1
    extra: dict = field(default_factory=dict)


# The five workloads of the method's problem statement.
TINY_PREFILL_FP32 = PrefillShape("tiny causal GQA prefill fp32", 1, 4, 2, 128, 128, 64, torch.float32)
LLAMA_GQA_PREFILL = PrefillShape("Llama-style GQA prefill, bottom-right causal", 1, 32, 4, 2048, 4096, 128,
                                 torch.bfloat16)
BATCHED_SQUARE_PREFILL = PrefillShape("batched square causal GQA prefill, K x2", 8, 32, 8, 4096, 4096, 128,
                                      torch.bfloat16, k_scale=2.0)
PAGED_DECODE_BF16 = DecodeShape("paged split-K decode bf16", 64, 32, 8, 128, 512, 32768, 256, 2048)
PAGED_DECODE_INT4 = DecodeShape("int4 paged split-K decode", 16, 32, 8, 128, 16384, 16384, 256, 2048,
                                kv_format="int4", n_groups=4)
# fp8 row-wise cache on the int4 workload's shape (an extension of the method, not one of its five workloads)
PAGED_DECODE_FP8 = DecodeShape("fp8 paged split-K decode", 16, 32, 8, 128, 16384, 16384, 256, 2048,
                               kv_format="fp8")

WORKLOADS = {
    "tiny_prefill_fp32": TINY_PREFILL_FP32,
    "llama_gqa_prefill": LLAMA_GQA_PREFILL,
    "batched_square_prefill": BATCHED_SQUARE_PREFILL,
    "paged_decode_bf16": PAGED_DECODE_BF16,
    "paged_decode_int4": PAGED_DECODE_INT4,
}


def generator(seed):
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    return g


def prefill_inputs(shape, seed=0):
    """Q, K, V for a prefill shape, drawn in the order Q, K, V.

    Each is i.i.d. N(0, 1) in float32, K is multiplied by ``shape.k_scale``,
    then all three are rounded to ``shape.dtype``.  Layouts:
    ``Q [B, Hq, q_len, D]``, ``K, V [B, Hkv, kv_len, D]``, contiguous.
    """
    g = generator(seed)
    q = torch.randn(shape.B, shape.Hq, shape.q_len, shape.D, generator=g)
    k = torch.randn(shape.B, shape.Hkv, shape.kv_len, shape.D, generator=g) * shape.k_scale
    v = torch.randn(shape.B, shape.Hkv, shape.kv_len, shape.D, generator=g)
    return q.to(shape.dtype), k.to(shape.dtype), v.to(shape.dtype)


def pack_int4_rows(codes, scale_bits, offset_bits, n_groups):
    """Encode rows in the int4 group format.

    ``codes`` uint8 ``[..., D]`` in 0..15, ``scale_bits`` / ``offset_bits``
    int32 ``[..., n_groups]`` holding fp16 bit patterns.  Output int32
    ``[..., n_groups + D // 8]``: one coefficient word per group (scale in the
    low 16 bits, offset in the high 16 bits), then the code words group by
    group, element ``8*w + j`` of a group in bits ``4j .. 4j+3`` of its word
    ``w``.  This is the input format, not part of the method.
    """
    d = codes.shape[-1]
    c = codes.to(torch.int64).reshape(*codes.shape[:-1], d // 8, 8)
    shifts = torch.arange(8, dtype=torch.int64) * 4
    words = (c << shifts).sum(dim=-1)                                  # [..., D/8] in [0, 2^32)
    coef = (scale_bits.to(torch.int64) & 0xFFFF) | ((offset_bits.to(torch.int64) & 0xFFFF) << 16)
    packed = torch.cat([coef, words], dim=-1)
    packed = torch.where(packed >= 2 ** 31, packed - 2 ** 32, packed)  # reinterpret as int32
    return packed.to(torch.int32)


def _fp16_bits(x):
    return x.to(torch.float16).view(torch.int16).to(torch.int32) & 0xFFFF


def decode_inputs(shape, seed=0, lens=None, pages_per_draw=64):
    """Inputs of one single-query paged decode problem.

    Draw order (one CPU generator):
      1. sequence lengths ``len_b`` ~ U{len_lo .. len_hi} (skipped when
         ``lens`` is given or ``len_lo == len_hi``);
      2. a permutation of the page pool, which holds exactly
         ``sum_b ceil(len_b / page_size)`` pages; sequence ``b`` owns the next
         ``ceil(len_b / page_size)`` entries of the permutation, in order;
      3. ``q [B, Hq, D]`` ~ N(0, 1), rounded to bf16;
      4. the K pool, then the V pool, ``pages_per_draw`` pages at a time:
         dense: N(0, 1) rounded to bf16, layout ``[pages, page_size, Hkv, D]``;
         int4: codes ~ U{0..15}, then scales ~ U[0.01, 0.1] and offsets
         ~ N(0, 0.1), both rounded to fp16, packed by :func:`pack_int4_rows`
         into ``[pages, page_size, Hkv, n_groups + D/8]`` int32;
         fp8: values ~ N(0, 16) rounded to float8 e4m3 (bytes
         ``[pages, page_size, Hkv, D]``), then scales ~ U[0.1, 0.5] and shifts
         ~ N(0, 0.1) rounded to fp16 and packed one word per row (scale low,
         shift high) into ``k/v_scale_shift [pages, page_size, Hkv]``.
    Block-table entries past a sequence's last page are -1.
    """
    g = generator(seed)
    if lens is None:
        if shape.len_lo == shape.len_hi:
            lens = [shape.len_lo] * shape.B
        else:
            lens = torch.randint(shape.len_lo, shape.len_hi + 1, (shape.B,), generator=g).tolist()
    lens = [int(x) for x in lens]
    ps = shape.page_size
    pages_per_seq = [-(-n // ps) for n in lens]
    n_pages = max(1, sum(pages_per_seq))
    perm = torch.randperm(n_pages, generator=g)
    max_pages = max(1, max(pages_per_seq))
    block_table = torch.full((shape.B, max_pages), -1, dtype=torch.int32)
    cursor = 0
    for b, n in enumerate(pages_per_seq):
        block_table[b, :n] = perm[cursor:cursor + n].to(torch.int32)
        cursor += n
    q = torch.randn(shape.B, shape.Hq, shape.D, generator=g).to(torch.bfloat16)

    def pool():
        chunks = []
        for start in range(0, n_pages, pages_per_draw):
            n = min(pages_per_draw, n_pages - start)
            if shape.kv_format == "dense":
                chunks.append(torch.randn(n, ps, shape.Hkv, shape.D, generator=g).to(torch.bfloat16))
            elif shape.kv_format == "fp8":
                x = torch.randn(n, ps, shape.Hkv, shape.D, generator=g) * 4.0
                codes = x.to(torch.float8_e4m3fn).view(torch.uint8)
                scales = torch.rand(n, ps, shape.Hkv, generator=g) * 0.4 + 0.1
                shifts = torch.randn(n, ps, shape.Hkv, generator=g) * 0.1
                words = _fp16_bits(scales).to(torch.int64) | (_fp16_bits(shifts).to(torch.int64) << 16)
                words = torch.where(words >= 2 ** 31, words - 2 ** 32, words).to(torch.int32)
                chunks.append((codes, words))
            elif shape.kv_format == "int4":
                codes = torch.randint(0, 16, (n, ps, shape.Hkv, shape.D), generator=g, dtype=torch.uint8)
                scales = torch.rand(n, ps, shape.Hkv, shape.n_groups, generator=g) * 0.09 + 0.01
                offsets = torch.randn(n, ps, shape.Hkv, shape.n_groups, generator=g) * 0.1
                chunks.append(pack_int4_rows(codes, _fp16_bits(scales), _fp16_bits(offsets), shape.n_groups))
            else:
                raise ValueError(shape.kv_format)
        if shape.kv_format == "fp8":
            return torch.cat([c for c, _ in chunks], dim=0), torch.cat([w for _, w in chunks], dim=0)
        return torch.cat(chunks, dim=0), None

    k_cache, k_scale_shift = pool()
    v_cache, v_scale_shift = pool()
    extra = {}
    if shape.kv_format == "fp8":
        extra = {"k_scale_shift": k_scale_shift, "v_scale_shift": v_scale_shift}
    return {**extra,
        "q": q,
        "k_cache": k_cache,
        "v_cache": v_cache,
        "block_table": block_table,
        "seq_lens": torch.tensor(lens, dtype=torch.int32),
        "lens": lens,
        "n_pages": n_pages,
        "max_pages": max_pages,
    }


def merge_inputs(n_rows, n_splits, d, seed=0, p_empty=0.25):
    """Random split partials for the merge: ``o_part [n_rows, n_splits, d]``
    ~ N(0, 1) and ``lse_part [n_rows, n_splits]`` ~ N(0, 3), drawn in that
    order, then a U[0, 1) draw per entry marks it empty (LSE = -inf, O = 0)
    with probability ``p_empty``; the first row is made entirely empty."""
    g = generator(seed)
    o_part = torch.randn(n_rows, n_splits, d, generator=g)
    lse_part = torch.randn(n_rows, n_splits, generator=g) * 3.0
    empty = torch.rand(n_rows, n_splits, generator=g) < p_empty
    if n_rows > 0:
        empty[0] = True
    lse_part = torch.where(empty, torch.full_like(lse_part, float("-inf")), lse_part)
    o_part = torch.where(empty[..., None], torch.zeros_like(o_part), o_part)
    return o_part, lse_part


@dataclass(frozen=True)
class VarlenShape:
    name: str
    B: int
    Hq: int
    Hkv: int
    D: int
    q_lo: int
    q_hi: int
    prefix_lo: int     # cached tokens before the new queries
    prefix_hi: int
    page_size: int = 1


# A ragged prefill batch over a token-granular paged cache, the layout of the
# FlashInfer-style GQA prefill (32 query heads, 4 KV heads, head dim 128,
# page size 1).  The page gives no batch sizes; these are chosen for the
# benchmark: 8 sequences, 256-2048 new tokens each on top of 0-2048 cached.
VARLEN_PAGED_PREFILL = VarlenShape("ragged paged GQA prefill, page size 1", 8, 32, 4, 128, 256, 2048, 0, 2048)


def varlen_inputs(shape, seed=0, q_lens=None, kv_lens=None):
    """Inputs of one ragged prefill over a paged cache.

    Draw order (one CPU generator): new-token counts ``q_len_b`` ~
    U{q_lo..q_hi} and cached-prefix lengths ~ U{prefix_lo..prefix_hi} (both
    skipped when given; ``kv_len_b = q_len_b + prefix_b``); a permutation of the
    page pool (exactly ``sum_b ceil(kv_len_b / page_size)`` pages, sequence b
    taking the next ones in order); ``q [total_q, Hq, D]`` ~ N(0, 1) as bf16;
    the K pool then the V pool ``[pages, page_size, Hkv, D]`` ~ N(0, 1) as bf16.
    Returns CSR ``qo_indptr``, ``kv_indptr`` (pages) and ``kv_indices`` plus
    ``kv_last_page_len``, all int32.
    """
    g = generator(seed)
    if q_lens is None:
        q_lens = torch.randint(shape.q_lo, shape.q_hi + 1, (shape.B,), generator=g).tolist()
    if kv_lens is None:
        pre = torch.randint(shape.prefix_lo, shape.prefix_hi + 1, (len(q_lens),), generator=g).tolist()
        kv_lens = [a + b for a, b in zip(q_lens, pre)]
    q_lens = [int(x) for x in q_lens]
    kv_lens = [int(x) for x in kv_lens]
    ps = shape.page_size
    n_pages_b = [-(-n // ps) for n in kv_lens]
    n_pages = max(1, sum(n_pages_b))
    perm = torch.randperm(n_pages, generator=g).to(torch.int32)
    qo = [0]
    for n in q_lens:
        qo.append(qo[-1] + n)
    kvp = [0]
    for n in n_pages_b:
        kvp.append(kvp[-1] + n)
    q = torch.randn(qo[-1], shape.Hq, shape.D, generator=g).to(torch.bfloat16)
    k_cache = torch.randn(n_pages, ps, shape.Hkv, shape.D, generator=g).to(torch.bfloat16)
    v_cache = torch.randn(n_pages, ps, shape.Hkv, shape.D, generator=g).to(torch.bfloat16)
    last = [n - (p - 1) * ps if p > 0 else 0 for n, p in zip(kv_lens, n_pages_b)]
    return {
        "q": q, "k_cache": k_cache, "v_cache": v_cache,
        "qo_indptr": torch.tensor(qo, dtype=torch.int32),
        "kv_indptr": torch.tensor(kvp, dtype=torch.int32),
        "kv_indices": perm[:kvp[-1]].clone() if kvp[-1] > 0 else torch.zeros(1, dtype=torch.int32),
        "kv_last_page_len": torch.tensor(last, dtype=torch.int32),
        "q_lens": q_lens, "kv_lens": kv_lens, "n_pages": n_pages,
    }
