"""fp64 definition of causal grouped-query attention, paged split-K decode and
the LSE merge (TEST INFRASTRUCTURE: tests, smoke check and CPU baseline only).

Sources, by page title and section:

* ``causal_forward_kernel.py`` (flash-attention-scratch),
  ``_flash_attention_forward_gqa_kernel``: the GQA head map
  (query head h reads KV head h // G, G = Hq / Hkv) and what the blockwise
  loop computes.
* ``gpt-o3 / triton6fd1ef`` (FlashInfer-style GQA prefill), ``_gqa_prefill_kernel``,
  the block that counts the KV tokens each query may see: bottom-right causal alignment,
  a key j is visible to query i iff ``j < min(kv_len, i + 1 + delta)`` with
  ``delta = kv_len - q_len``.
* ``splitk_kernels.py`` (xformers), ``_fwd_kernel_splitK``: split-K chunks,
  block-table indirection, the empty-chunk convention (O = 0, LSE = -inf) and
  the natural-log LSE written by its epilogue; its docstring and
  ``cast_uint32_to_half2`` / ``dequantize``: the int4 row format;
  ``_splitK_reduce``: the LSE-weighted merge.

Readings taken where the pages disagree or are silent:

* LSE is the natural log-sum-exp of the scaled scores, with no epsilon.
* Rows with no visible key yield O = 0 and LSE = -inf.
* Inputs are the exact low-precision values upcast to float64; nothing here
  rounds intermediate values.
"""

import math

import numpy as np

NEG_INF = -np.inf


# --------------------------------------------------------------------------
# Dense causal GQA prefill
# --------------------------------------------------------------------------

def visible_mask(q_len, kv_len, rows=None):
    """Boolean visibility matrix ``[len(rows), kv_len]``.

    Bottom-right causal alignment (``gpt-o3 / triton6fd1ef``,
    ``_gqa_prefill_kernel``, the count of keys each query may see): with
    ``delta = kv_len - q_len`` key ``j`` is visible to query ``i`` iff
    ``j <= i + delta`` (and ``j < kv_len``, which the range of ``j`` gives).
    """
    delta = kv_len - q_len
    i = np.arange(q_len) if rows is None else np.asarray(rows, dtype=np.int64)
    j = np.arange(kv_len)
    return j[None, :] <= (i[:, None] + delta)


def attend(q, k, v, mask, scale):
    """Masked softmax attention of one head, materialised in full: what the
    blockwise online-softmax loop of ``causal_forward_kernel.py``
    (``_flash_attention_forward_gqa_kernel``) computes, written directly.

    ``q [M, D]``, ``k [N, D]``, ``v [N, Dv]``, ``mask`` bool ``[M, N]``.
    Returns ``o [M, Dv]`` and the natural-log ``lse [M]``:

    1. ``S = scale * q k^T``, masked entries set to -inf;
    2. ``lse = m + log(sum_j exp(S - m))`` with ``m`` the row maximum;
    3. ``P = exp(S - lse)``, ``O = P v``;
    4. a row with no visible key gets ``O = 0`` and ``lse = -inf``.
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    m_rows, n_keys = q.shape[0], k.shape[0]
    s = scale * (q @ k.T)
    s = np.where(mask, s, NEG_INF)
    if n_keys == 0:
        return np.zeros((m_rows, v.shape[1])), np.full(m_rows, NEG_INF)
    m = s.max(axis=1)
    has_key = np.isfinite(m)
    m_safe = np.where(has_key, m, 0.0)
    l = np.exp(s - m_safe[:, None]).sum(axis=1)
    lse = np.where(has_key, m_safe + np.log(np.where(has_key, l, 1.0)), NEG_INF)
    p = np.where(has_key[:, None], np.exp(s - np.where(has_key, lse, 0.0)[:, None]), 0.0)
    return p @ v, lse


def _default_scale(d):
    # 1/sqrt(D), the wrappers' default softmax scale on every page.
    return 1.0 / math.sqrt(d)


def prefill(q, k, v, scale=None):
    """Causal GQA prefill: ``q [B, Hq, q_len, D]``, ``k, v [B, Hkv, kv_len, D]``.

    Returns ``o [B, Hq, q_len, D]`` and ``lse [B, Hq, q_len]`` in float64.
    K and V are expanded to Hq heads with an explicit ``np.repeat`` so that
    query head ``h`` reads key/value head ``h // (Hq // Hkv)``
    (``causal_forward_kernel.py``, ``_flash_attention_forward_gqa_kernel``,
    its GQA head-map block).
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    bsz, hq, q_len, d = q.shape
    hkv, kv_len = k.shape[1], k.shape[2]
    if hq % hkv != 0:
        raise ValueError("Hq must be a multiple of Hkv")
    group = hq // hkv
    scale = _default_scale(d) if scale is None else float(scale)
    k_rep = np.repeat(k, group, axis=1)
    v_rep = np.repeat(v, group, axis=1)
    mask = visible_mask(q_len, kv_len)
    o = np.zeros((bsz, hq, q_len, v.shape[3]))
    lse = np.zeros((bsz, hq, q_len))
    for b in range(bsz):
        for h in range(hq):
            o[b, h], lse[b, h] = attend(q[b, h], k_rep[b, h], v_rep[b, h], mask, scale)
    return o, lse


def prefill_rows(q, k, v, b, h, rows, scale=None):
    """The same definition as :func:`prefill`, for selected query rows
    ``rows`` of one (batch ``b``, query head ``h``); used to check sampled
    outputs of workloads too large to materialise whole."""
    d = q.shape[3]
    hq, hkv = q.shape[1], k.shape[1]
    q_len, kv_len = q.shape[2], k.shape[2]
    if hq % hkv != 0:
        raise ValueError("Hq must be a multiple of Hkv")
    group = hq // hkv
    scale = _default_scale(d) if scale is None else float(scale)
    rows = np.asarray(rows, dtype=np.int64)
    # explicit repeat of this batch entry's key/value heads
    k_rep = np.repeat(np.asarray(k[b], dtype=np.float64), group, axis=0)
    v_rep = np.repeat(np.asarray(v[b], dtype=np.float64), group, axis=0)
    qb = np.asarray(q[b, h], dtype=np.float64)[rows]
    return attend(qb, k_rep[h], v_rep[h], visible_mask(q_len, kv_len, rows), scale)


# --------------------------------------------------------------------------
# int4 row format (splitk_kernels.py: docstring of _fwd_kernel_splitK,
# cast_uint32_to_half2, dequantize)
# --------------------------------------------------------------------------

def fp16_from_bits(bits):
    """IEEE binary16 values from their 16-bit patterns, as float64."""
    return np.asarray(bits, dtype=np.uint16).view(np.float16).astype(np.float64)


def unpack_coef_word(word):
    """One quantisation coefficient word: the low 16 bits are the fp16 scale,
    the high 16 bits the fp16 offset (``cast_uint32_to_half2``)."""
    w = int(np.uint32(np.int64(word) & 0xFFFFFFFF))
    return float(fp16_from_bits(w & 0xFFFF)), float(fp16_from_bits(w >> 16))


def dequant_int4_row(words, d, n_groups):
    """Dequantise one packed row, element by element.

    ``words``: ``n_groups + d // 8`` 32-bit words.  The first ``n_groups`` are
    coefficient words (group order); then come the code words, group by group,
    ``d // 8 // n_groups`` words per group.  Inside a code word nibble ``j``
    (bits ``4j .. 4j+3``) holds element ``word_in_group * 8 + j`` of the group,
    and group ``g`` covers elements ``[g*d/n_groups, (g+1)*d/n_groups)``.
    Value = ``scale * code + offset`` in exact arithmetic.
    """
    if n_groups not in (1, 2, 4, 8) or d % (8 * n_groups) != 0:
        raise ValueError("unsupported int4 layout")
    words = [int(np.uint32(np.int64(x) & 0xFFFFFFFF)) for x in words]
    if len(words) != n_groups + d // 8:
        raise ValueError("row has the wrong number of words")
    per_group = d // n_groups
    words_per_group = per_group // 8
    out = np.zeros(d)
    for g in range(n_groups):
        scale, offset = unpack_coef_word(words[g])
        for w in range(words_per_group):
            word = words[n_groups + g * words_per_group + w]
            for j in range(8):
                code = (word >> (4 * j)) & 0xF
                out[g * per_group + w * 8 + j] = scale * code + offset
    return out


def dequant_int4_rows(words, d, n_groups):
    """The same layout as :func:`dequant_int4_row`, for an array of rows
    ``words [..., n_groups + d // 8]``, written with numpy broadcasting."""
    if n_groups not in (1, 2, 4, 8) or d % (8 * n_groups) != 0:
        raise ValueError("unsupported int4 layout")
    w = np.asarray(words).astype(np.int64) & 0xFFFFFFFF
    if w.shape[-1] != n_groups + d // 8:
        raise ValueError("row has the wrong number of words")
    coef = w[..., :n_groups]
    scale = fp16_from_bits(coef & 0xFFFF)                     # [..., G]
    offset = fp16_from_bits(coef >> 16)                       # [..., G]
    code_words = w[..., n_groups:]                            # [..., d/8]
    shifts = 4 * np.arange(8)
    codes = (code_words[..., :, None] >> shifts) & 0xF        # [..., d/8, 8]
    codes = codes.reshape(w.shape[:-1] + (d,)).astype(np.float64)
    per_group = d // n_groups
    scale_e = np.repeat(scale, per_group, axis=-1)
    offset_e = np.repeat(offset, per_group, axis=-1)
    return scale_e * codes + offset_e


# --------------------------------------------------------------------------
# fp8 row format (splitk_kernels.py: FP8_QUANTIZED in _fwd_kernel_splitK,
# the K/V_fp8_scale_shift tensors, the fp8 branch of dequantize)
# --------------------------------------------------------------------------

def fp8_e4m3_value(byte):
    """Value of one float8 e4m3 byte, the encoding ``splitk_kernels.py``'s
    ``dequantize`` bitcasts fp8 codes to (1 sign bit, 4 exponent bits with bias 7,
    3 mantissa bits, no infinities; exponent 15 with mantissa 7 is NaN)."""
    b = int(byte) & 0xFF
    sign = -1.0 if b >> 7 else 1.0
    e = (b >> 3) & 0xF
    m = b & 7
    if e == 15 and m == 7:
        return float("nan")
    if e == 0:
        return sign * m * 2.0 ** -9             # subnormal: m/8 * 2^(1-7)
    return sign * (1.0 + m / 8.0) * 2.0 ** (e - 7)


_FP8_TABLE = np.array([fp8_e4m3_value(b) for b in range(256)])


def dequant_fp8_rows(codes, scale_shift):
    """Row-wise fp8 dequantisation (``splitk_kernels.py``, ``_fwd_kernel_splitK``
    with a separate scale/shift tensor, and ``dequantize``).
    Rows of e4m3 bytes ``codes [..., D]`` with one coefficient word per row
    ``scale_shift [...]`` (fp16 scale in the low 16 bits, fp16 shift in the
    high 16 bits): value = decoded byte * scale + shift, in float64."""
    c = np.asarray(codes).astype(np.int64) & 0xFF
    w = np.asarray(scale_shift).astype(np.int64) & 0xFFFFFFFF
    scale = fp16_from_bits(w & 0xFFFF)[..., None]
    shift = fp16_from_bits(w >> 16)[..., None]
    return _FP8_TABLE[c] * scale + shift


# --------------------------------------------------------------------------
# Paged split-K decode (splitk_kernels.py: _fwd_kernel_splitK)
# --------------------------------------------------------------------------

def paged_row_index(block_table, b, t, page_size):
    """Physical row of logical token ``t`` of sequence ``b``:
    ``block_table[b, t // page_size] * page_size + t % page_size``
    (the page-offset computation, ``physical_page_idx``, in ``_fwd_kernel_splitK``)."""
    return int(block_table[b][t // page_size]) * page_size + t % page_size


def gather_paged_rows(cache, block_table, b, t_lo, t_hi, page_size):
    """Rows ``[t_lo, t_hi)`` of sequence ``b`` from a paged pool
    ``cache [num_pages, page_size, Hkv, W]``, one token at a time."""
    out = []
    for t in range(t_lo, t_hi):
        page = int(block_table[b][t // page_size])
        out.append(np.asarray(cache[page, t % page_size]))
    if not out:
        return np.zeros((0,) + tuple(cache.shape[2:]), dtype=np.asarray(cache[:0]).dtype)
    return np.stack(out)


def _kv_rows(cache, block_table, b, lo, hi, page_size, kv_format, d, n_groups, scale_shift=None):
    rows = gather_paged_rows(cache, block_table, b, lo, hi, page_size)
    if kv_format == "int4":
        return dequant_int4_rows(rows, d, n_groups)
    if kv_format == "fp8":
        words = gather_paged_rows(scale_shift, block_table, b, lo, hi, page_size)   # [n, Hkv]
        return dequant_fp8_rows(rows, words)
    if kv_format != "dense":
        raise ValueError("kv_format must be 'dense', 'int4' or 'fp8'")
    return rows.astype(np.float64)


def num_splits(max_kv_len, split_tokens):
    """Number of split-K chunks for the longest sequence (at least one); chunk
    ``s`` starts at ``s * split_tokens`` (``splitk_kernels.py``,
    ``_fwd_kernel_splitK``: each split's key range begins at its index times
    the per-split block size)."""
    return max(1, -(-int(max_kv_len) // int(split_tokens)))


def decode_split_partials(q, k_cache, v_cache, block_table, seq_lens, page_size,
                          split_tokens, scale=None, kv_format="dense", n_groups=1,
                          max_kv_len=None, batches=None, k_scale_shift=None, v_scale_shift=None):
    """Per-split partial results of single-query decode.

    ``q [B, Hq, D]``; caches ``[num_pages, page_size, Hkv, D]`` (dense values
    or fp8 e4m3 bytes, the latter with ``k/v_scale_shift [num_pages,
    page_size, Hkv]`` words) or ``[num_pages, page_size, Hkv, n_groups + D/8]``
    (int4 words).
    Split ``s`` of sequence ``b`` covers tokens
    ``[s*split_tokens, min((s+1)*split_tokens, len_b))``; with one query per
    sequence every cached token is visible.  An empty split gives ``O_s = 0``
    and ``LSE_s = -inf`` (the early exit and the ``l == 0`` guard of
    ``_fwd_kernel_splitK``).  Returns ``o_part [B, Hq, S, D]`` and
    ``lse_part [B, Hq, S]``; ``batches`` restricts the work to some sequences
    (the other entries stay zero / -inf).
    """
    q = np.asarray(q, dtype=np.float64)
    bsz, hq, d = q.shape
    hkv = k_cache.shape[2]
    if hq % hkv != 0:
        raise ValueError("Hq must be a multiple of Hkv")
    group = hq // hkv
    scale = _default_scale(d) if scale is None else float(scale)
    lens = [int(x) for x in np.asarray(seq_lens).reshape(-1)]
    if max_kv_len is None:
        max_kv_len = max(lens) if lens else 0
    n_split = num_splits(max_kv_len, split_tokens)
    o_part = np.zeros((bsz, hq, n_split, d))
    lse_part = np.full((bsz, hq, n_split), NEG_INF)
    for b in (range(bsz) if batches is None else batches):
        for s in range(n_split):
            lo = s * split_tokens
            hi = min(lo + split_tokens, lens[b])
            if hi <= lo:
                continue
            k_rows = _kv_rows(k_cache, block_table, b, lo, hi, page_size, kv_format, d, n_groups, k_scale_shift)
            v_rows = _kv_rows(v_cache, block_table, b, lo, hi, page_size, kv_format, d, n_groups, v_scale_shift)
            k_rep = np.repeat(k_rows, group, axis=1)          # [n, Hq, D]
            v_rep = np.repeat(v_rows, group, axis=1)
            every = np.ones((1, hi - lo), dtype=bool)
            for h in range(hq):
                o, lse = attend(q[b, h][None, :], k_rep[:, h], v_rep[:, h], every, scale)
                o_part[b, h, s] = o[0]
                lse_part[b, h, s] = lse[0]
    return o_part, lse_part


def decode_unsplit(q, k_cache, v_cache, block_table, seq_lens, page_size, scale=None,
                   kv_format="dense", n_groups=1, batches=None, k_scale_shift=None, v_scale_shift=None):
    """Single-query decode over each whole sequence in one piece (no split):
    the result every split of ``splitk_kernels.py``'s ``_fwd_kernel_splitK``
    followed by ``_splitK_reduce`` must reproduce.  Cache formats as in
    :func:`decode_split_partials` (an fp8 cache comes with its per-row
    ``k/v_scale_shift`` words)."""
    q = np.asarray(q, dtype=np.float64)
    bsz, hq, d = q.shape
    hkv = k_cache.shape[2]
    group = hq // hkv
    scale = _default_scale(d) if scale is None else float(scale)
    lens = [int(x) for x in np.asarray(seq_lens).reshape(-1)]
    o_out = np.zeros((bsz, hq, d))
    lse_out = np.full((bsz, hq), NEG_INF)
    for b in (range(bsz) if batches is None else batches):
        k_rows = _kv_rows(k_cache, block_table, b, 0, lens[b], page_size, kv_format, d, n_groups, k_scale_shift)
        v_rows = _kv_rows(v_cache, block_table, b, 0, lens[b], page_size, kv_format, d, n_groups, v_scale_shift)
        k_rep = np.repeat(k_rows, group, axis=1)
        v_rep = np.repeat(v_rows, group, axis=1)
        every = np.ones((1, lens[b]), dtype=bool)
        for h in range(hq):
            o, lse = attend(q[b, h][None, :], k_rep[:, h], v_rep[:, h], every, scale)
            o_out[b, h], lse_out[b, h] = o[0], lse[0]
    return o_out, lse_out


# --------------------------------------------------------------------------
# LSE-weighted merge (splitk_kernels.py: _splitK_reduce)
# --------------------------------------------------------------------------

def lse_merge(o_part, lse_part):
    """Merge split partials ``o_part [..., S, D]``, ``lse_part [..., S]``
    (``splitk_kernels.py``, ``_splitK_reduce``).

    ``M = max_s LSE_s``; ``w_s = exp(LSE_s - M)``;
    ``O = sum_s w_s O_s / sum_s w_s``; ``LSE = M + log(sum_s w_s)``;
    when every ``LSE_s`` is -inf the result is ``O = 0``, ``LSE = -inf``.
    """
    o_part = np.asarray(o_part, dtype=np.float64)
    lse_part = np.asarray(lse_part, dtype=np.float64)
    if lse_part.shape[-1] == 0:
        return np.zeros(o_part.shape[:-2] + o_part.shape[-1:]), np.full(lse_part.shape[:-1], NEG_INF)
    m = lse_part.max(axis=-1)
    alive = np.isfinite(m)
    m_safe = np.where(alive, m, 0.0)
    w = np.where(alive[..., None], np.exp(lse_part - m_safe[..., None]), 0.0)
    wsum = w.sum(axis=-1)
    o = np.where(alive[..., None],
                 (w[..., None] * o_part).sum(axis=-2) / np.where(alive, wsum, 1.0)[..., None],
                 0.0)
    lse = np.where(alive, m_safe + np.log(np.where(alive, wsum, 1.0)), NEG_INF)
    return o, lse


def decode(q, k_cache, v_cache, block_table, seq_lens, page_size, split_tokens, scale=None,
           kv_format="dense", n_groups=1, max_kv_len=None, batches=None, k_scale_shift=None,
           v_scale_shift=None):
    """Split-K decode: the per-split partials merged by :func:`lse_merge`."""
    o_part, lse_part = decode_split_partials(q, k_cache, v_cache, block_table, seq_lens,
                                             page_size, split_tokens, scale, kv_format,
                                             n_groups, max_kv_len, batches, k_scale_shift, v_scale_shift)
    return lse_merge(o_part, lse_part)


# --------------------------------------------------------------------------
# Gradient of the merge (splitk_kernels.py: _splitK_reduce_varargs_backward)
# --------------------------------------------------------------------------

def lse_merge_bwd(o_part, lse_part, d_o, d_lse=None):
    """Gradients of :func:`lse_merge` with respect to its inputs
    (``splitk_kernels.py``, ``_splitK_reduce_varargs_backward``).

    For each row with merged ``O`` and ``LSE`` (recomputed here by
    :func:`lse_merge`) and incoming gradients ``dO [..., D]``, ``dLSE [...]``:

    1. ``w_s = exp(LSE_s - LSE)``, the weight of split ``s`` in the merge;
    2. ``dO_s = w_s * dO``;
    3. ``dLSE_s = w_s * dLSE + sum_d (O_s - O)_d * w_s * dO_d``.

    A split with ``LSE_s = -inf`` (weight 0), and every split of a row whose
    merged LSE is ``-inf``, gets zero gradients.  Returns ``(d_o_part,
    d_lse_part)`` shaped like ``o_part`` and ``lse_part``.
    """
    o_part = np.asarray(o_part, dtype=np.float64)
    lse_part = np.asarray(lse_part, dtype=np.float64)
    d_o = np.asarray(d_o, dtype=np.float64)
    d_lse = np.zeros(lse_part.shape[:-1]) if d_lse is None else np.asarray(d_lse, dtype=np.float64)
    o, lse = lse_merge(o_part, lse_part)
    alive = np.isfinite(lse)[..., None] & np.isfinite(lse_part)
    w = np.where(alive, np.exp(np.where(alive, lse_part - np.where(np.isfinite(lse), lse, 0.0)[..., None], 0.0)),
                 0.0)                                                          # [..., S]
    d_o_part = w[..., None] * d_o[..., None, :]                                # [..., S, D]
    d_lse_part = w * d_lse[..., None] + w * ((o_part - o[..., None, :]) * d_o[..., None, :]).sum(axis=-1)
    return d_o_part, d_lse_part


# --------------------------------------------------------------------------
# Causal multi-query decode (splitk_kernels.py: _fwd_kernel_splitK with
# IS_CAUSAL and NUM_QUERIES_CAUSAL, and the kernel's own explanation of its
# causal mask)
# --------------------------------------------------------------------------

def decode_mq_split_partials(q, k_cache, v_cache, block_table, seq_lens, page_size, split_tokens, scale=None,
                             kv_format="dense", n_groups=1, max_kv_len=None, batches=None, k_scale_shift=None,
                             v_scale_shift=None):
    """Split partials of decode with ``q_len`` queries per sequence
    (``splitk_kernels.py``, ``_fwd_kernel_splitK``, its causal mask for several
    queries per sequence).

    ``q [B, Hq, q_len, D]``.  Query ``i`` of sequence ``b`` sees cached token
    ``t`` iff ``t <= len_b - q_len + i`` (bottom-right alignment, the queries
    being the last ``q_len`` positions).  Returns ``o_part [B, Hq, q_len, S,
    D]`` and ``lse_part [B, Hq, q_len, S]``; a split in which a query sees no
    token gives ``O_s = 0``, ``LSE_s = -inf``.
    """
    q = np.asarray(q, dtype=np.float64)
    bsz, hq, nq, d = q.shape
    hkv = k_cache.shape[2]
    if hq % hkv != 0:
        raise ValueError("Hq must be a multiple of Hkv")
    group = hq // hkv
    scale = _default_scale(d) if scale is None else float(scale)
    lens = [int(x) for x in np.asarray(seq_lens).reshape(-1)]
    if max_kv_len is None:
        max_kv_len = max(lens) if lens else 0
    n_split = num_splits(max_kv_len, split_tokens)
    o_part = np.zeros((bsz, hq, nq, n_split, d))
    lse_part = np.full((bsz, hq, nq, n_split), NEG_INF)
    for b in (range(bsz) if batches is None else batches):
        for s in range(n_split):
            lo = s * split_tokens
            hi = min(lo + split_tokens, lens[b])
            if hi <= lo:
                continue
            k_rows = _kv_rows(k_cache, block_table, b, lo, hi, page_size, kv_format, d, n_groups, k_scale_shift)
            v_rows = _kv_rows(v_cache, block_table, b, lo, hi, page_size, kv_format, d, n_groups, v_scale_shift)
            k_rep = np.repeat(k_rows, group, axis=1)
            v_rep = np.repeat(v_rows, group, axis=1)
            t = np.arange(lo, hi)
            mask = t[None, :] <= (lens[b] - nq + np.arange(nq))[:, None]      # [q_len, n]
            for h in range(hq):
                o, lse = attend(q[b, h], k_rep[:, h], v_rep[:, h], mask, scale)
                o_part[b, h, :, s] = o
                lse_part[b, h, :, s] = lse
    return o_part, lse_part


def decode_mq(q, k_cache, v_cache, block_table, seq_lens, page_size, split_tokens, scale=None,
              kv_format="dense", n_groups=1, max_kv_len=None, batches=None, k_scale_shift=None,
              v_scale_shift=None):
    """Causal multi-query decode: the per-split partials merged by :func:`lse_merge`."""
    o_part, lse_part = decode_mq_split_partials(q, k_cache, v_cache, block_table, seq_lens, page_size,
                                                split_tokens, scale, kv_format, n_groups, max_kv_len, batches,
                                                k_scale_shift, v_scale_shift)
    return lse_merge(o_part, lse_part)


# --------------------------------------------------------------------------
# Ragged (varlen) prefill over a paged KV cache ("gpt-o3 / triton6fd1ef",
# run: CSR qo_indptr / kv_indptr / kv_indices, one query head group per KV
# head, bottom-right causal per sequence)
# --------------------------------------------------------------------------

def prefill_paged_varlen(q, k_cache, v_cache, qo_indptr, kv_indptr, kv_indices, page_size=1,
                         kv_last_page_len=None, scale=None):
    """Causal GQA prefill of a ragged batch against a paged KV cache.

    ``q [total_q, Hq, D]``; sequence ``b`` owns query rows
    ``[qo_indptr[b], qo_indptr[b+1])`` and the pages
    ``kv_indices[kv_indptr[b] : kv_indptr[b+1]]`` of the pool
    ``k_cache, v_cache [num_pages, page_size, Hkv, D]``.  Its KV length is
    ``(n_pages - 1) * page_size + kv_last_page_len[b]`` (every page full when
    ``kv_last_page_len`` is None).  Each sequence is the dense causal GQA
    prefill of :func:`attend` with ``delta = kv_len - q_len``.  Returns
    ``o [total_q, Hq, D]`` and ``lse [total_q, Hq]``.
    """
    q = np.asarray(q, dtype=np.float64)
    total_q, hq, d = q.shape
    hkv = k_cache.shape[2]
    if hq % hkv != 0:
        raise ValueError("Hq must be a multiple of Hkv")
    group = hq // hkv
    scale = _default_scale(d) if scale is None else float(scale)
    qo = [int(x) for x in np.asarray(qo_indptr)]
    kvp = [int(x) for x in np.asarray(kv_indptr)]
    idx = [int(x) for x in np.asarray(kv_indices)]
    o = np.zeros((total_q, hq, d))
    lse = np.full((total_q, hq), NEG_INF)
    for b in range(len(qo) - 1):
        q_len = qo[b + 1] - qo[b]
        pages = idx[kvp[b]:kvp[b + 1]]
        last = page_size if kv_last_page_len is None else int(np.asarray(kv_last_page_len)[b])
        kv_len = (len(pages) - 1) * page_size + last if pages else 0
        if q_len == 0:
            continue
        rows_k, rows_v = [], []
        for t in range(kv_len):
            page = pages[t // page_size]
            rows_k.append(np.asarray(k_cache[page, t % page_size], dtype=np.float64))
            rows_v.append(np.asarray(v_cache[page, t % page_size], dtype=np.float64))
        kk = np.stack(rows_k) if rows_k else np.zeros((0, hkv, d))
        vv = np.stack(rows_v) if rows_v else np.zeros((0, hkv, d))
        k_rep = np.repeat(kk, group, axis=1)
        v_rep = np.repeat(vv, group, axis=1)
        mask = visible_mask(q_len, kv_len)
        for h in range(hq):
            ob, lb = attend(q[qo[b]:qo[b + 1], h], k_rep[:, h], v_rep[:, h], mask, scale)
            o[qo[b]:qo[b + 1], h] = ob
            lse[qo[b]:qo[b + 1], h] = lb
    return o, lse
