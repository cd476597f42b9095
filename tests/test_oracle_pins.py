"""Pins for the fp64 oracle, none of which re-types its formulas.

Each check ties the oracle to something outside itself: hand-derived fixtures
(tests/golden), brute force with scalar Python loops on tiny inputs, closed
forms, a library routine (torch's scaled_dot_product_attention with an explicit
boolean mask, and scipy's logsumexp), and invariants of the definition.  The
tests at the end plant plausible mistakes in the oracle (a wrong mask, scale, sign,
index, operand, bias or dropped term, one at a time) and check that a pin fails.
"""

import math

import numpy as np
import pytest
import torch

import oracle
from oracle import attention as oa


# ---------------------------------------------------------------- fixtures

def _f(vals):
    return np.array([float(x) for x in vals])


def test_golden_uniform_scores_bottom_right(golden):
    g = golden("uniform_scores_bottom_right.txt")
    v = _f(g["v"]).reshape(1, 1, 3, 1)
    q = np.zeros((1, 2, 2, 1))
    k = np.arange(3, dtype=np.float64).reshape(1, 1, 3, 1)   # any K: scores are all zero
    o, lse = oracle.prefill(q, k, v, scale=1.0)
    for h in range(2):
        np.testing.assert_allclose(o[0, h, :, 0], _f(g[f"o_head{h}"]), rtol=0, atol=1e-15)
        np.testing.assert_allclose(lse[0, h], _f(g[f"lse_head{h}"]), rtol=0, atol=1e-15)


def test_golden_two_key_softmax(golden):
    g = golden("two_key_softmax.txt")
    q = _f(g["q"]).reshape(1, 1, 1, 2)
    k = np.stack([_f(g["k0"]), _f(g["k1"])]).reshape(1, 1, 2, 2)
    v = np.stack([_f(g["v0"]), _f(g["v1"])]).reshape(1, 1, 2, 2)
    o, lse = oracle.prefill(q, k, v, scale=1.0)
    np.testing.assert_allclose(o[0, 0, 0], _f(g["o"]), rtol=0, atol=1e-14)
    np.testing.assert_allclose(lse[0, 0, 0], float(g["lse"][0]), rtol=0, atol=1e-15)


def test_golden_int4_rows(golden):
    g = golden("int4_rows.txt")
    for row, d, ng in (("rowA", 8, 1), ("rowB", 16, 2)):
        words = [int(x, 16) for x in g[f"{row}_words"]]
        want = _f(g[f"{row}_values"])
        got = oracle.dequant_int4_row(words, d, ng)
        np.testing.assert_array_equal(got, want)
        got_vec = oracle.dequant_int4_rows(np.array(words, dtype=np.uint32)[None], d, ng)[0]
        np.testing.assert_array_equal(got_vec, want)


def test_golden_block_table(golden):
    g = golden("block_table.txt")
    ps = int(g["page_size"][0])
    table = np.array([[int(x) for x in g["table0"]], [int(x) for x in g["table1"]]])
    rows0 = [oracle.paged_row_index(table, 0, t, ps) for t in range(4)]
    rows1 = [oracle.paged_row_index(table, 1, t, ps) for t in range(2)]
    assert rows0 == [int(x) for x in g["rows0"]]
    assert rows1 == [int(x) for x in g["rows1"]]
    # gathered rows are bit-identical to the rows of a pool that stores its
    # own physical row number
    pool = np.arange(3 * ps, dtype=np.int64).reshape(3, ps, 1, 1)
    got = oracle.gather_paged_rows(pool, table, 0, 0, 4, ps).reshape(-1)
    assert got.tolist() == rows0


def test_golden_merge_two_splits(golden):
    g = golden("merge_two_splits.txt")
    lse = _f(g["lse"])[None]
    o = _f(g["o"]).reshape(1, 2, 1)
    om, lm = oracle.lse_merge(o, lse)
    np.testing.assert_allclose(om[0], _f(g["o_merged"]), rtol=0, atol=1e-15)
    np.testing.assert_allclose(lm[0], float(g["lse_merged"][0]), rtol=0, atol=1e-15)
    # a -inf split carries no weight; an all -inf row merges to (0, -inf)
    om, lm = oracle.lse_merge(np.array([[[5.0], [7.0]]]), np.array([[-np.inf, 0.3]]))
    assert om[0, 0] == 7.0 and lm[0] == 0.3
    om, lm = oracle.lse_merge(np.zeros((1, 3, 2)), np.full((1, 3), -np.inf))
    assert np.all(om == 0) and lm[0] == -np.inf


# ------------------------------------------------------ brute force, tiny

def _brute_prefill(q, k, v, scale):
    """Scalar loops: for each (b, h, i) sum over visible j of exp(s_ij)."""
    bsz, hq, lq, d = q.shape
    hkv, lk = k.shape[1], k.shape[2]
    grp = hq // hkv
    delta = lk - lq
    o = np.zeros((bsz, hq, lq, v.shape[3]))
    lse = np.zeros((bsz, hq, lq))
    for b in range(bsz):
        for h in range(hq):
            kh = h // grp
            for i in range(lq):
                scores = []
                for j in range(lk):
                    if j <= i + delta:
                        s = 0.0
                        for c in range(d):
                            s += q[b, h, i, c] * k[b, kh, j, c]
                        scores.append((j, s * scale))
                if not scores:
                    lse[b, h, i] = -math.inf
                    continue
                mx = max(s for _, s in scores)
                tot = sum(math.exp(s - mx) for _, s in scores)
                lse[b, h, i] = mx + math.log(tot)
                for j, s in scores:
                    w = math.exp(s - mx) / tot
                    for c in range(v.shape[3]):
                        o[b, h, i, c] += w * v[b, kh, j, c]
    return o, lse


@pytest.mark.parametrize("bsz,hq,hkv,lq,lk,d", [
    (1, 2, 1, 4, 4, 3),
    (2, 4, 2, 3, 6, 2),   # bottom-right, delta = 3
    (1, 3, 3, 5, 5, 4),   # plain multi-head
    (1, 2, 2, 6, 3, 2),   # q_len > kv_len: the first rows see nothing
    (1, 4, 1, 1, 7, 3),   # single query row, sees every key
])
def test_brute_force_tiny(bsz, hq, hkv, lq, lk, d):
    rng = np.random.default_rng(bsz * 100 + lq * 10 + lk)
    q = rng.standard_normal((bsz, hq, lq, d))
    k = rng.standard_normal((bsz, hkv, lk, d))
    v = rng.standard_normal((bsz, hkv, lk, d))
    scale = 0.7
    o, lse = oracle.prefill(q, k, v, scale)
    ob, lb = _brute_prefill(q, k, v, scale)
    np.testing.assert_allclose(o, ob, rtol=1e-12, atol=1e-13)
    np.testing.assert_array_equal(np.isinf(lse), np.isinf(lb))
    fin = np.isfinite(lb)
    np.testing.assert_allclose(lse[fin], lb[fin], rtol=1e-12, atol=1e-13)
    if lq > lk:
        # rows with no visible key: O = 0, LSE = -inf
        dead = np.arange(lq) + (lk - lq) < 0
        assert np.all(o[:, :, dead] == 0) and np.all(lse[:, :, dead] == -np.inf)


# ---------------------------------------------------------- library check

@pytest.mark.parametrize("lq,lk", [(5, 5), (3, 9), (8, 8)])
def test_matches_torch_sdpa_with_explicit_mask(lq, lk):
    """torch's scaled_dot_product_attention in float64 on the CPU with an
    explicit boolean mask j <= i + (lk - lq) (not is_causal, which is
    top-left) and K/V heads expanded by repeat_interleave."""
    g = torch.Generator().manual_seed(7)
    bsz, hq, hkv, d = 2, 6, 2, 5
    q = torch.randn(bsz, hq, lq, d, generator=g, dtype=torch.float64)
    k = torch.randn(bsz, hkv, lk, d, generator=g, dtype=torch.float64)
    v = torch.randn(bsz, hkv, lk, d, generator=g, dtype=torch.float64)
    mask = torch.arange(lk)[None, :] <= torch.arange(lq)[:, None] + (lk - lq)
    kr = k.repeat_interleave(hq // hkv, dim=1)
    vr = v.repeat_interleave(hq // hkv, dim=1)
    ref = torch.nn.functional.scaled_dot_product_attention(q, kr, vr, attn_mask=mask, scale=0.37)
    s = (q @ kr.transpose(-1, -2)) * 0.37
    ref_lse = torch.logsumexp(s.masked_fill(~mask, float("-inf")), dim=-1)
    o, lse = oracle.prefill(q.numpy(), k.numpy(), v.numpy(), scale=0.37)
    np.testing.assert_allclose(o, ref.numpy(), rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(lse, ref_lse.numpy(), rtol=1e-12, atol=1e-12)


def test_default_scale_matches_torch_sdpa_default():
    """With no scale given, the prefill and the decode use torch's own default
    softmax scale (scaled_dot_product_attention without ``scale=``)."""
    g = torch.Generator().manual_seed(9)
    d = 16
    q = torch.randn(1, 4, 6, d, generator=g, dtype=torch.float64) * 3
    k = torch.randn(1, 2, 6, d, generator=g, dtype=torch.float64) * 3
    v = torch.randn(1, 2, 6, d, generator=g, dtype=torch.float64)
    kr, vr = k.repeat_interleave(2, dim=1), v.repeat_interleave(2, dim=1)
    mask = torch.ones(6, 6, dtype=torch.bool).tril()
    ref = torch.nn.functional.scaled_dot_product_attention(q, kr, vr, attn_mask=mask)
    o, _ = oracle.prefill(q.numpy(), k.numpy(), v.numpy())
    np.testing.assert_allclose(o, ref.numpy(), rtol=1e-12, atol=1e-12)
    # the decode: the last query row against a one-page cache of the 6 rows
    kc = k.numpy()[0].transpose(1, 0, 2)[None]       # [1 page, 6, Hkv, D]
    vc = v.numpy()[0].transpose(1, 0, 2)[None]
    od, _ = oracle.decode_unsplit(q.numpy()[:, :, -1], kc, vc, np.array([[0]]), [6], 6)
    np.testing.assert_allclose(od[0], ref.numpy()[0, :, -1], rtol=1e-12, atol=1e-12)


# ------------------------------------------------------------- invariants

def test_single_visible_key_returns_its_v_row():
    rng = np.random.default_rng(1)
    q = rng.standard_normal((1, 2, 6, 4))
    k = rng.standard_normal((1, 1, 6, 4))
    v = rng.standard_normal((1, 1, 6, 4))
    o, lse = oracle.prefill(q, k, v, scale=0.5)
    # square causal: row 0 sees only key 0
    np.testing.assert_array_equal(o[0, :, 0], np.stack([v[0, 0, 0]] * 2))
    np.testing.assert_allclose(lse[0, :, 0], 0.5 * (q[0, :, 0] @ k[0, 0, 0]), rtol=0, atol=1e-15)
    # and q_len = kv_len = 1
    o1, _ = oracle.prefill(q[:, :, :1], k[:, :, :1], v[:, :, :1])
    np.testing.assert_array_equal(o1[0, :, 0], np.stack([v[0, 0, 0]] * 2))


def test_constant_v_returns_the_constant():
    rng = np.random.default_rng(2)
    q = rng.standard_normal((2, 4, 5, 3)) * 3
    k = rng.standard_normal((2, 2, 9, 3)) * 3
    v = np.full((2, 2, 9, 3), -1.25)
    o, _ = oracle.prefill(q, k, v)
    np.testing.assert_allclose(o, -1.25, rtol=0, atol=1e-14)


def test_weight_rows_sum_to_one_and_respect_the_mask():
    """With V the identity (one column per key) O is the weight matrix."""
    rng = np.random.default_rng(3)
    lq, lk = 4, 7
    q = rng.standard_normal((1, 1, lq, 3))
    k = rng.standard_normal((1, 1, lk, 3))
    v = np.eye(lk).reshape(1, 1, lk, lk)
    p, _ = oracle.prefill(q, k, v)
    np.testing.assert_allclose(p[0, 0].sum(axis=1), 1.0, rtol=0, atol=1e-14)
    masked = ~oracle.visible_mask(lq, lk)
    assert np.all(p[0, 0][masked] == 0.0)
    assert np.all(p[0, 0][~masked] > 0.0)


def test_lse_is_a_direct_log_sum_exp():
    from scipy.special import logsumexp
    rng = np.random.default_rng(4)
    q = rng.standard_normal((1, 2, 6, 4)) * 4
    k = rng.standard_normal((1, 1, 8, 4)) * 4
    v = rng.standard_normal((1, 1, 8, 4))
    _, lse = oracle.prefill(q, k, v, scale=0.9)
    for h in range(2):
        for i in range(6):
            s = [0.9 * float(np.dot(q[0, h, i], k[0, 0, j])) for j in range(8) if j <= i + 2]
            assert abs(lse[0, h, i] - logsumexp(s)) < 1e-12


def test_gqa_equals_mha_with_repeated_heads():
    rng = np.random.default_rng(5)
    q = rng.standard_normal((2, 8, 5, 3))
    k = rng.standard_normal((2, 2, 7, 3))
    v = rng.standard_normal((2, 2, 7, 3))
    o, lse = oracle.prefill(q, k, v)
    # the repeat built by hand, head by head: q head h reads kv head h // 4
    k_mha = np.stack([k[:, h // 4] for h in range(8)], axis=1)
    v_mha = np.stack([v[:, h // 4] for h in range(8)], axis=1)
    o2, lse2 = oracle.prefill(q, k_mha, v_mha)
    np.testing.assert_array_equal(o, o2)
    np.testing.assert_array_equal(lse, lse2)


def test_prefill_rows_matches_prefill():
    rng = np.random.default_rng(6)
    q = rng.standard_normal((2, 4, 9, 3))
    k = rng.standard_normal((2, 2, 12, 3))
    v = rng.standard_normal((2, 2, 12, 3))
    o, lse = oracle.prefill(q, k, v)
    rows = [0, 4, 8]
    o2, lse2 = oracle.prefill_rows(q, k, v, 1, 3, rows)
    np.testing.assert_allclose(o2, o[1, 3, rows], rtol=1e-13, atol=1e-14)
    np.testing.assert_allclose(lse2, lse[1, 3, rows], rtol=1e-13, atol=1e-14)


# ------------------------------------------------------------------- int4

def test_int4_round_trip_of_every_code():
    """Codes 0..15 with a known fp16 scale and offset decode to exactly
    scale*code + offset (both are powers of two or short binary fractions)."""
    scale, offset = 0.375, -2.5
    s_bits = int(np.float16(scale).view(np.uint16))
    o_bits = int(np.float16(offset).view(np.uint16))
    coef = s_bits | (o_bits << 16)
    codes = list(range(16))
    words = [coef,
             sum(c << (4 * j) for j, c in enumerate(codes[:8])),
             sum(c << (4 * j) for j, c in enumerate(codes[8:]))]
    got = oracle.dequant_int4_row(words, 16, 1)
    np.testing.assert_array_equal(got, [scale * c + offset for c in codes])


def test_int4_vectorised_equals_elementwise():
    rng = np.random.default_rng(8)
    for ng in (1, 2, 4, 8):
        d = 128
        words = rng.integers(0, 2 ** 32, size=(5, ng + d // 8), dtype=np.uint64).astype(np.uint32)
        # keep the coefficient words finite fp16 numbers
        sc = np.float16(rng.uniform(0.01, 0.1, size=(5, ng))).view(np.uint16).astype(np.uint32)
        of = np.float16(rng.normal(0, 0.1, size=(5, ng))).view(np.uint16).astype(np.uint32)
        words[:, :ng] = sc | (of << 16)
        vec = oracle.dequant_int4_rows(words, d, ng)
        for r in range(5):
            np.testing.assert_array_equal(vec[r], oracle.dequant_int4_row(words[r], d, ng))


def test_int4_generator_round_trip():
    """The synthetic-input packer and the oracle's decoder agree on codes,
    scales and offsets drawn at random (int32 storage, sign bit included)."""
    from synth import pack_int4_rows
    g = torch.Generator().manual_seed(9)
    codes = torch.randint(0, 16, (3, 128), generator=g, dtype=torch.uint8)
    sc = torch.rand(3, 4, generator=g) * 0.09 + 0.01
    of = torch.randn(3, 4, generator=g) * 0.1
    sb = sc.half().view(torch.int16).to(torch.int32) & 0xFFFF
    ob = of.half().view(torch.int16).to(torch.int32) & 0xFFFF
    words = pack_int4_rows(codes, sb, ob, 4).numpy()
    got = oracle.dequant_int4_rows(words, 128, 4)
    want = (np.repeat(sc.half().double().numpy(), 32, axis=1) * codes.double().numpy()
            + np.repeat(of.half().double().numpy(), 32, axis=1))
    np.testing.assert_array_equal(got, want)


# ------------------------------------------------------------------ decode

def _decode_case(seed, lens, page_size=4, hq=4, hkv=2, d=8, kv_format="dense", ng=1):
    rng = np.random.default_rng(seed)
    n_pages = sum(-(-n // page_size) for n in lens)
    perm = rng.permutation(n_pages)
    max_pages = max(1, max(-(-n // page_size) for n in lens))
    table = np.full((len(lens), max_pages), -1, dtype=np.int64)
    cur = 0
    for b, n in enumerate(lens):
        np_b = -(-n // page_size)
        table[b, :np_b] = perm[cur:cur + np_b]
        cur += np_b
    q = rng.standard_normal((len(lens), hq, d))
    if kv_format == "dense":
        kc = rng.standard_normal((n_pages, page_size, hkv, d))
        vc = rng.standard_normal((n_pages, page_size, hkv, d))
    else:
        def pool():
            w = rng.integers(0, 2 ** 32, size=(n_pages, page_size, hkv, ng + d // 8), dtype=np.uint64)
            w = w.astype(np.uint32)
            sc = np.float16(rng.uniform(0.01, 0.1, size=w.shape[:-1] + (ng,))).view(np.uint16)
            of = np.float16(rng.normal(0, 0.1, size=w.shape[:-1] + (ng,))).view(np.uint16)
            w[..., :ng] = sc.astype(np.uint32) | (of.astype(np.uint32) << 16)
            return w
        kc, vc = pool(), pool()
    return q, kc, vc, table


@pytest.mark.parametrize("kv_format,ng", [("dense", 1), ("int4", 2)])
def test_decode_matches_dense_attention_on_gathered_rows(kv_format, ng):
    """Single-query decode equals plain attention (every key visible) over the
    logical rows rebuilt by walking each sequence page by page."""
    lens = [9, 1, 16, 5]
    ps, d = 4, 16
    q, kc, vc, table = _decode_case(11, lens, page_size=ps, d=d, kv_format=kv_format, ng=ng)
    o, lse = oracle.decode_unsplit(q, kc, vc, table, lens, ps, scale=0.3, kv_format=kv_format, n_groups=ng)
    for b, n in enumerate(lens):
        rows_k = [kc[table[b, t // ps], t % ps] for t in range(n)]
        rows_v = [vc[table[b, t // ps], t % ps] for t in range(n)]
        if kv_format == "int4":
            rows_k = [np.stack([oracle.dequant_int4_row(r[h], d, ng) for h in range(2)]) for r in rows_k]
            rows_v = [np.stack([oracle.dequant_int4_row(r[h], d, ng) for h in range(2)]) for r in rows_v]
        kk = np.stack(rows_k)[None].transpose(0, 2, 1, 3)   # [1, Hkv, n, D]
        vv = np.stack(rows_v)[None].transpose(0, 2, 1, 3)
        ob, lb = _brute_prefill(q[b][None, :, None, :], kk, vv, 0.3)
        np.testing.assert_allclose(o[b], ob[0, :, 0], rtol=1e-12, atol=1e-13)
        np.testing.assert_allclose(lse[b], lb[0, :, 0], rtol=1e-12, atol=1e-13)


def test_merge_of_any_split_partition_equals_unsplit():
    lens = [23, 0, 7, 64, 1]
    q, kc, vc, table = _decode_case(12, lens, page_size=4)
    ou, lu = oracle.decode_unsplit(q, kc, vc, table, lens, 4)
    for split in (1, 4, 5, 8, 64, 1000):
        o, lse = oracle.decode(q, kc, vc, table, lens, 4, split, max_kv_len=max(lens) + 17)
        np.testing.assert_allclose(o, ou, rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(lse[np.isfinite(lu)], lu[np.isfinite(lu)], rtol=1e-12, atol=1e-12)
        assert np.all(lse[1] == -np.inf) and np.all(o[1] == 0)
    # an arbitrary, uneven partition of [0, len) merged by hand-built partials
    rng = np.random.default_rng(13)
    b, n = 3, 64
    cuts = sorted(set(rng.integers(0, n, size=6).tolist()) | {0, n})
    cuts = [0, 0] + cuts     # an empty part too
    parts_o, parts_l = [], []
    krows = oracle.gather_paged_rows(kc, table, b, 0, n, 4)
    vrows = oracle.gather_paged_rows(vc, table, b, 0, n, 4)
    for lo, hi in zip(cuts[:-1], cuts[1:]):
        o_s, l_s = oracle.attend(q[b, :1], krows[lo:hi, 0], vrows[lo:hi, 0],
                                 np.ones((1, hi - lo), dtype=bool), 1 / math.sqrt(8))
        parts_o.append(o_s[0])
        parts_l.append(l_s[0])
    om, lm = oracle.lse_merge(np.stack(parts_o)[None], np.array(parts_l)[None])
    np.testing.assert_allclose(om[0], ou[b, 0], rtol=1e-12, atol=1e-12)
    assert abs(lm[0] - lu[b, 0]) < 1e-12


def test_merge_lse_is_logsumexp_of_split_lses():
    from scipy.special import logsumexp
    rng = np.random.default_rng(14)
    lse = rng.standard_normal((6, 5)) * 4
    lse[2, 1:] = -np.inf
    o = rng.standard_normal((6, 5, 3))
    _, lm = oracle.lse_merge(o, lse)
    np.testing.assert_allclose(lm, logsumexp(lse, axis=1), rtol=0, atol=1e-13)


def test_empty_split_partials_are_zero_and_minus_inf():
    lens = [5, 12]
    q, kc, vc, table = _decode_case(15, lens, page_size=4)
    o_p, l_p = oracle.decode_split_partials(q, kc, vc, table, lens, 4, 4)
    assert o_p.shape[2] == 3
    # sequence 0 has 2 non-empty splits, the third is empty
    assert np.all(l_p[0, :, 2] == -np.inf) and np.all(o_p[0, :, 2] == 0)
    assert np.all(np.isfinite(l_p[1]))


# -------------------------------------------------------- planted mistakes

def test_planted_top_left_mask_is_caught(monkeypatch, golden):
    """A top-left causal mask (the other convention on the pages) fails the
    bottom-right fixture."""
    def top_left(q_len, kv_len, rows=None):
        i = np.arange(q_len) if rows is None else np.asarray(rows)
        return np.arange(kv_len)[None, :] <= i[:, None]
    monkeypatch.setattr(oa, "visible_mask", top_left)
    with pytest.raises(AssertionError):
        test_golden_uniform_scores_bottom_right(golden)


def test_planted_base2_lse_is_caught(monkeypatch, golden):
    """An LSE in base 2 (another convention on the pages) fails the fixture."""
    real_log = np.log
    monkeypatch.setattr(oa.np, "log", lambda x: real_log(x) / math.log(2))
    try:
        with pytest.raises(AssertionError):
            test_golden_two_key_softmax(golden)
    finally:
        monkeypatch.undo()


def test_planted_wrong_nibble_order_is_caught(monkeypatch, golden):
    """Reading the high nibble first fails the int4 fixture."""
    real = oa.dequant_int4_row

    def reversed_nibbles(words, d, ng):
        words = list(words)
        flipped = []
        for i, w in enumerate(words):
            if i < ng:
                flipped.append(w)
            else:
                w = int(np.uint32(np.int64(w) & 0xFFFFFFFF))
                flipped.append(sum(((w >> (4 * j)) & 0xF) << (4 * (7 - j)) for j in range(8)))
        return real(flipped, d, ng)
    monkeypatch.setattr(oracle, "dequant_int4_row", reversed_nibbles)
    with pytest.raises(AssertionError):
        g = golden("int4_rows.txt")
        words = [int(x, 16) for x in g["rowA_words"]]
        np.testing.assert_array_equal(oracle.dequant_int4_row(words, 8, 1), _f(g["rowA_values"]))


def test_planted_wrong_gqa_map_is_caught(monkeypatch):
    """Mapping query head h to kv head h % Hkv (interleaved) fails the
    library cross-check's head repeat."""
    rng = np.random.default_rng(16)
    q = rng.standard_normal((1, 4, 3, 2))
    k = rng.standard_normal((1, 2, 3, 2))
    v = rng.standard_normal((1, 2, 3, 2))
    o, _ = oracle.prefill(q, k, v)
    real_repeat = np.repeat
    monkeypatch.setattr(oa.np, "repeat", lambda a, r, axis=None: np.tile(a, [r if i == axis else 1
                                                                               for i in range(a.ndim)])
                        if axis == 1 else real_repeat(a, r, axis=axis))
    o_bad, _ = oracle.prefill(q, k, v)
    monkeypatch.undo()
    qt = torch.from_numpy(q)
    kr = torch.from_numpy(k).repeat_interleave(2, dim=1)
    vr = torch.from_numpy(v).repeat_interleave(2, dim=1)
    mask = torch.ones(3, 3, dtype=torch.bool).tril()
    ref = torch.nn.functional.scaled_dot_product_attention(qt, kr, vr, attn_mask=mask).numpy()
    np.testing.assert_allclose(o, ref, rtol=1e-12, atol=1e-12)
    assert not np.allclose(o_bad, ref)


# ------------------------------------------------------------ merge backward

def test_merge_bwd_matches_finite_differences_of_the_merge():
    """Central differences of the (pinned) forward merge, in fp64."""
    rng = np.random.default_rng(21)
    n, s, d = 3, 4, 5
    o_part = rng.standard_normal((n, s, d))
    lse_part = rng.standard_normal((n, s)) * 2
    lse_part[1, 2] = -np.inf
    d_o = rng.standard_normal((n, d))
    d_lse = rng.standard_normal(n)
    g_o, g_l = oracle.lse_merge_bwd(o_part, lse_part, d_o, d_lse)

    def loss(op, lp):
        o, lse = oracle.lse_merge(op, lp)
        return float((o * d_o).sum() + (lse * d_lse).sum())
    h = 1e-6
    for idx in [(0, 0, 0), (1, 3, 4), (2, 1, 2), (1, 2, 0)]:
        op1, op2 = o_part.copy(), o_part.copy()
        op1[idx] += h
        op2[idx] -= h
        fd = (loss(op1, lse_part) - loss(op2, lse_part)) / (2 * h)
        assert abs(fd - g_o[idx]) < 1e-7
    for idx in [(0, 0), (0, 3), (2, 1), (1, 1)]:
        lp1, lp2 = lse_part.copy(), lse_part.copy()
        lp1[idx] += h
        lp2[idx] -= h
        fd = (loss(o_part, lp1) - loss(o_part, lp2)) / (2 * h)
        assert abs(fd - g_l[idx]) < 1e-7
    # the empty split carries no gradient
    assert g_l[1, 2] == 0 and np.all(g_o[1, 2] == 0)


def test_merge_bwd_matches_torch_autograd():
    rng = np.random.default_rng(22)
    o_part = torch.from_numpy(rng.standard_normal((6, 3, 8))).requires_grad_(True)
    lse_part = torch.from_numpy(rng.standard_normal((6, 3)) * 3).requires_grad_(True)
    lse = torch.logsumexp(lse_part, dim=-1)
    o = (torch.softmax(lse_part, dim=-1)[..., None] * o_part).sum(dim=1)
    d_o = torch.from_numpy(rng.standard_normal((6, 8)))
    d_lse = torch.from_numpy(rng.standard_normal(6))
    ((o * d_o).sum() + (lse * d_lse).sum()).backward()
    g_o, g_l = oracle.lse_merge_bwd(o_part.detach().numpy(), lse_part.detach().numpy(), d_o.numpy(), d_lse.numpy())
    np.testing.assert_allclose(g_o, o_part.grad.numpy(), rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(g_l, lse_part.grad.numpy(), rtol=1e-12, atol=1e-12)


def test_merge_bwd_all_empty_row_and_missing_dlse():
    o_part = np.ones((2, 2, 3))
    lse_part = np.array([[-np.inf, -np.inf], [0.0, 0.0]])
    g_o, g_l = oracle.lse_merge_bwd(o_part, lse_part, np.ones((2, 3)))
    assert np.all(g_o[0] == 0) and np.all(g_l[0] == 0)
    # two equal splits: each weight 1/2; O_s == O so the dLSE term vanishes
    np.testing.assert_allclose(g_o[1], 0.5)
    np.testing.assert_allclose(g_l[1], 0.0)


# ----------------------------------------------------- multi-query decode

def test_multi_query_decode_equals_prefill_over_the_gathered_sequence():
    """q_len queries against a paged cache of len tokens are the last q_len
    rows of a causal prefill with kv_len = len (bottom-right alignment);
    checked with the scalar brute force on the gathered rows."""
    lens = [9, 3, 16]
    ps, d, nq = 4, 8, 3
    qd, kc, vc, table = _decode_case(31, lens, page_size=ps, d=d)
    rng = np.random.default_rng(32)
    q = rng.standard_normal((len(lens), 4, nq, d))
    for split in (4, 5, 100):
        o, lse = oracle.decode_mq(q, kc, vc, table, lens, ps, split, scale=0.4)
        for b, n in enumerate(lens):
            kk = oracle.gather_paged_rows(kc, table, b, 0, n, ps).transpose(1, 0, 2)[None]   # [1, Hkv, n, D]
            vv = oracle.gather_paged_rows(vc, table, b, 0, n, ps).transpose(1, 0, 2)[None]
            ob, lb = _brute_prefill(q[b][None], kk, vv, 0.4)
            np.testing.assert_allclose(o[b], ob[0], rtol=1e-12, atol=1e-12)
            fin = np.isfinite(lb[0])
            np.testing.assert_allclose(lse[b][fin], lb[0][fin], rtol=1e-12, atol=1e-12)
            assert np.array_equal(np.isinf(lse[b]), np.isinf(lb[0]))


def test_multi_query_decode_with_one_query_is_single_query_decode():
    lens = [7, 12]
    qd, kc, vc, table = _decode_case(33, lens, page_size=4, d=8)
    o1, l1 = oracle.decode(qd, kc, vc, table, lens, 4, 5)
    o2, l2 = oracle.decode_mq(qd[:, :, None, :], kc, vc, table, lens, 4, 5)
    np.testing.assert_array_equal(o2[:, :, 0], o1)
    np.testing.assert_array_equal(l2[:, :, 0], l1)


# ------------------------------------------------------------------- fp8

def test_golden_fp8_e4m3(golden):
    g = golden("fp8_e4m3.txt")
    vals = [oracle.fp8_e4m3_value(int(x, 16)) for x in g["bytes"]]
    np.testing.assert_array_equal(vals, _f(g["values"]))
    row = oracle.dequant_fp8_rows(np.array([[int(x, 16) for x in g["row_bytes"]]]),
                                  np.array([int(g["row_word"][0], 16)]))
    np.testing.assert_array_equal(row[0], _f(g["row_values"]))


def test_fp8_decoder_matches_torch_float8_e4m3fn():
    """Every byte against torch's float8_e4m3fn (a library decoder)."""
    b = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = b.view(torch.float8_e4m3fn).double().numpy()
    ours = np.array([oracle.fp8_e4m3_value(x) for x in range(256)])
    nan = np.isnan(ref)
    assert np.array_equal(nan, np.isnan(ours)) and nan.sum() == 2    # 0x7F and 0xFF
    np.testing.assert_array_equal(ours[~nan], ref[~nan])


def test_fp8_decode_equals_dense_decode_on_dequantised_rows():
    lens = [9, 14]
    ps, d = 4, 8
    rng = np.random.default_rng(41)
    n_pages = sum(-(-n // ps) for n in lens)
    table = np.array([[0, 1, 2, -1], [3, 4, 5, 6]])
    codes_k = rng.integers(0, 256, size=(n_pages, ps, 2, d))
    codes_v = rng.integers(0, 256, size=(n_pages, ps, 2, d))
    codes_k[(codes_k & 0x7F) == 0x7F] = 0       # no NaN bytes
    codes_v[(codes_v & 0x7F) == 0x7F] = 0
    def words():
        sc = np.float16(rng.uniform(0.1, 0.5, size=(n_pages, ps, 2))).view(np.uint16).astype(np.int64)
        sh = np.float16(rng.normal(0, 0.1, size=(n_pages, ps, 2))).view(np.uint16).astype(np.int64)
        return sc | (sh << 16)
    wk, wv = words(), words()
    q = rng.standard_normal((2, 4, d))
    o, lse = oracle.decode(q, codes_k, codes_v, table, lens, ps, 5, kv_format="fp8", k_scale_shift=wk,
                           v_scale_shift=wv)
    kd = oracle.dequant_fp8_rows(codes_k, wk)
    vd = oracle.dequant_fp8_rows(codes_v, wv)
    o2, lse2 = oracle.decode(q, kd, vd, table, lens, ps, 5)
    np.testing.assert_allclose(o, o2, rtol=1e-13, atol=1e-13)
    np.testing.assert_allclose(lse, lse2, rtol=1e-13, atol=1e-13)


def test_fp8_unsplit_decode_against_brute_force_on_torch_decoded_rows():
    """decode_unsplit over an fp8 cache equals brute-force attention over rows
    rebuilt page by page, each byte decoded by torch's float8_e4m3fn and
    mapped by its row's fp16 scale and shift (a decoder independent of the
    oracle's own table)."""
    lens = [9, 14, 1]
    ps, d, hkv = 4, 8, 2
    rng = np.random.default_rng(43)
    n_pages = sum(-(-n // ps) for n in lens)
    perm = rng.permutation(n_pages)
    table = np.full((3, 4), -1, dtype=np.int64)
    cur = 0
    for b, n in enumerate(lens):
        table[b, :-(-n // ps)] = perm[cur:cur - (-n // ps)]
        cur += -(-n // ps)
    codes = [rng.integers(0, 256, size=(n_pages, ps, hkv, d)) for _ in range(2)]
    for c in codes:
        c[(c & 0x7F) == 0x7F] = 0                 # no NaN bytes
    words = []
    for _ in range(2):
        sc = np.float16(rng.uniform(0.1, 0.5, size=(n_pages, ps, hkv))).view(np.uint16).astype(np.int64)
        sh = np.float16(rng.normal(0, 0.1, size=(n_pages, ps, hkv))).view(np.uint16).astype(np.int64)
        words.append(sc | (sh << 16))
    q = rng.standard_normal((3, 4, d))
    o, lse = oracle.decode_unsplit(q, codes[0], codes[1], table, lens, ps, scale=0.4, kv_format="fp8",
                                   k_scale_shift=words[0], v_scale_shift=words[1])

    def rows(c, w, b, n):
        out = []
        for t in range(n):
            pg, sl = table[b, t // ps], t % ps
            x = torch.tensor(c[pg, sl].astype(np.uint8)).view(torch.float8_e4m3fn).double().numpy()
            sc = np.float64(np.uint16(w[pg, sl] & 0xFFFF).view(np.float16))
            sh = np.float64(np.uint16(w[pg, sl] >> 16).view(np.float16))
            out.append(x * sc[:, None] + sh[:, None])
        return np.stack(out)[None].transpose(0, 2, 1, 3)          # [1, Hkv, n, D]
    for b, n in enumerate(lens):
        kk, vv = rows(codes[0], words[0], b, n), rows(codes[1], words[1], b, n)
        ob, lb = _brute_prefill(q[b][None, :, None, :], kk, vv, 0.4)
        np.testing.assert_allclose(o[b], ob[0, :, 0], rtol=1e-12, atol=1e-13)
        np.testing.assert_allclose(lse[b], lb[0, :, 0], rtol=1e-12, atol=1e-13)


# ------------------------------------------------------- varlen paged prefill

@pytest.mark.parametrize("page_size", [1, 3])
def test_varlen_paged_prefill_equals_dense_prefill_per_sequence(page_size):
    """Each sequence of the ragged batch is the (pinned) dense causal prefill
    of its own Q against its gathered K/V (bottom-right, delta = kv - q)."""
    from synth import VarlenShape, varlen_inputs
    shape = VarlenShape("t", 3, 4, 2, 8, 1, 1, 0, 0, page_size=page_size)
    inp = varlen_inputs(shape, seed=3, q_lens=[5, 1, 7], kv_lens=[9, 4, 7])
    o, lse = oracle.prefill_paged_varlen(inp["q"].double().numpy(), inp["k_cache"].double().numpy(),
                                         inp["v_cache"].double().numpy(), inp["qo_indptr"].numpy(),
                                         inp["kv_indptr"].numpy(), inp["kv_indices"].numpy(), page_size,
                                         inp["kv_last_page_len"].numpy(), scale=0.3)
    qo, kvp, idx = inp["qo_indptr"].tolist(), inp["kv_indptr"].tolist(), inp["kv_indices"].tolist()
    for b in range(3):
        ql, kl = inp["q_lens"][b], inp["kv_lens"][b]
        pages = idx[kvp[b]:kvp[b + 1]]
        kk = np.stack([inp["k_cache"][pages[t // page_size], t % page_size].double().numpy() for t in range(kl)])
        vv = np.stack([inp["v_cache"][pages[t // page_size], t % page_size].double().numpy() for t in range(kl)])
        qb = inp["q"][qo[b]:qo[b + 1]].double().numpy().transpose(1, 0, 2)[None]     # [1, Hq, q, D]
        ob, lb = _brute_prefill(qb, kk.transpose(1, 0, 2)[None], vv.transpose(1, 0, 2)[None], 0.3)
        np.testing.assert_allclose(o[qo[b]:qo[b + 1]], ob[0].transpose(1, 0, 2), rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(lse[qo[b]:qo[b + 1]], lb[0].T, rtol=1e-12, atol=1e-12)


# ------------------------------------------- more planted mistakes, one each

def test_planted_default_scale_of_one_over_d_is_caught(monkeypatch):
    """A default scale of 1/D instead of 1/sqrt(D) fails the library default."""
    monkeypatch.setattr(oa, "_default_scale", lambda d: 1.0 / d)
    with pytest.raises(AssertionError):
        test_default_scale_matches_torch_sdpa_default()


def test_planted_strict_causal_mask_is_caught(monkeypatch):
    """A mask that hides the diagonal (j < i + delta) fails the brute force."""
    def strict(q_len, kv_len, rows=None):
        i = np.arange(q_len) if rows is None else np.asarray(rows)
        return np.arange(kv_len)[None, :] < i[:, None] + (kv_len - q_len)
    monkeypatch.setattr(oa, "visible_mask", strict)
    with pytest.raises(AssertionError):
        test_brute_force_tiny(2, 4, 2, 3, 6, 2)


def test_planted_k_in_place_of_v_is_caught(monkeypatch):
    """Weighting the key rows instead of the value rows fails the brute force."""
    real = oa.attend
    monkeypatch.setattr(oa, "attend", lambda q, k, v, mask, scale: real(q, k, k, mask, scale))
    with pytest.raises(AssertionError):
        test_brute_force_tiny(1, 2, 1, 4, 4, 3)


def test_planted_merge_weights_of_the_wrong_sign_are_caught(monkeypatch, golden):
    """Weights proportional to exp(-LSE_s) fail the merge fixture."""
    real = oracle.lse_merge
    monkeypatch.setattr(oracle, "lse_merge", lambda o, lse: real(o, -np.asarray(lse)))
    with pytest.raises(AssertionError):
        test_golden_merge_two_splits(golden)


def test_planted_page_and_slot_swapped_are_caught(monkeypatch, golden):
    """Taking the page from t % page_size and the slot from t // page_size
    fails the block-table fixture."""
    def swapped(block_table, b, t, page_size):
        return int(block_table[b][t % page_size]) * page_size + t // page_size
    monkeypatch.setattr(oracle, "paged_row_index", swapped)
    with pytest.raises(AssertionError):
        test_golden_block_table(golden)


def test_planted_gather_without_the_block_table_is_caught(monkeypatch):
    """Reading logical page t // page_size as if it were the physical page
    fails the decode's page-by-page brute force."""
    def no_table(cache, block_table, b, t_lo, t_hi, page_size):
        rows = [np.asarray(cache[t // page_size, t % page_size]) for t in range(t_lo, t_hi)]
        return np.stack(rows) if rows else np.zeros((0,) + tuple(cache.shape[2:]))
    monkeypatch.setattr(oa, "gather_paged_rows", no_table)
    with pytest.raises(AssertionError):
        test_decode_matches_dense_attention_on_gathered_rows("dense", 1)


def test_planted_one_split_short_is_caught(monkeypatch):
    """One split too few drops the tail of the longest sequence and fails the
    multi-query brute force."""
    real = oa.num_splits
    monkeypatch.setattr(oa, "num_splits", lambda n, s: max(1, real(n, s) - 1))
    with pytest.raises(AssertionError):
        test_multi_query_decode_equals_prefill_over_the_gathered_sequence()


def test_planted_fp8_exponent_bias_of_eight_is_caught(monkeypatch, golden):
    """An e4m3 decoder with exponent bias 8 fails the fp8 fixture."""
    real = oracle.fp8_e4m3_value
    monkeypatch.setattr(oracle, "fp8_e4m3_value", lambda b: real(b) / 2)
    with pytest.raises(AssertionError):
        test_golden_fp8_e4m3(golden)


def test_planted_merge_bwd_without_the_output_term_is_caught(monkeypatch):
    """Dropping sum_d (O_s - O)_d dO_d from dLSE_s fails torch autograd."""
    real = oracle.lse_merge_bwd

    def dropped(o_part, lse_part, d_o, d_lse=None):
        g_o, _ = real(o_part, lse_part, d_o, d_lse)
        _, g_l = real(o_part, lse_part, np.zeros_like(np.asarray(d_o)), d_lse)
        return g_o, g_l
    monkeypatch.setattr(oracle, "lse_merge_bwd", dropped)
    with pytest.raises(AssertionError):
        test_merge_bwd_matches_torch_autograd()


def test_planted_varlen_full_last_page_is_caught(monkeypatch):
    """Treating every last page as full fails the ragged prefill's per-sequence
    brute force on a cache of page size 3 (kv lengths 4 and 7 end mid-page)."""
    real = oracle.prefill_paged_varlen

    def full_pages(q, k_cache, v_cache, qo_indptr, kv_indptr, kv_indices, page_size=1,
                   kv_last_page_len=None, scale=None):
        return real(q, k_cache, v_cache, qo_indptr, kv_indptr, kv_indices, page_size, None, scale)
    monkeypatch.setattr(oracle, "prefill_paged_varlen", full_pages)
    with pytest.raises(AssertionError):
        test_varlen_paged_prefill_equals_dense_prefill_per_sequence(3)
