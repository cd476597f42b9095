"""Host checks of the number encodings the int4 and fp8 decode kernels rely on.

The int4 kernel never materialises dequantised K/V.  It builds tensor-core
operands whose values are the codes shifted into an exact range ("code
space"), and applies each group's affine map (value = scale * code + offset,
"splitk_kernels.py", dequantize) outside the MMA.  These tests pin, from the
IEEE binary16 / bfloat16 formats and CUDA's documented __byte_perm selector,
that the encodings are exact and that the per-group corrections recover the
dequantised products.  They read no kernel and no oracle code.
"""

import numpy as np


def f16(bits):
    return np.asarray(bits, dtype=np.uint16).view(np.float16).astype(np.float64)


def bf16(bits):
    return (np.asarray(bits, dtype=np.uint32) << 16).view(np.float32).astype(np.float64)


def byte_perm(x, y, s):
    """__byte_perm(x, y, s): result byte i is byte (s >> 4i) & 7 of the
    little-endian 8-byte value y:x (bytes 0-3 from x, 4-7 from y)."""
    src = [(x >> (8 * i)) & 0xFF for i in range(4)] + [(y >> (8 * i)) & 0xFF for i in range(4)]
    return sum(src[(s >> (4 * i)) & 7] << (8 * i) for i in range(4))


CODES = np.arange(16)


def test_bf16_score_codes_are_exact():
    """OR-ing a code into the bits of bf16 128.0 (0x4300) gives exactly 128 + c."""
    assert bf16(0x4300) == 128.0
    np.testing.assert_array_equal(bf16(0x4300 | CODES), 128.0 + CODES)


def test_fp16_value_codes_are_exact():
    """A code in bits 0-3 of fp16 1024.0 (0x6400) gives 1024 + c; one in bits
    4-7 gives 1024 + 16 c.  Both stay within the 10 mantissa bits."""
    assert f16(0x6400) == 1024.0
    np.testing.assert_array_equal(f16(0x6400 | CODES), 1024.0 + CODES)
    np.testing.assert_array_equal(f16(0x6400 | (CODES << 4)), 1024.0 + 16 * CODES)


def test_bf16_cannot_take_a_code_in_bits_4_to_7():
    """Why the score side shifts instead: in bf16 bit 7 is the exponent's
    lowest bit, so codes of 8 or more in bits 4-7 change the exponent."""
    vals = bf16(0x4300 | (CODES << 4))
    assert not np.array_equal(vals, 128.0 + 16 * CODES)


def test_upper_bytes_permute_moves_codes_2_and_3_down():
    """Selector 0x4341 puts byte 1 of x in byte 0 and byte 3 in byte 2, with
    zeros above, so codes 2 and 3 of each 16-bit half land in bits 0-3 and
    4-7, where the fp16 masks above take them."""
    rng = np.random.default_rng(0)
    for x in rng.integers(0, 2**32, size=200, dtype=np.uint64).tolist():
        y = byte_perm(x, 0, 0x4341)
        assert y == ((x >> 8) & 0xFF) | (((x >> 24) & 0xFF) << 16)
        for half in range(2):
            h_in = (x >> (16 * half)) & 0xFFFF
            h_out = (y >> (16 * half)) & 0xFFFF
            assert h_out & 0xF == (h_in >> 8) & 0xF          # code 2
            assert (h_out >> 4) & 0xF == (h_in >> 12) & 0xF  # code 3
            assert h_out >> 8 == 0


def test_byte_perm_pairs_tokens_in_one_register():
    """Selectors 0x5410 and 0x7632 take the low and the high halves of two
    words into one register, so the two tokens' codes share a 32-bit word."""
    a, b = 0x89ABCDEF, 0x01234567
    assert byte_perm(a, b, 0x5410) == (a & 0xFFFF) | ((b & 0xFFFF) << 16)
    assert byte_perm(a, b, 0x7632) == (a >> 16) | ((b >> 16) << 16)


def test_score_side_affine_terms_recover_the_dequantised_dot_product():
    """sum_g scale_g * sum_d q (128 + c) + (offset_g - 128 scale_g) * Qsum_g
    equals q . (scale * c + offset) for every group split."""
    rng = np.random.default_rng(1)
    d = 128
    for n_groups in (1, 2, 4, 8):
        q = rng.standard_normal(d)
        c = rng.integers(0, 16, d)
        scale = rng.uniform(0.01, 0.1, n_groups)
        off = rng.normal(0, 0.1, n_groups)
        e = d // n_groups
        direct = sum(q[g * e:(g + 1) * e] @ (scale[g] * c[g * e:(g + 1) * e] + off[g]) for g in range(n_groups))
        coded = 0.0
        for g in range(n_groups):
            qg, cg = q[g * e:(g + 1) * e], c[g * e:(g + 1) * e]
            t = qg @ bf16(0x4300 | cg)
            coded += scale[g] * t + (off[g] - 128 * scale[g]) * qg.sum()
        assert abs(coded - direct) < 1e-9 * max(1.0, abs(direct))


def test_value_side_corrections_recover_the_weighted_codes_exactly():
    """With w = fp16(p * scale) as the MMA sees it, SP = sum w and
    OFF = sum p * offset:
      sigma 1 rows:  sum w (1024 + c) - 1024 SP + OFF,
      sigma 16 rows: sum w (1024 + 16 c) / 16 - 64 SP + OFF,
    both equal sum w c + OFF, and sum p (scale c + offset) up to the fp16
    rounding of w."""
    rng = np.random.default_rng(2)
    t = 2368
    p = rng.uniform(0, 1, t)
    scale = rng.uniform(0.01, 0.1, t)
    off = rng.normal(0, 0.1, t)
    c = rng.integers(0, 16, t)
    w = (p * scale).astype(np.float16).astype(np.float64)
    sp, off_sum = w.sum(), (p * off).sum()
    want = (w * c).sum() + off_sum
    lo = (w * f16(0x6400 | c)).sum() - 1024 * sp + off_sum
    hi = (w * f16(0x6400 | (c << 4))).sum() / 16 - 64 * sp + off_sum
    assert abs(lo - want) < 1e-9 * abs(want) and abs(hi - want) < 1e-9 * abs(want)
    exact = (p * (scale * c + off)).sum()
    assert abs(want - exact) < 2.0 ** -11 * (p * scale * c).sum() + 1e-12


def test_fp8_e4m3_values_are_exact_in_fp16():
    """Every finite e4m3 value (3 mantissa bits, exponents -9 to 8 with
    subnormals) is an fp16 value, so the conversion to f16x2 is exact."""
    vals = []
    for b in range(256):
        s, e, m = b >> 7, (b >> 3) & 0xF, b & 7
        if e == 0xF and m == 7:
            continue                      # NaN
        v = (m / 8) * 2.0 ** -6 if e == 0 else (1 + m / 8) * 2.0 ** (e - 7)
        vals.append(-v if s else v)
    vals = np.array(vals)
    np.testing.assert_array_equal(vals.astype(np.float16).astype(np.float64), vals)
    assert np.abs(vals).max() == 448.0
