"""Pins for the oracle's two-word activation codes (lane page: a code that
crosses the array in two words is a signed high byte weighted by 256 and an
unsigned low byte; numerics page: Words).

Checked without trusting the oracle's two-word code: the lane page's per-word
delivery in excess form (an independent formulation of the same sums),
exact-rational dequantise-then-dot on small inputs, and the one-word product
for codes that fit one word.
"""
from fractions import Fraction

import numpy as np
import pytest

from block_quantized_weight_quantize_gb300 import synth
from test_oracle_pins import bits, round_f32_grid_then_flush

FMTS = [synth.FMT_Q8_0, synth.FMT_Q4K, synth.FMT_Q6K]


def _codes16(rng, ncols, K):
    """16-bit codes over the whole range, with the word boundaries and the
    extremes planted."""
    a = rng.integers(-32768, 32768, (ncols, K)).astype(np.int16)
    special = np.array([-32768, 32767, -1, 0, 1, 255, 256, -256, -255, 127, -128, 128], np.int16)
    a[0, :len(special)] = special
    if ncols > 1:
        a[1, :] = -32768
    if ncols > 2:
        a[2, :] = 32767
    return a


@pytest.mark.parametrize("fmt", FMTS)
def test_two_word_delivery_matches_direct_sums(orc, fmt):
    """Per unit, the high word in excess form (P' - 128Q - zS' + 2048z, weighted
    by 256) plus the low byte (P' - zS') gives the same block sums as taking
    sum coef*a and sum offs*a element by element (lane page, opening
    description, WordSums)."""
    rng = np.random.default_rng(60 + fmt)
    rows, K = 5, 512
    lg = synth.draw(fmt, rng, rows, K)
    if fmt == synth.FMT_Q4K:
        lg["q"][0, :] = 15; lg["sc"][0, :] = 63; lg["mn"][0, :] = 63      # the largest coefficients
    if fmt == synth.FMT_Q6K:
        lg["q"][0, :] = 0; lg["sc"][0, :] = -128                           # coefficient 4096
    if fmt == synth.FMT_Q8_0:
        lg["q"][0, :] = -127
    W = synth.pack(fmt, lg)
    a = _codes16(rng, 4, K)
    nb = K // synth.BLOCK[fmt]
    C, O, _ = orc.block_values_w2(fmt, W, rows, K, a, np.full((4, nb), 128, np.uint8), np.zeros((4, nb), np.int16))
    Ce, Oe = orc.block_sums_excess_w2(fmt, W, rows, K, a)
    assert np.array_equal(C, Ce) and np.array_equal(O, Oe)
    if fmt == synth.FMT_Q6K:
        assert C[1, 0, 0] == 4096 * -32768 * 256          # the largest magnitude a block sum takes


@pytest.mark.parametrize("fmt", FMTS)
def test_one_word_codes_give_the_one_word_product(orc, fmt):
    """Codes within -127..127 cross in one word; as two-word codes (high byte
    0 or -1) they must give the one-word product bit for bit."""
    rng = np.random.default_rng(70 + fmt)
    rows, K = 9, 1024
    lg = synth.draw(fmt, rng, rows, K)
    W = synth.pack(fmt, lg)
    x = synth.draw_act(rng, 3, K, outlier_frac=0.01)
    codes, m, e, _ = orc.quantize_blocks(x, synth.BLOCK[fmt])
    C1, O1, v1 = orc.block_values(fmt, W, rows, K, codes, m, e)
    C2, O2, v2 = orc.block_values_w2(fmt, W, rows, K, codes.astype(np.int16), m, e)
    assert np.array_equal(C1, C2) and np.array_equal(O1, O2) and np.array_equal(bits_arr(v1), bits_arr(v2))
    g1 = orc.gemv(fmt, W, rows, K, codes, m, e)
    g2 = orc.gemv_w2(fmt, W, rows, K, codes.astype(np.int16), m, e)
    assert np.array_equal(bits_arr(g1), bits_arr(g2))


def bits_arr(a):
    return np.ascontiguousarray(a, np.float32).view(np.uint32)


def _exact_value16(fmt, lg, r, b, a, m, e):
    f16 = lambda hb: Fraction(float(np.uint16(hb).view(np.float16)))
    s_a = Fraction(int(m)) * Fraction(2) ** int(e)
    X = Fraction(0)
    if fmt == synth.FMT_Q8_0:
        d = f16(lg["d"][r, b])
        for i in range(32):
            X += d * int(lg["q"][r, 32 * b + i]) * int(a[32 * b + i])
    elif fmt == synth.FMT_Q4K:
        d, dm = f16(lg["d"][r, b]), f16(lg["dmin"][r, b])
        for i in range(256):
            s = 8 * b + i // 32
            w = d * int(lg["sc"][r, s]) * int(lg["q"][r, 256 * b + i]) - dm * int(lg["mn"][r, s])
            X += w * int(a[256 * b + i])
    else:
        d = f16(lg["d"][r, b])
        for i in range(256):
            w = d * int(lg["sc"][r, 16 * b + i // 16]) * (int(lg["q"][r, 256 * b + i]) - 32)
            X += w * int(a[256 * b + i])
    return round_f32_grid_then_flush(X * s_a)


@pytest.mark.parametrize("fmt", FMTS)
def test_two_word_values_brute_force(orc, fmt):
    """Every block value bit for bit against exact-rational dequantise-then-dot
    with 16-bit codes, rounded once; rows as the in-order f32 fold of those
    values (numerics page, dot)."""
    rng = np.random.default_rng(80 + fmt)
    rows, K = 2, 512
    kw = {"d_range": (1e-7, 1e-1)} if fmt == synth.FMT_Q4K else {}
    lg = synth.draw(fmt, rng, rows, K, **kw)
    W = synth.pack(fmt, lg)
    a = _codes16(rng, 3, K)
    nb = K // synth.BLOCK[fmt]
    m = rng.integers(128, 256, (3, nb)).astype(np.uint8)
    e = rng.integers(-40, -10, (3, nb)).astype(np.int16)
    _, _, v = orc.block_values_w2(fmt, W, rows, K, a, m, e)
    out = orc.gemv_w2(fmt, W, rows, K, a, m, e)
    for c in range(3):
        for r in range(rows):
            acc = np.float32(0)
            for b in range(nb):
                ref = _exact_value16(fmt, lg, r, b, a[c], m[c, b], e[c, b])
                assert bits(v[c, r, b]) == ref, (c, r, b)
                s = np.float32(acc + np.uint32(ref).view(np.float32))
                acc = np.float32(0) if abs(float(s)) < 2.0 ** -126 else s   # ftz
            assert bits(out[c, r]) == bits(acc), (c, r)
