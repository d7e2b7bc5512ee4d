"""Pins of the oracle's ActScaling::Sub32 path against what the pages and the
mathematics fix: block_scale's minimality (numerics page, block_scale),
rne_div's nearest-ties-even codes per 32 elements (numerics page, quantize,
ACT_BLOCK), the exact sum of a group's terms rounded once (numerics page,
exact_sum, scaled_to_f32, GROUP; lane page, group) by exact-rational brute
force, a closed form, the in-order row fold (numerics page, dot) and the NaN
cases.  Exact rationals (fractions.Fraction) and numpy's binary16/binary32
casts are the independent references.
"""
from fractions import Fraction

import numpy as np
import pytest

from block_quantized_weight_quantize_gb300 import synth
from test_oracle_pins import bits, f32, frac, round_f32_grid_then_flush


@pytest.fixture(scope="module")
def orc():
    import oracle
    oracle.build()
    return oracle


def _check_block_scale(amax32, m, e):
    A = frac(amax32)
    assert 8 <= m <= 15
    s = Fraction(m) * Fraction(2) ** e
    assert 127 * s >= A
    prev = Fraction(m - 1) * Fraction(2) ** e if m > 8 else Fraction(15) * Fraction(2) ** (e - 1)
    assert 127 * prev < A, "not the least"


def test_block_scale_invariants(orc):
    """The least m*2^e, m in 8..15, with 127*m*2^e >= amax: the bound holds and
    the next-lower 4-bit value fails, over every binade and at exact products."""
    rng = np.random.default_rng(21)
    cases = [f32(0x00800000), f32(0x7F7FFFFF), np.float32(1.0), np.float32(127.0)]
    for E in range(1, 255):
        for mant in (0, 1, 0x7FFFFF, int(rng.integers(0, 1 << 23))):
            cases.append(f32((E << 23) | mant))
    for _ in range(300):
        mm = int(rng.integers(8, 16)); ee = int(rng.integers(-130, 110))
        v = np.float32(Fraction(127 * mm) * Fraction(2) ** ee)
        cases += [v, np.nextafter(v, np.float32(np.inf)), np.nextafter(v, np.float32(0))]
    for a in cases:
        a = np.float32(a)
        if not np.isfinite(a) or a < f32(0x00800000):
            continue
        m, e = orc.block_scale(a)
        _check_block_scale(a, m, e)


def test_quantize_sub32_codes(orc):
    """Per 32 elements: the scale is block_scale of the block's absmax and
    every code the nearest integer to x/s, ties to even (checked exactly);
    zero, infinite, NaN and denormal elements as in the PerBlock readings."""
    rng = np.random.default_rng(22)
    K = 512
    x = rng.standard_normal((2, K)).astype(np.float32)
    x[0, 32:64] *= np.float32(2.0 ** 60)                    # blocks far apart in magnitude
    x[0, 64:96] *= np.float32(2.0 ** -60)
    x[1, 96:128] = 0.0                                       # all-zero block
    x[1, 130] = np.inf                                       # a block with an infinity
    x[1, 170] = np.nan
    x[1, 171] = f32(0x00000123)                              # denormal
    for k in range(8):                                       # exact ties under a known scale
        x[0, 200 + k] = np.float32((k + 0.5) * 8 * 2.0 ** -3)
    x[0, 192] = np.float32(127 * 8 * 2.0 ** -3)              # makes the block's scale 8*2^-3
    codes, m, e, s16 = orc.quantize_sub32(x)
    for c in range(2):
        for b in range(K // 32):
            xb = x[c, 32 * b:32 * b + 32]
            if np.any(np.isinf(xb)):
                assert m[c, b] == 0 and np.all(codes[c, 32 * b:32 * b + 32] == 0)
                continue
            amax = orc.absmax(xb)
            if amax == 0:
                assert (m[c, b], e[c, b]) == (8, 0)
            else:
                assert (m[c, b], e[c, b]) == orc.block_scale(amax)
            s = Fraction(int(m[c, b])) * Fraction(2) ** int(e[c, b])
            for i in range(32):
                xi = xb[i]
                q = int(codes[c, 32 * b + i])
                if np.isnan(xi) or abs(xi) < f32(0x00800000):
                    assert q == 0
                    continue
                X = frac(xi) / s
                assert abs(X - q) <= Fraction(1, 2)
                if abs(X - q) == Fraction(1, 2):
                    assert q % 2 == 0, "ties to even"
    assert m[0, 6] == 8 and e[0, 6] == -3
    assert list(codes[0, 200:208]) == [0, 2, 2, 4, 4, 6, 6, 8]
    assert np.array_equal(s16, codes.reshape(2, -1, 16).astype(np.int32).sum(-1).astype(np.int16))


def test_exact_sum_against_rationals(orc):
    """exact_sum rounded once: random terms with exponent spreads up to ~250
    places, cancellation of the leading terms, ties, and the subnormal band."""
    rng = np.random.default_rng(23)
    for trial in range(3000):
        n = int(rng.integers(1, 17))
        sig = [int(v) for v in rng.integers(-(1 << 40), 1 << 40, n)]
        base = int(rng.integers(-170, 60))
        spread = [0, 5, 30, 120, 250][trial % 5]
        exps = [base + int(rng.integers(0, spread + 1)) for _ in range(n)]
        if trial % 7 == 0 and n >= 2:             # leading terms cancel exactly
            sig[1] = -sig[0]; exps[1] = exps[0]
        X = sum(Fraction(s) * Fraction(2) ** ex for s, ex in zip(sig, exps))
        assert bits(orc.exact_sum_f32(sig, exps)) == round_f32_grid_then_flush(X), (sig, exps)
    # ties: 2^24 + 1 (even below), 2^24 + 3 (even above), with a tiny term breaking the tie
    assert bits(orc.exact_sum_f32([(1 << 24) + 1], [0])) == bits(np.float32(2 ** 24))
    assert bits(orc.exact_sum_f32([(1 << 24) + 3], [0])) == bits(np.float32(2 ** 24 + 4))
    assert bits(orc.exact_sum_f32([(1 << 24) + 1, 1], [0, -200])) == bits(np.float32(2 ** 24 + 2))
    assert bits(orc.exact_sum_f32([], [])) == 0


def _exact_group_value(fmt, lg, r, g, codes, m, e):
    """Dequantise every weight of group g exactly (numerics page, CodedRow),
    dot with code times its 32-element block's scale, round once."""
    f16 = lambda hb: Fraction(float(np.uint16(hb).view(np.float16)))
    X = Fraction(0)
    for i in range(256):
        el = 256 * g + i
        sb = el // 32
        s_a = Fraction(int(m[sb])) * Fraction(2) ** int(e[sb])
        if fmt == synth.FMT_Q8_0:
            w = f16(lg["d"][r, sb]) * int(lg["q"][r, el])
        elif fmt == synth.FMT_Q4K:
            w = f16(lg["d"][r, g]) * int(lg["sc"][r, sb]) * int(lg["q"][r, el]) - f16(lg["dmin"][r, g]) * int(lg["mn"][r, sb])
        else:
            w = f16(lg["d"][r, g]) * int(lg["sc"][r, el // 16]) * (int(lg["q"][r, el]) - 32)
        X += w * int(codes[el]) * s_a
    return round_f32_grid_then_flush(X)


@pytest.mark.parametrize("fmt", [synth.FMT_Q8_0, synth.FMT_Q4K, synth.FMT_Q6K])
def test_group_values_brute_force(orc, fmt):
    """Every group's value bit for bit against exact-rational dequantise-then-dot
    and one rounding (lane page, group), with activation blocks of one group
    2^-60 .. 2^60 apart in magnitude."""
    rng = np.random.default_rng(24 + fmt)
    rows, K = 3, 512
    lg = synth.draw(fmt, rng, rows, K)
    W = synth.pack(fmt, lg)
    x = synth.draw_act(rng, 2, K, outlier_frac=0.01)
    for b in range(K // 32):
        x[0, 32 * b:32 * b + 32] *= np.float32(2.0 ** [0, 60, -60, 20, -7, 3, 40, -33][b % 8])
    codes, m, e, _ = orc.quantize_sub32(x)
    v = orc.group_values(fmt, W, rows, K, codes, m, e)
    for c in range(2):
        for r in range(rows):
            for g in range(K // 256):
                assert bits(v[c, r, g]) == _exact_group_value(fmt, lg, r, g, codes[c], m[c], e[c]), (c, r, g)


def test_group_closed_form(orc):
    """Q4_K-like, one group, every code q, sc, mn and activation code a constant
    and every activation block the same scale s_a: C_s = 32*sc*q*a and
    O_s = 32*mn*a per sub-block, so v = RNE(8 * s_a * (d*32*sc*q*a - dmin*32*mn*a))."""
    fmt, K = synth.FMT_Q4K, 256
    q, sc, mn, d16, dm16 = 11, 37, 5, 0x2E66, 0x1E00
    lg = {"q": np.full((1, K), q, np.uint8), "sc": np.full((1, 8), sc, np.uint8), "mn": np.full((1, 8), mn, np.uint8),
          "d": np.full((1, 1), d16, np.uint16), "dmin": np.full((1, 1), dm16, np.uint16)}
    W = synth.pack(fmt, lg)
    a, mm, ee = 77, 13, -9
    codes = np.full((1, K), a, np.int8)
    m = np.full((1, 8), mm, np.uint8)
    e = np.full((1, 8), ee, np.int16)
    v = orc.group_values(fmt, W, 1, K, codes, m, e)[0, 0, 0]
    f16 = lambda hb: Fraction(float(np.uint16(hb).view(np.float16)))
    X = 8 * Fraction(mm) * Fraction(2) ** ee * (f16(d16) * 32 * sc * q * a - f16(dm16) * 32 * mn * a)
    assert bits(v) == round_f32_grid_then_flush(X)


@pytest.mark.parametrize("fmt", [synth.FMT_Q8_0, synth.FMT_Q4K, synth.FMT_Q6K])
def test_sub32_row_fold_and_nan(orc, fmt):
    """A row is its groups' values added in order from +0 (f32, ftz); a group
    with an activation block holding an infinity, or an unreadable weight scale,
    makes the row the engine's NaN."""
    rng = np.random.default_rng(25 + fmt)
    rows, K = 4, 1024
    lg = synth.draw(fmt, rng, rows, K)
    lg["d"][2, 1] = 0x7C00                                    # unreadable scale in row 2
    W = synth.pack(fmt, lg)
    x = synth.draw_act(rng, 2, K)
    x[1, 700] = np.inf                                        # column 1: block 21 has no scale
    codes, m, e, _ = orc.quantize_sub32(x)
    v = orc.group_values(fmt, W, rows, K, codes, m, e)
    out = orc.gemv_sub32(fmt, W, rows, K, codes, m, e)
    for c in range(2):
        for r in range(rows):
            acc = np.float32(0)
            for g in range(K // 256):
                acc = orc.ftz(np.float32(acc + v[c, r, g]))
            want = 0x7FC00000 if np.isnan(acc) else bits(acc)
            assert bits(out[c, r]) == want, (c, r)
    assert np.all(out[1].view(np.uint32) == 0x7FC00000)
    assert out[0, 2].view(np.uint32) == 0x7FC00000
