"""Pins for the CPU oracle: what the pages and the mathematics fix, checked
without trusting the oracle's own code.

Each test names the passage it pins (decode engine pages: the numerics page
and the block-scale lane page).  The checks are library routines (numpy's
binary16/binary32 casts), exact rational arithmetic (fractions.Fraction),
closed forms with constant codes, invariants (minimality, nearest-ness),
hand-derived values under tests/golden/, and brute force on tiny inputs.
"""
import json
import os
from fractions import Fraction

import numpy as np
import pytest

from block_quantized_weight_quantize_gb300 import synth

GOLDEN = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "closed_forms.json")))
FLT_MIN = Fraction(2) ** -126


def f32(bits: int) -> np.float32:
    return np.uint32(bits).view(np.float32)


def bits(x) -> int:
    return int(np.float32(x).view(np.uint32))


def frac(x) -> Fraction:
    return Fraction(float(np.float32(x)))


def round_f32_grid_then_flush(X: Fraction) -> int:
    """f32 bits of the exact rational X: nearest on the f32 grid (ties even),
    a subnormal result flushed to a zero of its sign.  Independent check by
    neighbour search with numpy's nextafter and exact comparisons."""
    if X == 0:
        return 0
    neg = X < 0
    A = -X if neg else X
    if A >= Fraction(2) ** 128:
        return (0xFF800000 if neg else 0x7F800000)
    # candidate from a correctly rounded double, then walk neighbours exactly
    c = np.float32(float(A)) if float(A) < 3.4e38 else np.float32(3.4028234663852886e38)
    best = None
    for k in range(-3, 4):
        cand = c
        step = np.float32(np.inf) if k > 0 else np.float32(0)
        for _ in range(abs(k)):
            cand = np.nextafter(cand, step, dtype=np.float32)
        if np.isinf(cand):
            continue
        dist = abs(Fraction(float(cand)) - A)
        key = (dist, int(cand.view(np.uint32)) & 1)   # ties -> even significand
        if best is None or key < best[0]:
            best = (key, cand)
    r = best[1]
    # the largest finite value rounds to infinity past (2^24 - 1/2) * 2^104
    top = (Fraction(2 ** 24) - Fraction(1, 2)) * Fraction(2) ** 104
    if A >= top:
        return 0xFF800000 if neg else 0x7F800000
    rb = int(r.view(np.uint32))
    if Fraction(float(r)) < FLT_MIN:  # subnormal (or zero) result: flush
        rb = 0
    return rb | (0x80000000 if neg else 0)


# ---------------------------------------------------------------- Scale

def test_f16_scale_exhaustive(orc):
    """Scale is sig*2^exp exactly; Unreadable for inf/NaN (numerics page, structs
    Scale, Unreadable).  Pinned against numpy's binary16 decoding, all 65536 patterns."""
    allh = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    vals = allh.view(np.float16).astype(np.float64)
    for h in range(65536):
        r = orc.f16_scale(h)
        if not np.isfinite(vals[h]):
            assert r is None, hex(h)
        else:
            sig, ex = r
            assert Fraction(sig) * Fraction(2) ** ex == Fraction(vals[h]), hex(h)


def test_f16_to_f32_exhaustive(orc):
    """The oracle's binary16 -> f32 widening (used by fdot and the key-cache
    scales) against numpy's, all 65536 patterns: every finite value and the
    infinities exactly, subnormals included; NaN to NaN."""
    allh = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    want = allh.view(np.float16).astype(np.float32)
    for h in range(65536):
        got = orc.f16_to_f32(h)
        if np.isnan(want[h]):
            assert np.isnan(got), hex(h)
        else:
            assert bits(got) == bits(want[h]), hex(h)


def test_head_width_pads_to_whole_groups(orc):
    """A quantized query head holds d codes under PerBlock and d rounded up to
    whole 256-element groups under Sub32 (numerics page: quantize_head, GROUP)."""
    for d, sub32 in ((64, 256), (96, 256), (128, 256), (256, 256), (320, 512), (1024, 1024)):
        assert orc.head_width(0, d) == d
        assert orc.head_width(1, d) == sub32


# ---------------------------------------------------------------- absmax

def test_absmax_rules(orc):
    """absmax: largest magnitude, a denormal read as zero, folded from +0, NaN
    passed over (numerics page, absmax)."""
    den = f32(0x00400000)
    assert orc.absmax(np.array([den, -den], np.float32)) == 0.0
    assert bits(orc.absmax(np.array([-0.0], np.float32))) == 0          # folded from +0
    assert orc.absmax(np.array([np.nan, -3.0, 2.0], np.float32)) == 3.0
    assert orc.absmax(np.array([np.nan], np.float32)) == 0.0
    assert np.isinf(orc.absmax(np.array([1.0, -np.inf], np.float32)))
    rng = np.random.default_rng(5)
    for _ in range(50):
        x = (rng.standard_normal(64) * 10.0 ** rng.integers(-30, 30)).astype(np.float32)
        assert orc.absmax(x) == np.max(np.abs(x))


# ---------------------------------------------------------------- wide_scale

def _check_wide_scale(amax32, m, e):
    A = frac(amax32)
    assert 128 <= m <= 255
    s = Fraction(m) * Fraction(2) ** e
    assert 127 * s >= A
    prev = Fraction(m - 1) * Fraction(2) ** e if m > 128 else Fraction(255) * Fraction(2) ** (e - 1)
    assert 127 * prev < A, "not the least"


def test_wide_scale_invariants(orc):
    """The least m*2^e, m in 128..255, with 127*m*2^e >= amax (numerics page,
    wide_scale): bound holds and the next-lower 8-bit value fails, over every
    binade of normal f32 and at its edges."""
    rng = np.random.default_rng(1)
    cases = [f32(0x00800000), f32(0x7F7FFFFF), np.float32(1.0), np.float32(127.0)]
    for E in range(1, 255):
        for mant in (0, 1, 0x7FFFFF, int(rng.integers(0, 1 << 23))):
            cases.append(f32((E << 23) | mant))
    for k in range(1, 300):  # amax = 127 * m * 2^e exactly and one ulp either side
        mm = int(rng.integers(128, 256)); ee = int(rng.integers(-130, 110))
        v = np.float32(Fraction(127 * mm) * Fraction(2) ** ee)
        cases += [v, np.nextafter(v, np.float32(np.inf)), np.nextafter(v, np.float32(0))]
    for a in cases:
        a = np.float32(a)
        if not np.isfinite(a) or a < f32(0x00800000):
            continue
        m, e = orc.wide_scale(a)
        _check_wide_scale(a, m, e)


def test_wide_scale_golden(orc):
    for g in GOLDEN["wide_scale"]:
        a = np.float32(g["amax"]) if "amax" in g else f32(int(g["amax_bits"], 16))
        assert orc.wide_scale(a) == (g["m"], g["e"]), g


# ---------------------------------------------------------------- rne_div

def test_rne_div_nearest_ties_even(orc):
    """The nearest integer to x/(m*2^e), ties to even, exactly (numerics page,
    rne_div).  Exhaustive over all codes for several scales, constructed
    ties, and random x; checked with exact rationals."""
    rng = np.random.default_rng(2)
    for (m, e) in [(128, -7), (130, -14), (255, 0), (191, -20), (200, 40), (129, -135)]:
        s = Fraction(m) * Fraction(2) ** e
        for c in range(-127, 128):
            for t in (Fraction(c), Fraction(2 * c + 1, 2)):   # exact codes and ties
                X = t * s
                x = np.float32(X)
                if frac(x) != X or abs(frac(x)) < FLT_MIN:
                    continue
                q = orc.rne_div(x, m, e)
                if t.denominator == 1:
                    assert q == c
                else:
                    assert q % 2 == 0 and abs(Fraction(q) - t) == Fraction(1, 2)
        for x in (rng.uniform(-127.4, 127.4, 400) * float(s)).astype(np.float32):
            if abs(frac(x)) < FLT_MIN:
                continue
            q = orc.rne_div(x, m, e)
            d = abs(frac(x) - q * s)
            assert d <= s / 2
            if d == s / 2:
                assert q % 2 == 0


def test_rne_div_golden(orc):
    for g in GOLDEN["rne_div"]:
        assert orc.rne_div(np.float32(g["x"]), g["m"], g["e"]) == g["q"], g


# ---------------------------------------------------------------- quantize_blocks

@pytest.mark.parametrize("block", [32, 256])
def test_quantize_blocks_properties(orc, block):
    """quantize_blocks: per block, wide_scale of absmax, codes rne_div, |code|<=127
    (numerics page, quantize_blocks, ActScaling::PerBlock); the unit sums are the
    activation side's sums per 16 (lane page)."""
    rng = np.random.default_rng(3)
    x = synth.draw_act(rng, 3, 1024, outlier_frac=0.01)
    x[0, :block] = 0.0                               # zero block (reading R1)
    x[1, 5] = np.nan                                 # NaN element: code 0, skipped (R2)
    x[1, 7] = f32(0x00000123)                        # denormal element: code 0 (R2)
    x[2, block:2 * block] *= np.float32(1e-38)       # a block near the bottom of f32
    codes, m, e, s16 = orc.quantize_blocks(x, block)
    assert np.all(np.abs(codes.astype(int)) <= 127)
    assert np.array_equal(s16, codes.reshape(3, -1, 16).astype(np.int64).sum(-1))
    for c in range(3):
        for b in range(1024 // block):
            xb = x[c, b * block:(b + 1) * block]
            a = orc.absmax(xb)
            if a == 0:
                assert (m[c, b], e[c, b]) == (128, 0) and not codes[c, b * block:(b + 1) * block].any()
                continue
            _check_wide_scale(a, int(m[c, b]), int(e[c, b]))
            s = Fraction(int(m[c, b])) * Fraction(2) ** int(e[c, b])
            for i, xi in enumerate(xb):
                q = int(codes[c, b * block + i])
                if np.isnan(xi) or abs(frac(xi)) < FLT_MIN:
                    assert q == 0
                    continue
                d = abs(frac(xi) - q * s)
                assert d <= s / 2 and (d < s / 2 or q % 2 == 0)
            # the largest element codes to 126 or 127 (127*prev < amax <= 127*s)
            assert np.max(np.abs(codes[c, b * block:(b + 1) * block].astype(int))) in (126, 127)


def test_quantize_blocks_infinity_marks_block(orc):
    """Reading R3: a block holding an infinity has no scale (m = 0, codes 0)."""
    x = np.ones((1, 64), np.float32)
    x[0, 40] = np.inf
    codes, m, e, s16 = orc.quantize_blocks(x, 32)
    assert m[0, 1] == 0 and not codes[0, 32:].any() and m[0, 0] == 130


# ---------------------------------------------------------------- scaled_to_f32

def test_scaled_to_f32_vs_numpy_cast(orc):
    """v*2^ex rounded once to f32, RNE, denormal flushed keeping its sign
    (numerics page, scaled_to_f32).  For |v| < 2^53 the double v*2^ex is exact,
    so numpy's float64->float32 cast (IEEE RNE with gradual underflow) followed
    by a flush of subnormal results is the definition."""
    rng = np.random.default_rng(4)
    for _ in range(20000):
        nb = int(rng.integers(1, 54))
        v = int(rng.integers(0, 1 << min(nb, 62))) | (1 << (nb - 1))
        if rng.random() < 0.5:
            v = -v
        ex = int(rng.integers(-200, 110))
        dv = np.float64(v) * np.float64(2.0) ** ex if -1074 < ex + nb < 1020 else None
        if dv is None or not np.isfinite(dv):
            continue
        with np.errstate(over="ignore"):
            ref = np.float32(dv)
        rb = int(ref.view(np.uint32))
        if np.isfinite(ref) and 0 < abs(ref) < np.float32(2.0 ** -126):
            rb &= 0x80000000
        assert bits(orc.scaled_to_f32(v, ex)) == rb, (v, ex)


def test_scaled_to_f32_wide_exact(orc):
    """The same for values beyond 53 bits (up to 2^100), against the exact
    nearest-f32 neighbour search on rationals."""
    rng = np.random.default_rng(6)
    for _ in range(3000):
        nb = int(rng.integers(50, 101))
        v = int.from_bytes(rng.bytes(13), "little") % (1 << nb) | (1 << (nb - 1))
        if rng.random() < 0.5:
            v = -v
        ex = int(rng.integers(-240, 40))
        X = Fraction(v) * Fraction(2) ** ex
        assert bits(orc.scaled_to_f32(v, ex)) == round_f32_grid_then_flush(X), (v, ex)


def test_scaled_to_f32_golden(orc):
    for g in GOLDEN["scaled_to_f32"]:
        assert bits(orc.scaled_to_f32(g["v"], g["ex"])) == int(g["bits"], 16), g


def test_scaled_to_f32_flush_band(orc):
    """Reading R5 at the band just below 2^-126: every value (2^24 - k) * 2^-150
    rounds on the grid (quantum 2^-149) before the flush."""
    for k in range(1, 8):
        v = (1 << 24) - k
        X = Fraction(v) * Fraction(2) ** -150
        expect = round_f32_grid_then_flush(X)
        assert bits(orc.scaled_to_f32(v, -150)) == expect
    assert bits(orc.scaled_to_f32((1 << 24) - 1, -150)) == 0x00800000
    assert bits(orc.scaled_to_f32((1 << 24) - 2, -150)) == 0


# ---------------------------------------------------------------- f32_to_f16

def test_f32_to_f16_vs_numpy(orc):
    """f32_to_f16: RNE to binary16, subnormals kept, past the top infinite
    (numerics page, f32_to_f16).  Pinned against numpy's float32->float16 cast
    over random values, every half-way case between adjacent binary16 values
    of a sample, and the binary16 subnormal and overflow ranges."""
    rng = np.random.default_rng(7)
    xs = [rng.standard_normal(20000).astype(np.float32) * np.float32(10.0) ** rng.integers(-9, 6, 20000)]
    h = rng.integers(0, 0x7C00, 5000).astype(np.uint16)
    lo = h.view(np.float16).astype(np.float32)
    hi = (h + 1).astype(np.uint16).view(np.float16).astype(np.float32)
    mid = ((lo.astype(np.float64) + hi.astype(np.float64)) / 2).astype(np.float32)   # exact in f32
    xs += [mid, -mid, np.nextafter(mid, np.float32(np.inf)), np.nextafter(mid, np.float32(0))]
    xs += [rng.uniform(0, 2 ** -14, 5000).astype(np.float32), rng.uniform(60000, 70000, 5000).astype(np.float32)]
    x = np.concatenate(xs)
    with np.errstate(over="ignore"):
        ref = x.astype(np.float16).view(np.uint16)
    got = orc.quantize_f16(x)
    assert np.array_equal(got, ref)
    for g in GOLDEN["f32_to_f16"]:
        assert orc.f32_to_f16(f32(int(g["x_bits"], 16))) == int(g["h"], 16), g
    assert orc.f32_to_f16(np.float32(np.nan)) == 0x7E00


# ---------------------------------------------------------------- lane / block values

def test_lane_golden(orc):
    for g in GOLDEN["lane"]:
        v = orc.lane_value(g["C"], g["O"], int(g["s1"], 16), int(g["s2"], 16), g["kind"], g["m"], g["e"])
        assert bits(v) == int(g["bits"], 16), g


def _exact_block_value(fmt, lg, r, b, codes, m, e):
    """Brute force in exact rationals: dequantise every weight (numerics page,
    CodedRow: a*coef + b*offs), dot with the activation code times its scale,
    then round once (lane page, lane)."""
    f16 = lambda hb: Fraction(float(np.uint16(hb).view(np.float16)))
    s_a = Fraction(int(m)) * Fraction(2) ** int(e)
    X = Fraction(0)
    if fmt == synth.FMT_Q8_0:
        d = f16(lg["d"][r, b])
        for i in range(32):
            X += d * int(lg["q"][r, 32 * b + i]) * int(codes[32 * b + i])
    elif fmt == synth.FMT_Q4K:
        d, dm = f16(lg["d"][r, b]), f16(lg["dmin"][r, b])
        for i in range(256):
            s = 8 * b + i // 32
            w = d * int(lg["sc"][r, s]) * int(lg["q"][r, 256 * b + i]) - dm * int(lg["mn"][r, s])
            X += w * int(codes[256 * b + i])
    else:
        d = f16(lg["d"][r, b])
        for i in range(256):
            u = 16 * b + i // 16
            w = d * int(lg["sc"][r, u]) * (int(lg["q"][r, 256 * b + i]) - 32)
            X += w * int(codes[256 * b + i])
    return round_f32_grid_then_flush(X * s_a)


@pytest.mark.parametrize("fmt", [synth.FMT_Q8_0, synth.FMT_Q4K, synth.FMT_Q6K])
def test_block_values_brute_force(orc, fmt):
    """Every block's value, bit for bit, against exact-rational dequantise-then-dot
    and a once-only rounding (lane page: the block's two terms summed exactly and
    rounded once; numerics page, dot under PerBlock)."""
    rng = np.random.default_rng(8 + fmt)
    rows, K = 3, 512
    kw = {} if fmt != synth.FMT_Q4K else {"d_range": (1e-7, 1e-1)}   # wide exponent spread
    lg = synth.draw(fmt, rng, rows, K, **kw)
    W = synth.pack(fmt, lg)
    x = synth.draw_act(rng, 2, K, outlier_frac=0.01)
    blk = synth.BLOCK[fmt]
    codes, m, e, _ = orc.quantize_blocks(x, blk)
    C, O, v = orc.block_values(fmt, W, rows, K, codes, m, e)
    for c in range(2):
        for r in range(rows):
            for b in range(K // blk):
                ref = _exact_block_value(fmt, lg, r, b, codes[c], m[c, b], e[c, b])
                assert bits(v[c, r, b]) == ref, (c, r, b)


def test_block_value_fp64_dequant(orc):
    """Where the exact dot fits in 53 bits (Q4_K, K = 256, d = dmin), a plain
    float64 dequantise-then-dot is exact; numpy's cast then rounds it once."""
    rng = np.random.default_rng(9)
    for _ in range(20):
        lg = synth.draw_q4k(rng, 1, 256)
        lg["dmin"] = lg["d"].copy()
        W = synth.pack_q4k(**lg)
        x = synth.draw_act(rng, 1, 256)
        codes, m, e, _ = orc.quantize_blocks(x, 256)
        d = float(lg["d"].view(np.float16)[0, 0])
        sc = np.repeat(lg["sc"][0].astype(np.float64), 32)
        mn = np.repeat(lg["mn"][0].astype(np.float64), 32)
        w = d * sc * lg["q"][0].astype(np.float64) - d * mn
        dot = float(np.dot(w, codes[0].astype(np.float64)))   # |terms| < 2^40 * ulp(d): exact
        ref = np.float32(dot * float(m[0, 0]) * 2.0 ** float(e[0, 0]))
        _, _, v = orc.block_values(synth.FMT_Q4K, W, 1, 256, codes, m, e)
        assert bits(v[0, 0, 0]) == bits(ref)


@pytest.mark.parametrize("fmt", [synth.FMT_Q8_0, synth.FMT_Q4K, synth.FMT_Q6K])
def test_closed_form_constant_codes(orc, fmt):
    """All codes, sub-scales and activation codes constant: C and O have closed
    forms (Q8_0: 32*q*a; Q4_K: 256*sc*q*a and 256*mn*a; Q6_K: 256*sc*(q-32)*a)."""
    K = 256
    for (q, sc, mn, a) in [(15, 63, 63, 127), (1, 1, 0, -1), (7, 33, 5, -100), (0, 63, 63, 127)]:
        if fmt == synth.FMT_Q8_0:
            qq = int(np.clip(q * 8 - 60, -127, 127))
            lg = {"q": np.full((1, K), qq, np.int8), "d": np.full((1, K // 32), 0x3C00, np.uint16)}
            Cx, Ox = 32 * qq * a, 0
        elif fmt == synth.FMT_Q4K:
            lg = {"q": np.full((1, K), q, np.uint8), "sc": np.full((1, 8), sc, np.uint8),
                  "mn": np.full((1, 8), mn, np.uint8), "d": np.full((1, 1), 0x3C00, np.uint16),
                  "dmin": np.full((1, 1), 0x3800, np.uint16)}
            Cx, Ox = 256 * sc * q * a, 256 * mn * a
        else:
            qq, s6 = 4 * q + 3, sc - 64
            lg = {"q": np.full((1, K), qq, np.uint8), "sc": np.full((1, 16), s6, np.int8),
                  "d": np.full((1, 1), 0x3C00, np.uint16)}
            Cx, Ox = 256 * s6 * (qq - 32) * a, 0
        W = synth.pack(fmt, lg)
        codes = np.full((1, K), a, np.int8)
        blk = synth.BLOCK[fmt]
        m = np.full((1, K // blk), 128, np.uint8); e = np.full((1, K // blk), -7, np.int16)   # scale 1
        C, O, v = orc.block_values(fmt, W, 1, K, codes, m, e)
        assert np.all(C == Cx) and np.all(O == Ox)
        dmin = Fraction(1, 2)
        X = Fraction(Cx) - (dmin * Ox if fmt == synth.FMT_Q4K else 0)
        if fmt == synth.FMT_Q8_0:
            X = Fraction(32 * qq * a)
        assert bits(v[0, 0, 0]) == round_f32_grid_then_flush(X)


@pytest.mark.parametrize("fmt", [synth.FMT_Q8_0, synth.FMT_Q4K, synth.FMT_Q6K])
def test_excess_identity_matches_direct_sums(orc, fmt):
    """The lane's delivery -- unit sums P', Q, S' in one-word excess form and the
    identity sum(q-z)*a = P' - 128*Q - z*S' + 128*16*z (lane page) -- gives the
    same block sums as the direct element-by-element sum (lane page,
    block_sums), including codes at the extremes of every format."""
    rng = np.random.default_rng(10 + fmt)
    rows, K = 4, 1024
    lg = synth.draw(fmt, rng, rows, K)
    if fmt == synth.FMT_Q6K:
        lg["sc"][0, :] = -128; lg["q"][0, :] = 0              # COEF_BOUND: -128 * -32
    W = synth.pack(fmt, lg)
    codes = rng.integers(-127, 128, (3, K)).astype(np.int8)
    codes[0, :] = -127
    Cd, Od, _ = orc.block_values(fmt, W, rows, K, codes, np.full((3, K // synth.BLOCK[fmt]), 128, np.uint8),
                                 np.zeros((3, K // synth.BLOCK[fmt]), np.int16))
    Ce, Oe = orc.block_sums_excess(fmt, W, rows, K, codes)
    assert np.array_equal(Cd, Ce) and np.array_equal(Od, Oe)
    if fmt == synth.FMT_Q6K:
        assert Cd[0, 0, 0] == 4096 * -127 * 256                # COEF_BOUND * (-127) * 256


def test_excess_identity_pure():
    """The identity itself, exhaustively over small units and in its two-word
    form (lane page): a 16-bit code a = 256*hi + lo crosses as hi+128 (excess)
    and lo (unsigned); the low word gives P' - z*S', the high word is weighted
    by 256."""
    rng = np.random.default_rng(11)
    for z, qmax in ((0, 15), (32, 63), (128, 255)):
        for _ in range(2000):
            q = rng.integers(0, qmax + 1, 16)
            a = rng.integers(-127, 128, 16)
            ap = a + 128
            P1, Q, S1 = int(np.dot(q, ap)), int(q.sum()), int(ap.sum())
            assert int(np.dot(q - z, a)) == P1 - 128 * Q - z * S1 + 128 * 16 * z
            assert int(a.sum()) == S1 - 128 * 16
            a16 = rng.integers(-32768, 32768, 16)
            hi, lo = a16 >> 8, a16 & 0xFF
            hp = hi + 128
            Ph, Sh = int(np.dot(q, hp)), int(hp.sum())
            Pl, Sl = int(np.dot(q, lo)), int(lo.sum())
            hi_dot = Ph - 128 * Q - z * Sh + 128 * 16 * z
            lo_dot = Pl - z * Sl
            assert int(np.dot(q - z, a16)) == 256 * hi_dot + lo_dot
            assert int(a16.sum()) == 256 * (Sh - 128 * 16) + Sl


# ---------------------------------------------------------------- row fold / dot

@pytest.mark.parametrize("fmt", [synth.FMT_Q8_0, synth.FMT_Q4K, synth.FMT_Q6K])
def test_row_fold(orc, fmt):
    """dot: the rounded pieces of a row added in order from +0 in f32 with ftz
    (numerics page, dot and the f32 rules).  One block: the row is the block's
    value; many blocks: numpy float32 adds in block order."""
    rng = np.random.default_rng(12 + fmt)
    blk = synth.BLOCK[fmt]
    for K in (blk, 2 * blk, 7 * blk):
        lg = synth.draw(fmt, rng, 5, K)
        W = synth.pack(fmt, lg)
        x = synth.draw_act(rng, 2, K)
        codes, m, e, _ = orc.quantize_blocks(x, blk)
        _, _, v = orc.block_values(fmt, W, 5, K, codes, m, e)
        out = orc.gemv(fmt, W, 5, K, codes, m, e)
        acc = np.zeros((2, 5), np.float32)
        for b in range(K // blk):
            acc = acc + v[:, :, b]
            acc[np.abs(acc) < np.float32(2.0 ** -126)] *= np.float32(0)
        assert np.array_equal(out.view(np.uint32), acc.view(np.uint32))


def test_unreadable_rows_are_nan(orc):
    """Unreadable: a block with an infinite or NaN scale (numerics page, struct
    Unreadable); its row is the engine's NaN 0x7FC00000 (numerics page, NAN)."""
    rng = np.random.default_rng(13)
    lg = synth.draw_q4k(rng, 4, 512)
    lg["d"][1, 1] = 0x7C00        # +inf
    lg["dmin"][2, 0] = 0x7E01     # NaN with payload
    W = synth.pack_q4k(**lg)
    assert orc.count_unreadable(synth.FMT_Q4K, W, 4, 512) == 2
    x = synth.draw_act(rng, 1, 512)
    codes, m, e, _ = orc.quantize_blocks(x, 256)
    out = orc.gemv(synth.FMT_Q4K, W, 4, 512, codes, m, e)
    assert out.view(np.uint32)[0, 1] == 0x7FC00000 and out.view(np.uint32)[0, 2] == 0x7FC00000
    assert np.isfinite(out[0, 0]) and np.isfinite(out[0, 3])
    m[0, 1] = 0                    # reading R3: an activation block with no scale
    out = orc.gemv(synth.FMT_Q4K, W, 4, 512, codes, m, e)
    assert np.all(out.view(np.uint32) == 0x7FC00000)


@pytest.mark.parametrize("fmt", [synth.FMT_Q8_0, synth.FMT_Q4K, synth.FMT_Q6K])
def test_batch_invariance(orc, fmt):
    """Each column of a many-column product equals the one-column product bit
    for bit (the definition is per column)."""
    rng = np.random.default_rng(14 + fmt)
    K = 512
    lg = synth.draw(fmt, rng, 6, K)
    W = synth.pack(fmt, lg)
    x = synth.draw_act(rng, 5, K)
    codes, m, e, _ = orc.quantize_blocks(x, synth.BLOCK[fmt])
    all5 = orc.gemv(fmt, W, 6, K, codes, m, e)
    for c in range(5):
        one = orc.gemv(fmt, W, 6, K, codes[c:c + 1], m[c:c + 1], e[c:c + 1])
        assert np.array_equal(one[0].view(np.uint32), all5[c].view(np.uint32))


# ---------------------------------------------------------------- F16 path

def _lanes_tree_numpy(w16, x16):
    """An independent float32 statement of fdot with 8 lanes and the tree."""
    p = w16.view(np.float16).astype(np.float32) * x16.view(np.float16).astype(np.float32)
    K = p.shape[-1]
    lanes = np.zeros(p.shape[:-1] + (8,), np.float32)
    for i in range(0, K, 8):
        lanes = lanes + p[..., i:i + 8]
    t = (lanes[..., 0] + lanes[..., 1]) + (lanes[..., 2] + lanes[..., 3])
    u = (lanes[..., 4] + lanes[..., 5]) + (lanes[..., 6] + lanes[..., 7])
    return t + u


def test_f16_gemv_pins(orc):
    """fdot in LANES=8 lanes, element i in lane i mod 8 in index order, then the
    balanced tree (numerics page, fdot, tree; reading R6), the activation
    first rounded to f16 (numerics page, f32_to_f16)."""
    rng = np.random.default_rng(15)
    rows, K = 13, 576
    W = synth.draw_f16(rng, rows, K)
    x = synth.draw_act(rng, 3, K)
    x16 = orc.quantize_f16(x)
    out = orc.gemv_f16(W, rows, K, x16)
    ref = _lanes_tree_numpy(W[None, :, :], x16[:, None, :])
    assert np.array_equal(out.view(np.uint32), ref.view(np.uint32))
    # one-hot activation: the weight itself, exactly
    oh = np.zeros((1, K), np.uint16); oh[0, 77] = 0x3C00
    o1 = orc.gemv_f16(W, rows, K, oh)
    assert np.array_equal(o1[0], W[:, 77].view(np.float16).astype(np.float32))
    # K = 8: the tree of the 8 exact products
    W8, x8 = W[:, :8].copy(), x16[:1, :8].copy()
    p = W8.view(np.float16).astype(np.float32) * x8.view(np.float16).astype(np.float32)
    tr = ((p[:, 0] + p[:, 1]) + (p[:, 2] + p[:, 3])) + ((p[:, 4] + p[:, 5]) + (p[:, 6] + p[:, 7]))
    assert np.array_equal(orc.gemv_f16(W8, rows, 8, x8)[0], tr)
    # within the order's error bound of the exact dot (depth 72 + 3 adds)
    exact = W.view(np.float16).astype(np.float64) @ x16[0].view(np.float16).astype(np.float64)
    bound = (K // 8 + 3) * 2.0 ** -24 * (np.abs(W.view(np.float16).astype(np.float64))
                                         @ np.abs(x16[0].view(np.float16).astype(np.float64)))
    assert np.all(np.abs(out[0] - exact) <= bound)


# ---------------------------------------------------------------- layout

@pytest.mark.parametrize("fmt", [synth.FMT_Q8_0, synth.FMT_Q4K, synth.FMT_Q6K])
def test_oracle_unpack_reads_the_layout(orc, fmt):
    """The oracle's own unpacker reads back the logical arrays the generator
    packed (the byte layout is this library's own; the pages fix none)."""
    rng = np.random.default_rng(16 + fmt)
    for K in (256, 768):
        lg = synth.draw(fmt, rng, 3, K)
        W = synth.pack(fmt, lg)
        assert W.size == 3 * synth.record_bytes(fmt, K) == 3 * orc.record_bytes(fmt, K)
        back = orc.unpack(fmt, W, 3, K)
        for key, val in lg.items():
            assert np.array_equal(back[key].view(val.dtype), val), key
