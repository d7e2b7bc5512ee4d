"""Pins of the oracle's FP8 path against what the colizig OPS page (FP8:
e4m3ToF32, dequantRow, matmulFp8) and the mathematics fix: the page's own bit
formula for E4M3 normals and its rule for subnormals, the format's extreme
values, exact sums where double arithmetic is exact, one-hot activations that
read single weights (and so the 128x128 scale indexing), and a bound check
on random data against exact rationals.
"""
from fractions import Fraction

import numpy as np
import pytest

from test_oracle_pins import bits, round_f32_grid_then_flush


@pytest.fixture(scope="module")
def orc():
    import oracle
    oracle.build()
    return oracle


def test_e4m3_decode_all_bytes(orc):
    """Normals map onto f32 fields as (s << 31) | ((e + 120) << 23) | (m << 20);
    subnormals are m * 2^-9 with the sign; S.1111.111 is NaN (no infinity)."""
    for b in range(256):
        s, e, m = b >> 7, (b >> 3) & 15, b & 7
        v = orc.e4m3_to_f32(b)
        if e == 15 and m == 7:
            assert np.isnan(v)
        elif e == 0:
            want = np.float32(m * 2.0 ** -9)
            assert bits(v) == bits(-want if s else want), b
        else:
            assert bits(v) == (s << 31) | ((e + 120) << 23) | (m << 20), b
    assert orc.e4m3_to_f32(0x7E) == 448.0 and orc.e4m3_to_f32(0x01) == 2.0 ** -9
    assert orc.e4m3_to_f32(0x38) == 1.0 and orc.e4m3_to_f32(0x08) == 2.0 ** -6
    finite = [float(orc.e4m3_to_f32(b)) for b in range(0x7F)]
    assert all(a < c for a, c in zip(finite, finite[1:]))          # increasing over 0x00..0x7E


def _draw(rng, rows, K):
    W = rng.integers(0, 256, size=(rows, K), dtype=np.uint8)
    W[(W & 0x7F) == 0x7F] = 0x3C                                     # no NaN codes here
    scales = (2.0 ** rng.uniform(-12, -4, size=((rows + 127) // 128, (K + 127) // 128))).astype(np.float32)
    return W, scales


def test_one_hot_reads_weights_and_scale_blocks(orc):
    """x = e_i gives column i of the dequantized matrix: decode(W[r][i]) times
    the scale of block (r // 128, i // 128), one f32 rounding."""
    rng = np.random.default_rng(70)
    rows, K = 200, 384
    W, scales = _draw(rng, rows, K)
    for i in (0, 127, 128, 255, 256, 383):
        x = np.zeros((1, K), np.float32)
        x[0, i] = 1.0
        out, _ = orc.gemv_fp8(W, scales, rows, K, x)
        for r in (0, 127, 128, 199):
            want = np.float32(orc.e4m3_to_f32(W[r, i])) * scales[r // 128, i // 128]
            assert bits(out[0, r]) == bits(np.float32(want)), (r, i)


def test_exact_sums(orc):
    """Integer activations and unit scales: every product and partial sum is an
    integer below 2^53, so the oracle's result is RNE(exact sum)."""
    rng = np.random.default_rng(71)
    rows, K = 40, 512
    W, _ = _draw(rng, rows, K)
    W[:] = rng.integers(0x30, 0x5F, size=(rows, K)).astype(np.uint8)        # values 2^-1 .. 2^4: multiples of 2^-4
    scales = np.ones(((rows + 127) // 128, (K + 127) // 128), np.float32)
    x = rng.integers(-1000, 1001, size=(2, K)).astype(np.float32)
    out, ab = orc.gemv_fp8(W, scales, rows, K, x)
    for c in range(2):
        for r in range(rows):
            X = sum(Fraction(float(x[c, i])) * Fraction(float(orc.e4m3_to_f32(W[r, i]))) for i in range(K))
            assert bits(out[c, r]) == round_f32_grid_then_flush(X) or X == 0, (c, r)
            assert ab[c, r] == float(sum(abs(Fraction(float(x[c, i])) * Fraction(float(orc.e4m3_to_f32(W[r, i]))))
                                         for i in range(K)))


def round_f32_nearest(X: Fraction) -> int:
    """f32 bits of the exact rational X, nearest even on the f32 grid with
    subnormals kept (IEEE), infinite past the top: the neighbour search of
    round_f32_grid_then_flush without its flush, written out again here."""
    if X == 0:
        return 0
    neg = X < 0
    A = -X if neg else X
    top = (Fraction(2 ** 24) - Fraction(1, 2)) * Fraction(2) ** 104
    if A >= top:
        return 0xFF800000 if neg else 0x7F800000
    c = np.float32(float(A)) if float(A) < 3.4e38 else np.float32(3.4028234663852886e38)
    best = None
    for k in range(-3, 4):
        cand = c
        step = np.float32(np.inf) if k > 0 else np.float32(0)
        for _ in range(abs(k)):
            cand = np.nextafter(cand, step, dtype=np.float32)
        if np.isinf(cand):
            continue
        key = (abs(Fraction(float(cand)) - A), int(cand.view(np.uint32)) & 1)   # ties -> even significand
        if best is None or key < best[0]:
            best = (key, cand)
    return int(best[1].view(np.uint32)) | (0x80000000 if neg else 0)


def test_random_exact(orc):
    """Random data: the oracle's result is the exact rational dot of the f32
    activation with the f32-rounded dequantized weights, rounded once to the
    nearest f32 (ties even) -- bit for bit; its absdot is the sum of |x_i w_i|
    within K double roundings."""
    rng = np.random.default_rng(72)
    rows, K = 8, 384
    W, scales = _draw(rng, rows, K)
    x = rng.standard_normal((1, K)).astype(np.float32)
    out, ab = orc.gemv_fp8(W, scales, rows, K, x)
    for r in range(rows):
        ws = [Fraction(float(np.float32(np.float32(orc.e4m3_to_f32(W[r, i])) * scales[r // 128, i // 128])))
              for i in range(K)]
        X = sum(Fraction(float(x[0, i])) * ws[i] for i in range(K))
        S = sum(abs(Fraction(float(x[0, i])) * ws[i]) for i in range(K))
        assert bits(out[0, r]) == round_f32_nearest(X), r
        assert abs(Fraction(ab[0, r]) - S) <= K * Fraction(2) ** -52 * S


def test_cancellation_and_range(orc):
    """Sums that a double accumulation gets wrong, and the ends of the range:
    2^60 + 1 - 2^60 is exactly 1; a result below 2^-126 stays subnormal (no
    flush on this path); a sum past the top is infinite; opposite infinities
    give NaN."""
    def dot(xs, ws):
        return orc.exact_dot_f32(np.array(xs, np.float32), np.array(ws, np.float32))
    assert dot([2.0 ** 30, 1.0, -2.0 ** 30], [2.0 ** 30, 1.0, 2.0 ** 30]) == 1.0
    assert bits(dot([2.0 ** -100], [2.0 ** -40])) == 0x00000200                # 2^-140: subnormal kept
    # 2^-149 + 2^-150: 1.5 quanta of the subnormal grid, a tie, to even (2 quanta);
    # 2^-149 + 2^-151: 1.25 quanta, down to 1
    assert bits(dot([2.0 ** -100, 2.0 ** -100], [2.0 ** -49, 2.0 ** -50])) == 0x00000002
    assert bits(dot([2.0 ** -100, 2.0 ** -100], [2.0 ** -49, 2.0 ** -51])) == 0x00000001
    assert np.isinf(dot([3e38, 3e38], [1.0, 1.0])) and dot([3e38, 3e38], [1.0, 1.0]) > 0
    assert np.isnan(dot([np.inf, 1.0], [1.0, -np.inf]))
    assert np.isnan(dot([np.inf], [0.0]))
    assert bits(dot([1.0, -1.0], [5.0, 5.0])) == 0                             # an exact zero is +0


def test_nan_weight(orc):
    W = np.full((3, 256), 0x38, np.uint8)
    W[1, 17] = 0xFF
    out, _ = orc.gemv_fp8(W, np.ones((1, 2), np.float32), 3, 256, np.ones((1, 256), np.float32))
    assert bits(out[0, 1]) == 0x7FC00000 and out[0, 0] == 256.0 and out[0, 2] == 256.0
