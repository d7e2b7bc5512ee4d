"""Pins of the oracle's int8-cache score path against what the pages and the
mathematics fix (numerics page: cache_row, int8_codes, INV_127,
quantize_head, int8_score): numpy's IEEE binary32 arithmetic and binary16
cast for the cache rows, exact rationals (fractions.Fraction) for the scores,
a closed form, and the NaN and zero cases.
"""
from fractions import Fraction

import numpy as np
import pytest

from test_oracle_pins import bits, f32, frac, round_f32_grid_then_flush


@pytest.fixture(scope="module")
def orc():
    import oracle
    oracle.build()
    return oracle


def _numpy_cache_row(x):
    """cache_row restated with numpy's IEEE f32 operations and binary16 cast:
    scale = f16(amax * f32(1/127)); codes = clip(rint(x * (1/scale)), +-127),
    NaN products 0, all zero when the scale is 0."""
    ax = np.abs(x.astype(np.float32))
    ax = np.where(np.isnan(ax) | (ax < f32(0x00800000)), np.float32(0), ax)
    amax = np.float32(ax.max()) if ax.size else np.float32(0)
    inv127 = np.float32(1) / np.float32(127)
    with np.errstate(over="ignore"):
        s16 = np.float16(np.float32(amax) * inv127)
    s = np.float32(s16)
    with np.errstate(divide="ignore", invalid="ignore", over="ignore"):
        inv = np.float32(1) / s
        if np.isinf(inv):
            return np.zeros(x.size, np.int8), s16.view(np.uint16)
        p = x.astype(np.float32) * inv
    p = np.where(np.isnan(p), np.float32(0), p)
    q = np.clip(np.rint(p), -127, 127).astype(np.int8)
    return q, s16.view(np.uint16)


def test_inv_127_bits(orc):
    """INV_127 is 1/127 rounded to f32: 2^-7 * 1.0000001000000100000010..._2 -> 0x3C010204."""
    assert orc.int8_code(127.0, np.uint32(0x3C010204).view(np.float32)) == 1
    assert (np.float32(1) / np.float32(127)).view(np.uint32) == 0x3C010204


def test_cache_rows_against_numpy(orc):
    rng = np.random.default_rng(41)
    rows = []
    for mag in (1.0, 1e-3, 1e3, 7e6, 1e-20, 3e-8):
        rows.append((rng.standard_normal(128) * mag).astype(np.float32))
    r = rng.standard_normal(128).astype(np.float32)
    r[5] = np.nan
    r[6] = np.float32(1e-41)                          # denormal
    rows.append(r)
    rows.append(np.zeros(128, np.float32))            # zero row: scale 0, codes 0
    r = rng.standard_normal(128).astype(np.float32)
    r[9] = np.inf                                     # scale overflows binary16: codes 0
    rows.append(r)
    r = rng.standard_normal(128).astype(np.float32)
    r[:] = np.float32(2.5)                            # ties under the scale: x*inv near 127 for all
    rows.append(r)
    for k in range(40):                               # random magnitudes across f32
        rows.append((rng.standard_normal(128) * np.float32(2.0 ** rng.integers(-140, 100))).astype(np.float32))
    x = np.stack(rows)
    codes, scales = orc.cache_rows(x)
    for i in range(x.shape[0]):
        q, s = _numpy_cache_row(x[i])
        assert scales[i] == s, i
        assert np.array_equal(codes[i], q), i
    assert scales[7] == 0 and not codes[7].any()
    assert scales[8] == 0x7C00 and not codes[8].any()
    assert scales[4] == 0 and not codes[4].any()      # 1e-20 * 127^-1 rounds to a zero f16


def test_int8_codes_ties_and_clamp(orc):
    inv = np.float32(0.5)
    assert [orc.int8_code(v, inv) for v in (1.0, 3.0, 5.0, -1.0, -3.0)] == [0, 2, 2, 0, -2]  # 0.5, 1.5, 2.5 ties even
    assert orc.int8_code(1000.0, inv) == 127 and orc.int8_code(-1000.0, inv) == -127
    assert orc.int8_code(np.nan, inv) == 0
    assert orc.int8_code(3.0, np.float32(np.inf)) == 0


def _exact_score(qc, m, e, blk, d, kc, ks):
    s_k = Fraction(float(np.uint16(ks).view(np.float16)))
    X = Fraction(0)
    for b in range(len(m)):
        D = sum(int(qc[i]) * int(kc[i]) for i in range(b * blk, min((b + 1) * blk, d)))
        X += Fraction(int(m[b])) * Fraction(2) ** int(e[b]) * D * s_k
    return round_f32_grid_then_flush(X)


@pytest.mark.parametrize("scaling", [0, 1])
@pytest.mark.parametrize("d", [64, 96, 128, 256, 320])
def test_int8_score_brute_force(orc, scaling, d):
    """Every score bit for bit against the exact rational sum over the query's
    blocks, rounded once; query blocks of one head up to 2^100 apart."""
    rng = np.random.default_rng(50 + d + scaling)
    q = rng.standard_normal((4, d)).astype(np.float32)
    if scaling == 1:
        for b in range(d // 32):
            q[1, 32 * b:32 * b + 32] *= np.float32(2.0 ** [0, 50, -50, 9, -3, 30, 1, 0, -1, 2][b % 10])
    k = (rng.standard_normal((6, d)) * np.float32(2.0 ** rng.integers(-20, 10, (6, 1)))).astype(np.float32)
    kc, ks = orc.cache_rows(k)
    qc, m, e = orc.quantize_heads(scaling, q)
    blk = 32 if scaling == 1 else d
    for h in range(4):
        for p in range(6):
            got = orc.int8_score(qc[h], m[h], e[h], blk, d, kc[p], ks[p])
            assert bits(got) == _exact_score(qc[h], m[h], e[h], blk, d, kc[p], ks[p]), (h, p)


def test_quantize_heads_padding_and_blocks(orc):
    """Sub32: the head padded with zeros to a whole group, scales per 32 as
    quantize gives them for the padded row; PerBlock: one block of d."""
    rng = np.random.default_rng(60)
    q = rng.standard_normal((3, 96)).astype(np.float32)
    qc, m, e = orc.quantize_heads(1, q)
    pad = np.zeros((3, 256), np.float32)
    pad[:, :96] = q
    c2, m2, e2, _ = orc.quantize_sub32(pad)
    assert np.array_equal(qc, c2) and np.array_equal(m, m2) and np.array_equal(e, e2)
    assert np.all(m[:, 3:] == 8) and np.all(e[:, 3:] == 0) and not qc[:, 96:].any()
    qc, m, e = orc.quantize_heads(0, q)
    c3, m3, e3, _ = orc.quantize_blocks(q, 96)
    assert np.array_equal(qc, c3) and np.array_equal(m, m3) and np.array_equal(e, e3)


def test_int8_score_closed_form(orc):
    """Every query code a under one scale m*2^e, every key code k: the score is
    RNE(ks * m * 2^e * a * k * d)."""
    d, a, kk, mm, ee, ks = 128, 77, -91, 13, -9, 0x2E66
    qc = np.full(256, 0, np.int8)
    qc[:d] = a
    m = np.full(8, mm, np.uint8)
    e = np.full(8, ee, np.int16)
    kc = np.full(d, kk, np.int8)
    got = orc.int8_score(qc, m, e, 32, d, kc, ks)
    s_k = Fraction(float(np.uint16(ks).view(np.float16)))
    assert bits(got) == round_f32_grid_then_flush(s_k * mm * Fraction(2) ** ee * a * kk * d)


def test_int8_score_nan_and_zero(orc):
    rng = np.random.default_rng(61)
    q = rng.standard_normal((2, 128)).astype(np.float32)
    q[1, 40] = np.inf                                  # query block without a scale
    qc, m, e = orc.quantize_heads(1, q)
    k = rng.standard_normal((3, 128)).astype(np.float32)
    k[1] = 0.0                                         # zero key row: scale 0, codes 0 -> +0
    k[2, 3] = np.inf                                   # key scale overflows: unreadable -> NaN
    kc, ks = orc.cache_rows(k)
    assert bits(orc.int8_score(qc[0], m[0], e[0], 32, 128, kc[1], ks[1])) == 0
    assert bits(orc.int8_score(qc[0], m[0], e[0], 32, 128, kc[2], ks[2])) == 0x7FC00000
    assert bits(orc.int8_score(qc[1], m[1], e[1], 32, 128, kc[0], ks[0])) == 0x7FC00000


@pytest.mark.parametrize("scaling", [0, 1])
def test_kv_scores_heads_and_scale(orc, scaling):
    """Query head h reads key head h / (nh / nkv); each score is the f32 product
    of int8_score and the attention scale (numpy's f32 multiply, flushed)."""
    rng = np.random.default_rng(62 + scaling)
    nh, nkv, d, L, lcap = 8, 2, 128, 37, 40
    q = rng.standard_normal((nh, d)).astype(np.float32)
    k = rng.standard_normal((nkv * lcap, d)).astype(np.float32)
    kc, ks = orc.cache_rows(k)
    kc = kc.reshape(nkv, lcap, d)
    ks = ks.reshape(nkv, lcap)
    qc, m, e = orc.quantize_heads(scaling, q)
    scale = np.float32(1.0 / np.sqrt(d))
    out = orc.kv_scores(scaling, qc, m, e, d, kc, ks, L, nkv, scale)
    blk = 32 if scaling == 1 else d
    for h in range(nh):
        for p in range(L):
            s = orc.int8_score(qc[h], m[h], e[h], blk, d, kc[h // 4, p], ks[h // 4, p])
            want = np.float32(s) * scale
            if want != 0 and abs(want) < f32(0x00800000):
                want = np.float32(0.0) * np.sign(want)
            assert bits(out[h, p]) == bits(want), (h, p)
