"""The int8 cache's score path on the GPU against the oracle, bit for bit
(numerics page: cache_row, int8_codes, INV_127, quantize_head, int8_score).

Cache rows (codes and f16 scales) and quantized query heads are compared
element for element; the scores are computed on the GPU from the ORACLE's
cache rows and query codes (so the score kernel is tested on its own) and
compared score for score, for both scalings, head sizes on the tensor-core
path (64, 128, 256) and off it (96, 320, 1024), grouped-query layouts with
one, several and a padded second chunk of query heads per key head, ragged
lengths, a key-head stride past the length, query blocks far apart (the exact
routine), blocks without a scale and key rows whose scale overflowed.
"""
import numpy as np
import pytest

import oracle
import block_quantized_weight_quantize_gb300 as qb
from helpers import bits, dev, host

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    import torch
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    qb.lib()
    yield
    torch.cuda.synchronize()
    assert qb.q_device_status() == qb.QB_OK


def _packed(m, e):
    return (m.astype(np.uint32) | (e.astype(np.int32).astype(np.uint32) << 16)).view(np.int32)


def _rows(rng, n, d, specials=True):
    x = (rng.standard_normal((n, d)) * np.float32(2.0) ** rng.integers(-30, 30, (n, 1))).astype(np.float32)
    if specials and n >= 8:
        x[0] = 0.0                                   # scale 0, codes 0
        x[1, 3] = np.inf                             # scale overflows binary16, codes 0
        x[2, 5] = np.nan
        x[2, 6] = np.float32(1e-41)                  # denormal
        x[3] *= np.float32(1e-30)                    # scale rounds to zero
        x[4] *= np.float32(1e6)                      # scale near the top of binary16
        x[5] = np.float32(2.5)                       # every x*inv near 127
    return x


@pytest.mark.parametrize("d", [64, 96, 128, 256, 1024])
def test_kv_cache_rows_bit_exact(d):
    import torch
    rng = np.random.default_rng(d)
    x = _rows(rng, 300, d)
    codes, scales = oracle.cache_rows(x)
    gc = torch.empty((300, d), dtype=torch.int8, device="cuda")
    gs = torch.empty(300, dtype=torch.int16, device="cuda")
    qb.kv_cache_rows(dev(x), gc, gs)
    torch.cuda.synchronize()
    assert np.array_equal(host(gs).view(np.uint16), scales)
    assert np.array_equal(host(gc), codes)


@pytest.mark.parametrize("scaling", [qb.PERBLOCK, qb.SUB32])
@pytest.mark.parametrize("d", [64, 96, 128, 256, 320, 1024])
def test_kv_quantize_heads_bit_exact(scaling, d):
    import torch
    rng = np.random.default_rng(d + 7 * scaling)
    q = rng.standard_normal((13, d)).astype(np.float32)
    q[1] *= np.float32(2.0 ** -120)
    q[2, 7] = np.inf
    q[3] = 0.0
    q[4, ::2] *= np.float32(2.0 ** 40)
    codes, m, e = oracle.quantize_heads(scaling, q)
    dp = qb.kv_head_codes(scaling, d)
    nbq = dp // 32 if scaling == qb.SUB32 else 1
    gc = torch.empty((13, dp), dtype=torch.int8, device="cuda")
    gs = torch.empty((13, nbq), dtype=torch.int32, device="cuda")
    qb.kv_quantize_heads(scaling, dev(q), gc, gs)
    torch.cuda.synchronize()
    assert np.array_equal(host(gs), _packed(m, e))
    assert np.array_equal(host(gc), codes)


def _scores_case(scaling, d, nh, nkv, L, lcap, seed, spread_heads=False):
    import torch
    rng = np.random.default_rng(seed)
    q = rng.standard_normal((nh, d)).astype(np.float32)
    if spread_heads:
        for b in range(d // 32):
            q[0, 32 * b:32 * b + 32] *= np.float32(2.0 ** [0, 40, -40, 5, -90, 2, 1, 0][b % 8])
        q[1, 3] = np.inf                             # query block without a scale
    k = _rows(rng, nkv * lcap, d)
    kc, ks = oracle.cache_rows(k)
    kc = kc.reshape(nkv, lcap, d)
    ks = ks.reshape(nkv, lcap)
    qc, m, e = oracle.quantize_heads(scaling, q)
    scale = np.float32(1.0 / np.sqrt(d))
    want = oracle.kv_scores(scaling, qc, m, e, d, kc, ks, L, nkv, scale)
    out = torch.full((nh, L), float("nan"), dtype=torch.float32, device="cuda")
    qb.kv_scores(scaling, dev(qc), dev(_packed(m, e)), d, dev(kc), dev(ks.view(np.int16)), L, float(scale), out)
    torch.cuda.synchronize()
    return host(out), want


@pytest.mark.parametrize("scaling", [qb.PERBLOCK, qb.SUB32])
@pytest.mark.parametrize("d", [64, 128, 256, 96, 320])
@pytest.mark.parametrize("nh,nkv", [(8, 2), (32, 8), (12, 1), (4, 4)])
def test_kv_scores_bit_exact(scaling, d, nh, nkv):
    got, want = _scores_case(scaling, d, nh, nkv, L=37, lcap=45, seed=d + nh + 3 * scaling)
    assert np.array_equal(bits(got), bits(want))


@pytest.mark.parametrize("scaling", [qb.PERBLOCK, qb.SUB32])
@pytest.mark.parametrize("d", [128, 256, 1024])
def test_kv_scores_exact_routine_and_nan(scaling, d):
    got, want = _scores_case(scaling, d, nh=16, nkv=2, L=300, lcap=300, seed=99 + d, spread_heads=True)
    assert np.array_equal(bits(got), bits(want))
    assert np.all(bits(want[1]) == 0x7FC00000)


@pytest.mark.parametrize("scaling", [qb.PERBLOCK, qb.SUB32])
def test_kv_scores_long_context(scaling):
    """32 query heads on 8 key heads of 128, 32768 cached positions."""
    got, want = _scores_case(scaling, 128, nh=32, nkv=8, L=32768 - 5, lcap=32768, seed=5 + scaling)
    assert np.array_equal(bits(got), bits(want))


@pytest.mark.parametrize("rows_last", [False, True])
def test_kv_pipeline(rows_last):
    """kv_cache_rows and kv_quantize_heads on the GPU, then kv_scores, against
    the oracle's cache_row, quantize_head and scores.  rows_last: the cache
    rows are written by the launch right before kv_scores, on the same stream
    with no synchronisation between (the score kernel requests key tiles
    before its dependency wait; kv_cache_rows lets it start only once the rows
    are written), the cache filled with stale bytes beforehand."""
    import torch
    rng = np.random.default_rng(123)
    nh, nkv, d, L = 16, 4, 128, 1000
    q = rng.standard_normal((nh, d)).astype(np.float32)
    k = rng.standard_normal((nkv * L, d)).astype(np.float32)
    for scaling in (qb.PERBLOCK, qb.SUB32):
        kc = torch.full((nkv, L, d), 77, dtype=torch.int8, device="cuda")
        ks = torch.full((nkv, L), 0x3C00, dtype=torch.int16, device="cuda")
        dp = qb.kv_head_codes(scaling, d)
        qc = torch.empty((nh, dp), dtype=torch.int8, device="cuda")
        qs = torch.empty((nh, dp // 32 if scaling == qb.SUB32 else 1), dtype=torch.int32, device="cuda")
        torch.cuda.synchronize()
        if rows_last:
            qb.kv_quantize_heads(scaling, dev(q), qc, qs)
            qb.kv_cache_rows(dev(k), kc.view(nkv * L, d), ks.view(-1))
        else:
            qb.kv_cache_rows(dev(k), kc.view(nkv * L, d), ks.view(-1))
            qb.kv_quantize_heads(scaling, dev(q), qc, qs)
        out = torch.empty((nh, L), dtype=torch.float32, device="cuda")
        qb.kv_scores(scaling, qc, qs, d, kc, ks, L, 0.125, out)
        torch.cuda.synchronize()
        okc, oks = oracle.cache_rows(k)
        oqc, om, oe = oracle.quantize_heads(scaling, q)
        want = oracle.kv_scores(scaling, oqc, om, oe, d, okc.reshape(nkv, L, d), oks.reshape(nkv, L), L, nkv, 0.125)
        assert np.array_equal(bits(host(out)), bits(want))


def test_kv_argument_checks():
    import torch
    x = torch.zeros((4, 72), dtype=torch.float32, device="cuda")
    with pytest.raises(qb.QbError):   # d % 16 != 0
        qb.kv_cache_rows(x, torch.empty((4, 72), dtype=torch.int8, device="cuda"),
                         torch.empty(4, dtype=torch.int16, device="cuda"))
    qc = torch.zeros((6, 128), dtype=torch.int8, device="cuda")
    qs = torch.zeros((6, 1), dtype=torch.int32, device="cuda")
    kc = torch.zeros((4, 8, 128), dtype=torch.int8, device="cuda")
    ks = torch.zeros((4, 8), dtype=torch.int16, device="cuda")
    out = torch.zeros((6, 8), dtype=torch.float32, device="cuda")
    with pytest.raises(qb.QbError):   # 6 query heads on 4 key heads
        qb.kv_scores(qb.PERBLOCK, qc, qs, 128, kc, ks, 8, 1.0, out)
    with pytest.raises(qb.QbError):   # L past the key stride
        qb.kv_scores(qb.PERBLOCK, qc[:4], qs[:4], 128, kc, ks, 9, 1.0, out)
