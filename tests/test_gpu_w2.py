"""Parity of q_gemv_w2 (activation codes that cross in two words: a 16-bit
code a = 256*hi + lo, lane page) with the CPU oracle, bit for bit: every
output is the in-order fold of once-rounded block values, as q_gemv's are."""
import numpy as np
import pytest

import oracle
import block_quantized_weight_quantize_gb300 as qb
from block_quantized_weight_quantize_gb300 import synth
from helpers import bits, dev, host, make_case, oracle_act

pytestmark = pytest.mark.gpu

FMTS = [synth.FMT_Q8_0, synth.FMT_Q4K, synth.FMT_Q6K]


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


def _codes16(rng, ncols, K):
    a = rng.integers(-32768, 32768, (ncols, K)).astype(np.int16)
    special = np.array([-32768, 32767, -1, 0, 1, 255, 256, -256, -255, 127, -128, 128], np.int16)
    a[0, :len(special)] = special
    if ncols > 1:
        a[1, :] = -32768
    if ncols > 2:
        a[2, :] = 32767
    return a


def _gpu(fmt, W, rows, K, a16, m, e):
    import torch
    ncols = a16.shape[0]
    out = torch.full((ncols, rows), float("nan"), dtype=torch.float32, device="cuda")
    qb.q_gemv_w2(fmt, dev(W), rows, K, dev(a16), dev(_packed(m, e)), ncols, out)
    torch.cuda.synchronize()
    return host(out)


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("ncols", [1, 3, 16])
@pytest.mark.parametrize("rows,K", [(1, 256), (37, 1024), (261, 4096), (19, 14336)])
def test_w2_bit_exact(fmt, ncols, rows, K):
    rng = np.random.default_rng(rows + K + ncols + 3 * fmt)
    lg = synth.draw(fmt, rng, rows, K)
    W = synth.pack(fmt, lg)
    a = _codes16(rng, ncols, K)
    nb = K // synth.BLOCK[fmt]
    m = rng.integers(128, 256, (ncols, nb)).astype(np.uint8)
    e = rng.integers(-40, -10, (ncols, nb)).astype(np.int16)
    want = oracle.gemv_w2(fmt, W, rows, K, a, m, e)
    got = _gpu(fmt, W, rows, K, a, m, e)
    assert np.array_equal(bits(got), bits(want))


@pytest.mark.parametrize("fmt", FMTS)
def test_w2_one_word_codes_match_q_gemv(fmt):
    """Codes of one word given as two-word codes: the same bits as q_gemv."""
    import torch
    rows, K, ncols = 300, 2048, 5
    lg, W, x = make_case(fmt, rows, K, ncols, seed=90 + fmt, outliers=0.001)
    codes, m, e, s16, packed = oracle_act(x, synth.BLOCK[fmt])
    want = oracle.gemv(fmt, W, rows, K, codes, m, e)
    out = torch.full((ncols, rows), float("nan"), dtype=torch.float32, device="cuda")
    qb.q_gemv(fmt, dev(W), rows, K, (dev(codes), dev(packed), dev(s16)), ncols, out)
    got1 = _gpu(fmt, W, rows, K, codes.astype(np.int16), m, e)
    assert np.array_equal(bits(host(out)), bits(want))
    assert np.array_equal(bits(got1), bits(want))


@pytest.mark.parametrize("fmt", FMTS)
def test_w2_scales_at_the_edges(fmt):
    """Activation scales across the f32 range (values rounding to subnormal and
    flushed, to infinity), a block without a scale (m = 0), an unreadable
    weight scale: each as the oracle has it."""
    rng = np.random.default_rng(33 + fmt)
    rows, K, ncols = 64, 1024, 4
    lg = synth.draw(fmt, rng, rows, K)
    lg["d"][5, 1] = 0x7C00        # an unreadable block scale
    W = synth.pack(fmt, lg)
    a = _codes16(rng, ncols, K)
    nb = K // synth.BLOCK[fmt]
    m = rng.integers(1, 256, (ncols, nb)).astype(np.uint8)
    e = rng.integers(-40, -10, (ncols, nb)).astype(np.int16)
    e[0, :] = -160                # values far below the f32 range: flushed to zero
    e[1, :] = -140                # values near the bottom of the f32 range
    e[2, 0] = 60                  # values past the top: infinities
    m[3, 1] = 0                   # a block without a scale
    want = oracle.gemv_w2(fmt, W, rows, K, a, m, e)
    got = _gpu(fmt, W, rows, K, a, m, e)
    assert np.array_equal(bits(got), bits(want))
    assert np.all(bits(got[3]) == 0x7FC00000) and np.all(bits(got[:, 5]) == 0x7FC00000)
