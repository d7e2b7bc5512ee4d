"""FP8 E4M3 weights with 128x128 block scales on the GPU (colizig OPS page,
FP8: e4m3ToF32, dequantRow, matmulFp8) against the oracle.

The decode is checked bit for bit on every byte value (one-hot activations
read single weights exactly); the products are a float path, held to the f32
summation bound (K + 4) * 2^-24 * sum |x_i * w_i| (plus K subnormal quanta)
around the oracle's exact dot of the dequantized weights, over shapes with a
partial last round of chunks, a single chunk, the longest rows (one column a
launch) and 1..16 columns; NaN weights and infinite activations propagate as
on the oracle.
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


def _draw(rng, rows, K):
    W = rng.integers(0, 256, size=(rows, K), dtype=np.uint8)
    W[(W & 0x7F) == 0x7F] = 0x3C                      # no NaN codes
    scales = (2.0 ** rng.uniform(-12, -4, size=((rows + 127) // 128, (K + 127) // 128))).astype(np.float32)
    return W, scales


def _gpu(W, scales, rows, K, x):
    import torch
    out = torch.full((x.shape[0], rows), float("nan"), dtype=torch.float32, device="cuda")
    qb.q_gemv_fp8(dev(W), dev(scales), rows, K, dev(x), out)
    torch.cuda.synchronize()
    return host(out)


def _within_bound(got, want, ab, K, sq=None):
    """The rigorous bound; with sq (sum of squared terms) also the random-walk
    scale 8 * 2^-24 * sqrt(K * sq) for 99 % of the outputs, which a dropped or
    misscaled 16-element chunk exceeds by orders of magnitude."""
    tol = (K + 4) * 2.0 ** -24 * ab + K * 2.0 ** -149
    fin = np.isfinite(want)
    assert np.array_equal(fin, np.isfinite(got))
    err = np.abs(got[fin].astype(np.float64) - want[fin].astype(np.float64))
    assert np.all(err <= tol[fin])
    if sq is not None:
        assert np.mean(err > 8 * 2.0 ** -24 * np.sqrt(K * sq[fin])) < 0.01


def _sum_sq(W, scales, x):
    """sum over i of (x_i * w_i)^2 for every (column, row), the weights dequantized by the oracle."""
    lut = np.array([oracle.e4m3_to_f32(b) for b in range(256)], np.float64)
    rows, K = W.shape
    w = lut[W] * np.repeat(np.repeat(scales.astype(np.float64), 128, 0)[:rows], 128, 1)[:, :K]
    return (x.astype(np.float64) ** 2) @ (w ** 2).T


def test_fp8_decode_every_byte():
    """Rows 0 and 1 hold every finite byte value (the NaN codes replaced by
    zeros, in two orders); with unit scales, x = e_i reads W[r][i] exactly (one
    product), so each output is the decoded byte, bit for bit.  Row 2 holds
    NaN codes only: NaN for every column."""
    K, rows = 256, 3
    W = np.tile(np.arange(256, dtype=np.uint8), (rows, 1))
    W[:2, 0x7F] = 0
    W[:2, 0xFF] = 0
    W[1] = W[1][::-1]
    W[2, :128] = 0x7F
    W[2, 128:] = 0xFF
    scales = np.ones((1, 2), np.float32)
    for i0 in range(0, 256, 16):
        x = np.zeros((16, K), np.float32)
        for c in range(16):
            x[c, i0 + c] = 1.0
        got = _gpu(W, scales, rows, K, x)
        want, _ = oracle.gemv_fp8(W, scales, rows, K, x)
        assert np.array_equal(bits(got), bits(want)), i0
        assert np.all(bits(got[:, 2]) == 0x7FC00000)


@pytest.mark.parametrize("ncols", [1, 3, 16])
@pytest.mark.parametrize("rows,K", [(4096, 4096), (300, 1024), (1000, 640), (129, 16), (77, 32768)])
def test_fp8_gemv_within_bound(rows, K, ncols):
    rng = np.random.default_rng(rows + K + ncols)
    W, scales = _draw(rng, rows, K)
    x = rng.standard_normal((ncols, K)).astype(np.float32)
    got = _gpu(W, scales, rows, K, x)
    want, ab = oracle.gemv_fp8(W, scales, rows, K, x)
    _within_bound(got, want, ab, K, _sum_sq(W, scales, x) if rows * K <= 4096 * 4096 else None)


def test_fp8_nan_and_infinity():
    rng = np.random.default_rng(9)
    rows, K = 260, 512
    W, scales = _draw(rng, rows, K)
    W[7, 100] = 0x7F                                  # a NaN weight: row 7 NaN
    x = rng.standard_normal((3, K)).astype(np.float32)
    x[1, 200] = np.inf                                # column 1: +-inf or NaN as the oracle has it
    got = _gpu(W, scales, rows, K, x)
    want, ab = oracle.gemv_fp8(W, scales, rows, K, x)
    assert np.all(bits(got[:, 7]) == 0x7FC00000)
    assert np.array_equal(np.isnan(got), np.isnan(want))
    inf = np.isinf(want)
    assert np.array_equal(got[inf], want[inf])
    fin = np.isfinite(want)
    tol = (K + 4) * 2.0 ** -24 * ab + K * 2.0 ** -149
    assert np.all(np.abs(got[fin].astype(np.float64) - want[fin]) <= tol[fin])


def test_fp8_argument_checks():
    import torch
    W = torch.zeros((4, 48), dtype=torch.uint8, device="cuda")
    s = torch.ones((1, 1), dtype=torch.float32, device="cuda")
    x = torch.zeros((1, 40), dtype=torch.float32, device="cuda")
    out = torch.zeros((1, 4), dtype=torch.float32, device="cuda")
    with pytest.raises(qb.QbError):   # K % 16 != 0
        qb.q_gemv_fp8(W, s, 4, 40, x, out)
    x17 = torch.zeros((17, 48), dtype=torch.float32, device="cuda")
    with pytest.raises(qb.QbError):   # 17 columns
        qb.q_gemv_fp8(W, s, 4, 48, x17, torch.zeros((17, 4), dtype=torch.float32, device="cuda"))
