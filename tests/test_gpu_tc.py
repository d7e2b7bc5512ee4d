"""Parity of the tensor-core (tcgen05) product of many columns with the CPU
oracle, bit for bit.

The kernel takes Q4_K-like and Q6_K-like matrices from five columns on: the
weights' coefficients and the activation codes go through f16 MMAs with f32
accumulation, which is exact only because every partial sum is an integer
below 2^24.  These cases drive the accumulators to the top of that range and
arrange for the block value to expose the low bits of the integer sums: a
Q4_K-like block whose two terms cancel exactly (d*C = dmin*O) except for a
few perturbed codes, and Q6_K-like blocks whose value is the sum itself times
a power of two.  A single lost bit anywhere changes an output.
"""
import numpy as np
import pytest

import oracle
import block_quantized_weight_quantize_gb300 as qb
from block_quantized_weight_quantize_gb300 import synth
from helpers import bits, dev, host, make_case, oracle_act

pytestmark = pytest.mark.gpu

Q4K, Q6K = synth.FMT_Q4K, synth.FMT_Q6K


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    import torch
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    qb.lib()
    yield
    torch.cuda.synchronize()
    assert qb.q_device_status() == qb.QB_OK


def _gpu(fmt, W, rows, K, x, ncols):
    import torch
    blk = synth.BLOCK[fmt]
    codes, scales, sums = qb.alloc_act(ncols, K, blk)
    qb.quantize_act(blk, dev(x), codes, scales, sums)
    out = torch.full((ncols, rows), float("nan"), dtype=torch.float32, device="cuda")
    qb.q_gemv(fmt, dev(W), rows, K, (codes, scales, sums), ncols, out)
    torch.cuda.synchronize()
    return host(out)


def _want(fmt, W, rows, K, x):
    codes, m, e, s16, packed = oracle_act(x, synth.BLOCK[fmt])
    return oracle.gemv(fmt, W, rows, K, codes, m, e)


@pytest.mark.parametrize("fmt", [Q4K, Q6K])
@pytest.mark.parametrize("ncols", [5, 9, 16])
@pytest.mark.parametrize("rows,K", [(1, 256), (127, 512), (128, 1024), (129, 2304), (300, 4096), (4101, 4096),
                                    (260, 8192), (200, 14336)])
def test_tc_shapes(fmt, ncols, rows, K):
    """One or several 128-row tiles (a ragged last one), one block a row up
    to 56, and the cluster splits of the blocks those give."""
    lg, W, x = make_case(fmt, rows, K, ncols, seed=3 * rows + K + ncols + fmt, outliers=0.001)
    got = _gpu(fmt, W, rows, K, x, ncols)
    want = _want(fmt, W, rows, K, x)
    assert np.array_equal(bits(got), bits(want))


def _extreme_activation(ncols, K, rng):
    """Codes at +-127 under m = 128 (x = +-127/128): all positive, all
    negative, alternating, half-block halves of opposite sign, then random."""
    x = rng.standard_normal(size=(ncols, K)).astype(np.float32)
    a = np.float32(127.0 / 128.0)
    idx = np.arange(K)
    x[0] = a
    x[1] = -a
    x[2] = np.where(idx % 2 == 0, a, -a)
    x[3] = np.where((idx // 64) % 2 == 0, a, -a)
    x[4] = a
    x[4, rng.integers(0, K, size=K // 64)] = np.float32(0.25)
    return x


def test_tc_q4k_cancelling_extremes():
    """Q4_K-like: sc = mn = 63, q = 15 and dmin = 15*d, so d*C - dmin*O is
    zero unless a few codes are perturbed; half-block sums reach
    945*127*128 = 15,362,560 and O reaches 8*63*4064."""
    rows, K, ncols = 256, 1024, 16
    rng = np.random.default_rng(11)
    lg = synth.draw(Q4K, rng, rows, K)
    nb = K // 256
    lg["q"][:] = 15
    lg["sc"][:] = 63
    lg["mn"][:] = 63
    lg["d"][:] = 0x1400      # 2^-10
    lg["dmin"][:] = 0x2380   # 15 * 2^-10
    for r in range(rows):
        kind = r % 4
        if kind == 1:        # a few codes one lower: a small, exactly visible value
            lg["q"][r, rng.integers(0, K, size=3)] = 14
        elif kind == 2:      # random codes under the extreme scales
            lg["q"][r] = rng.integers(0, 16, size=K)
        elif kind == 3:      # random codes, some zero half blocks
            lg["q"][r] = rng.integers(0, 16, size=K)
            lg["q"][r, 128:256] = 0
    W = synth.pack(Q4K, lg)
    x = _extreme_activation(ncols, K, rng)
    got = _gpu(Q4K, W, rows, K, x, ncols)
    want = _want(Q4K, W, rows, K, x)
    assert np.any(bits(want[:5, 1::4]) != 0)   # the perturbed rows are not zero
    assert np.array_equal(bits(got), bits(want))


def test_tc_q6k_accumulator_extremes():
    """Q6_K-like with d = 2^-24 (the least subnormal) and m = 128: a block's
    value is C * 2^(e-17), exact while |C| < 2^24, so each sum shows in the
    output.  sc = -128 (hi = -8, lo = 0) with q = 0 drives the hi accumulator
    to 8*32*127*256; sc = 15 (hi = 0, lo = 15) the lo one to 15*32*127*256."""
    rows, K, ncols = 200, 1024, 16
    rng = np.random.default_rng(12)
    lg = synth.draw(Q6K, rng, rows, K)
    lg["d"][:] = 0x0001
    for r in range(rows):
        kind = r % 5
        if kind == 0:
            lg["sc"][r] = -128
            lg["q"][r] = 0
        elif kind == 1:
            lg["sc"][r] = 15
            lg["q"][r] = 0
        elif kind == 2:
            lg["sc"][r] = -128
            lg["q"][r] = 0
            lg["q"][r, rng.integers(0, K, size=5)] = 1
        elif kind == 3:
            lg["sc"][r] = 127
            lg["q"][r] = 63
    W = synth.pack(Q6K, lg)
    x = _extreme_activation(ncols, K, rng)
    got = _gpu(Q6K, W, rows, K, x, ncols)
    want = _want(Q6K, W, rows, K, x)
    assert np.array_equal(bits(got), bits(want))


@pytest.mark.parametrize("fmt", [Q4K, Q6K])
def test_tc_column_subsets_match_single_columns(fmt):
    """Column c of a 16-column product equals the one-column product of that
    column (the one-column kernels share no code with the tensor-core one)."""
    rows, K = 333, 2048
    lg, W, x = make_case(fmt, rows, K, 16, seed=90 + fmt, outliers=0.001)
    allc = _gpu(fmt, W, rows, K, x, 16)
    for c in (0, 7, 15):
        one = _gpu(fmt, W, rows, K, x[c:c + 1].copy(), 1)
        assert np.array_equal(bits(one[0]), bits(allc[c]))


@pytest.mark.parametrize("fmt", [Q4K, Q6K])
def test_tc_grouped_matrices(fmt):
    """Three matrices sharing an activation in one call (q_gemv_many)."""
    import torch
    K, ncols = 2048, 12
    rows_l = [300, 129, 1]
    rng = np.random.default_rng(40 + fmt)
    Ws = [synth.pack(fmt, synth.draw(fmt, rng, r, K)) for r in rows_l]
    x = synth.draw_act(rng, ncols, K, outlier_frac=0.001)
    blk = synth.BLOCK[fmt]
    codes, scales, sums = qb.alloc_act(ncols, K, blk)
    qb.quantize_act(blk, dev(x), codes, scales, sums)
    outs = [torch.full((ncols, r), float("nan"), dtype=torch.float32, device="cuda") for r in rows_l]
    qb.q_gemv_many(fmt, [dev(W) for W in Ws], rows_l, K, (codes, scales, sums), ncols, outs)
    torch.cuda.synchronize()
    for W, r, o in zip(Ws, rows_l, outs):
        assert np.array_equal(bits(host(o)), bits(_want(fmt, W, r, K, x)))
