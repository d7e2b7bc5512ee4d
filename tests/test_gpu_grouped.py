"""Several matrices sharing one activation (bankML forward page: mv_many, qkv;
bankML f16 page: mat_vec_multi_par), through the C ABI's grouped calls.

Each matrix's output must be bit for bit what the oracle gives for that
matrix alone (and so what a separate q_gemv gives): grouping changes launches,
not arithmetic.  Shapes put matrix boundaries inside CTAs' row ranges and
inside one bulk fill, include an empty matrix, and include shapes the
streaming kernels do not take (the per-matrix fallback).
"""
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


def _mats(fmt, rows_list, K, seed):
    rng = np.random.default_rng(seed)
    out = []
    for rows in rows_list:
        if rows == 0:
            out.append(np.zeros(0, np.uint8))
            continue
        lg = synth.draw(fmt, rng, rows, K)
        out.append(synth.pack(fmt, lg))
    return out


def _outs(rows_list, ncols):
    import torch
    # an empty matrix still gets a valid (unused) output pointer
    return [torch.full((ncols, max(r, 1)), float("nan"), dtype=torch.float32, device="cuda") for r in rows_list]


def _dev_w(Wh):
    import torch
    # an empty matrix still needs a (16-byte aligned) device pointer
    return dev(Wh) if Wh.size else torch.zeros(16, dtype=torch.uint8, device="cuda")


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("ncols", [1, 3, 16])
@pytest.mark.parametrize("rows_list,K", [([300, 77, 0, 129], 2048), ([4096, 1024, 1024], 4096), ([5, 3], 256),
                                         ([1001, 2000, 513], 4096), ([333, 21, 150], 14336)])
def test_gemv_many_bit_exact(fmt, ncols, rows_list, K):
    import torch
    Ws = _mats(fmt, rows_list, K, seed=sum(rows_list) + ncols + fmt)
    rng = np.random.default_rng(K + ncols)
    x = synth.draw_act(rng, ncols, K, outlier_frac=0.001)
    blk = synth.BLOCK[fmt]
    codes, m, e, s16, packed = oracle_act(x, blk)
    act = qb.alloc_act(ncols, K, blk)
    qb.quantize_act(blk, dev(x), *act)
    outs = _outs(rows_list, ncols)
    qb.q_gemv_many(fmt, [_dev_w(W) for W in Ws], rows_list, K, act, ncols, outs)
    torch.cuda.synchronize()
    for Wh, rows, o in zip(Ws, rows_list, outs):
        if rows == 0:
            continue
        want = oracle.gemv(fmt, Wh, rows, K, codes, m, e)
        assert np.array_equal(bits(host(o)), bits(want)), (rows, K)


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("ncols", [1, 3])
@pytest.mark.parametrize("rows_list,K", [([700, 152 * 2 + 3, 64], 1024), ([1001, 2000, 513], 4096),
                                         ([1001, 20, 513], 14336), ([77, 130], 10240)])
def test_matvec_many_matches_separate_calls(fmt, ncols, rows_list, K):
    """q_matvec_many (one launch for one column) against q_matvec per matrix;
    the warp-ring one-column kernel takes K = 4096 (under 49 rows a CTA),
    10240 and 14336 (rows in passes, the last one partial), with matrix
    boundaries inside row pairs."""
    import torch
    Ws = [dev(W) for W in _mats(fmt, rows_list, K, seed=11 + fmt)]
    x = dev(synth.draw_act(np.random.default_rng(3), ncols, K, outlier_frac=0.001))
    ws = torch.empty(qb.q_matvec_workspace_bytes(fmt, K, ncols) + 16, dtype=torch.uint8, device="cuda")
    outs = _outs(rows_list, ncols)
    qb.q_matvec_many(fmt, Ws, rows_list, K, x, outs, workspace=ws)
    torch.cuda.synchronize()
    for W, rows, o in zip(Ws, rows_list, outs):
        one = torch.full((ncols, rows), float("nan"), dtype=torch.float32, device="cuda")
        qb.q_matvec(fmt, W, rows, K, x, one, workspace=ws)
        torch.cuda.synchronize()
        assert np.array_equal(bits(host(o)), bits(host(one)))


def test_gemv_many_fallback_shapes():
    """Q8_0 with K % 256 != 0 (no streaming kernel): one launch per matrix, same bits."""
    import torch
    fmt, rows_list, K, ncols = synth.FMT_Q8_0, [40, 9], 96, 2
    Ws = _mats(fmt, rows_list, K, seed=5)
    x = synth.draw_act(np.random.default_rng(9), ncols, K)
    codes, m, e, s16, packed = oracle_act(x, 32)
    act = qb.alloc_act(ncols, K, 32)
    qb.quantize_act(32, dev(x), *act)
    outs = _outs(rows_list, ncols)
    qb.q_gemv_many(fmt, [dev(W) for W in Ws], rows_list, K, act, ncols, outs)
    torch.cuda.synchronize()
    for Wh, rows, o in zip(Ws, rows_list, outs):
        assert np.array_equal(bits(host(o)), bits(oracle.gemv(fmt, Wh, rows, K, codes, m, e)))


@pytest.mark.parametrize("ncols", [1, 2, 6])
@pytest.mark.parametrize("rows_list,K", [([1536, 576, 0, 300], 576), ([129, 13], 1536), ([5, 40], 16384)])
def test_gemv_f16_many_bit_exact(ncols, rows_list, K):
    """F16 (the pages' mat_vec_multi_par shape: Q, K, V of one layer); K = 16384
    takes the row-per-thread kernel, one launch per matrix."""
    import torch
    if ncols * K * 4 > 227 * 1024:
        ncols = 1
    rng = np.random.default_rng(K + ncols)
    Ws = [synth.draw_f16(rng, max(r, 0), K) for r in rows_list]
    x = synth.draw_act(rng, ncols, K)
    x16 = oracle.quantize_f16(x)
    outs = _outs(rows_list, ncols)
    Wd = [dev(W.view(np.int16)) if W.size else torch.zeros(8, dtype=torch.int16, device="cuda") for W in Ws]
    qb.q_gemv_f16_many(Wd, rows_list, K, dev(x16.view(np.int16)), ncols, outs)
    torch.cuda.synchronize()
    for W, rows, o in zip(Ws, rows_list, outs):
        if rows == 0:
            continue
        want = oracle.gemv_f16(W, rows, K, x16)
        assert np.array_equal(bits(host(o)), bits(want)), (rows, K)


def test_grouped_argument_checks():
    import torch
    K = 256
    W = torch.zeros(synth.record_bytes(synth.FMT_Q4K, K) * 4, dtype=torch.uint8, device="cuda")
    act = qb.alloc_act(1, K, 256)
    outs = _outs([4] * 5, 1)
    with pytest.raises(qb.QbError):   # more than QB_MAX_MATS matrices
        qb.q_gemv_many(qb.Q4K, [W] * 5, [4] * 5, K, act, 1, outs)
    with pytest.raises(qb.QbError):   # a misaligned weight pointer
        qb.q_gemv_many(qb.Q4K, [W, W[1:]], [4, 3], K, act, 1, outs[:2])
