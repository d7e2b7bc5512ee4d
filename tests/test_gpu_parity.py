"""Parity of the CUDA path (through the C ABI) with the CPU oracle.

Integer results (activation codes, scales, unit sums, block sums C and O) and
every block's once-rounded f32 value must match bit for bit.  Rows must match
within |delta| <= 1e-5 * sum_b |v_b| (the product's stated tolerance, which
allows a tree fold of the block values); the kernels fold in block order as
the oracle does, so the tests demand -- and check -- bit equality.
"""
import numpy as np
import pytest

import oracle
import block_quantized_weight_quantize_gb300 as qb
from block_quantized_weight_quantize_gb300 import synth
from helpers import bits, dev, host, make_case, oracle_act, unpack_scales

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


def gpu_quantize(x: np.ndarray, block: int):
    import torch
    ncols, K = x.shape
    codes, scales, sums = qb.alloc_act(ncols, K, block)
    qb.quantize_act(block, dev(x), codes, scales, sums)
    torch.cuda.synchronize()
    return codes, scales, sums


def gpu_rows(fmt, W, rows, K, act, ncols):
    import torch
    out = torch.full((ncols, rows), float("nan"), dtype=torch.float32, device="cuda")
    qb.q_gemv(fmt, dev(W) if isinstance(W, np.ndarray) else W, rows, K, act, ncols, out)
    torch.cuda.synchronize()
    return host(out)


def tolerance_ok(got, want, v_abs_sum):
    return np.all(np.abs(got.astype(np.float64) - want.astype(np.float64)) <= 1e-5 * v_abs_sum)


# ---------------------------------------------------------------- quantize_act

def _edge_activation(ncols, K, block, seed):
    rng = np.random.default_rng(seed)
    x = synth.draw_act(rng, ncols, K, outlier_frac=0.001)
    nb = K // block
    planted = [
        lambda b: 0.0,                                           # all-zero block
        lambda b: np.float32(1e-38) * x[0, b],                   # bottom of the f32 range
        lambda b: np.float32(1e37) * x[0, b],                    # top of the f32 range
        lambda b: np.round(x[0, b] * 4) / 4,                     # many exact ties
    ]
    for i, f in enumerate(planted):
        if i < nb:
            sl = slice(i * block, (i + 1) * block)
            x[0, sl] = f(sl)
    if nb > 4:
        x[0, 4 * block + 3] = np.nan                             # NaN element
        x[0, 4 * block + 5] = np.uint32(0x00012345).view(np.float32)   # denormal element
    if nb > 5:
        x[0, 5 * block + 1] = np.inf                              # a block with an infinity
    if nb > 6:
        x[0, 6 * block:7 * block] = np.uint32(0x00000042).view(np.float32)  # only denormals
    return x


@pytest.mark.parametrize("block,K", [(32, 1024), (256, 4096), (32, 96), (256, 256)])
@pytest.mark.parametrize("ncols", [1, 3, 16])
def test_quantize_act_bit_exact(block, K, ncols):
    x = _edge_activation(ncols, K, block, seed=block + ncols + K)
    codes, m, e, s16, packed = oracle_act(x, block)
    gc, gs, gsum = gpu_quantize(x, block)
    assert np.array_equal(host(gc), codes)
    gm, ge = unpack_scales(host(gs))
    assert np.array_equal(gm, m) and np.array_equal(ge, e)
    assert np.array_equal(host(gsum), s16)


def test_quantize_every_scale_significand():
    """Blocks whose absmax is exactly 127*m*2^e for every m in 128..255 (so
    wide_scale picks that m), filled with values drawn over the whole range and
    with halfway points k*s + s/2, quantized by quantize_act and inside the
    single-launch product's prologue (q_matvec), equal the oracle's codes and
    rows: the reciprocal of each m the fast path scales by is the right one."""
    import torch
    rng = np.random.default_rng(4242)
    nb = 128
    K = 256 * nb
    x = np.empty((1, K), np.float32)
    for i, m in enumerate(range(128, 256)):
        e = int(rng.integers(-20, 10))
        s = np.float64(m) * 2.0 ** e
        blk = rng.uniform(-127 * s, 127 * s, 256)
        blk[:64] = (rng.integers(-127, 127, 64) + 0.5) * s        # halfway points, exact in f32
        blk[64] = 127 * s                                           # the block's absmax
        x[0, 256 * i:256 * (i + 1)] = blk.astype(np.float32)
    codes, m, e, s16, packed = oracle_act(x, 256)
    assert sorted(set(m.ravel().tolist())) == list(range(128, 256))
    gc, gs, gsum = gpu_quantize(x, 256)
    assert np.array_equal(host(gc), codes)
    gm, ge = unpack_scales(host(gs))
    assert np.array_equal(gm, m) and np.array_equal(ge, e)
    assert np.array_equal(host(gsum), s16)
    # the same blocks through the single-launch product (K = 4096 slices)
    for j in range(nb // 16):
        xs = np.ascontiguousarray(x[:, 4096 * j:4096 * (j + 1)])
        W = synth.pack_q4k(**synth.draw_q4k(rng, 300, 4096))
        cj, mj, ej, _, _ = oracle_act(xs, 256)
        want = oracle.gemv(synth.FMT_Q4K, W, 300, 4096, cj, mj, ej)
        out = torch.full((1, 300), float("nan"), dtype=torch.float32, device="cuda")
        qb.q_matvec(synth.FMT_Q4K, dev(W), 300, 4096, dev(xs), out)
        torch.cuda.synchronize()
        assert np.array_equal(bits(host(out)), bits(want)), j


# ---------------------------------------------------------------- block values (the lane)

SHAPES = {synth.FMT_Q8_0: [(37, 1024), (129, 2048), (5, 32)],
          synth.FMT_Q4K: [(37, 1024), (130, 4096), (3, 256)],
          synth.FMT_Q6K: [(37, 1024), (130, 4096), (3, 256)]}


@pytest.mark.parametrize("fmt", FMTS)
def test_block_values_bit_exact(fmt):
    import torch
    for si, (rows, K) in enumerate(SHAPES[fmt]):
        for ncols in (1, 4):
            lg, W, x = make_case(fmt, rows, K, ncols, seed=100 * fmt + si, outliers=0.001)
            blk = synth.BLOCK[fmt]
            codes, m, e, s16, packed = oracle_act(x, blk)
            C, O, v = oracle.block_values(fmt, W, rows, K, codes, m, e)
            nb = K // blk
            gC = torch.empty((ncols, rows, nb), dtype=torch.int32, device="cuda")
            gO = torch.empty_like(gC)
            gv = torch.empty((ncols, rows, nb), dtype=torch.float32, device="cuda")
            qb.q_block_values(fmt, dev(W), rows, K, (dev(codes), dev(packed), dev(s16)), ncols, gC, gO, gv)
            torch.cuda.synchronize()
            assert np.array_equal(host(gC), C), (rows, K, ncols)
            assert np.array_equal(host(gO), O), (rows, K, ncols)
            assert np.array_equal(bits(host(gv)), bits(v)), (rows, K, ncols)


def test_block_values_wide_exponent_spread():
    """Q4_K blocks whose d and dmin exponents lie far apart (up to the whole f16
    range, subnormals included) take the 128-bit combine; still bit-exact."""
    import torch
    rng = np.random.default_rng(77)
    rows, K = 64, 1024
    lg = synth.draw_q4k(rng, rows, K)
    extremes = np.array([0x0001, 0x0003, 0x03FF, 0x0400, 0x7BFF, 0x7800, 0x3C00, 0x1234], np.uint16)
    lg["d"] = rng.choice(extremes, size=lg["d"].shape).astype(np.uint16)
    lg["dmin"] = rng.choice(extremes, size=lg["dmin"].shape).astype(np.uint16)
    lg["d"][0, 0], lg["dmin"][0, 0] = 0x0001, 0x7BFF          # spread 2^-24 vs 65504
    lg["d"][1, 0], lg["dmin"][1, 0] = 0x7BFF, 0x0001
    W = synth.pack_q4k(**lg)
    x = synth.draw_act(rng, 2, K) * np.float32(1e-30)         # push values toward the f32 bottom too
    x[1] *= np.float32(1e35)
    codes, m, e, s16, packed = oracle_act(x, 256)
    C, O, v = oracle.block_values(synth.FMT_Q4K, W, rows, K, codes, m, e)
    gv = torch.empty((2, rows, K // 256), dtype=torch.float32, device="cuda")
    qb.q_block_values(synth.FMT_Q4K, dev(W), rows, K, (dev(codes), dev(packed), dev(s16)), 2, None, None, gv)
    torch.cuda.synchronize()
    assert np.array_equal(bits(host(gv)), bits(v))


# ---------------------------------------------------------------- rows

@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("ncols", [1, 2, 3, 4, 5, 8, 13, 16])
def test_gemv_rows_bit_exact(fmt, ncols):
    K = 2048 if fmt == synth.FMT_Q8_0 else 4096
    rows = 261   # several tiles and a ragged tail
    lg, W, x = make_case(fmt, rows, K, ncols, seed=7 * fmt + ncols, outliers=0.001)
    blk = synth.BLOCK[fmt]
    codes, m, e, s16, packed = oracle_act(x, blk)
    want = oracle.gemv(fmt, W, rows, K, codes, m, e)
    act = gpu_quantize(x, blk)   # the product consumes the GPU's own quantization
    got = gpu_rows(fmt, W, rows, K, act, ncols)
    assert np.array_equal(bits(got), bits(want))
    _, _, v = oracle.block_values(fmt, W, rows, K, codes, m, e)
    assert tolerance_ok(got, want, np.abs(v.astype(np.float64)).sum(-1))


@pytest.mark.parametrize("fmt", FMTS)
def test_batch_invariance(fmt):
    K = 1024
    rows = 97
    lg, W, x = make_case(fmt, rows, K, 16, seed=31 + fmt)
    act = gpu_quantize(x, synth.BLOCK[fmt])
    allc = gpu_rows(fmt, W, rows, K, act, 16)
    for c in (0, 5, 15):
        one = tuple(t[c:c + 1].contiguous() for t in act)
        got = gpu_rows(fmt, W, rows, K, one, 1)
        assert np.array_equal(bits(got[0]), bits(allc[c]))


@pytest.mark.parametrize("fmt", FMTS)
def test_long_rows_and_chunked_activation(fmt):
    """K = 14336 (the down projection) at 16 columns: the activation is staged
    in several chunks of at most 64 KB."""
    K, rows, ncols = 14336, 45, 16
    if fmt == synth.FMT_Q8_0:
        K = 14336
    lg, W, x = make_case(fmt, rows, K, ncols, seed=55 + fmt)
    blk = synth.BLOCK[fmt]
    codes, m, e, s16, packed = oracle_act(x, blk)
    want = oracle.gemv(fmt, W, rows, K, codes, m, e)
    got = gpu_rows(fmt, W, rows, K, gpu_quantize(x, blk), ncols)
    assert np.array_equal(bits(got), bits(want))


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("ncols", [2, 6, 16])
@pytest.mark.parametrize("rows,K", [(152 * 9 + 77, 1024), (700, 8192), (300, 12288)])
def test_skinny_launch_shapes(fmt, ncols, rows, K):
    """2..16 columns through the multi-column streaming kernel: several ring
    iterations per CTA with a ragged last one, four- and two-column groups,
    and (K = 8192, 12288 at 16 columns) several launches over column chunks.
    Non-finite and unreadable cases ride along in one column and one row."""
    lg, W, x = make_case(fmt, rows, K, ncols, seed=rows + K + 17 * ncols + fmt, outliers=0.001)
    blk = synth.BLOCK[fmt]
    lg["d"][rows // 2, 1] = 0x7C00                           # one unreadable block scale
    W = synth.pack(fmt, lg)
    x[ncols - 1, 2 * blk + 5] = np.inf                       # last column: a block with no scale
    codes, m, e, s16, packed = oracle_act(x, blk)
    want = oracle.gemv(fmt, W, rows, K, codes, m, e)
    got = gpu_rows(fmt, W, rows, K, gpu_quantize(x, blk), ncols)
    assert np.array_equal(bits(got), bits(want))
    assert np.all(bits(got[ncols - 1]) == 0x7FC00000)
    assert np.all(bits(got[:, rows // 2]) == 0x7FC00000)


@pytest.mark.parametrize("ncols", [11, 12, 16])
@pytest.mark.parametrize("rows,K", [(152 * 33 + 5, 4096), (300, 256), (1000, 2304)])
def test_tensor_path_shapes(ncols, rows, K):
    """Q4_K-like at 11..16 columns, the tensor-core sub-block path: several
    row chunks per CTA, one block per row (one busy warp), nine blocks (idle
    warps); rows whose two scales' exponents differ by 29 (the combine's
    out-of-line exact path), an unreadable dmin, and a column with an
    infinite activation."""
    fmt = synth.FMT_Q4K
    lg, W, x = make_case(fmt, rows, K, ncols, seed=rows + K + ncols, outliers=0.001)
    nb = K // 256
    for r in range(3, rows, max(1, rows // 7)):      # d subnormal, dmin near the top: spread 29
        lg["d"][r, r % nb] = 0x0001
        lg["dmin"][r, r % nb] = 0x7BFF
    lg["dmin"][rows // 2, nb - 1] = 0x7E00               # unreadable
    W = synth.pack(fmt, lg)
    x[ncols // 2, 5] = -np.inf                           # that column: a block with no scale
    codes, m, e, s16, packed = oracle_act(x, 256)
    want = oracle.gemv(fmt, W, rows, K, codes, m, e)
    got = gpu_rows(fmt, W, rows, K, gpu_quantize(x, 256), ncols)
    assert np.array_equal(bits(got), bits(want))
    assert np.all(bits(got[ncols // 2]) == 0x7FC00000)
    assert np.all(bits(got[:, rows // 2]) == 0x7FC00000)


# ---------------------------------------------------------------- full-size workloads

def test_q8_0_512x1024_full():
    lg, W, x = make_case(synth.FMT_Q8_0, 512, 1024, 1, seed=0)
    codes, m, e, s16, packed = oracle_act(x, 32)
    want = oracle.gemv(synth.FMT_Q8_0, W, 512, 1024, codes, m, e)
    got = gpu_rows(synth.FMT_Q8_0, W, 512, 1024, gpu_quantize(x, 32), 1)
    assert np.array_equal(bits(got), bits(want))


def test_q4k_4096x4096_full():
    mats, x = synth.workload_inputs("q4k_4096x4096")
    rows, K, lg, W = mats[0]
    codes, m, e, s16, packed = oracle_act(x, 256)
    want = oracle.gemv(synth.FMT_Q4K, W, rows, K, codes, m, e)
    got = gpu_rows(synth.FMT_Q4K, W, rows, K, gpu_quantize(x, 256), 1)
    assert np.array_equal(bits(got), bits(want))


def test_q6k_ffn_full():
    """gate and up (14336x4096, one shared activation) and down (4096x14336)."""
    rng = np.random.default_rng(2)
    gate = synth.draw_q6k(rng, 14336, 4096)
    up = synth.draw_q6k(rng, 14336, 4096)
    down = synth.draw_q6k(rng, 4096, 14336)
    x = synth.draw_act(rng, 1, 4096)
    h = synth.draw_act(rng, 1, 14336)
    for lg, xx in ((gate, x), (up, x), (down, h)):
        rows, K = lg["q"].shape
        W = synth.pack_q6k(**lg)
        codes, m, e, s16, packed = oracle_act(xx, 256)
        want = oracle.gemv(synth.FMT_Q6K, W, rows, K, codes, m, e)
        got = gpu_rows(synth.FMT_Q6K, W, rows, K, gpu_quantize(xx, 256), 1)
        assert np.array_equal(bits(got), bits(want)), (rows, K)


@pytest.mark.parametrize("ncols", [1, 4, 16])
def test_8b_stack_shapes_sampled(ncols):
    """The decode-stack shapes at 1, 4 and 16 columns, in the launch shape the
    benchmark uses; the oracle checks a sample of rows of each matrix."""
    import torch
    rng = np.random.default_rng(5 + ncols)
    shapes = [(synth.FMT_Q4K, 6144, 4096), (synth.FMT_Q4K, 4096, 4096), (synth.FMT_Q4K, 28672, 4096),
              (synth.FMT_Q4K, 4096, 14336), (synth.FMT_Q6K, 128256, 4096)]
    for fmt, rows, K in shapes:
        lg = synth.draw(fmt, rng, rows, K)
        W = synth.pack(fmt, lg)
        x = synth.draw_act(rng, ncols, K)
        codes, m, e, s16, packed = oracle_act(x, 256)
        got = gpu_rows(fmt, W, rows, K, gpu_quantize(x, 256), ncols)
        sample = np.unique(np.concatenate([rng.integers(0, rows, 48), [0, rows - 1]]))
        rec = synth.record_bytes(fmt, K)
        Ws = np.concatenate([W[r * rec:(r + 1) * rec] for r in sample])
        want = oracle.gemv(fmt, Ws, len(sample), K, codes, m, e)
        assert np.array_equal(bits(got[:, sample]), bits(want)), (fmt, rows, K)
        del W, lg
        torch.cuda.empty_cache()


# ---------------------------------------------------------------- edge cases

@pytest.mark.parametrize("fmt", FMTS)
def test_edge_shapes(fmt):
    blk = synth.BLOCK[fmt]
    K1 = blk if fmt == synth.FMT_Q8_0 else 256
    for rows, K in ((1, K1), (2, K1), (33, K1), (1, 4096), (7, 3 * 256)):
        lg, W, x = make_case(fmt, rows, K, 2, seed=rows * 13 + K)
        codes, m, e, s16, packed = oracle_act(x, blk)
        want = oracle.gemv(fmt, W, rows, K, codes, m, e)
        got = gpu_rows(fmt, W, rows, K, gpu_quantize(x, blk), 2)
        assert np.array_equal(bits(got), bits(want)), (rows, K)
        if K == blk:   # one block: the row is that block's value
            _, _, v = oracle.block_values(fmt, W, rows, K, codes, m, e)
            assert np.array_equal(bits(got), bits(v[:, :, 0]))


def test_empty_and_degenerate():
    import torch
    act = qb.alloc_act(1, 256, 256)
    out = torch.full((1, 4), 7.0, device="cuda")
    W = torch.zeros(144 * 4, dtype=torch.uint8, device="cuda")
    qb.q_gemv(qb.Q4K, W, 0, 256, act, 1, out)               # no rows: nothing written
    torch.cuda.synchronize()
    assert torch.all(out == 7.0)
    qb.q_gemv(qb.Q4K, W, 4, 0, act, 1, out)                 # rows of no blocks: +0
    torch.cuda.synchronize()
    assert np.all(bits(host(out)) == 0)
    # an all-zero activation gives +0 in every row
    lg, Wn, _ = make_case(synth.FMT_Q4K, 9, 512, 1, seed=3)
    z = np.zeros((1, 512), np.float32)
    got = gpu_rows(synth.FMT_Q4K, Wn, 9, 512, gpu_quantize(z, 256), 1)
    assert np.all(bits(got) == 0)


@pytest.mark.parametrize("fmt", FMTS)
def test_unreadable_scales_and_nonfinite_activation(fmt):
    rows, K = 6, 512
    lg, _, x = make_case(fmt, rows, K, 2, seed=91 + fmt)
    lg["d"][2, 1] = 0x7C00
    lg["d"][4, 0] = 0xFE01
    if fmt == synth.FMT_Q4K:
        lg["dmin"][5, 0] = 0x7C00
    W = synth.pack(fmt, lg)
    blk = synth.BLOCK[fmt]
    x[1, 3] = np.inf                                         # column 1: a block with no scale
    codes, m, e, s16, packed = oracle_act(x, blk)
    want = oracle.gemv(fmt, W, rows, K, codes, m, e)
    got = gpu_rows(fmt, W, rows, K, gpu_quantize(x, blk), 2)
    assert np.array_equal(bits(got), bits(want))
    assert np.all(bits(got[1]) == 0x7FC00000)
    assert bits(got[0, 2]) == 0x7FC00000 and bits(got[0, 4]) == 0x7FC00000
    assert qb.q_check_weights(fmt, dev(W), rows, K) == qb.QB_E_UNREADABLE
    assert oracle.count_unreadable(fmt, W, rows, K) >= 2
    lg2, W2, _ = make_case(fmt, rows, K, 1, seed=5)
    assert qb.q_check_weights(fmt, dev(W2), rows, K) == qb.QB_OK


# ---------------------------------------------------------------- F16

def test_quantize_act_f16_bit_exact():
    import torch
    rng = np.random.default_rng(21)
    x = synth.draw_act(rng, 3, 4096)
    x[0, :64] *= np.float32(1e-6)     # binary16 subnormals
    x[0, 64:128] *= np.float32(4000)  # past the top
    x[1, 7] = np.nan
    x[1, 8] = -np.inf
    x[2, :] = np.round(x[2, :] * 1024) / 1024 + np.float32(2.0 ** -11)   # ties
    want = oracle.quantize_f16(x)
    g = torch.empty((3, 4096), dtype=torch.int16, device="cuda")
    qb.quantize_act_f16(dev(x), g)
    torch.cuda.synchronize()
    assert np.array_equal(host(g).view(np.uint16), want)


@pytest.mark.parametrize("rows,K", [(49152, 576), (1536, 576), (13, 8), (129, 1536), (300, 64), (40, 8192),
                                    (1000, 56), (151 * 64 + 3, 128)])
@pytest.mark.parametrize("ncols", [1, 2, 3, 6])
def test_f16_gemv_bit_exact(rows, K, ncols):
    import torch
    rng = np.random.default_rng(rows + K + ncols)
    W = synth.draw_f16(rng, rows, K)
    x = synth.draw_act(rng, ncols, K)
    x16 = oracle.quantize_f16(x)
    want = oracle.gemv_f16(W, rows, K, x16)
    gx = torch.empty((ncols, K), dtype=torch.int16, device="cuda")
    qb.quantize_act_f16(dev(x), gx)
    out = torch.empty((ncols, rows), dtype=torch.float32, device="cuda")
    qb.q_gemv_f16(dev(W), rows, K, gx, ncols, out)
    torch.cuda.synchronize()
    assert np.array_equal(bits(host(out)), bits(want))


def test_f16_sixteen_columns_and_nonfinite():
    import torch
    rng = np.random.default_rng(8)
    rows, K = 200, 512
    W = synth.draw_f16(rng, rows, K)
    W[3, 9] = 0x7C00                      # +inf weight
    W[4, 0] = 0x7E00                      # NaN weight
    x = synth.draw_act(rng, 16, K)
    x[2, 9] = 0.0                         # inf * 0 -> NaN in column 2, row 3
    x16 = oracle.quantize_f16(x)
    want = oracle.gemv_f16(W, rows, K, x16)
    out = torch.empty((16, rows), dtype=torch.float32, device="cuda")
    qb.q_gemv_f16(dev(W), rows, K, dev(x16.view(np.int16)), 16, out)
    torch.cuda.synchronize()
    assert np.array_equal(bits(host(out)), bits(want))


# ---------------------------------------------------------------- q_matvec (one call from f32)

@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("ncols", [1, 3])
@pytest.mark.parametrize("rows,K", [(261, 4096), (1000, 1024), (7, 256), (152 * 3 + 5, 2048), (5021, 4096),
                                    (1200, 14336)])
def test_matvec_bit_exact(fmt, ncols, rows, K):
    """q_matvec -- in one launch for one column (the activation quantized inside
    the product kernel), through a workspace otherwise -- equals the oracle's
    quantize_blocks + dot, including activation blocks that are zero, hold a
    NaN, a denormal or an infinity.  The last two shapes take several ring
    iterations a CTA: the 256-element formats' one-column launch then runs in
    the multi-column kernel's organisation."""
    import torch
    blk = synth.BLOCK[fmt]
    x = _edge_activation(ncols, K, blk, seed=rows + K + ncols + fmt)
    rng = np.random.default_rng(rows * 3 + fmt)
    lg = synth.draw(fmt, rng, rows, K)
    W = synth.pack(fmt, lg)
    codes, m, e, s16, packed = oracle_act(x, blk)
    want = oracle.gemv(fmt, W, rows, K, codes, m, e)
    out = torch.full((ncols, rows), float("nan"), dtype=torch.float32, device="cuda")
    ws = torch.empty(qb.q_matvec_workspace_bytes(fmt, K, ncols), dtype=torch.uint8, device="cuda")
    qb.q_matvec(fmt, dev(W), rows, K, dev(x), out, workspace=ws if ncols > 1 else None)
    torch.cuda.synchronize()
    assert np.array_equal(bits(host(out)), bits(want))
    if ncols > 1:  # without a workspace: one launch where the shape allows it, else refused
        out.fill_(float("nan"))
        try:
            qb.q_matvec(fmt, dev(W), rows, K, dev(x), out, workspace=None)
        except qb.QbError as exc:
            assert exc.status == qb.QB_E_ARG
        else:
            torch.cuda.synchronize()
            assert fmt != synth.FMT_Q8_0 and K == 4096 and ncols <= 4
            assert np.array_equal(bits(host(out)), bits(want))


@pytest.mark.parametrize("fmt", [synth.FMT_Q4K, synth.FMT_Q6K])
@pytest.mark.parametrize("rows,K", [(307, 8192), (157, 10240), (2 * 152 + 3, 14336), (95, 16384), (3, 14336),
                                    (4096, 14336)])
def test_one_column_long_rows(fmt, rows, K):
    """One column at K = 8192 .. 16384 (the down projection's 14336 among them):
    rows streamed in passes of 16 blocks, the last pass partial at 10240 and
    14336 (8 blocks), CTAs with an odd row count; both the product from a
    quantized activation and the single-launch q_matvec equal the oracle."""
    import torch
    rng = np.random.default_rng(rows + K + fmt)
    W = synth.pack(fmt, synth.draw(fmt, rng, rows, K))
    x = synth.draw_act(rng, 1, K, outlier_frac=0.001)
    x[0, 5 * 256:6 * 256] = 0.0                                 # a zero block
    codes, m, e, s16, packed = oracle_act(x, 256)
    want = oracle.gemv(fmt, W, rows, K, codes, m, e)
    act = qb.alloc_act(1, K, 256)
    qb.quantize_act(256, dev(x), *act)
    out = torch.full((1, rows), float("nan"), dtype=torch.float32, device="cuda")
    qb.q_gemv(fmt, dev(W), rows, K, act, 1, out)
    torch.cuda.synchronize()
    assert np.array_equal(bits(host(out)), bits(want))
    out.fill_(float("nan"))
    qb.q_matvec(fmt, dev(W), rows, K, dev(x), out)
    torch.cuda.synchronize()
    assert np.array_equal(bits(host(out)), bits(want))


@pytest.mark.parametrize("fmt", [synth.FMT_Q4K, synth.FMT_Q6K])
@pytest.mark.parametrize("K", [4352, 6400, 14336, 16384])
@pytest.mark.parametrize("rows", [1, 152 * 27 - 8, 4096, 152 * 32, 152 * 32 + 1])
def test_long_k_row_ranges(fmt, K, rows):
    """One column of rows longer than K = 4096 from a quantized activation (17,
    25, 56 and 64 blocks a row) over row counts around 27 and 32 rows a CTA;
    an unreadable block scale in the last block and a zero activation block."""
    import torch
    rng = np.random.default_rng(rows + 3 * K + fmt)
    lg = synth.draw(fmt, rng, rows, K)
    lg["d"][rows // 2, K // 256 - 1] = 0x7E00                   # unreadable, in the last chunk
    W = synth.pack(fmt, lg)
    x = synth.draw_act(rng, 1, K, outlier_frac=0.001)
    x[0, 256:512] = 0.0
    codes, m, e, s16, packed = oracle_act(x, 256)
    want = oracle.gemv(fmt, W, rows, K, codes, m, e)
    act = qb.alloc_act(1, K, 256)
    qb.quantize_act(256, dev(x), *act)
    out = torch.full((1, rows), float("nan"), dtype=torch.float32, device="cuda")
    qb.q_gemv(fmt, dev(W), rows, K, act, 1, out)
    torch.cuda.synchronize()
    got = host(out)
    assert np.array_equal(bits(got), bits(want))
    assert bits(got)[0, rows // 2] == 0x7FC00000


@pytest.mark.parametrize("fmt", [synth.FMT_Q4K, synth.FMT_Q6K])
@pytest.mark.parametrize("ncols", [1, 2, 3, 4])
@pytest.mark.parametrize("rows", [1, 31, 152, 152 * 31 + 7, 152 * 32, 152 * 32 + 1, 152 * 64, 152 * 64 + 1])
def test_k4096_row_ranges(fmt, ncols, rows):
    """1..4 columns at K = 4096 across the row counts where the kernel changes
    form: up to 32 rows a CTA (a lane per row; one column: each lane's block
    held in registers from before the dependency wait), 33..64 (blocks read
    from shared memory, two rows a lane), and past the shared-memory budget (the
    ring kernels) -- from a quantized activation and from the f32 activation
    (one launch up to 4 columns), both equal to the oracle."""
    import torch
    K = 4096
    x = _edge_activation(ncols, K, 256, seed=rows + fmt + 10 * ncols)
    x[0, 5 * 256 + 1] = 3.0   # no infinity: every row a finite value, not the engine's NaN
    rng = np.random.default_rng(rows * 7 + fmt + ncols)
    W = synth.pack(fmt, synth.draw(fmt, rng, rows, K))
    codes, m, e, s16, packed = oracle_act(x, 256)
    want = oracle.gemv(fmt, W, rows, K, codes, m, e)
    act = qb.alloc_act(ncols, K, 256)
    qb.quantize_act(256, dev(x), *act)
    out = torch.full((ncols, rows), float("nan"), dtype=torch.float32, device="cuda")
    qb.q_gemv(fmt, dev(W), rows, K, act, ncols, out)
    torch.cuda.synchronize()
    assert np.array_equal(bits(host(out)), bits(want))
    out.fill_(float("nan"))
    ws = torch.empty(qb.q_matvec_workspace_bytes(fmt, K, ncols), dtype=torch.uint8, device="cuda")
    qb.q_matvec(fmt, dev(W), rows, K, dev(x), out, workspace=ws)
    torch.cuda.synchronize()
    assert np.array_equal(bits(host(out)), bits(want))


_RING_CASES = [(n, r, 4096) for n in (2, 3, 4) for r in (152 * 65, 152 * 189 + 17, 152 * 96 - 5)] + \
              [(n, r, K) for n in (2, 3, 4) for r, K in ((4096, 14336), (152 * 33 + 7, 14336), (300, 8192))]


@pytest.mark.parametrize("ncols,rows,K", _RING_CASES)
def test_ring_rows_and_chunks(ncols, rows, K):
    """Q4_K-like through the ring form: 2..4 columns at K = 4096 past 64 rows
    a CTA, and at longer K (chunks of 14 or 16 blocks a tile,
    the fold carried across a row's chunks): full tiles, a ragged last one,
    CTAs with one row more than others; from codes and from x; and the same
    rows as a table of three matrices sharing the activation."""
    import torch
    fmt = synth.FMT_Q4K
    rng = np.random.default_rng(rows + ncols + K)
    lg = synth.draw(fmt, rng, rows, K)
    W = synth.pack(fmt, lg)
    x = synth.draw_act(rng, ncols, K, outlier_frac=0.001)
    codes, m, e, s16, packed = oracle_act(x, 256)
    want = oracle.gemv(fmt, W, rows, K, codes, m, e)
    act = gpu_quantize(x, 256)
    out = torch.full((ncols, rows), float("nan"), dtype=torch.float32, device="cuda")
    qb.q_gemv(fmt, dev(W), rows, K, act, ncols, out)
    torch.cuda.synchronize()
    assert np.array_equal(bits(host(out)), bits(want))
    out.fill_(float("nan"))
    ws = torch.empty(qb.q_matvec_workspace_bytes(fmt, K, ncols), dtype=torch.uint8, device="cuda")
    qb.q_matvec(fmt, dev(W), rows, K, dev(x), out, workspace=ws)
    torch.cuda.synchronize()
    assert np.array_equal(bits(host(out)), bits(want))
    # three matrices: the first rows, a middle part, the last 7 rows
    cut = [0, rows // 2 + 3, rows - 7, rows]
    Wr = W.reshape(rows, -1)
    parts = [np.ascontiguousarray(Wr[cut[i]:cut[i + 1]]) for i in range(3)]
    outs = [torch.full((ncols, cut[i + 1] - cut[i]), float("nan"), dtype=torch.float32, device="cuda")
            for i in range(3)]
    qb.q_gemv_many(fmt, [dev(P) for P in parts], [cut[i + 1] - cut[i] for i in range(3)], K, act, ncols, outs)
    torch.cuda.synchronize()
    for i in range(3):
        assert np.array_equal(bits(host(outs[i])), bits(want[:, cut[i]:cut[i + 1]])), i


@pytest.mark.parametrize("ncols", [1, 2, 3, 4])
@pytest.mark.parametrize("rows,K", [(300, 4096), (152 * 64 + 1, 4096), (200, 14336)])
def test_scale_exponent_gaps(ncols, rows, K):
    """Q4_K-like blocks whose d and dmin exponents differ by every gap on
    either side of the combine's thresholds (d's term shifted up by at most
    17 places, dmin's by at most 21, a 128-bit combine past those), one gap a
    block and the gaps of neighbouring rows different, so that the lanes of a
    warp take different shifts: through the product and the single-launch form."""
    import torch
    fmt = synth.FMT_Q4K
    rng = np.random.default_rng(rows + K + ncols)
    lg = synth.draw(fmt, rng, rows, K)
    gaps = np.array([-29, -22, -21, -20, -7, -1, 0, 1, 9, 16, 17, 18, 29])
    nb = K // 256
    g = gaps[(np.arange(rows)[:, None] * 5 + np.arange(nb)[None, :] * 3) % len(gaps)]
    E2 = rng.integers(1, 31, size=g.shape)
    E2 = np.clip(E2, np.maximum(1, 1 - g), np.minimum(30, 30 - g))   # both exponents normal
    E1 = E2 + g
    lg["d"] = ((E1 << 10) | rng.integers(0, 1024, size=g.shape)).astype(np.uint16)
    lg["dmin"] = ((E2 << 10) | rng.integers(0, 1024, size=g.shape)).astype(np.uint16)
    W = synth.pack(fmt, lg)
    x = synth.draw_act(rng, ncols, K, outlier_frac=0.001)
    codes, m, e, s16, packed = oracle_act(x, 256)
    want = oracle.gemv(fmt, W, rows, K, codes, m, e)
    out = torch.full((ncols, rows), float("nan"), dtype=torch.float32, device="cuda")
    qb.q_gemv(fmt, dev(W), rows, K, gpu_quantize(x, 256), ncols, out)
    torch.cuda.synchronize()
    assert np.array_equal(bits(host(out)), bits(want))
    out.fill_(float("nan"))
    ws = torch.empty(qb.q_matvec_workspace_bytes(fmt, K, ncols), dtype=torch.uint8, device="cuda")
    qb.q_matvec(fmt, dev(W), rows, K, dev(x), out, workspace=ws)
    torch.cuda.synchronize()
    assert np.array_equal(bits(host(out)), bits(want))


def test_matvec_repeated_launches_graph():
    """Many single-launch products back to back (programmatic dependent launch
    overlapping each launch's weight stream with the previous one) on distinct
    weights and activations, replayed from a CUDA graph: every output exact."""
    import torch
    rng = np.random.default_rng(99)
    rows, K, n = 777, 4096, 6
    Ws = [synth.pack_q4k(**synth.draw_q4k(rng, rows, K)) for _ in range(n)]
    xs = [synth.draw_act(rng, 1, K, outlier_frac=0.001) for _ in range(n)]
    Wd = [dev(w) for w in Ws]
    xd = [dev(x) for x in xs]
    outs = [torch.empty((1, rows), dtype=torch.float32, device="cuda") for _ in range(n)]
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        qb.q_matvec(qb.Q4K, Wd[0], rows, K, xd[0], outs[0], stream=s)
    s.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        g.capture_begin()
        for i in range(n):
            qb.q_matvec(qb.Q4K, Wd[i], rows, K, xd[i], outs[i], stream=s)
        g.capture_end()
    for o in outs:
        o.fill_(float("nan"))
    g.replay()
    s.synchronize()
    for i in range(n):
        codes, m, e, _, _ = oracle_act(xs[i], 256)
        want = oracle.gemv(synth.FMT_Q4K, Ws[i], rows, K, codes, m, e)
        assert np.array_equal(bits(host(outs[i])), bits(want)), i


@pytest.mark.parametrize("rows,K,ncols", [(1536, 576, 2), (49152, 576, 1), (777, 576, 6), (300, 2048, 3),
                                         (9, 8, 1), (64, 16384, 1)])
def test_matvec_f16(rows, K, ncols):
    """q_matvec for F16 -- one launch that rounds x to f16 in the prologue where
    the warp-ring kernel takes the shape (no workspace), else quantize_act_f16
    + q_gemv_f16 -- equals the oracle's f32_to_f16 + fdot, including elements
    that round to f16 infinities, subnormals and NaN."""
    import torch
    rng = np.random.default_rng(4 + rows + K)
    W = synth.draw_f16(rng, rows, K)
    x = synth.draw_act(rng, ncols, K)
    x[0, 0] = np.float32(70000.0)          # past the f16 top: +inf
    x[0, min(1, K - 1)] = np.float32(3e-6)  # an f16 subnormal
    if K > 2:
        x[-1, 2] = np.nan
    want = oracle.gemv_f16(W, rows, K, oracle.quantize_f16(x))
    out = torch.full((ncols, rows), float("nan"), dtype=torch.float32, device="cuda")
    ws = torch.empty(qb.q_matvec_workspace_bytes(qb.F16, K, ncols), dtype=torch.uint8, device="cuda")
    qb.q_matvec(qb.F16, dev(W), rows, K, dev(x), out, workspace=ws)
    torch.cuda.synchronize()
    assert np.array_equal(bits(host(out)), bits(want))
    if ncols * K * 4 <= 16 * 1024:  # the one-launch form needs no workspace
        out2 = torch.full((ncols, rows), float("nan"), dtype=torch.float32, device="cuda")
        qb.q_matvec(qb.F16, dev(W), rows, K, dev(x), out2, workspace=None)
        torch.cuda.synchronize()
        assert np.array_equal(bits(host(out2)), bits(want))


# ---------------------------------------------------------------- host to host in one call

@pytest.mark.parametrize("scaling,fmt,ncols", [(qb.PERBLOCK, synth.FMT_Q4K, 1), (qb.PERBLOCK, synth.FMT_Q6K, 3),
                                               (qb.PERBLOCK, synth.FMT_Q8_0, 1), (qb.SUB32, synth.FMT_Q4K, 2),
                                               (qb.PERBLOCK, synth.FMT_F16, 2)])
def test_matvec_host_matches_device_call(scaling, fmt, ncols):
    """q_matvec_host (pinned x in, pinned out back, one call) gives the bits of
    the device-buffer call on the same stream."""
    import torch
    rows, K = 1000, 1024
    rng = np.random.default_rng(31 + fmt + ncols + scaling)
    if fmt == synth.FMT_F16:
        W = synth.draw_f16(rng, rows, K)
        Wd = dev(W.view(np.int16))
    else:
        W = synth.pack(fmt, synth.draw(fmt, rng, rows, K))
        Wd = dev(W)
    x = synth.draw_act(rng, ncols, K, outlier_frac=0.001)
    xh = torch.from_numpy(x).pin_memory()
    oh = torch.full((ncols, rows), float("nan"), dtype=torch.float32).pin_memory()
    ws = torch.empty(qb.q_matvec_host_workspace_bytes(scaling, fmt, rows, K, ncols), dtype=torch.uint8, device="cuda")
    s = torch.cuda.Stream()
    qb.q_matvec_host(fmt, Wd, rows, K, xh, oh, ws, scaling=scaling, stream=s)
    s.synchronize()
    od = torch.full((ncols, rows), float("nan"), dtype=torch.float32, device="cuda")
    if scaling == qb.SUB32:
        qb.q_matvec_sub32(fmt, Wd, rows, K, dev(x), od)
    else:
        ws2 = torch.empty(qb.q_matvec_workspace_bytes(fmt, K, ncols), dtype=torch.uint8, device="cuda")
        qb.q_matvec(fmt, Wd, rows, K, dev(x), od, workspace=ws2)
    torch.cuda.synchronize()
    assert np.array_equal(bits(oh.numpy()), bits(host(od)))
