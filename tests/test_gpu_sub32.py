"""ActScaling::Sub32 on the GPU against the oracle, bit for bit (numerics page:
block_scale, quantize, ACT_BLOCK, GROUP, exact_sum, dot; lane page: group).

The quantizer is compared code for code, scale for scale and unit sum for unit
sum; the product is fed the ORACLE's quantized activation (so it is tested on
its own) and every output row compared; the one-call path (quantize, then the
product) against the oracle's pipeline.  Inputs put activation blocks of one
group up to 2^170 apart (the exact routine), Q8_0 weight scales many binades
apart, blocks without a scale, unreadable weight scales and subnormal f16
scales in the way; shapes span several CTAs, a ragged last iteration, one
group, many column launches and the plain kernel.
"""
import numpy as np
import pytest

import oracle
import block_quantized_weight_quantize_gb300 as qb
from block_quantized_weight_quantize_gb300 import synth
from helpers import bits, dev, host

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


def _oracle_act(x):
    codes, m, e, s16 = oracle.quantize_sub32(x)
    return codes, m, e, s16, _packed(m, e)


def _gpu_product(fmt, W, rows, K, codes, packed, s16, ncols):
    import torch
    out = torch.full((ncols, rows), float("nan"), dtype=torch.float32, device="cuda")
    qb.q_gemv_sub32(fmt, dev(W), rows, K, (dev(codes), dev(packed), dev(s16)), ncols, out)
    torch.cuda.synchronize()
    return host(out)


def _spread_blocks(x, exps):
    """Scale 32-element block b of every column by 2^exps[b % len(exps)]."""
    for b in range(x.shape[1] // 32):
        x[:, 32 * b:32 * b + 32] *= np.float32(2.0 ** exps[b % len(exps)])
    return x


# ------------------------------------------------------------------ quantizer

@pytest.mark.parametrize("ncols,K", [(1, 256), (3, 4096), (16, 1024), (2, 65536)])
def test_quantize_sub32_bit_exact(ncols, K):
    import torch
    rng = np.random.default_rng(K + ncols)
    x = synth.draw_act(rng, ncols, K, outlier_frac=0.01)
    _spread_blocks(x, [0, 60, -60, 20, -7, 3, 100, -110, -124, 118])
    c = ncols - 1
    x[c, 0:32] = 0.0                                              # all-zero block: m=8, e=0
    x[c, 40] = np.inf                                             # a block with an infinity: m=0
    x[c, 70] = np.nan
    x[c, 71] = np.float32(1e-40)                                  # denormal: read as zero, code 0
    x[0, 96:128] = np.float32(1e-40)                              # a block of denormals only
    for k in range(8):                                            # exact ties under the scale 8*2^-3
        x[0, 128 + k] = np.float32((k + 0.5) * 8 * 2.0 ** -3)
    x[0, 128 + 31] = np.float32(127 * 8 * 2.0 ** -3)
    x[0, 160:192] = np.float32(2.0 ** -127) * np.arange(1, 33, dtype=np.float32)   # e < -130: the exact routine
    codes, m, e, s16, packed = _oracle_act(x)
    g_codes, g_scales, g_sums = qb.alloc_act(ncols, K, 32)
    qb.quantize_act_sub32(dev(x), g_codes, g_scales, g_sums)
    torch.cuda.synchronize()
    assert np.array_equal(host(g_scales), packed)
    assert np.array_equal(host(g_codes), codes)
    assert np.array_equal(host(g_sums), s16)
    assert m[0, 4] == 8 and e[0, 4] == -3
    assert list(codes[0, 128:136]) == [0, 2, 2, 4, 4, 6, 6, 8]


def test_quantize_sub32_binades():
    """One block per binade of amax (every exponent field 1..254), with amax's
    significand at the edges where block_scale moves to the next exponent."""
    import torch
    rng = np.random.default_rng(5)
    # 0x6E2000 / 0x6E2001: m = 15 / the next exponent; 0x7E0000 / 0x7E0001: m = 8 / 9 there
    mants = [0, 1, 0x7FFFFF, 0x6E2000, 0x6E2001, 0x7E0000, 0x7E0001, int(rng.integers(0, 1 << 23))]
    rows = []
    for E in range(1, 255):
        for mt in mants:
            blk = rng.standard_normal(32).astype(np.float32)
            blk = blk / np.float32(np.max(np.abs(blk)))
            amax = np.uint32((E << 23) | mt).view(np.float32)
            blk = (blk * amax).astype(np.float32)
            blk[int(rng.integers(0, 32))] = amax
            rows.append(blk)
    x = np.concatenate(rows)
    K = (x.size // 256) * 256
    x = x[:K].reshape(1, K)
    codes, m, e, s16, packed = _oracle_act(x)
    g = qb.alloc_act(1, K, 32)
    qb.quantize_act_sub32(dev(x), *g)
    torch.cuda.synchronize()
    assert np.array_equal(host(g[1]), packed)
    assert np.array_equal(host(g[0]), codes)
    assert np.array_equal(host(g[2]), s16)


# ------------------------------------------------------------------ product

@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("ncols", [1, 2, 3, 16])
@pytest.mark.parametrize("rows,K", [(300, 4096), (1000, 256), (77, 1024), (2 * 152 + 5, 2048)])
def test_gemv_sub32_bit_exact(fmt, ncols, rows, K):
    rng = np.random.default_rng(rows * 7 + K + ncols + fmt)
    lg = synth.draw(fmt, rng, rows, K)
    W = synth.pack(fmt, lg)
    x = synth.draw_act(rng, ncols, K, outlier_frac=0.002)
    codes, m, e, s16, packed = _oracle_act(x)
    got = _gpu_product(fmt, W, rows, K, codes, packed, s16, ncols)
    want = oracle.gemv_sub32(fmt, W, rows, K, codes, m, e)
    assert np.array_equal(bits(got), bits(want))


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("ncols", [1, 5])
def test_gemv_sub32_exact_routine(fmt, ncols):
    """Groups whose activation blocks lie far apart (2^-110 .. 2^60: the exact
    384-bit routine), next to groups the fast path takes; Q8_0 weight scales
    from 2^-24 to 2^15 (spreads past 13 binades); subnormal f16 scales."""
    rows, K = 400, 2048
    rng = np.random.default_rng(31 + fmt + ncols)
    kw = {"d_range": (1e-7, 3e4)} if fmt == synth.FMT_Q8_0 else {"d_range": (1e-7, 1e-1)}
    lg = synth.draw(fmt, rng, rows, K, **kw)
    W = synth.pack(fmt, lg)
    x = synth.draw_act(rng, ncols, K, outlier_frac=0.01)
    # groups 0, 2, 4, 6: blocks far apart; 1, 3, 5, 7: within a few binades
    for g in range(0, K // 256, 2):
        for s in range(8):
            x[:, 256 * g + 32 * s:256 * g + 32 * s + 32] *= np.float32(2.0 ** [0, 60, -110, 13, -13, 40, -70, 7][s])
    codes, m, e, s16, packed = _oracle_act(x)
    got = _gpu_product(fmt, W, rows, K, codes, packed, s16, ncols)
    want = oracle.gemv_sub32(fmt, W, rows, K, codes, m, e)
    assert np.array_equal(bits(got), bits(want))
    assert np.isfinite(want).mean() > 0.5


@pytest.mark.parametrize("fmt", FMTS)
def test_gemv_sub32_nan_and_edges(fmt):
    """A block without a scale makes its column's rows NaN; an unreadable weight
    scale its row; scale multipliers at the 16-bit edge (spread exactly 12, m =
    15) take the fast path; spread 13 the exact routine; all-zero columns give +0."""
    rows, K, ncols = 260, 1536, 4
    rng = np.random.default_rng(77 + fmt)
    lg = synth.draw(fmt, rng, rows, K)
    lg["d"][5, 0] = 0x7C00                                   # inf scale in row 5
    lg["d"][9, lg["d"].shape[1] - 1] = 0xFE00                # NaN scale in row 9
    if fmt == synth.FMT_Q4K:
        lg["dmin"][11, 2] = 0x7C00                           # inf dmin in row 11
    W = synth.pack(fmt, lg)
    x = synth.draw_act(rng, ncols, K)
    x[0, 300] = -np.inf                                      # column 0: NaN rows
    x[2, :] = 0.0                                            # column 2: every code 0
    codes, m, e, s16, packed = _oracle_act(x)
    # column 3: handcrafted scales at the fast path's edges (codes as drawn)
    m[3, 0:8] = [15, 8, 15, 8, 15, 8, 15, 8]
    e[3, 0:8] = [0, 12, 12, 3, 0, 1, 5, 12]                  # spread 12, M = 15 << 12 < 2^16
    m[3, 8:16] = [15, 8, 9, 8, 15, 8, 15, 8]
    e[3, 8:16] = [0, 13, 1, 3, 0, 1, 5, 13]                  # spread 13: exact routine
    m[3, 16:24] = [255, 128, 15, 8, 200, 8, 15, 1]
    e[3, 16:24] = [9, 8, 1, 3, 0, 1, 5, 2]                   # m past 4 bits: 255 << 9 >= 2^16 -> exact routine
    packed = _packed(m, e)
    got = _gpu_product(fmt, W, rows, K, codes, packed, s16, ncols)
    want = oracle.gemv_sub32(fmt, W, rows, K, codes, m, e)
    assert np.array_equal(bits(got), bits(want))
    assert np.all(bits(want[0]) == 0x7FC00000)
    assert np.all(bits(want[1, [5, 9]]) == 0x7FC00000)
    assert np.all(bits(want[2])[~np.isin(np.arange(rows), [5, 9, 11])] == 0)


@pytest.mark.parametrize("fmt", FMTS)
def test_gemv_sub32_plain_kernel(fmt):
    """K = 131072: past the streaming kernel's team size, the plain kernel."""
    rows, K, ncols = 9, 131072, 2
    rng = np.random.default_rng(3 + fmt)
    lg = synth.draw(fmt, rng, rows, K)
    W = synth.pack(fmt, lg)
    x = synth.draw_act(rng, ncols, K, outlier_frac=0.001)
    _spread_blocks(x, [0, 2, -1, 30, 0, 1, -3, 2, 0, 1, 1, 0, -2, 0, 0, 0])
    codes, m, e, s16, packed = _oracle_act(x)
    got = _gpu_product(fmt, W, rows, K, codes, packed, s16, ncols)
    want = oracle.gemv_sub32(fmt, W, rows, K, codes, m, e)
    assert np.array_equal(bits(got), bits(want))


@pytest.mark.parametrize("fmt", FMTS)
def test_gemv_sub32_many_launches(fmt):
    """16 columns at K = 16384: four columns a launch, four launches."""
    rows, K, ncols = 200, 16384, 16
    rng = np.random.default_rng(8 + fmt)
    lg = synth.draw(fmt, rng, rows, K)
    W = synth.pack(fmt, lg)
    x = synth.draw_act(rng, ncols, K, outlier_frac=0.001)
    codes, m, e, s16, packed = _oracle_act(x)
    got = _gpu_product(fmt, W, rows, K, codes, packed, s16, ncols)
    want = oracle.gemv_sub32(fmt, W, rows, K, codes, m, e)
    assert np.array_equal(bits(got), bits(want))


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("ncols", [1, 16])
def test_matvec_sub32_pipeline(fmt, ncols):
    """The one-call path (quantize_act_sub32, then q_gemv_sub32) against the
    oracle's quantize then dot, at the 4096 x 4096 decode shape."""
    import torch
    rows, K = 4096, 4096
    rng = np.random.default_rng(100 + fmt + ncols)
    lg = synth.draw(fmt, rng, rows, K)
    W = synth.pack(fmt, lg)
    x = synth.draw_act(rng, ncols, K, outlier_frac=0.001)
    out = torch.full((ncols, rows), float("nan"), dtype=torch.float32, device="cuda")
    qb.q_matvec_sub32(fmt, dev(W), rows, K, dev(x), out)
    torch.cuda.synchronize()
    codes, m, e, _ = oracle.quantize_sub32(x)
    want = oracle.gemv_sub32(fmt, W, rows, K, codes, m, e)
    assert np.array_equal(bits(host(out)), bits(want))


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("rows,K", [(300, 4096), (1000, 256), (77, 1024), (2 * 152 + 5, 2048), (40, 14336)])
def test_matvec_sub32_one_launch(fmt, rows, K):
    """One column of q_matvec_sub32 without a workspace: the product kernel
    quantizes x in its prologue.  Bit for bit the oracle's quantize then dot,
    with 32-element blocks many binades apart in one group (the exact group
    sum), a zero block, a NaN, a denormal and an infinity among the inputs;
    the same call given a workspace agrees."""
    import torch
    rng = np.random.default_rng(rows + K + fmt)
    W = synth.pack(fmt, synth.draw(fmt, rng, rows, K))
    x = _spread_blocks(synth.draw_act(rng, 1, K, outlier_frac=0.001), [0, -40, 37, 5, -90, 0, 60, -3])
    x[0, 64:96] = 0.0                                   # a zero block
    x[0, 100] = np.nan
    x[0, 130] = np.uint32(0x00012345).view(np.float32)  # a denormal element
    if K == 2048:
        x[0, 700] = np.inf                              # a block with an infinity: every row NaN
    codes, m, e, _ = oracle.quantize_sub32(x)
    want = oracle.gemv_sub32(fmt, W, rows, K, codes, m, e)
    out = torch.full((1, rows), float("nan"), dtype=torch.float32, device="cuda")
    qb.q_matvec_sub32(fmt, dev(W), rows, K, dev(x), out, workspace=None)
    torch.cuda.synchronize()
    assert np.array_equal(bits(host(out)), bits(want))
    ws = torch.empty(qb.q_matvec_sub32_workspace_bytes(K, 1), dtype=torch.uint8, device="cuda")
    out.fill_(float("nan"))
    qb.q_matvec_sub32(fmt, dev(W), rows, K, dev(x), out, workspace=ws)
    torch.cuda.synchronize()
    assert np.array_equal(bits(host(out)), bits(want))


def test_sub32_argument_checks():
    import torch
    K = 512
    W = torch.zeros(synth.record_bytes(synth.FMT_Q4K, K) * 4, dtype=torch.uint8, device="cuda")
    act = qb.alloc_act(1, K, 32)
    out = torch.zeros((1, 4), dtype=torch.float32, device="cuda")
    with pytest.raises(qb.QbError):   # K not a whole number of groups
        qb.q_gemv_sub32(qb.Q4K, W, 4, 480, act, 1, out)
    with pytest.raises(qb.QbError):   # 17 columns
        qb.q_gemv_sub32(qb.Q4K, W, 4, K, act, 17, out)
    with pytest.raises(qb.QbError):   # F16 has no Sub32 form
        qb.q_gemv_sub32(qb.F16, W, 4, K, act, 1, out)
    x = torch.zeros((1, 480), dtype=torch.float32, device="cuda")
    with pytest.raises(qb.QbError):
        qb.quantize_act_sub32(x, *qb.alloc_act(1, 480, 32))
    qb.q_gemv_sub32(qb.Q4K, W, 0, K, act, 1, out)    # no rows: nothing to do
    torch.cuda.synchronize()
