"""Out-of-range writes on the GPU: every call writes its outputs (and, for the
two-launch forms, its workspace) and nothing else.

Outputs and workspaces sit in the middle of larger buffers whose bytes were
set to a canary pattern; after each call the canary bytes on both sides must
be intact, and the outputs must equal those of the same call on plain
buffers.  The calls and shapes are those of the parity tests: the one-column
kernels (warp rings, the one-column gemv3 form for long rows, Q8_0's), two
launches through a workspace, 2..4 columns (the warp-per-block kernel and its
ring form), the grouped launch, 16 columns, Sub32, F16, FP8 and the score
kernel.
"""
import numpy as np
import pytest

import block_quantized_weight_quantize_gb300 as qb
from block_quantized_weight_quantize_gb300 import synth
from helpers import bits, dev, host

pytestmark = pytest.mark.gpu

CANARY = np.uint32(0x7FBADBAD)
PAD = 64            # floats (256 bytes) each side of an output
WPAD = 256          # bytes each side of a workspace
WBYTE = np.uint8(0xA5)


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    import torch
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    qb.lib()
    yield
    torch.cuda.synchronize()
    assert qb.q_device_status() == qb.QB_OK


def _out(shape):
    """(whole buffer, the output view) -- f32, 256-byte margins of canary words."""
    import torch
    n = int(np.prod(shape))
    buf = torch.empty(PAD + n + PAD, dtype=torch.float32, device="cuda")
    buf.view(torch.int32).fill_(int(CANARY))
    return buf, buf[PAD:PAD + n].view(*shape)


def _ws(nbytes):
    import torch
    buf = torch.full((WPAD + nbytes + WPAD,), int(WBYTE), dtype=torch.uint8, device="cuda")
    return buf, buf[WPAD:WPAD + nbytes]


def _out_intact(buf, n):
    b = host(buf).view(np.uint32)
    return bool(np.all(b[:PAD] == CANARY) and np.all(b[PAD + n:] == CANARY))


def _ws_intact(buf, nbytes):
    b = host(buf)
    return bool(np.all(b[:WPAD] == WBYTE) and np.all(b[WPAD + nbytes:] == WBYTE))


def _plain(shape):
    import torch
    return torch.full(shape, float("nan"), dtype=torch.float32, device="cuda")


@pytest.mark.parametrize("fmt", [synth.FMT_Q8_0, synth.FMT_Q4K, synth.FMT_Q6K])
@pytest.mark.parametrize("rows,K,ncols,use_ws", [(4096, 4096, 1, False), (1200, 14336, 1, False),
                                                 (1200, 14336, 1, True), (261, 4096, 3, True),
                                                 (1000, 1024, 3, True), (152 * 65 + 3, 4096, 4, True),
                                                 (1200, 14336, 3, True)])
def test_matvec_writes_only_its_outputs(fmt, rows, K, ncols, use_ws):
    import torch
    rng = np.random.default_rng(rows + K + ncols + fmt)
    W = dev(synth.pack(fmt, synth.draw(fmt, rng, rows, K)))
    x = dev(synth.draw_act(rng, ncols, K, outlier_frac=0.001))
    need = qb.q_matvec_workspace_bytes(fmt, K, ncols)
    ref = _plain((ncols, rows))
    wsp = torch.empty(need, dtype=torch.uint8, device="cuda")
    qb.q_matvec(fmt, W, rows, K, x, ref, workspace=wsp if use_ws else None)
    buf, out = _out((ncols, rows))
    wbuf, ws = _ws(need)
    qb.q_matvec(fmt, W, rows, K, x, out, workspace=ws if use_ws else None)
    torch.cuda.synchronize()
    assert _out_intact(buf, ncols * rows)
    assert _ws_intact(wbuf, need)
    assert np.array_equal(bits(host(out)), bits(host(ref)))


@pytest.mark.parametrize("fmt", [synth.FMT_Q4K, synth.FMT_Q6K])
def test_grouped_writes_only_its_outputs(fmt):
    import torch
    rows_list, K = [1001, 2000, 513], 4096
    rng = np.random.default_rng(5 + fmt)
    Ws = [dev(synth.pack(fmt, synth.draw(fmt, rng, r, K))) for r in rows_list]
    x = dev(synth.draw_act(rng, 1, K, outlier_frac=0.001))
    need = qb.q_matvec_workspace_bytes(fmt, K, 1)
    refs = [_plain((1, r)) for r in rows_list]
    qb.q_matvec_many(fmt, Ws, rows_list, K, x, refs, workspace=torch.empty(need, dtype=torch.uint8, device="cuda"))
    padded = [_out((1, r)) for r in rows_list]
    wbuf, ws = _ws(need)
    qb.q_matvec_many(fmt, Ws, rows_list, K, x, [o for _, o in padded], workspace=ws)
    torch.cuda.synchronize()
    assert _ws_intact(wbuf, need)
    for (buf, o), ref, r in zip(padded, refs, rows_list):
        assert _out_intact(buf, r)
        assert np.array_equal(bits(host(o)), bits(host(ref)))


@pytest.mark.parametrize("fmt,ncols", [(synth.FMT_Q4K, 16), (synth.FMT_Q6K, 16), (synth.FMT_Q8_0, 5)])
def test_multi_column_writes_only_its_outputs(fmt, ncols):
    import torch
    rows, K = 4096 if fmt == synth.FMT_Q4K else 777, 4096
    rng = np.random.default_rng(ncols + fmt)
    W = dev(synth.pack(fmt, synth.draw(fmt, rng, rows, K)))
    x = dev(synth.draw_act(rng, ncols, K, outlier_frac=0.001))
    blk = synth.BLOCK[fmt]
    act = qb.alloc_act(ncols, K, blk)
    qb.quantize_act(blk, x, *act)
    ref = _plain((ncols, rows))
    qb.q_gemv(fmt, W, rows, K, act, ncols, ref)
    buf, out = _out((ncols, rows))
    qb.q_gemv(fmt, W, rows, K, act, ncols, out)
    torch.cuda.synchronize()
    assert _out_intact(buf, ncols * rows)
    assert np.array_equal(bits(host(out)), bits(host(ref)))


@pytest.mark.parametrize("fmt", [synth.FMT_Q8_0, synth.FMT_Q4K, synth.FMT_Q6K])
def test_sub32_writes_only_its_outputs(fmt):
    import torch
    rows, K = 300, 4096
    rng = np.random.default_rng(40 + fmt)
    W = dev(synth.pack(fmt, synth.draw(fmt, rng, rows, K)))
    for ncols in (1, 3):
        x = dev(synth.draw_act(rng, ncols, K, outlier_frac=0.001))
        need = qb.q_matvec_sub32_workspace_bytes(K, ncols)
        ref = _plain((ncols, rows))
        qb.q_matvec_sub32(fmt, W, rows, K, x, ref, workspace=torch.empty(need, dtype=torch.uint8, device="cuda"))
        buf, out = _out((ncols, rows))
        wbuf, ws = _ws(need)
        qb.q_matvec_sub32(fmt, W, rows, K, x, out, workspace=ws)
        torch.cuda.synchronize()
        assert _out_intact(buf, ncols * rows)
        assert _ws_intact(wbuf, need)
        assert np.array_equal(bits(host(out)), bits(host(ref)))


@pytest.mark.parametrize("rows,K,ncols", [(1536, 576, 2), (49152, 576, 1), (300, 2048, 3)])
def test_f16_writes_only_its_outputs(rows, K, ncols):
    import torch
    rng = np.random.default_rng(3 + rows)
    W = dev(synth.draw_f16(rng, rows, K))
    x = dev(synth.draw_act(rng, ncols, K))
    need = qb.q_matvec_workspace_bytes(qb.F16, K, ncols)
    ref = _plain((ncols, rows))
    qb.q_matvec(qb.F16, W, rows, K, x, ref, workspace=torch.empty(need, dtype=torch.uint8, device="cuda"))
    buf, out = _out((ncols, rows))
    wbuf, ws = _ws(need)
    qb.q_matvec(qb.F16, W, rows, K, x, out, workspace=ws)
    torch.cuda.synchronize()
    assert _out_intact(buf, ncols * rows)
    assert _ws_intact(wbuf, need)
    assert np.array_equal(bits(host(out)), bits(host(ref)))


@pytest.mark.parametrize("ncols", [1, 3, 16])
def test_fp8_writes_only_its_outputs(ncols):
    import torch
    rows, K = 300, 1024
    rng = np.random.default_rng(ncols)
    W = rng.integers(0, 256, size=(rows, K), dtype=np.uint8)
    W[(W & 0x7F) == 0x7F] = 0x3C
    scales = (2.0 ** rng.uniform(-12, -4, size=((rows + 127) // 128, K // 128))).astype(np.float32)
    x = dev(rng.standard_normal((ncols, K)).astype(np.float32))
    Wd, sd = dev(W), dev(scales)
    ref = _plain((ncols, rows))
    qb.q_gemv_fp8(Wd, sd, rows, K, x, ref)
    buf, out = _out((ncols, rows))
    qb.q_gemv_fp8(Wd, sd, rows, K, x, out)
    torch.cuda.synchronize()
    assert _out_intact(buf, ncols * rows)
    assert np.array_equal(bits(host(out)), bits(host(ref)))


@pytest.mark.parametrize("scaling", [qb.PERBLOCK, qb.SUB32])
def test_kv_scores_write_only_their_outputs(scaling):
    import torch
    nh, nkv, d, L, lcap = 32, 8, 128, 1000, 1024
    rng = np.random.default_rng(7 + scaling)
    q = dev(rng.standard_normal((nh, d)).astype(np.float32))
    k = dev(rng.standard_normal((nkv * lcap, d)).astype(np.float32))
    kc = torch.empty((nkv, lcap, d), dtype=torch.int8, device="cuda")
    ks = torch.empty((nkv, lcap), dtype=torch.int16, device="cuda")
    qb.kv_cache_rows(k, kc.view(nkv * lcap, d), ks.view(-1))
    dp = qb.kv_head_codes(scaling, d)
    qc = torch.empty((nh, dp), dtype=torch.int8, device="cuda")
    qs = torch.empty((nh, dp // 32 if scaling == qb.SUB32 else 1), dtype=torch.int32, device="cuda")
    qb.kv_quantize_heads(scaling, q, qc, qs)
    ref = _plain((nh, L))
    qb.kv_scores(scaling, qc, qs, d, kc, ks, L, 0.125, ref)
    buf, out = _out((nh, L))
    qb.kv_scores(scaling, qc, qs, d, kc, ks, L, 0.125, out)
    torch.cuda.synchronize()
    assert _out_intact(buf, nh * L)
    assert np.array_equal(bits(host(out)), bits(host(ref)))
