"""The C-ABI library on a host without a GPU: it loads, exports every entry
point include/*.h declares, and its host-side argument checks answer before
any CUDA call."""
import ctypes
import glob
import os
import re

import pytest

import block_quantized_weight_quantize_gb300 as qb
from block_quantized_weight_quantize_gb300 import synth

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_entry_points():
    names = []
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        src = open(h).read()
        names += re.findall(r"QB_API\s+[\w\s\*]+?\b(\w+)\s*\(", src)
    return names


def test_library_exports_every_declared_symbol():
    L = qb.lib()
    names = declared_entry_points()
    assert len(names) >= 9
    for n in names:
        assert hasattr(L, n), n
    assert set(qb.EXPORTS) <= set(names)


def test_weight_bytes_match_the_layout():
    for fmt in (synth.FMT_Q8_0, synth.FMT_Q4K, synth.FMT_Q6K, synth.FMT_F16):
        for K in (256, 512, 1024, 4096, 14336):
            for rows in (1, 7, 4096):
                assert qb.q_weight_bytes(fmt, rows, K) == synth.weight_bytes(fmt, rows, K)
    assert qb.lib().q_weight_bytes(3, 4, 256) == qb.QB_E_FORMAT
    assert qb.lib().q_weight_bytes(qb.Q4K, 4, 100) == qb.QB_E_ARG


def test_host_argument_checks():
    L = qb.lib()
    act = qb._Act(256, 16, 16, 16)
    W = ctypes.c_void_p(4096)  # never dereferenced: every call below fails its checks first
    out = ctypes.c_void_p(4096)
    assert L.q_gemv(qb.Q4K, None, 4, 256, ctypes.byref(act), 1, out, None) == qb.QB_E_ARG
    assert L.q_gemv(qb.Q4K, W, 4, 256, None, 1, out, None) == qb.QB_E_ARG
    assert L.q_gemv(qb.Q4K, W, 4, 256, ctypes.byref(act), 0, out, None) == qb.QB_E_ARG
    a16 = qb._Act16(256, 16, 16)
    assert L.q_gemv_w2(qb.Q4K, W, 4, 256, ctypes.byref(a16), 17, out, None) == qb.QB_E_ARG
    assert L.q_gemv_w2(qb.Q4K, W, 4, 100, ctypes.byref(a16), 1, out, None) == qb.QB_E_ARG
    assert L.q_gemv_w2(qb.Q8_0, W, 4, 256, ctypes.byref(a16), 1, out, None) == qb.QB_E_BLOCK
    assert L.q_gemv_w2(3, W, 4, 256, ctypes.byref(a16), 1, out, None) == qb.QB_E_FORMAT
    assert L.q_gemv_w2(qb.Q4K, W, 0, 256, ctypes.byref(a16), 1, out, None) == qb.QB_OK   # no rows: nothing to do
    assert L.q_gemv(qb.Q4K, W, 4, 256, ctypes.byref(act), 17, out, None) == qb.QB_E_ARG
    assert L.q_gemv(qb.Q4K, W, 4, 100, ctypes.byref(act), 1, out, None) == qb.QB_E_ARG
    assert L.q_gemv(qb.Q4K, ctypes.c_void_p(4097), 4, 256, ctypes.byref(act), 1, out, None) == qb.QB_E_ARG
    assert L.q_gemv(qb.Q4K, W, -1, 256, ctypes.byref(act), 1, out, None) == qb.QB_E_ARG
    assert L.q_gemv(qb.F16, W, 4, 256, ctypes.byref(act), 1, out, None) == qb.QB_E_FORMAT
    assert L.q_gemv(99, W, 4, 256, ctypes.byref(act), 1, out, None) == qb.QB_E_FORMAT
    act32 = qb._Act(32, 16, 16, 16)
    assert L.q_gemv(qb.Q4K, W, 4, 256, ctypes.byref(act32), 1, out, None) == qb.QB_E_BLOCK
    assert L.q_gemv(qb.Q8_0, W, 4, 256, ctypes.byref(act), 1, out, None) == qb.QB_E_BLOCK
    assert L.quantize_act(64, W, 256, 1, W, W, W, None) == qb.QB_E_BLOCK
    assert L.quantize_act(32, W, 48, 1, W, W, W, None) == qb.QB_E_ARG
    assert L.quantize_act(32, None, 64, 1, W, W, W, None) == qb.QB_E_ARG
    assert L.q_gemv_f16(W, 4, 12, W, 1, out, None) == qb.QB_E_ARG      # K % 8
    assert L.q_check_weights(7, W, 4, 256, None) == qb.QB_E_FORMAT
    for s in (0, -1, -2, -3, -4, -5, -6, -99):
        assert isinstance(qb.strerror(s), str)


def test_binding_fails_loudly_without_library(monkeypatch):
    monkeypatch.setattr(qb, "_lib", None)
    monkeypatch.setattr(qb, "LIB_PATH", "/nonexistent/libqgemv.so")
    with pytest.raises(RuntimeError):
        qb.lib()


def test_matvec_host_argument_checks():
    L = qb.lib()
    P = ctypes.c_void_p
    assert L.q_matvec_host_workspace_bytes(2, qb.Q4K, 4, 256, 1) == qb.QB_E_ARG
    assert L.q_matvec_host_workspace_bytes(qb.SUB32, qb.F16, 4, 256, 1) == qb.QB_E_FORMAT
    assert L.q_matvec_host_workspace_bytes(qb.PERBLOCK, qb.Q4K, 4, 256, 17) == qb.QB_E_ARG
    n = L.q_matvec_host_workspace_bytes(qb.PERBLOCK, qb.Q4K, 4, 256, 1)
    assert n >= 4 * 256 + 4 * 4
    # null host buffers and a short workspace are refused before any CUDA call
    assert L.q_matvec_host(qb.PERBLOCK, qb.Q4K, P(4096), 4, 256, None, 1, P(4096), P(4096), n, None) == qb.QB_E_ARG
    assert L.q_matvec_host(qb.PERBLOCK, qb.Q4K, P(4096), 4, 256, P(4096), 1, P(4096), P(4096), n - 16,
                           None) == qb.QB_E_ARG


def _a16(n):
    return (n + 15) // 16 * 16


def test_workspace_sizes_follow_the_layout():
    """q_matvec / q_matvec_sub32 workspaces: codes, scales and unit sums, each
    16-byte aligned (F16: the rounded activation); bad requests refused."""
    L = qb.lib()
    for fmt, blk in ((qb.Q8_0, 32), (qb.Q4K, 256), (qb.Q6K, 256)):
        for K, nc in ((256, 1), (4096, 1), (14336, 3), (1024, 16)):
            want = _a16(K * nc) + _a16(4 * (K // blk) * nc) + _a16(2 * (K // 16) * nc)
            assert L.q_matvec_workspace_bytes(fmt, K, nc) == want
    assert L.q_matvec_workspace_bytes(qb.F16, 576, 2) == _a16(2 * 576 * 2)
    assert L.q_matvec_workspace_bytes(qb.F16, 12, 1) == qb.QB_E_ARG
    assert L.q_matvec_workspace_bytes(qb.Q4K, 100, 1) == qb.QB_E_ARG
    assert L.q_matvec_workspace_bytes(qb.Q4K, 256, 17) == qb.QB_E_ARG
    assert L.q_matvec_workspace_bytes(99, 256, 1) == qb.QB_E_FORMAT
    for K, nc in ((256, 1), (4096, 1), (14336, 16)):
        assert L.q_matvec_sub32_workspace_bytes(K, nc) == _a16(K * nc) + _a16(4 * (K // 32) * nc) + \
            _a16(2 * (K // 16) * nc)
    assert L.q_matvec_sub32_workspace_bytes(288, 1) == qb.QB_E_ARG
    assert L.q_matvec_sub32_workspace_bytes(256, 0) == qb.QB_E_ARG


def test_sub32_kv_fp8_grouped_host_checks():
    """The later entry points' argument checks answer on the host, before any
    CUDA call; empty requests return 0 without a launch."""
    L = qb.lib()
    P = ctypes.c_void_p
    a, odd = P(4096), P(4097)
    # Sub32
    assert L.quantize_act_sub32(a, 288, 1, a, a, a, None) == qb.QB_E_ARG
    assert L.quantize_act_sub32(a, 256, 17, a, a, a, None) == qb.QB_E_ARG
    assert L.quantize_act_sub32(odd, 256, 1, a, a, a, None) == qb.QB_E_ARG
    assert L.quantize_act_sub32(a, 0, 1, a, a, a, None) == qb.QB_OK
    act256 = qb._Act(256, 4096, 4096, 4096)
    act32 = qb._Act(32, 4096, 4096, 4096)
    assert L.q_gemv_sub32(qb.Q4K, a, 4, 256, ctypes.byref(act256), 1, a, None) == qb.QB_E_BLOCK
    assert L.q_gemv_sub32(qb.F16, a, 4, 256, ctypes.byref(act32), 1, a, None) == qb.QB_E_FORMAT
    assert L.q_gemv_sub32(qb.Q4K, a, 4, 288, ctypes.byref(act32), 1, a, None) == qb.QB_E_ARG
    assert L.q_matvec_sub32(99, a, 4, 256, a, 1, a, None, 0, None) == qb.QB_E_FORMAT
    assert L.q_matvec_sub32(qb.Q4K, a, 0, 256, a, 1, a, None, 0, None) == qb.QB_OK      # no rows
    assert L.q_matvec_sub32(qb.Q4K, a, 4, 256, a, 3, a, None, 0, None) == qb.QB_E_ARG   # 3 columns need a workspace
    # the int8 cache
    assert L.kv_head_codes(qb.SUB32, 128) == 256 and L.kv_head_codes(qb.PERBLOCK, 128) == 128
    assert L.kv_head_codes(qb.SUB32, 320) == 512
    for bad in ((2, 128), (qb.PERBLOCK, 8), (qb.PERBLOCK, 1040), (qb.SUB32, 100)):
        assert L.kv_head_codes(*bad) == qb.QB_E_ARG
    assert L.kv_cache_rows(None, 4, 128, a, a, None) == qb.QB_E_ARG
    assert L.kv_cache_rows(a, 4, 100, a, a, None) == qb.QB_E_ARG
    assert L.kv_cache_rows(odd, 4, 128, a, a, None) == qb.QB_E_ARG
    assert L.kv_cache_rows(a, 0, 128, a, a, None) == qb.QB_OK
    assert L.kv_quantize_heads(qb.SUB32, a, 0, 128, a, a, None) == qb.QB_E_ARG
    assert L.kv_quantize_heads(qb.SUB32, a, 4, 100, a, a, None) == qb.QB_E_ARG
    args = dict(scaling=qb.PERBLOCK, nh=32, d=128, L=100, lcap=128, nkv=8)
    def scores(**kw):
        k = dict(args, **kw)
        return L.kv_scores(k["scaling"], a, a, k["nh"], k["d"], a, a, k["L"], k["lcap"], k["nkv"], 1.0, a, None)
    assert scores(nkv=6) == qb.QB_E_ARG          # 32 heads do not share 6 key heads evenly
    assert scores(lcap=99) == qb.QB_E_ARG        # the cache holds fewer rows than L
    assert scores(d=100) == qb.QB_E_ARG
    assert scores(L=0) == qb.QB_OK               # no positions: nothing launched
    # FP8
    assert L.q_gemv_fp8(a, a, 4, 40, a, 1, a, None) == qb.QB_E_ARG       # K % 16
    assert L.q_gemv_fp8(a, a, 4, 48, a, 17, a, None) == qb.QB_E_ARG      # 17 columns
    assert L.q_gemv_fp8(a, a, 4, 65536, a, 1, a, None) == qb.QB_E_ARG    # K past 32768
    assert L.q_gemv_fp8(odd, a, 4, 48, a, 1, a, None) == qb.QB_E_ARG
    assert L.q_gemv_fp8(a, a, 0, 48, a, 1, a, None) == qb.QB_OK
    # grouped: 1..QB_MAX_MATS matrices, host arrays
    Ws = (ctypes.c_void_p * 5)(*([4096] * 5))
    rows = (ctypes.c_int64 * 5)(*([4] * 5))
    outs = (ctypes.c_void_p * 5)(*([4096] * 5))
    act = qb._Act(256, 4096, 4096, 4096)
    assert L.q_gemv_many(qb.Q4K, 0, Ws, rows, 256, ctypes.byref(act), 1, outs, None) == qb.QB_E_ARG
    assert L.q_gemv_many(qb.Q4K, 5, Ws, rows, 256, ctypes.byref(act), 1, outs, None) == qb.QB_E_ARG
    assert L.q_gemv_many(qb.Q4K, 2, None, rows, 256, ctypes.byref(act), 1, outs, None) == qb.QB_E_ARG


def test_binding_refuses_host_tensors_for_device_arguments():
    """A CPU tensor where the library reads or writes device memory is refused
    by the binding (ValueError) before the library is called -- a kernel handed
    its host address would fault."""
    import torch
    W = torch.zeros(144 * 4, dtype=torch.uint8)
    x = torch.zeros((1, 256), dtype=torch.float32)
    out = torch.zeros((1, 4), dtype=torch.float32)
    with pytest.raises(ValueError):
        qb.q_matvec(qb.Q4K, W, 4, 256, x, out)
    act = (torch.zeros((1, 256), dtype=torch.int8), torch.zeros((1, 1), dtype=torch.int32),
           torch.zeros((1, 16), dtype=torch.int16))
    with pytest.raises(ValueError):
        qb.q_gemv(qb.Q4K, W, 4, 256, act, 1, out)
    with pytest.raises(ValueError):
        qb.q_gemv_many(qb.Q4K, [W, W], [4, 4], 256, act, 1, [out, out])
    with pytest.raises(ValueError):
        qb.q_gemv_fp8(W, torch.ones((1, 2)), 4, 256, x, out)
    with pytest.raises(ValueError):
        qb.kv_cache_rows(torch.zeros((4, 128)), torch.zeros((4, 128), dtype=torch.int8),
                         torch.zeros(4, dtype=torch.int16))
    with pytest.raises(ValueError):
        qb.q_matvec_static(qb.Q4K, W, 4, 256, x, out)
