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
