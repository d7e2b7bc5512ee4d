"""q_matvec_static -- the product for callers that cannot allocate device
memory (a process whose device memory all belongs to its own pool, a loop that
must not call cudaMalloc).  It keeps the quantized activation in a fixed array
inside the library instead of a caller-provided workspace.

Checked through the C ABI against q_matvec (the entry point with a caller
workspace) bit for bit, on two calls in a row, so that the second call runs on
the scratch contents the first one left.  This file is collected last: if it
fails, every other test has already run.
"""
import ctypes

import numpy as np
import pytest

import block_quantized_weight_quantize_gb300 as qb
from block_quantized_weight_quantize_gb300 import synth

pytestmark = pytest.mark.gpu


def _dev(a):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def _c_static(fmt, W, rows, K, x, out):
    """Calls the C entry point directly (not the Python wrapper)."""
    import torch
    L = qb.lib()
    fn = L.q_matvec_static
    fn.argtypes = [ctypes.c_int, ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64, ctypes.c_void_p, ctypes.c_int,
                   ctypes.c_void_p, ctypes.c_void_p]
    fn.restype = ctypes.c_int
    s = torch.cuda.current_stream().cuda_stream
    return fn(fmt, W.data_ptr(), rows, K, x.data_ptr(), x.shape[0], out.data_ptr(), s)


CASES = [(synth.FMT_Q4K, 4096, 4096, 1), (synth.FMT_Q4K, 261, 4096, 4), (synth.FMT_Q6K, 300, 4096, 2),
         (synth.FMT_Q8_0, 512, 1024, 3), (synth.FMT_F16, 1536, 576, 2)]


@pytest.mark.parametrize("fmt,rows,K,ncols", CASES)
def test_static_scratch_matches_q_matvec(fmt, rows, K, ncols):
    import torch
    assert torch.cuda.is_available()
    rng = np.random.default_rng(1000 + fmt + ncols)
    for call in range(2):  # two calls in a row on the shared scratch
        lg = synth.draw(fmt, rng, rows, K)
        W = _dev(synth.pack(fmt, lg))
        x = _dev(synth.draw_act(rng, ncols, K, outlier_frac=0.001))
        got = torch.full((ncols, rows), float("nan"), dtype=torch.float32, device="cuda")
        want = torch.full((ncols, rows), float("nan"), dtype=torch.float32, device="cuda")
        assert _c_static(fmt, W, rows, K, x, got) == qb.QB_OK
        ws = torch.empty(qb.q_matvec_workspace_bytes(fmt, K, ncols), dtype=torch.uint8, device="cuda")
        qb.q_matvec(fmt, W, rows, K, x, want, workspace=ws)
        torch.cuda.synchronize()
        g = got.cpu().numpy().view(np.uint32)
        w = want.cpu().numpy().view(np.uint32)
        assert np.array_equal(g, w), (call, int((g != w).sum()))
    assert qb.q_device_status() == qb.QB_OK


def test_python_wrapper_matches_q_matvec():
    """The binding's q_matvec_static (argument marshalling only) gives q_matvec's bits."""
    import torch
    fmt, rows, K, ncols = synth.FMT_Q4K, 4096, 4096, 1
    rng = np.random.default_rng(77)
    W = _dev(synth.pack(fmt, synth.draw(fmt, rng, rows, K)))
    x = _dev(synth.draw_act(rng, ncols, K, outlier_frac=0.001))
    got = torch.full((ncols, rows), float("nan"), dtype=torch.float32, device="cuda")
    want = torch.full((ncols, rows), float("nan"), dtype=torch.float32, device="cuda")
    for _ in range(2):
        qb.q_matvec_static(fmt, W, rows, K, x, got)
        qb.q_matvec(fmt, W, rows, K, x, want)
        torch.cuda.synchronize()
        assert np.array_equal(got.cpu().numpy().view(np.uint32), want.cpu().numpy().view(np.uint32))


@pytest.mark.parametrize("fmt", [synth.FMT_Q4K, synth.FMT_Q8_0, synth.FMT_F16])
def test_static_scratch_empty_shapes(fmt):
    """rows == 0 writes nothing; K == 0 writes +0 to every output (the fold of
    no terms), as q_matvec does."""
    import torch
    W = torch.zeros(64, dtype=torch.uint8, device="cuda")
    x = torch.zeros((2, 16), dtype=torch.float32, device="cuda")
    sentinel = torch.full((2, 8), -1.0, dtype=torch.float32, device="cuda")
    assert _c_static(fmt, W, 0, 0, x, sentinel) == qb.QB_OK
    K = 256 if fmt != synth.FMT_F16 else 8
    xk = torch.zeros((2, K), dtype=torch.float32, device="cuda")
    assert _c_static(fmt, W, 0, K, xk, sentinel) == qb.QB_OK
    torch.cuda.synchronize()
    assert bool((sentinel == -1.0).all())
    assert _c_static(fmt, W, 8, 0, x, sentinel) == qb.QB_OK
    torch.cuda.synchronize()
    assert sentinel.cpu().numpy().view(np.uint32).tolist() == [[0] * 8] * 2


def test_static_scratch_rejects_oversize_requests():
    import torch
    K, ncols = 1 << 18, 16   # needs ~4.6 MiB of scratch: beyond the 1 MiB array
    assert qb.q_matvec_workspace_bytes(synth.FMT_Q4K, K, ncols) > qb.STATIC_SCRATCH_BYTES
    W = torch.zeros(16, dtype=torch.uint8, device="cuda")
    x = torch.zeros((ncols, 16), dtype=torch.float32, device="cuda")
    out = torch.zeros((ncols, 1), dtype=torch.float32, device="cuda")
    L = qb.lib()
    rc = L.q_matvec_static(synth.FMT_Q4K, ctypes.c_void_p(W.data_ptr()), 1, K, ctypes.c_void_p(x.data_ptr()),
                           ncols, ctypes.c_void_p(out.data_ptr()), None)
    assert rc == qb.QB_E_SCRATCH
    assert "scratch" in qb.strerror(rc)
