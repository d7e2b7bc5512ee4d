"""Block-quantized weight x quantized activation GEMV for GB300 (sm_103a).

The compute path is the C-ABI library ``libqgemv.so`` (hand-written CUDA
kernels; declared in ``include/qgemv.h``).  This module is its thin Python
binding: it marshals torch tensors (device memory, streams) into the C calls
and raises on a non-zero status.  Every step of the product runs in the
library's kernels.  Importing the package does not load the library; the
first call does, and raises if it is missing -- there is no fallback.

Layouts are those of ``include/qgemv.h``: weights as bytes (uint8 tensors of
``q_weight_bytes`` bytes, or uint16 [rows, K] for F16); activation codes int8
[ncols, K], scales int32 [ncols, K/block] (each the 4-byte struct {m u8, pad
u8, e i16}), unit sums int16 [ncols, K/16]; outputs f32 [ncols, rows].
"""
from __future__ import annotations

import ctypes
import os

F16, Q8_0, Q4K, Q6K = 1, 8, 12, 14
BLOCK = {Q8_0: 32, Q4K: 256, Q6K: 256}
FORMATS = {"f16": F16, "q8_0": Q8_0, "q4k": Q4K, "q6k": Q6K}

QB_OK, QB_E_ARG, QB_E_FORMAT, QB_E_BLOCK, QB_E_CUDA, QB_E_UNREADABLE, QB_E_DEVICE = 0, -1, -2, -3, -4, -5, -6
QB_E_SCRATCH = -7
STATIC_SCRATCH_BYTES = 1 << 20  # QB_STATIC_SCRATCH_BYTES
MAX_MATS = 4  # QB_MAX_MATS

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libqgemv.so")

# every entry point include/qgemv.h declares
EXPORTS = ("quantize_act", "q_gemv", "quantize_act_f16", "q_gemv_f16", "q_check_weights", "q_weight_bytes",
           "q_block_values", "q_device_status", "q_strerror", "q_matvec", "q_matvec_workspace_bytes",
           "q_matvec_static", "q_gemv_many", "q_gemv_f16_many", "q_matvec_many", "quantize_act_sub32",
           "q_gemv_sub32", "q_matvec_sub32_workspace_bytes", "q_matvec_sub32", "kv_head_codes", "kv_cache_rows",
           "kv_quantize_heads", "kv_scores", "q_gemv_fp8", "q_matvec_host_workspace_bytes", "q_matvec_host", "q_gemv_w2")
PERBLOCK, SUB32 = 0, 1  # QB_PERBLOCK, QB_SUB32: how an activation (or a query head) is scaled


class QbError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {strerror(status)} ({status})")


class _Act(ctypes.Structure):
    _fields_ = [("block", ctypes.c_int), ("codes", ctypes.c_void_p), ("scales", ctypes.c_void_p),
                ("sums16", ctypes.c_void_p)]


class _Act16(ctypes.Structure):
    _fields_ = [("block", ctypes.c_int), ("codes", ctypes.c_void_p), ("scales", ctypes.c_void_p)]


_lib = None


def lib() -> ctypes.CDLL:
    """The loaded C-ABI library (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with __graft_entry__.build() "
                               "(there is no non-CUDA fallback)")
        L = ctypes.CDLL(LIB_PATH)
        P, i64, i32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
        L.quantize_act.argtypes, L.quantize_act.restype = [i32, P, i64, i32, P, P, P, P], i32
        L.q_gemv.argtypes, L.q_gemv.restype = [i32, P, i64, i64, ctypes.POINTER(_Act), i32, P, P], i32
        L.quantize_act_f16.argtypes, L.quantize_act_f16.restype = [P, i64, i32, P, P], i32
        L.q_gemv_f16.argtypes, L.q_gemv_f16.restype = [P, i64, i64, P, i32, P, P], i32
        L.q_check_weights.argtypes, L.q_check_weights.restype = [i32, P, i64, i64, P], i32
        L.q_weight_bytes.argtypes, L.q_weight_bytes.restype = [i32, i64, i64], i64
        L.q_gemv_w2.argtypes, L.q_gemv_w2.restype = [i32, P, i64, i64, ctypes.POINTER(_Act16), i32, P, P], i32
        L.q_block_values.argtypes = [i32, P, i64, i64, ctypes.POINTER(_Act), i32, P, P, P, P]
        L.q_block_values.restype = i32
        L.q_device_status.argtypes, L.q_device_status.restype = [P], i32
        L.q_strerror.argtypes, L.q_strerror.restype = [i32], ctypes.c_char_p
        L.q_matvec_workspace_bytes.argtypes, L.q_matvec_workspace_bytes.restype = [i32, i64, i32], i64
        L.q_matvec.argtypes = [i32, P, i64, i64, P, i32, P, P, ctypes.c_size_t, P]
        L.q_matvec.restype = i32
        L.q_matvec_static.argtypes, L.q_matvec_static.restype = [i32, P, i64, i64, P, i32, P, P], i32
        L.q_gemv_many.argtypes = [i32, i32, P, P, i64, ctypes.POINTER(_Act), i32, P, P]
        L.q_gemv_many.restype = i32
        L.q_gemv_f16_many.argtypes, L.q_gemv_f16_many.restype = [i32, P, P, i64, P, i32, P, P], i32
        L.q_matvec_many.argtypes = [i32, i32, P, P, i64, P, i32, P, P, ctypes.c_size_t, P]
        L.q_matvec_many.restype = i32
        L.quantize_act_sub32.argtypes, L.quantize_act_sub32.restype = [P, i64, i32, P, P, P, P], i32
        L.q_gemv_sub32.argtypes, L.q_gemv_sub32.restype = [i32, P, i64, i64, ctypes.POINTER(_Act), i32, P, P], i32
        L.q_matvec_sub32_workspace_bytes.argtypes, L.q_matvec_sub32_workspace_bytes.restype = [i64, i32], i64
        L.q_matvec_sub32.argtypes = [i32, P, i64, i64, P, i32, P, P, ctypes.c_size_t, P]
        L.q_matvec_sub32.restype = i32
        L.kv_head_codes.argtypes, L.kv_head_codes.restype = [i32, i32], i32
        L.kv_cache_rows.argtypes, L.kv_cache_rows.restype = [P, i64, i32, P, P, P], i32
        L.kv_quantize_heads.argtypes, L.kv_quantize_heads.restype = [i32, P, i32, i32, P, P, P], i32
        L.kv_scores.argtypes = [i32, P, P, i32, i32, P, P, i64, i64, i32, ctypes.c_float, P, P]
        L.kv_scores.restype = i32
        L.q_gemv_fp8.argtypes, L.q_gemv_fp8.restype = [P, P, i64, i64, P, i32, P, P], i32
        L.q_matvec_host_workspace_bytes.argtypes = [i32, i32, i64, i64, i32]
        L.q_matvec_host_workspace_bytes.restype = i64
        L.q_matvec_host.argtypes = [i32, i32, P, i64, i64, P, i32, P, P, ctypes.c_size_t, P]
        L.q_matvec_host.restype = i32
        _lib = L
    return _lib


def strerror(status: int) -> str:
    return lib().q_strerror(status).decode()


def _check(rc: int, where: str):
    if rc != QB_OK:
        raise QbError(rc, where)


def _ptr(t):
    """Device pointer of a CUDA tensor (None -> NULL).  A CPU tensor is refused
    here: a kernel handed its host address would fault."""
    if t is None:
        return ctypes.c_void_p(0)
    if not t.is_cuda:
        raise ValueError("device memory expected, got a CPU tensor")
    return ctypes.c_void_p(t.data_ptr())


def _hptr(t):
    """Host pointer of a CPU tensor (q_matvec_host's activation and result)."""
    if t.is_cuda:
        raise ValueError("host memory expected, got a CUDA tensor")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    import torch
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


# ------------------------------------------------------------------ activations

def alloc_act(ncols: int, K: int, block: int, device="cuda"):
    """Device buffers (codes, scales, sums16) for a quantized activation."""
    import torch
    codes = torch.empty((ncols, K), dtype=torch.int8, device=device)
    scales = torch.empty((ncols, K // block), dtype=torch.int32, device=device)
    sums16 = torch.empty((ncols, K // 16), dtype=torch.int16, device=device)
    return codes, scales, sums16


def quantize_act(block: int, x, codes, scales, sums16, stream=None) -> None:
    """quantize_blocks under PerBlock: x f32 [ncols, K] -> codes, scales, sums16."""
    ncols, K = x.shape
    _check(lib().quantize_act(block, _ptr(x), K, ncols, _ptr(codes), _ptr(scales), _ptr(sums16), _stream(stream)),
           "quantize_act")


def quantize_act_sub32(x, codes, scales, sums16, stream=None) -> None:
    """quantize under ActScaling::Sub32: x f32 [ncols, K] -> codes, scales (per
    32 elements, m in 8..15), sums16.  Buffers from alloc_act(ncols, K, 32)."""
    ncols, K = x.shape
    _check(lib().quantize_act_sub32(_ptr(x), K, ncols, _ptr(codes), _ptr(scales), _ptr(sums16), _stream(stream)),
           "quantize_act_sub32")


def q_gemv_sub32(fmt: int, W, rows: int, K: int, act, ncols: int, out, stream=None) -> None:
    """dot under Sub32 for every row and column: out f32 [ncols, rows].
    act = (codes, scales, sums16) as written by quantize_act_sub32."""
    codes, scales, sums16 = act
    a = _act(32, codes, scales, sums16)
    _check(lib().q_gemv_sub32(fmt, _ptr(W), rows, K, ctypes.byref(a), ncols, _ptr(out), _stream(stream)),
           "q_gemv_sub32")


def q_matvec_sub32_workspace_bytes(K: int, ncols: int) -> int:
    n = lib().q_matvec_sub32_workspace_bytes(K, ncols)
    if n < 0:
        raise QbError(int(n), "q_matvec_sub32_workspace_bytes")
    return int(n)


def q_matvec_sub32(fmt: int, W, rows: int, K: int, x, out, workspace=None, stream=None) -> None:
    """quantize_act_sub32 then q_gemv_sub32 in one call: x f32 [ncols, K] ->
    out f32 [ncols, rows].  workspace: a 16-byte aligned device buffer of at
    least q_matvec_sub32_workspace_bytes(K, ncols) bytes (allocated here when
    None)."""
    import torch
    ncols = x.shape[0]
    if workspace is None:
        workspace = torch.empty(q_matvec_sub32_workspace_bytes(K, ncols), dtype=torch.uint8, device=x.device)
    _check(lib().q_matvec_sub32(fmt, _ptr(W), rows, K, _ptr(x), ncols, _ptr(out), _ptr(workspace),
                                workspace.numel() * workspace.element_size(), _stream(stream)), "q_matvec_sub32")


def kv_head_codes(scaling: int, d: int) -> int:
    """Codes a quantized query head holds (d rounded up to whole groups under SUB32)."""
    n = lib().kv_head_codes(scaling, d)
    if n < 0:
        raise QbError(n, "kv_head_codes")
    return n


def kv_cache_rows(x, codes, scales, stream=None) -> None:
    """cache_row of every row of x f32 [n, d] -> codes int8 [n, d], scales (f16 bits) int16/uint16 [n]."""
    n, d = x.shape
    _check(lib().kv_cache_rows(_ptr(x), n, d, _ptr(codes), _ptr(scales), _stream(stream)), "kv_cache_rows")


def kv_quantize_heads(scaling: int, q, codes, scales, stream=None) -> None:
    """quantize_head of q f32 [nh, d] -> codes int8 [nh, dp], scales int32 [nh, dp/32] (SUB32) or [nh, 1]."""
    nh, d = q.shape
    _check(lib().kv_quantize_heads(scaling, _ptr(q), nh, d, _ptr(codes), _ptr(scales), _stream(stream)),
           "kv_quantize_heads")


def kv_scores(scaling: int, qcodes, qscales, d: int, kcodes, kscales, L: int, scale: float, out,
              stream=None) -> None:
    """int8_score of every query head against key rows 0..L-1 of its key head, times scale:
    out f32 [nh, L].  kcodes int8 [nkv, lcap, d], kscales [nkv, lcap]."""
    nh = qcodes.shape[0]
    nkv, lcap = kcodes.shape[0], kcodes.shape[1]
    _check(lib().kv_scores(scaling, _ptr(qcodes), _ptr(qscales), nh, d, _ptr(kcodes), _ptr(kscales), L, lcap, nkv,
                           ctypes.c_float(scale), _ptr(out), _stream(stream)), "kv_scores")


def q_gemv_fp8(W, scales, rows: int, K: int, x, out, stream=None) -> None:
    """FP8 E4M3 weights (uint8 [rows, K]) with 128x128 block scales (f32
    [ceil(rows/128), ceil(K/128)]) times x f32 [ncols, K]: out f32 [ncols, rows]."""
    ncols = x.shape[0]
    _check(lib().q_gemv_fp8(_ptr(W), _ptr(scales), rows, K, _ptr(x), ncols, _ptr(out), _stream(stream)),
           "q_gemv_fp8")


def q_matvec_host_workspace_bytes(scaling: int, fmt: int, rows: int, K: int, ncols: int) -> int:
    n = lib().q_matvec_host_workspace_bytes(scaling, fmt, rows, K, ncols)
    if n < 0:
        raise QbError(int(n), "q_matvec_host_workspace_bytes")
    return int(n)


def q_matvec_host(fmt: int, W, rows: int, K: int, x_host, out_host, workspace, scaling: int = PERBLOCK,
                  stream=None) -> None:
    """One call from host to host: x_host f32 [ncols, K] (a pinned CPU tensor for
    an asynchronous call) is copied to the device, multiplied (q_matvec, or
    q_matvec_sub32 with scaling=SUB32) and the result copied into out_host f32
    [ncols, rows] (CPU); synchronize the stream before reading it."""
    ncols = x_host.shape[0]
    _check(lib().q_matvec_host(scaling, fmt, _ptr(W), rows, K, _hptr(x_host), ncols, _hptr(out_host), _ptr(workspace),
                               workspace.numel() * workspace.element_size(), _stream(stream)), "q_matvec_host")


def _act(block, codes, scales, sums16):
    return _Act(block, _ptr(codes).value or 0, _ptr(scales).value or 0, _ptr(sums16).value or 0)


def q_gemv(fmt: int, W, rows: int, K: int, act, ncols: int, out, stream=None) -> None:
    """dot under PerBlock for every row and column: out f32 [ncols, rows].
    act = (codes, scales, sums16) as written by quantize_act."""
    codes, scales, sums16 = act
    a = _act(BLOCK[fmt], codes, scales, sums16)
    _check(lib().q_gemv(fmt, _ptr(W), rows, K, ctypes.byref(a), ncols, _ptr(out), _stream(stream)), "q_gemv")


def q_gemv_w2(fmt: int, W, rows: int, K: int, codes16, scales, ncols: int, out, stream=None) -> None:
    """q_gemv with two-word activation codes: codes16 int16 [ncols, K], scales
    int32 [ncols, K/block] (qb_scale), out f32 [ncols, rows]."""
    a = _Act16(BLOCK[fmt], _ptr(codes16).value, _ptr(scales).value)
    _check(lib().q_gemv_w2(fmt, _ptr(W), rows, K, ctypes.byref(a), ncols, _ptr(out), _stream(stream)), "q_gemv_w2")


def q_block_values(fmt: int, W, rows: int, K: int, act, ncols: int, C=None, O=None, v=None, stream=None) -> None:
    codes, scales, sums16 = act
    a = _act(BLOCK[fmt], codes, scales, sums16)
    _check(lib().q_block_values(fmt, _ptr(W), rows, K, ctypes.byref(a), ncols, _ptr(C), _ptr(O), _ptr(v),
                                _stream(stream)), "q_block_values")


def quantize_act_f16(x, x16, stream=None) -> None:
    ncols, K = x.shape
    _check(lib().quantize_act_f16(_ptr(x), K, ncols, _ptr(x16), _stream(stream)), "quantize_act_f16")


def q_gemv_f16(W, rows: int, K: int, x16, ncols: int, out, stream=None) -> None:
    _check(lib().q_gemv_f16(_ptr(W), rows, K, _ptr(x16), ncols, _ptr(out), _stream(stream)), "q_gemv_f16")


def q_check_weights(fmt: int, W, rows: int, K: int, stream=None) -> int:
    """QB_OK, or QB_E_UNREADABLE if a block scale is inf/NaN (synchronizes)."""
    rc = lib().q_check_weights(fmt, _ptr(W), rows, K, _stream(stream))
    if rc not in (QB_OK, QB_E_UNREADABLE):
        raise QbError(rc, "q_check_weights")
    return rc


def q_weight_bytes(fmt: int, rows: int, K: int) -> int:
    n = lib().q_weight_bytes(fmt, rows, K)
    if n < 0:
        raise QbError(int(n), "q_weight_bytes")
    return int(n)


def q_device_status(stream=None) -> int:
    return lib().q_device_status(_stream(stream))


# ------------------------------------------------------------------ one call

def q_matvec_workspace_bytes(fmt: int, K: int, ncols: int) -> int:
    n = lib().q_matvec_workspace_bytes(fmt, K, ncols)
    if n < 0:
        raise QbError(int(n), "q_matvec_workspace_bytes")
    return int(n)


def q_matvec(fmt: int, W, rows: int, K: int, x, out, workspace=None, stream=None) -> None:
    """The whole product from an f32 activation x [ncols, K]: out f32 [ncols, rows].
    One launch for a single column of a block format (K % 256 == 0); otherwise
    `workspace` (a uint8 device tensor of q_matvec_workspace_bytes) holds the
    quantized activation between the two launches."""
    ncols = x.shape[0]
    nbytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    _check(lib().q_matvec(fmt, _ptr(W), rows, K, _ptr(x), ncols, _ptr(out), _ptr(workspace), nbytes,
                          _stream(stream)), "q_matvec")


def q_matvec_static(fmt: int, W, rows: int, K: int, x, out, stream=None) -> None:
    """q_matvec for callers that cannot allocate device memory: the quantized
    activation goes through a fixed 1 MiB array inside the library (no
    workspace argument, nothing allocated).  Calls on one device share that
    array, so calls that may run at the same time on the GPU must be ordered
    (one stream, or events).  The first call on a device looks up the array's
    address; make it before any stream capture."""
    ncols = x.shape[0]
    _check(lib().q_matvec_static(fmt, _ptr(W), rows, K, _ptr(x), ncols, _ptr(out), _stream(stream)),
           "q_matvec_static")


# ------------------------------------------------------------------ several matrices, one activation

def _tables(Ws, rows, outs):
    n = len(Ws)
    if not (len(rows) == n == len(outs)):
        raise ValueError("Ws, rows and outs must have the same length")
    Wa = (ctypes.c_void_p * n)(*[_ptr(W).value for W in Ws])
    Ra = (ctypes.c_int64 * n)(*[int(r) for r in rows])
    Oa = (ctypes.c_void_p * n)(*[_ptr(o).value for o in outs])
    return n, Wa, Ra, Oa


def q_gemv_many(fmt: int, Ws, rows, K: int, act, ncols: int, outs, stream=None) -> None:
    """q_gemv for several matrices sharing one quantized activation (one launch
    where the shape allows): outs[i] f32 [ncols, rows[i]]."""
    n, Wa, Ra, Oa = _tables(Ws, rows, outs)
    codes, scales, sums16 = act
    a = _act(BLOCK[fmt], codes, scales, sums16)
    _check(lib().q_gemv_many(fmt, n, Wa, Ra, K, ctypes.byref(a), ncols, Oa, _stream(stream)), "q_gemv_many")


def q_gemv_f16_many(Ws, rows, K: int, x16, ncols: int, outs, stream=None) -> None:
    n, Wa, Ra, Oa = _tables(Ws, rows, outs)
    _check(lib().q_gemv_f16_many(n, Wa, Ra, K, _ptr(x16), ncols, Oa, _stream(stream)), "q_gemv_f16_many")


def q_matvec_many(fmt: int, Ws, rows, K: int, x, outs, workspace=None, stream=None) -> None:
    """q_matvec for several matrices sharing the f32 activation x [ncols, K]."""
    n, Wa, Ra, Oa = _tables(Ws, rows, outs)
    ncols = x.shape[0]
    nbytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    _check(lib().q_matvec_many(fmt, n, Wa, Ra, K, _ptr(x), ncols, Oa, _ptr(workspace), nbytes, _stream(stream)),
           "q_matvec_many")


def matvec(fmt: int, W, rows: int, K: int, x, out=None, act=None, stream=None):
    """quantize_act then q_gemv (or quantize_act_f16 then q_gemv_f16): x f32
    [ncols, K] on the device -> out f32 [ncols, rows].  `act` may pass
    preallocated activation buffers (from alloc_act, or a uint16 [ncols, K]
    tensor for F16)."""
    import torch
    ncols = x.shape[0]
    if out is None:
        out = torch.empty((ncols, rows), dtype=torch.float32, device=x.device)
    if fmt == F16:
        x16 = act if act is not None else torch.empty((ncols, K), dtype=torch.int16, device=x.device)
        quantize_act_f16(x, x16, stream)
        q_gemv_f16(W, rows, K, x16, ncols, out, stream)
        return out
    act = act if act is not None else alloc_act(ncols, K, BLOCK[fmt], x.device)
    quantize_act(BLOCK[fmt], x, *act, stream=stream)
    q_gemv(fmt, W, rows, K, act, ncols, out, stream)
    return out
