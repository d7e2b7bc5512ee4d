"""The CPU oracle -- TEST INFRASTRUCTURE ONLY.

A thin numpy/ctypes wrapper around ``qb_oracle.c``, the plain scalar statement
of what the block-quantized weight x quantized activation product computes
(the decode engine's numerics and lane pages).  Only ``tests/``,
``__graft_entry__.smoke()`` and the benchmark's CPU-baseline leg may import
it; the library never does, and nothing here imports the library.

Every function takes and returns numpy arrays in the library's own layouts:
codes int8 [ncols][K], activation scales (m uint8, e int16) [ncols][K/block],
unit sums int16 [ncols][K/16], outputs f32 [ncols][rows].
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "qb_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_CFLAGS = ["-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fno-strict-aliasing",
           "-shared", "-fPIC"]

F16, Q8_0, Q4K, Q6K = 1, 8, 12, 14
_BLOCK = {Q8_0: 32, Q4K: 256, Q6K: 256}


def build(force: bool = False) -> str:
    """Compile the oracle with the host's gcc (plain C11, no SIMD intrinsics)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", *_CFLAGS, _SRC, "-o", tmp, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


_lib = None


def lib():
    global _lib
    if _lib is None:
        _lib = ctypes.CDLL(build())
        L = _lib
        P = ctypes.c_void_p
        i64, i32 = ctypes.c_int64, ctypes.c_int
        L.or_ftz.argtypes, L.or_ftz.restype = [ctypes.c_float], ctypes.c_float
        L.or_f16_scale.argtypes, L.or_f16_scale.restype = [ctypes.c_uint16, P, P], i32
        L.or_absmax.argtypes, L.or_absmax.restype = [P, i32], ctypes.c_float
        L.or_wide_scale.argtypes, L.or_wide_scale.restype = [ctypes.c_float, P, P], None
        L.or_rne_div.argtypes, L.or_rne_div.restype = [ctypes.c_float, i32, i32], i32
        L.or_quantize_blocks.argtypes = [P, i64, i32, i32, P, P, P, P]
        L.or_quantize_blocks.restype = None
        L.or_scaled_to_f32_2x64.argtypes = [ctypes.c_int64, ctypes.c_uint64, i32]
        L.or_scaled_to_f32_2x64.restype = ctypes.c_float
        L.or_record_bytes.argtypes, L.or_record_bytes.restype = [i32, i64], i64
        L.or_unpack_q4k.argtypes, L.or_unpack_q4k.restype = [P, i64, P, P, P, P, P], None
        L.or_unpack_q6k.argtypes, L.or_unpack_q6k.restype = [P, i64, P, P, P], None
        L.or_unpack_q8_0.argtypes, L.or_unpack_q8_0.restype = [P, i64, P, P], None
        L.or_lane_value.argtypes = [ctypes.c_int64, ctypes.c_int64, ctypes.c_uint16, ctypes.c_uint16,
                                    i32, i32, i32]
        L.or_lane_value.restype = ctypes.c_float
        L.or_block_values.argtypes, L.or_block_values.restype = [i32, P, i64, i64, P, P, P, i32, P, P, P], i32
        L.or_gemv_rows.argtypes, L.or_gemv_rows.restype = [i32, P, i64, i64, i64, i64, P, P, P, i32, P], i32
        L.or_gemv.argtypes, L.or_gemv.restype = [i32, P, i64, i64, P, P, P, i32, P], i32
        L.or_block_sums_excess.argtypes, L.or_block_sums_excess.restype = [i32, P, i64, i64, P, i32, P, P], i32
        L.or_count_unreadable.argtypes, L.or_count_unreadable.restype = [i32, P, i64, i64], i64
        L.or_block_values_w2.argtypes = [i32, P, i64, i64, P, P, P, i32, P, P, P]
        L.or_block_values_w2.restype = i32
        L.or_gemv_w2_rows.argtypes = [i32, P, i64, i64, i64, i64, P, P, P, i32, P]
        L.or_gemv_w2_rows.restype = i32
        L.or_block_sums_excess_w2.argtypes = [i32, P, i64, i64, P, i32, P, P]
        L.or_block_sums_excess_w2.restype = i32
        L.or_f32_to_f16.argtypes, L.or_f32_to_f16.restype = [ctypes.c_float], ctypes.c_uint16
        L.or_f16_to_f32.argtypes, L.or_f16_to_f32.restype = [ctypes.c_uint16], ctypes.c_float
        L.or_gemv_f16.argtypes, L.or_gemv_f16.restype = [P, i64, i64, P, i32, P], i32
        L.or_quantize_f16.argtypes, L.or_quantize_f16.restype = [P, i64, P], None
        L.or_block_scale.argtypes, L.or_block_scale.restype = [ctypes.c_float, P, P], None
        L.or_quantize_sub32.argtypes, L.or_quantize_sub32.restype = [P, i64, i32, P, P, P, P], None
        L.or_exact_sum_f32.argtypes, L.or_exact_sum_f32.restype = [P, P, i32], ctypes.c_float
        L.or_gemv_sub32_rows.argtypes = [i32, P, i64, i64, i64, i64, P, P, P, i32, P]
        L.or_gemv_sub32_rows.restype = i32
        L.or_group_values.argtypes, L.or_group_values.restype = [i32, P, i64, i64, P, P, P, i32, P], i32
        L.or_int8_code.argtypes, L.or_int8_code.restype = [ctypes.c_float, ctypes.c_float], i32
        L.or_cache_rows.argtypes, L.or_cache_rows.restype = [P, i64, i32, P, P], None
        L.or_quantize_heads.argtypes, L.or_quantize_heads.restype = [i32, P, i32, i32, P, P, P], i32
        L.or_int8_score.argtypes = [P, P, P, i32, i32, i32, P, ctypes.c_uint16]
        L.or_int8_score.restype = ctypes.c_float
        L.or_kv_scores.argtypes = [i32, P, P, P, i32, i32, P, P, i64, i64, i32, ctypes.c_float, P]
        L.or_kv_scores.restype = i32
        L.or_e4m3_to_f32.argtypes, L.or_e4m3_to_f32.restype = [ctypes.c_uint8], ctypes.c_float
        L.or_gemv_fp8.argtypes, L.or_gemv_fp8.restype = [P, P, i64, i64, P, i32, P, P], i32
        L.or_exact_dot_f32.argtypes, L.or_exact_dot_f32.restype = [P, P, i64], ctypes.c_float
    return _lib


def _p(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data_as(ctypes.c_void_p)


# ---------------------------------------------------------------- scalars

def ftz(x: float) -> np.float32:
    return np.float32(lib().or_ftz(np.float32(x)))


def f16_scale(h: int):
    """(sig, exp) with value sig*2^exp, or None if the f16 scale is unreadable."""
    sig, ex = ctypes.c_int64(), ctypes.c_int()
    if lib().or_f16_scale(h, ctypes.byref(sig), ctypes.byref(ex)):
        return None
    return sig.value, ex.value


def absmax(x: np.ndarray) -> np.float32:
    x = np.ascontiguousarray(x, dtype=np.float32)
    return np.float32(lib().or_absmax(_p(x), x.size))


def wide_scale(amax: float):
    m, e = ctypes.c_int(), ctypes.c_int()
    lib().or_wide_scale(np.float32(amax), ctypes.byref(m), ctypes.byref(e))
    return m.value, e.value


def rne_div(x: float, m: int, e: int) -> int:
    return lib().or_rne_div(np.float32(x), m, e)


def scaled_to_f32(v: int, ex: int) -> np.float32:
    """v*2^ex rounded once to f32 (RNE, subnormal flushed); |v| < 2^127."""
    hi, lo = v >> 64, v & ((1 << 64) - 1)
    return np.float32(lib().or_scaled_to_f32_2x64(hi, lo, ex))


def lane_value(C: int, O: int, s1: int, s2: int, kind: int, m: int, e: int) -> np.float32:
    return np.float32(lib().or_lane_value(C, O, s1, s2, kind, m, e))


def f32_to_f16(x: float) -> int:
    return int(lib().or_f32_to_f16(np.float32(x)))


def f16_to_f32(h: int) -> np.float32:
    return np.float32(lib().or_f16_to_f32(h))


# ---------------------------------------------------------------- arrays

def quantize_blocks(x: np.ndarray, block: int):
    """x f32 [ncols][K] -> (codes int8, m uint8, e int16, sums16 int16)."""
    x = np.ascontiguousarray(np.atleast_2d(x), dtype=np.float32)
    ncols, K = x.shape
    codes = np.zeros((ncols, K), np.int8)
    m = np.zeros((ncols, K // block), np.uint8)
    e = np.zeros((ncols, K // block), np.int16)
    s16 = np.zeros((ncols, K // 16), np.int16)
    lib().or_quantize_blocks(_p(x), K, ncols, block, _p(codes), _p(m), _p(e), _p(s16))
    return codes, m, e, s16


def record_bytes(fmt: int, K: int) -> int:
    return int(lib().or_record_bytes(fmt, K))


def unpack(fmt: int, W: np.ndarray, rows: int, K: int) -> dict:
    """The oracle's own reading of the packed row records back to logical arrays."""
    W = np.ascontiguousarray(W, dtype=np.uint8)
    rec = record_bytes(fmt, K)
    out = {}
    if fmt == Q4K:
        q = np.zeros((rows, K), np.uint8); sc = np.zeros((rows, K // 32), np.uint8)
        mn = np.zeros((rows, K // 32), np.uint8); d = np.zeros((rows, K // 256), np.uint16)
        dm = np.zeros((rows, K // 256), np.uint16)
        for r in range(rows):
            row = np.ascontiguousarray(W[r * rec:(r + 1) * rec])
            qr, scr, mnr = q[r].copy(), sc[r].copy(), mn[r].copy()
            dr, dmr = d[r].copy(), dm[r].copy()
            lib().or_unpack_q4k(_p(row), K, _p(qr), _p(scr), _p(mnr), _p(dr), _p(dmr))
            q[r], sc[r], mn[r], d[r], dm[r] = qr, scr, mnr, dr, dmr
        out = {"q": q, "sc": sc, "mn": mn, "d": d, "dmin": dm}
    elif fmt == Q6K:
        q = np.zeros((rows, K), np.uint8); sc = np.zeros((rows, K // 16), np.int8)
        d = np.zeros((rows, K // 256), np.uint16)
        for r in range(rows):
            row = np.ascontiguousarray(W[r * rec:(r + 1) * rec])
            qr, scr, dr = q[r].copy(), sc[r].copy(), d[r].copy()
            lib().or_unpack_q6k(_p(row), K, _p(qr), _p(scr), _p(dr))
            q[r], sc[r], d[r] = qr, scr, dr
        out = {"q": q, "sc": sc, "d": d}
    elif fmt == Q8_0:
        q = np.zeros((rows, K), np.int8); d = np.zeros((rows, K // 32), np.uint16)
        for r in range(rows):
            row = np.ascontiguousarray(W[r * rec:(r + 1) * rec])
            qr, dr = q[r].copy(), d[r].copy()
            lib().or_unpack_q8_0(_p(row), K, _p(qr), _p(dr))
            q[r], d[r] = qr, dr
        out = {"q": q, "d": d}
    else:
        raise ValueError(fmt)
    return out


def block_values(fmt: int, W: np.ndarray, rows: int, K: int, codes, m, e):
    """Per (column, row, block): exact sums C, O (int64) and the rounded f32 value."""
    codes = np.ascontiguousarray(np.atleast_2d(codes), np.int8)
    m = np.ascontiguousarray(np.atleast_2d(m), np.uint8)
    e = np.ascontiguousarray(np.atleast_2d(e), np.int16)
    W = np.ascontiguousarray(W, np.uint8)
    ncols = codes.shape[0]
    nb = K // _BLOCK[fmt]
    C = np.zeros((ncols, rows, nb), np.int64); O = np.zeros_like(C)
    v = np.zeros((ncols, rows, nb), np.float32)
    rc = lib().or_block_values(fmt, _p(W), rows, K, _p(codes), _p(m), _p(e), ncols, _p(C), _p(O), _p(v))
    assert rc == 0
    return C, O, v


def block_sums_excess(fmt: int, W: np.ndarray, rows: int, K: int, codes):
    codes = np.ascontiguousarray(np.atleast_2d(codes), np.int8)
    W = np.ascontiguousarray(W, np.uint8)
    ncols = codes.shape[0]
    nb = K // _BLOCK[fmt]
    C = np.zeros((ncols, rows, nb), np.int64); O = np.zeros_like(C)
    assert lib().or_block_sums_excess(fmt, _p(W), rows, K, _p(codes), ncols, _p(C), _p(O)) == 0
    return C, O


def block_values_w2(fmt: int, W: np.ndarray, rows: int, K: int, codes16, m, e):
    """Two-word (16-bit) activation codes: per (column, row, block) the exact
    sums C, O (int64) and the rounded f32 value."""
    codes16 = np.ascontiguousarray(np.atleast_2d(codes16), np.int16)
    m = np.ascontiguousarray(np.atleast_2d(m), np.uint8)
    e = np.ascontiguousarray(np.atleast_2d(e), np.int16)
    W = np.ascontiguousarray(W, np.uint8)
    ncols = codes16.shape[0]
    nb = K // _BLOCK[fmt]
    C = np.zeros((ncols, rows, nb), np.int64); O = np.zeros_like(C)
    v = np.zeros((ncols, rows, nb), np.float32)
    assert lib().or_block_values_w2(fmt, _p(W), rows, K, _p(codes16), _p(m), _p(e), ncols, _p(C), _p(O), _p(v)) == 0
    return C, O, v


def block_sums_excess_w2(fmt: int, W: np.ndarray, rows: int, K: int, codes16):
    """The lane's two-word delivery: block sums rebuilt from the per-word unit sums."""
    codes16 = np.ascontiguousarray(np.atleast_2d(codes16), np.int16)
    W = np.ascontiguousarray(W, np.uint8)
    ncols = codes16.shape[0]
    nb = K // _BLOCK[fmt]
    C = np.zeros((ncols, rows, nb), np.int64); O = np.zeros_like(C)
    assert lib().or_block_sums_excess_w2(fmt, _p(W), rows, K, _p(codes16), ncols, _p(C), _p(O)) == 0
    return C, O


def gemv_w2(fmt: int, W: np.ndarray, rows: int, K: int, codes16, m, e, r0: int = 0, r1: int | None = None,
            out: np.ndarray | None = None) -> np.ndarray:
    """out f32 [ncols][rows] for two-word codes: the in-order fold of the rounded block values."""
    codes16 = np.ascontiguousarray(np.atleast_2d(codes16), np.int16)
    m = np.ascontiguousarray(np.atleast_2d(m), np.uint8)
    e = np.ascontiguousarray(np.atleast_2d(e), np.int16)
    W = np.ascontiguousarray(W, np.uint8)
    ncols = codes16.shape[0]
    if out is None:
        out = np.zeros((ncols, rows), np.float32)
    r1 = rows if r1 is None else r1
    assert lib().or_gemv_w2_rows(fmt, _p(W), rows, r0, r1, K, _p(codes16), _p(m), _p(e), ncols, _p(out)) == 0
    return out


def gemv(fmt: int, W: np.ndarray, rows: int, K: int, codes, m, e, r0: int = 0, r1: int | None = None,
         out: np.ndarray | None = None) -> np.ndarray:
    """out f32 [ncols][rows]: the in-order fold of the rounded block values."""
    codes = np.ascontiguousarray(np.atleast_2d(codes), np.int8)
    m = np.ascontiguousarray(np.atleast_2d(m), np.uint8)
    e = np.ascontiguousarray(np.atleast_2d(e), np.int16)
    W = np.ascontiguousarray(W, np.uint8)
    ncols = codes.shape[0]
    if out is None:
        out = np.zeros((ncols, rows), np.float32)
    r1 = rows if r1 is None else r1
    rc = lib().or_gemv_rows(fmt, _p(W), rows, r0, r1, K, _p(codes), _p(m), _p(e), ncols, _p(out))
    assert rc == 0
    return out


def count_unreadable(fmt: int, W: np.ndarray, rows: int, K: int) -> int:
    W = np.ascontiguousarray(W, np.uint8)
    return int(lib().or_count_unreadable(fmt, _p(W), rows, K))


def quantize_f16(x: np.ndarray) -> np.ndarray:
    x = np.ascontiguousarray(x, np.float32)
    out = np.zeros(x.shape, np.uint16)
    lib().or_quantize_f16(_p(x), x.size, _p(out))
    return out


def gemv_f16(W16: np.ndarray, rows: int, K: int, x16: np.ndarray) -> np.ndarray:
    W16 = np.ascontiguousarray(W16, np.uint16).reshape(rows, K)
    x16 = np.ascontiguousarray(np.atleast_2d(x16), np.uint16)
    ncols = x16.shape[0]
    out = np.zeros((ncols, rows), np.float32)
    assert lib().or_gemv_f16(_p(W16), rows, K, _p(x16), ncols, _p(out)) == 0
    return out


# ---------------------------------------------------------------- ActScaling::Sub32

def block_scale(amax: float):
    """The least m*2^e, m in 8..15, with 127*m*2^e >= amax (numerics page, block_scale)."""
    m, e = ctypes.c_int(), ctypes.c_int()
    lib().or_block_scale(np.float32(amax), ctypes.byref(m), ctypes.byref(e))
    return m.value, e.value


def quantize_sub32(x: np.ndarray):
    """quantize (numerics page) per 32 elements: codes [ncols][K], m, e [ncols][K/32], unit sums."""
    x = np.ascontiguousarray(np.atleast_2d(x), np.float32)
    ncols, K = x.shape
    codes = np.zeros((ncols, K), np.int8)
    m = np.zeros((ncols, K // 32), np.uint8)
    e = np.zeros((ncols, K // 32), np.int16)
    s16 = np.zeros((ncols, K // 16), np.int16)
    lib().or_quantize_sub32(_p(x), K, ncols, _p(codes), _p(m), _p(e), _p(s16))
    return codes, m, e, s16


def exact_sum_f32(sigs, exps) -> np.float32:
    """exact_sum (numerics page) of sig*2^exp terms (|sig| < 2^63), rounded once to f32."""
    sg = np.ascontiguousarray(np.asarray(sigs, np.int64))
    ex = np.ascontiguousarray(np.asarray(exps, np.int32))
    return np.float32(lib().or_exact_sum_f32(_p(sg), _p(ex), len(sg)))


def gemv_sub32(fmt: int, W: np.ndarray, rows: int, K: int, codes, m, e, r0: int = 0, r1: int | None = None,
               out: np.ndarray | None = None) -> np.ndarray:
    """dot under ActScaling::Sub32 for every row and column: out f32 [ncols][rows]."""
    codes = np.ascontiguousarray(np.atleast_2d(codes), np.int8)
    m = np.ascontiguousarray(np.atleast_2d(m), np.uint8)
    e = np.ascontiguousarray(np.atleast_2d(e), np.int16)
    W = np.ascontiguousarray(W, np.uint8)
    ncols = codes.shape[0]
    if out is None:
        out = np.zeros((ncols, rows), np.float32)
    r1 = rows if r1 is None else r1
    rc = lib().or_gemv_sub32_rows(fmt, _p(W), rows, r0, r1, K, _p(codes), _p(m), _p(e), ncols, _p(out))
    assert rc == 0
    return out


def group_values(fmt: int, W: np.ndarray, rows: int, K: int, codes, m, e) -> np.ndarray:
    """Each group's value rounded once (lane page, group): v f32 [ncols][rows][K/256]."""
    codes = np.ascontiguousarray(np.atleast_2d(codes), np.int8)
    m = np.ascontiguousarray(np.atleast_2d(m), np.uint8)
    e = np.ascontiguousarray(np.atleast_2d(e), np.int16)
    W = np.ascontiguousarray(W, np.uint8)
    ncols = codes.shape[0]
    v = np.zeros((ncols, rows, K // 256), np.float32)
    rc = lib().or_group_values(fmt, _p(W), rows, K, _p(codes), _p(m), _p(e), ncols, _p(v))
    assert rc == 0
    return v


# ---------------------------------------------------------------- the int8 cache's score path

def int8_code(x: float, inv: float) -> int:
    """int8_codes (numerics page) of one element under the inverse scale inv."""
    return int(lib().or_int8_code(np.float32(x), np.float32(inv)))


def cache_rows(x: np.ndarray):
    """cache_row (numerics page) of every row of x f32 [n][d]: codes int8 [n][d], f16 scale bits uint16 [n]."""
    x = np.ascontiguousarray(np.atleast_2d(x), np.float32)
    n, d = x.shape
    codes = np.zeros((n, d), np.int8)
    scales = np.zeros(n, np.uint16)
    lib().or_cache_rows(_p(x), n, d, _p(codes), _p(scales))
    return codes, scales


def head_width(scaling: int, d: int) -> int:
    """Codes a quantized head holds: d rounded up to whole groups under Sub32 (1), d under PerBlock (0)."""
    return (d + 255) // 256 * 256 if scaling == 1 else d


def quantize_heads(scaling: int, q: np.ndarray):
    """quantize_head (numerics page) of q f32 [nh][d]: codes [nh][dp], m, e [nh][dp/32] (Sub32) or [nh][1]."""
    q = np.ascontiguousarray(np.atleast_2d(q), np.float32)
    nh, d = q.shape
    dp = head_width(scaling, d)
    nb = dp // 32 if scaling == 1 else 1
    codes = np.zeros((nh, dp), np.int8)
    m = np.zeros((nh, nb), np.uint8)
    e = np.zeros((nh, nb), np.int16)
    assert lib().or_quantize_heads(scaling, _p(q), nh, d, _p(codes), _p(m), _p(e)) == 0
    return codes, m, e


def int8_score(qc, m, e, blk: int, d: int, kc, ks: int) -> np.float32:
    """int8_score (numerics page) of one quantized query head against one cached key row."""
    qc = np.ascontiguousarray(qc, np.int8)
    m = np.ascontiguousarray(m, np.uint8)
    e = np.ascontiguousarray(e, np.int16)
    kc = np.ascontiguousarray(kc, np.int8)
    return np.float32(lib().or_int8_score(_p(qc), _p(m), _p(e), blk, len(m), d, _p(kc), int(ks)))


def kv_scores(scaling: int, qc, qm, qe, d: int, kc, ks, L: int, nkv: int, scale: float) -> np.ndarray:
    """Scores of every query head against L cached key rows: out f32 [nh][L].
    kc int8 [nkv][lcap][d], ks uint16 [nkv][lcap]."""
    qc = np.ascontiguousarray(qc, np.int8)
    qm = np.ascontiguousarray(qm, np.uint8)
    qe = np.ascontiguousarray(qe, np.int16)
    kc = np.ascontiguousarray(kc, np.int8)
    ks = np.ascontiguousarray(ks, np.uint16)
    nh = qc.shape[0]
    lcap = kc.shape[1]
    out = np.zeros((nh, L), np.float32)
    assert lib().or_kv_scores(scaling, _p(qc), _p(qm), _p(qe), nh, d, _p(kc), _p(ks), L, lcap, nkv,
                              np.float32(scale), _p(out)) == 0
    return out


# ---------------------------------------------------------------- FP8 E4M3 with 128x128 block scales

def e4m3_to_f32(b: int) -> np.float32:
    """e4m3ToF32 (colizig OPS page, FP8) of one byte."""
    return np.float32(lib().or_e4m3_to_f32(int(b) & 0xFF))


def exact_dot_f32(x: np.ndarray, w: np.ndarray) -> np.float32:
    """The exact dot of two f32 vectors rounded once to the nearest f32 (the FP8
    path's sum)."""
    x = np.ascontiguousarray(x, np.float32)
    w = np.ascontiguousarray(w, np.float32)
    assert x.shape == w.shape and x.ndim == 1
    return np.float32(lib().or_exact_dot_f32(_p(x), _p(w), x.size))


def gemv_fp8(W: np.ndarray, scales: np.ndarray, rows: int, K: int, x: np.ndarray):
    """matmulFp8 as dequantize-then-dot (exact dot, one rounding): out f32 [ncols][rows] and
    absdot f64 [ncols][rows] = sum |x_i * w_i| (the scale of a summation-error bound)."""
    W = np.ascontiguousarray(W, np.uint8)
    scales = np.ascontiguousarray(scales, np.float32)
    x = np.ascontiguousarray(np.atleast_2d(x), np.float32)
    ncols = x.shape[0]
    out = np.zeros((ncols, rows), np.float32)
    ab = np.zeros((ncols, rows), np.float64)
    assert lib().or_gemv_fp8(_p(W), _p(scales), rows, K, _p(x), ncols, _p(out), _p(ab)) == 0
    return out, ab
