"""Seeded synthetic inputs and the byte packing of the weight formats.

This module draws random logical arrays (integer codes, sub-block scales,
f16 block scales, f32 activations) and packs codes and scales into the row
records the library reads.  It holds none of the method's arithmetic: no
quantisation, no dot product, no rounding other than numpy's own f32->f16 cast
of freshly drawn scales.  Both the CUDA path and the CPU oracle consume what it
produces; neither is imported here.

Byte layouts (little endian; the decode engine's pages fix the logical form of
a coded row -- "every weight is a.coef + b.offs of its segment", numerics page,
structs CodedRow / Segment / Scale -- but no byte layout, so these are this
library's own).  A matrix is `rows` row records laid end to end; a record's
size is `record_bytes(fmt, K)`, always a multiple of 16 bytes.

Q8_0, block 32:       codes int8[K] | d f16[K/32] | zero pad to 16 B
Q4_K-like, block 256: K/256 blocks of 144 B, each
                        [0:2) d f16 | [2:4) dmin f16 |
                        [4:10) sc, eight 6-bit fields, field s = bits 6s..6s+5
                               of the 48-bit little-endian integer |
                        [10:16) mn, the same packing |
                        [16:144) qs: 16 B per 32-element sub-block s; byte j
                               holds q[32s+j] in its low nibble and
                               q[32s+16+j] in its high nibble.
                      weight = d*sc[s]*q - dmin*mn[s], q in 0..15.
Q6_K-like, block 256: K/256 blocks of 208 B | d f16[K/256] | zero pad to 16 B.
                      A 208 B block is
                        [0:128) ql: 16 B per 32-element chunk c; byte j holds
                               the low 4 bits of q[32c+j] (low nibble) and of
                               q[32c+16+j] (high nibble) |
                        [128:192) qh: 8 B per chunk c; in bytes 0..3 byte b
                               holds the high 2 bits of q[32c+4k+b] at bits
                               2k..2k+1 (k = 0..3); bytes 4..7 the same for
                               q[32c+16+4k+b] |
                        [192:208) sc int8[16], one per 16-element unit.
                      weight = d*sc[u]*(q-32), q in 0..63.
F16:                  K f16 values (K % 8 == 0).
"""
from __future__ import annotations

import numpy as np

FMT_F16, FMT_Q8_0, FMT_Q4K, FMT_Q6K = 1, 8, 12, 14
FORMAT_NAMES = {FMT_F16: "f16", FMT_Q8_0: "q8_0", FMT_Q4K: "q4k", FMT_Q6K: "q6k"}
BLOCK = {FMT_Q8_0: 32, FMT_Q4K: 256, FMT_Q6K: 256, FMT_F16: 8}


def _round16(n: int) -> int:
    return (n + 15) // 16 * 16


def record_bytes(fmt: int, K: int) -> int:
    """Bytes of one row record of a K-element row."""
    if fmt == FMT_Q8_0:
        return _round16(K + 2 * (K // 32))
    if fmt == FMT_Q4K:
        return 144 * (K // 256)
    if fmt == FMT_Q6K:
        return _round16(210 * (K // 256))
    if fmt == FMT_F16:
        return 2 * K
    raise ValueError(fmt)


def weight_bytes(fmt: int, rows: int, K: int) -> int:
    return rows * record_bytes(fmt, K)


# --------------------------------------------------------------------------
# draws
# --------------------------------------------------------------------------

def log_uniform_f16_bits(rng: np.random.Generator, lo: float, hi: float, shape) -> np.ndarray:
    """exp(U(ln lo, ln hi)) cast to binary16 (numpy's cast rounds to nearest even)."""
    v = np.exp(rng.uniform(np.log(lo), np.log(hi), size=shape))
    return v.astype(np.float16).view(np.uint16)


def draw_q8_0(rng, rows, K, d_range=(1e-3, 1e-2)):
    q = rng.integers(-127, 128, size=(rows, K), dtype=np.int8)
    d = log_uniform_f16_bits(rng, *d_range, (rows, K // 32))
    return {"q": q, "d": d}


def draw_q4k(rng, rows, K, d_range=(1e-4, 1e-2)):
    q = rng.integers(0, 16, size=(rows, K), dtype=np.uint8)
    sc = rng.integers(0, 64, size=(rows, K // 32), dtype=np.uint8)
    mn = rng.integers(0, 64, size=(rows, K // 32), dtype=np.uint8)
    d = log_uniform_f16_bits(rng, *d_range, (rows, K // 256))
    dmin = log_uniform_f16_bits(rng, *d_range, (rows, K // 256))
    return {"q": q, "sc": sc, "mn": mn, "d": d, "dmin": dmin}


def draw_q6k(rng, rows, K, d_range=(1e-5, 1e-3)):
    q = rng.integers(0, 64, size=(rows, K), dtype=np.uint8)
    sc = rng.integers(-128, 128, size=(rows, K // 16), dtype=np.int8)
    d = log_uniform_f16_bits(rng, *d_range, (rows, K // 256))
    return {"q": q, "sc": sc, "d": d}


def draw_f16(rng, rows, K, std=0.02):
    return rng.normal(0.0, std, size=(rows, K)).astype(np.float16).view(np.uint16)


def draw_act(rng, ncols, K, outlier_frac=0.0, outlier_mult=50.0):
    x = rng.standard_normal(size=(ncols, K)).astype(np.float32)
    if outlier_frac > 0:
        mask = rng.random(size=(ncols, K)) < outlier_frac
        x[mask] *= np.float32(outlier_mult)
    return x


# --------------------------------------------------------------------------
# packing (layout only)
# --------------------------------------------------------------------------

def _pack6(vals: np.ndarray) -> np.ndarray:
    """[..., 8] values < 64 -> [..., 6] bytes of a 48-bit little-endian field stream."""
    v = vals.astype(np.uint64)
    acc = np.zeros(vals.shape[:-1], dtype=np.uint64)
    for s in range(8):
        acc |= v[..., s] << np.uint64(6 * s)
    out = np.empty(vals.shape[:-1] + (6,), dtype=np.uint8)
    for b in range(6):
        out[..., b] = ((acc >> np.uint64(8 * b)) & np.uint64(0xFF)).astype(np.uint8)
    return out


def _pad_records(body: np.ndarray, rec: int) -> np.ndarray:
    rows = body.shape[0]
    out = np.zeros((rows, rec), dtype=np.uint8)
    out[:, : body.shape[1]] = body
    return out


def pack_q8_0(q: np.ndarray, d: np.ndarray) -> np.ndarray:
    rows, K = q.shape
    body = np.concatenate([q.view(np.uint8), d.astype("<u2").view(np.uint8).reshape(rows, -1)], axis=1)
    return _pad_records(body, record_bytes(FMT_Q8_0, K)).reshape(-1)


def _nibble_chunks(lo4: np.ndarray) -> np.ndarray:
    """[rows, K] values < 16 -> [rows, K/32, 16] bytes: byte j of chunk c = v[32c+j] | v[32c+16+j] << 4."""
    rows, K = lo4.shape
    v = lo4.reshape(rows, K // 32, 2, 16).astype(np.uint8)
    return (v[:, :, 0, :] | (v[:, :, 1, :] << 4)).astype(np.uint8)


def pack_q4k(q, sc, mn, d, dmin) -> np.ndarray:
    rows, K = q.shape
    nsb = K // 256
    blk = np.zeros((rows, nsb, 144), dtype=np.uint8)
    blk[:, :, 0:2] = d.astype("<u2").view(np.uint8).reshape(rows, nsb, 2)
    blk[:, :, 2:4] = dmin.astype("<u2").view(np.uint8).reshape(rows, nsb, 2)
    blk[:, :, 4:10] = _pack6(sc.reshape(rows, nsb, 8))
    blk[:, :, 10:16] = _pack6(mn.reshape(rows, nsb, 8))
    blk[:, :, 16:144] = _nibble_chunks(q).reshape(rows, nsb, 128)
    return blk.reshape(-1)


def pack_q6k(q, sc, d) -> np.ndarray:
    rows, K = q.shape
    nsb = K // 256
    blk = np.zeros((rows, nsb, 208), dtype=np.uint8)
    blk[:, :, 0:128] = _nibble_chunks(q & 0xF).reshape(rows, nsb, 128)
    hi = (q >> 4).astype(np.uint8).reshape(rows, K // 32, 2, 4, 4)  # [.., half, k, b]
    qh = np.zeros((rows, K // 32, 2, 4), dtype=np.uint8)              # [.., half, b]
    for k in range(4):
        qh |= (hi[:, :, :, k, :] << (2 * k)).astype(np.uint8)
    blk[:, :, 128:192] = qh.reshape(rows, nsb, 64)
    blk[:, :, 192:208] = sc.view(np.uint8).reshape(rows, nsb, 16)
    body = np.concatenate([blk.reshape(rows, -1), d.astype("<u2").view(np.uint8).reshape(rows, -1)], axis=1)
    return _pad_records(body, record_bytes(FMT_Q6K, K)).reshape(-1)


def pack_f16(w16: np.ndarray) -> np.ndarray:
    return np.ascontiguousarray(w16.astype("<u2")).view(np.uint8).reshape(-1)


def pack(fmt: int, logical: dict) -> np.ndarray:
    if fmt == FMT_Q8_0:
        return pack_q8_0(logical["q"], logical["d"])
    if fmt == FMT_Q4K:
        return pack_q4k(logical["q"], logical["sc"], logical["mn"], logical["d"], logical["dmin"])
    if fmt == FMT_Q6K:
        return pack_q6k(logical["q"], logical["sc"], logical["d"])
    if fmt == FMT_F16:
        return pack_f16(logical["w"])
    raise ValueError(fmt)


def draw(fmt: int, rng, rows: int, K: int, **kw) -> dict:
    if fmt == FMT_Q8_0:
        return draw_q8_0(rng, rows, K, **kw)
    if fmt == FMT_Q4K:
        return draw_q4k(rng, rows, K, **kw)
    if fmt == FMT_Q6K:
        return draw_q6k(rng, rows, K, **kw)
    if fmt == FMT_F16:
        return {"w": draw_f16(rng, rows, K, **kw)}
    raise ValueError(fmt)


# --------------------------------------------------------------------------
# the workloads (shapes, value distributions, seeds)
# --------------------------------------------------------------------------

WORKLOADS = {
    # Q8_0 GEMV 512x1024, one column, seed 0
    "q8_0_512x1024": dict(fmt=FMT_Q8_0, mats=[(512, 1024)], ncols=1, seed=0, outliers=0.0),
    # Q4_K-like GEMV 4096x4096, one column, 0.1 % activation outliers x50
    "q4k_4096x4096": dict(fmt=FMT_Q4K, mats=[(4096, 4096)], ncols=1, seed=1, outliers=0.001),
    # Q6_K-like FFN: gate and up 14336x4096 (one shared activation), down 4096x14336
    "q6k_ffn": dict(fmt=FMT_Q6K, mats=[(14336, 4096), (14336, 4096), (4096, 14336)], ncols=1, seed=2,
                    outliers=0.0),
    # F16 tied-embedding logits 49152x576 and a 1536x576 projection, 1..6 columns
    "f16_49152x576": dict(fmt=FMT_F16, mats=[(49152, 576), (1536, 576)], ncols=1, seed=3, outliers=0.0),
}


def workload_inputs(name: str, rows_limit: int | None = None):
    """Logical arrays + packed bytes for each matrix of a workload, and its activation."""
    w = WORKLOADS[name]
    rng = np.random.default_rng(w["seed"])
    mats = []
    for rows, K in w["mats"]:
        r = rows if rows_limit is None else min(rows, rows_limit)
        lg = draw(w["fmt"], rng, r, K)
        mats.append((r, K, lg, pack(w["fmt"], lg)))
    K0 = w["mats"][0][1]
    x = draw_act(rng, w["ncols"], K0, outlier_frac=w["outliers"])
    return mats, x
