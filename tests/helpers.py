"""Shared helpers of the GPU parity tests: seeded inputs from the synth module,
the oracle on the CPU, the library's kernels on cuda:0 through the C ABI."""
import numpy as np

import oracle
from block_quantized_weight_quantize_gb300 import synth


def dev(a: np.ndarray):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def host(t) -> np.ndarray:
    return t.cpu().numpy()


def bits(a) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=np.float32).view(np.uint32)


def oracle_act(x: np.ndarray, block: int):
    """codes, m, e, sums16 and the scales packed as the library's int32 struct."""
    codes, m, e, s16 = oracle.quantize_blocks(x, block)
    packed = (m.astype(np.uint32) | (e.astype(np.int32).astype(np.uint32) << 16)).view(np.int32)
    return codes, m, e, s16, packed


def unpack_scales(packed: np.ndarray):
    u = packed.view(np.uint32)
    return (u & 0xFF).astype(np.uint8), (u >> 16).astype(np.uint16).view(np.int16)


def gpu_act_from_oracle(codes, packed, s16):
    return dev(codes), dev(packed), dev(s16)


def make_case(fmt: int, rows: int, K: int, ncols: int, seed: int, outliers: float = 0.0, **kw):
    rng = np.random.default_rng(seed)
    lg = synth.draw(fmt, rng, rows, K, **kw)
    W = synth.pack(fmt, lg)
    x = synth.draw_act(rng, ncols, K, outlier_frac=outliers)
    return lg, W, x
