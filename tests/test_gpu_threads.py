"""The library driven from several host threads at once (one process, cuda:0).

Each thread has its own stream and inputs and runs a different kind of call
(one-column single launch, several columns, the Q6_K-like and Q8_0 formats,
F16); the kernels' shared-memory limits are raised per (kernel, device) under a
lock, so concurrent first launches are safe.  Every output must equal, bit for
bit, the same call made from a single thread beforehand.
"""
import threading

import numpy as np
import pytest

import block_quantized_weight_quantize_gb300 as qb
from block_quantized_weight_quantize_gb300 import synth

pytestmark = pytest.mark.gpu


def _case(fmt, rows, K, ncols, seed):
    import torch
    rng = np.random.default_rng(seed)
    W = torch.from_numpy(synth.pack(fmt, synth.draw(fmt, rng, rows, K))).cuda()
    x = torch.from_numpy(synth.draw_act(rng, ncols, K, outlier_frac=0.001)).cuda()
    ws = torch.empty(max(16, qb.q_matvec_workspace_bytes(fmt, K, ncols)), dtype=torch.uint8, device="cuda")
    return W, x, ws


def test_library_from_several_host_threads():
    import torch
    cases = [(synth.FMT_Q4K, 4096, 4096, 1), (synth.FMT_Q4K, 1000, 4096, 3), (synth.FMT_Q6K, 777, 4096, 1),
             (synth.FMT_Q8_0, 512, 1024, 2), (synth.FMT_F16, 1536, 576, 2), (synth.FMT_Q4K, 300, 14336, 1)]
    inputs = [_case(f, r, k, n, 500 + i) for i, (f, r, k, n) in enumerate(cases)]
    want = []
    for (f, r, k, n), (W, x, ws) in zip(cases, inputs):
        out = torch.empty((n, r), dtype=torch.float32, device="cuda")
        qb.q_matvec(f, W, r, k, x, out, workspace=ws)
        torch.cuda.synchronize()
        want.append(out.cpu().numpy().view(np.uint32).copy())

    errors = []
    results = [None] * len(cases)

    def worker(i):
        try:
            f, r, k, n = cases[i]
            W, x, ws = inputs[i]
            s = torch.cuda.Stream()
            out = torch.full((n, r), float("nan"), dtype=torch.float32, device="cuda")
            for _ in range(20):
                qb.q_matvec(f, W, r, k, x, out, workspace=ws, stream=s)
            s.synchronize()
            results[i] = out.cpu().numpy().view(np.uint32).copy()
        except Exception as exc:  # reported by the main thread
            errors.append((i, repr(exc)))

    threads = [threading.Thread(target=worker, args=(i,)) for i in range(len(cases))]
    for t in threads:
        t.start()
    for t in threads:
        t.join(timeout=120)
    assert not any(t.is_alive() for t in threads)
    assert not errors, errors
    for i in range(len(cases)):
        assert np.array_equal(results[i], want[i]), cases[i]
    assert qb.q_device_status() == qb.QB_OK
