"""The benchmark's mirror of the library's kernel choice (host logic, no GPU):
the kernel a bench line names for its roofline and the launches a step it
claims follow the dispatch for the workloads it runs."""
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from block_quantized_weight_quantize_gb300 import synth  # noqa: E402

Q4K, Q6K = synth.FMT_Q4K, synth.FMT_Q6K


@pytest.mark.parametrize("fmt,rows,K,ncols,kernel", [
    (Q4K, 4096, 4096, 4, "gemv7m_kernel"),     # 27 rows a CTA: two CTAs a SM
    (Q4K, 6144, 4096, 4, "gemv7m_kernel"),     # 41 rows a CTA: one CTA a SM
    (Q4K, 28672, 4096, 4, "gemv7r_kernel"),    # past 64 rows a CTA: the ring form
    (Q4K, 4096, 14336, 4, "gemv7r_kernel"),    # K = 14336: chunks of 14 blocks
    (Q4K, 4096, 14336, 2, "gemv7r_kernel"),
    (Q6K, 128256, 4096, 4, "gemv3_kernel"),    # Q6_K-like past the warp-per-block kernel: dp4a CTA ring
    (Q4K, 4096, 4096, 8, "gemv3_kernel"),      # 5..8 columns
    (Q4K, 4096, 4096, 16, "tc_kernel"),        # 9..16 columns: tcgen05
    (Q6K, 4096, 4096, 12, "tc_kernel"),
    (Q4K, 4096, 14336, 16, "gemv3_kernel"),    # K = 14336 does not fit the tensor-core kernel's shared memory
])
def test_multi_column_kernel_choice(fmt, rows, K, ncols, kernel):
    assert bench.multi_col_kernel(fmt, rows, K, ncols).startswith(kernel)


def test_one_column_kernel_choice():
    assert bench.one_col_gemv7(Q4K, 4096, 4096)          # the headline: a warp per block, a lane per row
    assert bench.one_col_gemv7(Q4K, 6144, 4096)          # 41 rows a SM, CTAs of at most 32 rows
    assert not bench.one_col_gemv7(Q6K, 14336, 4096)     # 95 rows a CTA: the warp-ring kernel
    assert not bench.one_col_gemv7(Q4K, 4096, 14336)     # K = 4096 only


def test_tc_needs_nine_columns():
    assert not bench.tc_applies(Q4K, 4096, bench.TC_MIN_COLS - 1)
    assert bench.tc_applies(Q4K, 4096, bench.TC_MIN_COLS)
    assert not bench.tc_applies(synth.FMT_Q8_0, 4096, 16)
