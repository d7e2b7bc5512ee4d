"""Block-quantized weight x quantized activation GEMV for GB300 (sm_103a).

The compute path is the C-ABI library ``libqgemv.so`` (CUDA kernels); this
package is its thin Python binding.  Importing the package does not load the
library; the first call does, and fails loudly if it is missing.
"""
