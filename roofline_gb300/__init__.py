"""FP32 GEMM library for one NVIDIA GB300 (sm_103a).

The compute path is the C-ABI shared library built from ``csrc/``
(``libgb300gemm.so``); ``gemm`` is its thin ctypes binding.  Importing the
binding raises if the library has not been built: there is no CPU fallback.
"""
