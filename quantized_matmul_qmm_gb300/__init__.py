"""Quantized projection matmul for one GB300 (sm_103a).

The compute lives in ``libqmm.so`` (hand-written CUDA, C ABI in include/qmm.h).
``quantized_matmul_qmm_gb300.qmm`` is its Python binding.  Build the library
with ``quantized_matmul_qmm_gb300.build.build()``.
"""
