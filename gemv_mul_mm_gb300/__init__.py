"""Fused block-quantized GEMV/GEMM for GB300 (sm_103a).

The compute lives in the CUDA library ``libqmm.so`` (C ABI declared in
``include/qmm.h``); ``gemv_mul_mm_gb300.qmm`` is the thin ctypes binding and
``gemv_mul_mm_gb300.synth`` the seeded input generators.
"""
__all__ = ["qmm", "synth"]
