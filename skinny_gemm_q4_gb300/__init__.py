"""GB300-native fused 4-bit block-quantized GEMV / skinny GEMM.

The compute path is the C-ABI CUDA library ``libqgemv.so`` (sources in
``csrc/``, declarations in ``include/qgemv.h``); ``qgemv`` is its thin ctypes
binding.  ``synth`` holds the seeded synthetic input generators.
"""
__all__ = ["qgemv", "synth"]
