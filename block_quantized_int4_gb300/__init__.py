"""GB300-native block-quantized int4 x int8 matrix products (Q4_0 x Q8_0).

The compute lives in ``libqmm.so`` (hand-written sm_103a CUDA behind the C
ABI of ``include/qmm.h``); ``qmm`` is its thin ctypes binding.  Build with
``block_quantized_int4_gb300._build.build()``.
"""
from ._build import LIB as LIB_PATH, build  # noqa: F401
