"""GB300 (sm_103a) per-head INT8 attention quantization: calibration, quantize-append, decode attention.

The compute path is libfa3.so (C ABI in include/fa3.h); ``fa3`` is its Python binding.
"""
from . import fa3  # noqa: F401
from .build import build  # noqa: F401
