"""GB300-native batch-1 decode of block-quantized Llama models.

The compute lives in libnt.so (CUDA, sm_103a) behind the C ABI of
include/nt.h; ``nt`` is its ctypes binding.
"""
from . import nt  # noqa: F401  (loads libnt.so; raises if it cannot)

__all__ = ["nt"]
