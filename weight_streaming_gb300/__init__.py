"""weight_streaming_gb300: the speculative-decoding verify pass as one weight stream on a GB300.

The compute path is libverify.so (hand-written CUDA for sm_103a behind the C ABI in
include/verify.h); this package holds its build script, the ctypes binding (same names as the C
entry points) and helpers that place packed weights in device memory.
"""
from .build import build  # noqa: F401


def binding():
    """The ctypes binding module (loads libverify.so; raises ImportError if it is not built)."""
    from . import _lib
    return _lib
