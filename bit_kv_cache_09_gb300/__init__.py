"""Quantized KV cache with fused-dequant decode attention for GB300 (sm_103a).

``kvq`` is the ctypes binding of the C ABI (include/kvq.h) and ``cache`` a
PyTorch device-memory harness around it; ``build`` compiles ``libkvq.so``.
"""

from . import kvq  # noqa: F401

__all__ = ["kvq"]
