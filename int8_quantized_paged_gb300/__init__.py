"""kvq: quantized, paged KV-cache decode attention for one GB300 (sm_103a).

The compute path is the C-ABI library ``libkvq.so`` (``include/kvq.h``): CUDA
kernels for quantize-on-append, split-K GQA decode attention with a log-sum-exp
combine, and ring-buffer window decode, plus a C++ host page pool and block
tables.  ``kvq`` is its ctypes binding; ``cache.LayerCache`` holds the torch
tensors one layer's cache needs.
"""
from . import kvq  # noqa: F401
from .kvq import KvqError, Config, config  # noqa: F401

__all__ = ["kvq", "KvqError", "Config", "config"]
