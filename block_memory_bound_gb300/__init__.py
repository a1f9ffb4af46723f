"""GB300-native RMSNorm forward and rotate-half RoPE.

The compute path is the CUDA library ``libcamp.so`` (sources in ``csrc/``, C ABI in
``include/camp.h``); :mod:`block_memory_bound_gb300.camp` is its Python binding. Importing
this package loads nothing: the library is opened on first use, and every call raises if
it is missing. There is no CPU or torch fallback.
"""

__all__ = ["camp", "inputs"]
