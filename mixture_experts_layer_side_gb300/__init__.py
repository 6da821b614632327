"""GB300-native deterministic MoE layer (forward + backward, BF16 / MXFP8).

The compute path is ``libmok.so`` (hand-written CUDA for sm_103a behind the
C ABI in ``include/mok.h``); ``_lib`` is its ctypes binding and ``layer`` a
thin host-side convenience wrapper that owns the workspace tensors.
"""

__version__ = "0.1.0"
