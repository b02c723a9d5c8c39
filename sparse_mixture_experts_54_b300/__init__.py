"""Mixtral sparse MoE feed-forward layer on B300 (sm_103a).

The layer runs in hand-written CUDA kernels behind a C ABI (``include/moe.h``,
built into ``libmoe_b300.so`` next to this file).  ``_lib`` is the thin ctypes
binding with the same names as the C entry points; ``layer.MoELayer`` wraps it
for torch tensors (device memory and streams only).  Importing this package
does not load the library; the first call does, and it fails loudly when the
library is missing.
"""

__all__ = ["inputs"]
