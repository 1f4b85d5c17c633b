"""GB300-native paged KV cache decode attention.

The compute path is the C-ABI library ``libpkv.so`` (hand-written CUDA for
sm_103a plus a C++ block manager); ``capi`` is a thin ctypes binding with
the same names, and ``engine`` drives a paged cache through it with torch
for device memory and streams.  Importing the package loads nothing; the
library is loaded on first use and a missing library raises.
"""

__all__ = ["capi", "engine", "workloads", "build"]
