"""GB300-native single-query grouped-query decode attention.

The CUDA kernels and their C ABI live in ``csrc/`` (built into ``libgqadecode.so`` by
``build_lib.py``); ``gqa_decode`` is the thin ctypes binding over that ABI and ``workloads``
draws the seeded synthetic inputs.  Import ``gqa_decode`` explicitly: it loads the shared
library and raises if it has not been built.
"""

__all__ = ["gqa_decode", "workloads"]
