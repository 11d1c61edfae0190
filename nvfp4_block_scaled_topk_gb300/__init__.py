"""GB300-native NVFP4 MegaMoE routed-expert forward.

The compute lives in a C-ABI shared library of hand-written sm_103a CUDA
kernels (``csrc/``, declared in ``include/megamoe.h``).  ``megamoe`` is the
thin ctypes binding over it; ``inputs`` draws the seeded synthetic workloads.
Importing this package loads nothing; ``megamoe.load()`` loads the library
and raises if it is missing.
"""

__all__ = ["inputs", "megamoe"]
