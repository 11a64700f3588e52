"""Block-sparse decode-step attention for GB300 (sm_103a).

The compute path is liblsa.so (hand-written CUDA kernels behind a C ABI,
declared in include/lsa.h); ``lsa`` is its thin ctypes binding.  Importing
this package does not load the library; the first call does, and fails
loudly if it has not been built.
"""
from . import lsa  # noqa: F401
from .lsa import *  # noqa: F401,F403
