"""ECHO decode hot path on one GB300 (sm_103a).

The product is the C-ABI CUDA library libecho.so (include/echo.h); this package
holds its sources (csrc/), the in-tree build (build.py), the ctypes binding (echo.py),
the buffer plumbing of a decode step (runtime.py) and the seeded synthetic inputs
(synth.py).  Importing the package does not load the library; the first call does,
and fails if it has not been built.
"""
