"""GB300-native (sm_103a) sparse MLA attention forward.

The compute path is the CUDA library ``libsparse_mla.so`` (built from
``csrc/``) behind a C ABI declared in ``include/sparse_mla.h``. This package
holds its thin ctypes binding (``binding``) and the seeded synthetic input
recipes (``inputs``). Importing the package loads nothing; the binding loads
the library on first use and raises if it is missing.
"""
