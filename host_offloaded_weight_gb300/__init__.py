"""Layer-streamed execution for GB300: parameters in pinned host memory, a
fixed-slot device pool filled ahead of compute, tcgen05 GEMMs for the segments.

The library is the C ABI in include/ls_api.h (liblstream.so); ``lstream`` is its
ctypes binding under the same names. Importing this package fails if the
library has not been built: there is no other code path.
"""
from . import lstream  # noqa: F401
from .lstream import *  # noqa: F401,F403
