"""GB300 (sm_103a) small-T Mixture-of-Experts FFN layer with MXFP4 experts.

The layer runs in the CUDA library libmoe_fp4.so (C ABI declared in
include/moe_fp4.h); ``moe`` is its Python binding and ``inputs`` the seeded
synthetic workloads.  Importing the package does not load the library; the
first call does, and raises if the library has not been built.
"""
from . import inputs  # noqa: F401
