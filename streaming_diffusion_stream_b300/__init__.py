"""Stream-batch diffusion hot path for B300 (sm_103a).

The compute runs in the CUDA library libsds.so (C ABI, include/sds.h);
this package only marshals arguments to it.  Importing the package does not
load the library; the first call into the binding does, and raises if the
library or a CUDA device is missing -- there is no CPU fallback.
"""
from . import workloads  # noqa: F401

__all__ = ["workloads"]
