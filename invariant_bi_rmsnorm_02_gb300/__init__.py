"""Batch-invariant reduction kernels (RMSNorm, GEMM, paged attention) for
GB300, behind a C ABI (``libbi.so``, declared in ``include/bi.h``)."""
from ._binding import *  # noqa: F401,F403
from ._binding import load  # noqa: F401
