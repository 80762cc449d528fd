"""GB300-native (sm_103a) capacity-boundary engine for GrowPage over a paged
KV cache.

The engine is the C-ABI library ``libgrowpage.so`` (include/growpage.h,
kernels in csrc/); ``binding`` is a ctypes layer with the same function
names.  Every hot-path step runs in the CUDA kernels; there is no CPU path.
"""

from .binding import *  # noqa: F401,F403
from .binding import EXPORTS, Request, load  # noqa: F401

__all__ = ["load", "Request", "EXPORTS"]
