"""GB300-native LazyAttention hot path: paged pre-RoPE KV, RoPE inside the kernels.

The compute lives in liblazyattn.so (C ABI, include/lazyattn.h); this package is
its thin Python binding plus host-side plumbing for device buffers and block
tables. Importing it fails if the library has not been built.
"""
from . import lazyattn  # noqa: F401  (raises ImportError when the library is missing)
from .lazyattn import *  # noqa: F401,F403
from .paged import Batch, DevicePool, Segment, pack_entries  # noqa: F401
