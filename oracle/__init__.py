"""fp64 CPU oracle for the LazyAttention hot path (test infrastructure only).

Only tests/, __graft_entry__.smoke() and bench.py's cpu_baseline / reference leg
may import this package. The CUDA library never calls it, and it shares no code
with the library: it re-derives everything it needs (RoPE, block-table
decoding, softmax attention) from the paper's definitions.
"""
from .lazyattn_oracle import *  # noqa: F401,F403
from .hit_ratio import *  # noqa: F401,F403
