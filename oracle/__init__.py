"""CPU oracle for the sparse-MoE feed-forward layer (test infrastructure).

Only the test suite, ``__graft_entry__.smoke()`` and the benchmark's CPU
baseline leg may import this package.  The product path (the CUDA library
and its binding) never touches it, and it never touches the product path.
"""
from .oracle import (  # noqa: F401
    build,
    dispatch,
    expert_ffn,
    forward,
    max_threads,
    route_stats,
    route,
)
