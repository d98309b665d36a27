"""CPU oracle for the sparse-MoE feed-forward layer (test infrastructure).

Only the test suite, ``__graft_entry__.smoke()`` and the benchmark's CPU
baseline leg may import this package.  The product path (the CUDA library
and its binding) never touches it, and it never touches the product path.
"""
from .oracle import (  # noqa: F401
    build,
    dispatch,
    e4m3_decode,
    e4m3_encode,
    expert_ffn,
    forward,
    forward_fp8,
    max_threads,
    quantize_e4m3,
    route_stats,
    route,
)
