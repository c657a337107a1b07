"""FP64 CPU oracle for the local MoE forward.

TEST INFRASTRUCTURE ONLY: the test suite, the smoke check and the benchmark's
CPU-baseline leg are the only users.  The product library never imports,
links or calls anything here, and this package imports nothing from it.
"""
from .oracle import (  # noqa: F401
    DTYPE_CODES,
    build,
    combine,
    combine_backward,
    decode,
    dispatch,
    dispatch_backward,
    experts,
    experts_backward,
    forward_tokens,
    num_threads,
    round_to_dtype,
    route,
    route_sigmoid_grouped,
    router_backward,
    selected_router_weights,
    set_threads,
)
