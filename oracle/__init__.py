"""CPU oracle for Depth-Staggered Fibonacci Spacing sparse attention (test infrastructure).

Only the tests, the smoke check and the benchmark's CPU-baseline / reference leg may use
this package.  The product library never imports it; it shares no code with the CUDA path.
"""
from .fib_oracle import (  # noqa: F401
    MODE_INTERP, MODE_MASK, attend, attend_bwd, fibonacci_base,
    index_sets, interp_rungs, mask_distances, pow2_base, rope, rope_angles,
    round_half_even, schedule, virtual_keys,
)
