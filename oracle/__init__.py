"""fp64 CPU oracle of the W4A16 routed-expert MoE layer (test infrastructure only),
and in ``w4a8_oracle`` of its W4A8-FP8 variant (no CUDA path yet).

Only the tests, the smoke check and the CPU-baseline leg of the benchmark use
this package; the CUDA path neither imports it nor shares code with it.
"""
from .moe_oracle import *  # noqa: F401,F403
