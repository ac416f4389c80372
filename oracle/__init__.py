"""fp64 CPU oracle of the W4A16 routed-expert MoE layer (test infrastructure only).

Only the tests, the smoke check and the CPU-baseline leg of the benchmark use
this package; the CUDA path neither imports it nor shares code with it.
"""
from .moe_oracle import *  # noqa: F401,F403
