"""fp64 CPU oracle of the sparse MoE layer forward.

TEST INFRASTRUCTURE ONLY: imported by the tests, by the package smoke check
and by the benchmark's CPU-baseline leg, never by the product path.
"""

from .moe_oracle import *  # noqa: F401,F403
