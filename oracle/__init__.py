"""fp64 CPU oracle of the MoE decode path.  Test infrastructure: imported only by
tests, the smoke check and the benchmark's CPU-baseline leg, never by the product."""
from .moe_oracle import *  # noqa: F401,F403
