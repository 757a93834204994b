"""fp64 CPU oracle for the sparse MoE layer.  Test infrastructure only: imported
by the tests, the package's smoke entry and the benchmark's CPU-baseline leg,
never by the library's product path."""
from .moe_oracle import *  # noqa: F401,F403
