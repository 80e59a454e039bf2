"""CPU fp64 oracle of the MoE SwiGLU FFN forward pass (test infrastructure).

Only the tests, the package's smoke check and the benchmark's CPU-baseline /
reference arm may import this package.  It shares no code with the CUDA
library and imports nothing from it.
"""
from .moe_oracle import *  # noqa: F401,F403
