"""Float64 CPU oracle of the diffusion-transformer block (test infrastructure only).

Only tests, the smoke check and the CPU-baseline leg of the benchmark import this package.
"""
from .mi_oracle import *  # noqa: F401,F403
