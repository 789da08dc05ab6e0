"""Test infrastructure: the fp64 CPU oracle of the MLA latent pre-projection.

Only the tests, the package's smoke check and the benchmark's CPU-baseline leg
may import this package.  It shares no code with the CUDA path.
"""
from .dsnq_oracle import *  # noqa: F401,F403
from . import dsnq_oracle  # noqa: F401
