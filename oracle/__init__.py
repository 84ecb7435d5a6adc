"""fp64 CPU oracle for the Gated DeltaNet decode step.

Test infrastructure, not product code: only the test suite, the smoke check
and the benchmark's CPU-baseline leg may import this package.  It shares no
code with the CUDA path and never consumes anything the CUDA path produced.
"""
from .oracle import *  # noqa: F401,F403
