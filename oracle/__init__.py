"""fp64 CPU oracle for causal / sliding-window GQA attention.

TEST INFRASTRUCTURE ONLY: imported by the tests, the smoke check and the
benchmark's CPU-baseline leg, never by the product path.  It shares no code
with the CUDA library.
"""
from .oracle import (  # noqa: F401
    build,
    forward,
    backward,
    rows,
    key_rows,
    num_threads,
)
