"""fp64 CPU oracle for the fused flash-attention training op (test infrastructure only).

Only the tests, the package smoke check and the benchmark's CPU-baseline leg
may import this package. The product path never does.
"""
from .attention import backward, backward_accumulate, forward, probabilities, visibility  # noqa: F401
