"""fp64 CPU oracle for jagged softmax attention (test infrastructure only).

Only tests, the smoke check and the benchmark's CPU-baseline arm may import
this package; the CUDA library never does.
"""
from .jfa_oracle import forward, backward, delta_rowsum  # noqa: F401
