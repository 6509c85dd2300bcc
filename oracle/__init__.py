"""fp64 CPU oracle for causal flash attention (test infrastructure only).

Importable from the tests, the smoke check and the benchmark's CPU-baseline leg;
never from the CUDA path.
"""
from .attention import (backward, forward, forward_tiled, head_probs,  # noqa: F401
                        key_columns, rows, softmax_jacobian)
