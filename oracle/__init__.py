"""fp64 CPU oracle for exact attention: test infrastructure, not part of the product.

Only the tests, ``__graft_entry__.smoke()`` and the bench's CPU-baseline leg may import this package.
The CUDA library never calls it and shares no code with it.

Every function is pinned by checks in ``tests/test_oracle.py`` against closed forms, invariants,
brute force and library routines; none of its expected values comes from the CUDA path.
"""
from .sdpa import (backward, backward_rows, forward, forward_from_scores, forward_rows,
                   online_forward, scores, softmax_rows)

__all__ = ["backward", "backward_rows", "forward", "forward_from_scores", "forward_rows",
           "online_forward", "scores", "softmax_rows"]
