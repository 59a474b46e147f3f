"""Float64 CPU oracle for fused linear cross-entropy (test infrastructure only).

Only the tests, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline / reference arm may
import this package. The product path never imports it.
"""
from .flce_oracle import (  # noqa: F401
    REDUCTIONS,
    backward,
    dlogits,
    flce,
    forward,
    grad_scale,
    grad_weight_rows,
    log_sum_exp,
    logits,
    sampled_rows,
)
