"""Algorithmic work and traffic of the FLCE hot path (FLOPs and bytes per call).

These counts are what the roofline fractions are computed from; they are properties of the
problem, not of any kernel.

* FLOPs: the forward is one T x V x H contraction (2 T H V); the backward recomputes the logits
  and runs the two gradient contractions (6 T H V), so forward + backward is 8 T H V.
* Bytes: "Fused linear + cross-entropy" (KernelIndex operation page), record panel "Estimated
  floor", counts every declared tensor (x, weight, int64 target, fp32 loss) crossing HBM once.
  The forward also writes the fp32 per-token lse that the backward reads back; the backward
  reads x, weight, target and lse and writes both gradients.
"""
from __future__ import annotations

__all__ = ["flops", "declared_tensor_bytes", "forward_bytes", "backward_bytes"]


def flops(T: int, H: int, V: int, mode: str = "fwd_bwd") -> float:
    """Tensor-core FLOPs: 'fwd' 2THV, 'bwd' 6THV (recompute + 2 contractions), 'fwd_bwd' 8THV,
    'model' 6THV (forward + the two gradient contractions, no recompute)."""
    k = {"fwd": 2, "bwd": 6, "fwd_bwd": 8, "model": 6}[mode]
    return float(k) * T * H * V


def declared_tensor_bytes(T: int, H: int, V: int, elem_bytes: int) -> int:
    """x + weight + int64 target + fp32 loss scalar, each crossing HBM once."""
    return T * H * elem_bytes + V * H * elem_bytes + T * 8 + 4


def forward_bytes(T: int, H: int, V: int, elem_bytes: int) -> int:
    """Forward: the declared tensors plus the saved fp32 lse[T] written once."""
    return declared_tensor_bytes(T, H, V, elem_bytes) + 4 * T


def backward_bytes(T: int, H: int, V: int, elem_bytes: int) -> int:
    """Backward: read x, weight, target, lse and grad_loss; write grad_x and grad_weight."""
    return (2 * T * H * elem_bytes + 2 * V * H * elem_bytes + T * 8 + 4 * T + 4)
