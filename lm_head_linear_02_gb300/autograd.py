"""PyTorch-facing wrapper of libflce: device memory and streams from torch, compute in libflce.

``flce(x, weight, target, reduction)`` returns the scalar loss and supports ``.backward()``.
torch supplies only the buffers (outputs, workspace, status word) and the current CUDA stream;
every step of the forward and backward runs in the library's kernels. There is no CPU or
PyTorch fallback: without the built library the first call raises.
"""
from __future__ import annotations

import torch

from . import binding as B

__all__ = ["FLCEFunction", "flce", "flce_forward", "flce_backward", "flce_forward_backward",
           "check_status", "FlceDeviceError"]

_DTYPES = {torch.bfloat16: B.FLCE_DTYPE_BF16, torch.float32: B.FLCE_DTYPE_F32}


class FlceDeviceError(RuntimeError):
    """A kernel reported a problem through the device status word."""


def _prep(x: torch.Tensor, weight: torch.Tensor, target: torch.Tensor):
    if not (x.is_cuda and weight.is_cuda and target.is_cuda):
        raise ValueError("x, weight and target must be CUDA tensors")
    if x.device != weight.device or x.device != target.device:
        raise ValueError("x, weight and target must be on the same device")
    if x.dim() != 2 or weight.dim() != 2 or target.dim() != 1:
        raise ValueError("expected x[T,H], weight[V,H], target[T]")
    if x.dtype != weight.dtype or x.dtype not in _DTYPES:
        raise ValueError("x and weight must both be bfloat16 or both float32")
    if target.dtype != torch.int64:
        raise ValueError("target must be int64")
    T, H = x.shape
    V, H2 = weight.shape
    if H2 != H or target.shape[0] != T:
        raise ValueError("shape mismatch")
    return x.contiguous(), weight.contiguous(), target.contiguous(), T, H, V, _DTYPES[x.dtype]


def _saved_lse(lse: torch.Tensor, T: int, device) -> torch.Tensor:
    """The forward's lse as the backward reads it: T fp32 values on the device of x. The C
    entry point cannot see the buffer's length, so a short one is refused here."""
    if lse.device != device:
        raise ValueError("lse must be on the device of x")
    if lse.dim() != 1 or lse.shape[0] != T:
        raise ValueError(f"lse must have shape [{T}] (one value per token)")
    return lse.to(torch.float32).contiguous()


def _reduction(name: str) -> int:
    if name not in ("sum", "mean", "none"):
        raise ValueError(f"reduction must be 'sum', 'mean' or 'none', not {name!r}")
    return B.reduction_code(name)


def _stream(device) -> int:
    return torch.cuda.current_stream(device).cuda_stream


def check_status(status: torch.Tensor) -> None:
    """Synchronise on the status word and raise if any kernel flagged an error."""
    v = int(status.item())
    if v & B.FLCE_STATUS_TARGET_RANGE:
        raise FlceDeviceError("a target lies outside [0, vocab)")
    if v & B.FLCE_STATUS_TIMEOUT:
        raise FlceDeviceError("a kernel pipeline wait timed out; outputs are undefined")
    if v:
        raise FlceDeviceError(f"device status {v}")


def flce_forward(x, weight, target, reduction: str = "mean", status: torch.Tensor | None = None):
    """Enqueue the forward on the current stream. Returns (loss, lse[T], status[1]); loss has
    one element, or T (the per-token losses) for reduction 'none'."""
    x, weight, target, T, H, V, dt = _prep(x, weight, target)
    red = _reduction(reduction)
    dev = x.device
    ws_bytes = B.flce_forward_workspace_size(T, H, V, dt)
    ws = torch.empty(max(ws_bytes, 1), dtype=torch.uint8, device=dev)
    loss = torch.empty(T if reduction == "none" else 1, dtype=torch.float32, device=dev)
    lse = torch.empty(T, dtype=torch.float32, device=dev)
    if status is None:
        status = torch.zeros(1, dtype=torch.int32, device=dev)
    B.flce_forward(x.data_ptr(), weight.data_ptr(), target.data_ptr(), T, H, V, dt,
                   red, loss.data_ptr(), lse.data_ptr(), ws.data_ptr(),
                   ws_bytes, status.data_ptr(), _stream(dev))
    return loss, lse, status


def flce_backward(x, weight, target, lse, grad_loss, reduction: str = "mean",
                  status: torch.Tensor | None = None):
    """Enqueue the backward on the current stream. Returns (grad_x, grad_weight, status).
    grad_loss has one element, or one per token for reduction 'none'."""
    x, weight, target, T, H, V, dt = _prep(x, weight, target)
    red = _reduction(reduction)
    dev = x.device
    lse = _saved_lse(lse, T, dev)
    n = T if reduction == "none" else 1
    grad_loss = grad_loss.reshape(n).to(device=dev, dtype=torch.float32).contiguous()
    ws_bytes = B.flce_backward_workspace_size(T, H, V, dt)
    ws = torch.empty(max(ws_bytes, 1), dtype=torch.uint8, device=dev)
    grad_x = torch.empty_like(x)
    grad_w = torch.empty_like(weight)
    if status is None:
        status = torch.zeros(1, dtype=torch.int32, device=dev)
    B.flce_backward(x.data_ptr(), weight.data_ptr(), target.data_ptr(), lse.data_ptr(), T, H, V,
                    dt, red, grad_loss.data_ptr(), grad_x.data_ptr(),
                    grad_w.data_ptr(), ws.data_ptr(), ws_bytes, status.data_ptr(), _stream(dev))
    return grad_x, grad_w, status


def flce_forward_backward(x, weight, target, grad_loss, reduction: str = "mean",
                          status: torch.Tensor | None = None):
    """Forward and backward in one call on the current stream, for an upstream gradient known in
    advance (one element, or one per token for 'none'). Returns (loss, lse, grad_x,
    grad_weight, status)."""
    x, weight, target, T, H, V, dt = _prep(x, weight, target)
    red = _reduction(reduction)
    dev = x.device
    n = T if reduction == "none" else 1
    grad_loss = grad_loss.reshape(n).to(device=dev, dtype=torch.float32).contiguous()
    ws_bytes = B.flce_forward_backward_workspace_size(T, H, V, dt)
    ws = torch.empty(max(ws_bytes, 1), dtype=torch.uint8, device=dev)
    loss = torch.empty(n, dtype=torch.float32, device=dev)
    lse = torch.empty(T, dtype=torch.float32, device=dev)
    grad_x = torch.empty_like(x)
    grad_w = torch.empty_like(weight)
    if status is None:
        status = torch.zeros(1, dtype=torch.int32, device=dev)
    B.flce_forward_backward(x.data_ptr(), weight.data_ptr(), target.data_ptr(), T, H, V, dt,
                            red, grad_loss.data_ptr(), loss.data_ptr(),
                            lse.data_ptr(), grad_x.data_ptr(), grad_w.data_ptr(), ws.data_ptr(),
                            ws_bytes, status.data_ptr(), _stream(dev))
    return loss, lse, grad_x, grad_w, status


class FLCEFunction(torch.autograd.Function):
    """loss = FLCE(x, weight, target); backward yields grad_x and grad_weight."""

    @staticmethod
    def forward(ctx, x, weight, target, reduction="mean"):
        loss, lse, status = flce_forward(x, weight, target, reduction)
        ctx.save_for_backward(x, weight, target, lse)
        ctx.reduction = reduction
        ctx.status = status
        return loss if reduction == "none" else loss.reshape(())

    @staticmethod
    def backward(ctx, grad_loss):
        x, weight, target, lse = ctx.saved_tensors
        grad_x, grad_w, _ = flce_backward(x, weight, target, lse, grad_loss, ctx.reduction,
                                          status=ctx.status)
        return grad_x, grad_w, None, None


def flce(x, weight, target, reduction: str = "mean"):
    """Fused linear cross-entropy loss with autograd support: a scalar for 'sum' and 'mean',
    the per-token losses [T] for 'none' (fp32)."""
    return FLCEFunction.apply(x, weight, target, reduction)
