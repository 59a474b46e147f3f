"""GB300-native fused linear cross-entropy (FLCE).

The compute path is the C-ABI library ``libflce.so`` (hand-written sm_103a CUDA) and the thin
ctypes binding in ``lm_head_linear_02_gb300.binding``; ``lm_head_linear_02_gb300.autograd``
wraps it as a ``torch.autograd.Function``. Nothing is imported eagerly here so that the input
generators can be used on machines without the built library.
"""
__all__ = ["binding", "autograd", "inputs", "roofline"]
