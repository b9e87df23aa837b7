"""CPU fp64 oracle for exact attention (test infrastructure only).

Imported by the tests, the smoke check and the bench's CPU-baseline leg; the
product path never imports it.
"""
from .attention import (BLOCK, backward, forward, head_backward, head_backward_jacobian,
                        head_forward, head_probs, loss, to_f64, visible)
from .dropout import draw_bytes, keep_mask, multiplier, philox4x32_10, rescale, threshold

__all__ = ["BLOCK", "backward", "forward", "head_backward", "head_backward_jacobian",
           "head_forward", "head_probs", "loss", "to_f64", "visible", "draw_bytes", "keep_mask",
           "multiplier", "philox4x32_10", "rescale", "threshold"]
