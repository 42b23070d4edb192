"""PyTorch-facing entry point with autograd, mirroring the page's interface.

"CANN ops-transformer 的 aclnnInplacePartialRotaryMul 算子…", section Python 接口与
自动微分: ``inplace_partial_rotary_mul(x, r1, r2, *, rotary_mode="interleave",
partial_slice=None) -> None`` rewrites x in place; when x requires grad the call
goes through an autograd Function that marks x dirty, keeps r1/r2 (cos/sin) and
computes only x's gradient in the backward (cos/sin get None).  As on the page,
x must not be a leaf that requires grad (apply it to e.g. ``y = x * 1.0``).
"""
from __future__ import annotations

from typing import Optional, Sequence

import torch

from . import _capi


class InplacePartialRotaryMulFn(torch.autograd.Function):
    @staticmethod
    def forward(ctx, x, r1, r2, mode: int, start: int, end: int):
        _capi.rope_inplace_partial(x, r1, r2, mode, [start, end])
        ctx.mark_dirty(x)
        ctx.save_for_backward(r1, r2)
        ctx.mode = mode
        ctx.slice = (start, end)
        return x

    @staticmethod
    def backward(ctx, grad_out):
        r1, r2 = ctx.saved_tensors
        g = grad_out.contiguous().clone()  # the backward op works in place; never touch grad_out
        _capi.rope_inplace_partial_backward(g, r1, r2, ctx.mode, list(ctx.slice))
        return g, None, None, None, None, None


def inplace_partial_rotary_mul(x: torch.Tensor, r1: torch.Tensor, r2: torch.Tensor, *,
                               rotary_mode="interleave", partial_slice: Optional[Sequence[int]] = None) -> None:
    """Rotate ``x[..., start:end]`` in place (r1 = cos, r2 = sin); returns None."""
    mode = _capi._mode(rotary_mode)
    start, end = _capi._slice(partial_slice)
    if torch.is_grad_enabled() and x.requires_grad:
        InplacePartialRotaryMulFn.apply(x, r1, r2, mode, start, end)
    else:
        _capi.rope_inplace_partial(x, r1, r2, mode, [start, end])
    return None
