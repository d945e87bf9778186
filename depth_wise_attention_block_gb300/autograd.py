"""One layer of depth-wise attention as a differentiable torch operation.

`aggregate(H, w)` returns r = sum_s softmax_s(w . RMSNorm(H_s)) H_s for a
[S, T, d] stack of sources (float32 or bfloat16) and an fp32 pseudo-query
[d], and takes part in torch autograd: the forward runs attnres_aggregate,
the backward attnres_aggregate_backward (the forward recomputed inside it,
as under activation checkpointing: only H and w are kept).  Both run in the
library's kernels; torch only allocates the outputs and the backward's
workspace.  Gradients: dH in the sources' dtype, dw in fp32 (summed over
tokens in a fixed order, so bit-reproducible).  The incoming gradient of r
is taken in the sources' dtype (the backward kernel reads it so): an fp32
gradient for bf16 sources is rounded to bf16 first.
"""
from __future__ import annotations

import torch

from . import ATTNRES_DEFAULT_EPS, attnres_aggregate, attnres_aggregate_backward

__all__ = ["AttnResAggregate", "aggregate"]


class AttnResAggregate(torch.autograd.Function):
    @staticmethod
    def forward(ctx, H: torch.Tensor, w: torch.Tensor, eps: float) -> torch.Tensor:
        if H.dim() != 3:
            raise ValueError("H must be [S, T, d]")
        H = H.contiguous()
        S, T, d = H.shape
        r = torch.empty((T, d), dtype=H.dtype, device=H.device)
        attnres_aggregate(H, w, r, None, eps=eps)
        ctx.save_for_backward(H, w)
        ctx.eps = eps
        return r

    @staticmethod
    def backward(ctx, grad_r: torch.Tensor):
        H, w = ctx.saved_tensors
        grad_r = grad_r.to(H.dtype).contiguous()
        grad_H = torch.empty_like(H)
        grad_w = torch.empty_like(w)
        attnres_aggregate_backward(H, w, grad_r, grad_H, grad_w, eps=ctx.eps)
        return (grad_H if ctx.needs_input_grad[0] else None,
                grad_w if ctx.needs_input_grad[1] else None, None)


def aggregate(H: torch.Tensor, w: torch.Tensor, eps: float = ATTNRES_DEFAULT_EPS) -> torch.Tensor:
    """r = sum_s softmax_s(w . RMSNorm(H_s)) H_s, differentiable in H and w."""
    return AttnResAggregate.apply(H, w, eps)
