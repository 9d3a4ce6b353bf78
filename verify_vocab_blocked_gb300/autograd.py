"""torch.autograd integration of the fused head (page "mlx-bun 0.0.9 ->
0.0.10", src/train/loss.ts: the custom-VJP wrapper whose forward returns the
log-probabilities and keeps the lse, and whose backward turns the incoming
cotangent into dh).

Marshalling only: the forward is one qhead_fwd call, the backward one qhead_bwd
call with dlogp = the incoming gradient; nothing is computed in torch.  The
head is frozen (no gradient for it); dh is computed in fp32 and returned in the
dtype of h (bf16), as autograd requires.
"""
from __future__ import annotations

import torch

from . import qhead


class HeadLogp(torch.autograd.Function):
    """logp[m] = z[m, targets[m]] - lse[m] for every row of h (0 for rows the
    mask turns off); differentiable in h."""

    @staticmethod
    def forward(ctx, h: torch.Tensor, head: qhead.Head, targets: torch.Tensor,
                mask: torch.Tensor | None = None):
        logp, lse, _ = qhead.fwd(head, h, targets, mask, want_argmax=False)
        ctx.head = head
        ctx.mask = mask
        ctx.save_for_backward(h, targets, lse)
        return logp

    @staticmethod
    def backward(ctx, grad_logp: torch.Tensor):
        h, targets, lse = ctx.saved_tensors
        dlogp = grad_logp.to(torch.float32).contiguous()
        dh = qhead.bwd(ctx.head, h, targets, lse, dlogp, ctx.mask)
        return dh.to(h.dtype), None, None, None


def head_logp(h: torch.Tensor, head: qhead.Head, targets: torch.Tensor,
              mask: torch.Tensor | None = None) -> torch.Tensor:
    """Differentiable per-row log-probabilities of the targets under the
    quantized head: a loss such as -head_logp(...).sum() backpropagates into h
    through the fused backward."""
    return HeadLogp.apply(h, head, targets, mask)
