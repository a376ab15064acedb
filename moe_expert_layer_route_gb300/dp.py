"""Token data parallelism over G ranks: every rank holds all experts and its own
share of the tokens.

The block's forward needs no exchange at all under this split (a token's route,
experts and combine touch only that token), and the input gradient dX stays on the
token's rank; only the expert weight gradients are sums over every rank's tokens, so
the backward adds one all-reduce of dW_gu and dW_down. `allreduce_weight_grads`
performs it in fp32 (the library's bf16 gradients are widened, summed across ranks,
and rounded back once), so the result does not depend on how the tokens were split
beyond one rounding of each rank's share.
"""
from __future__ import annotations

import torch


def allreduce_weight_grads(grads, group=None) -> None:
    """Sum each tensor of `grads` (e.g. (dw_gu, dw_down)) over the ranks of `group`, in
    place, accumulating in fp32."""
    import torch.distributed as dist
    for g in grads:
        acc = g.float() if g.dtype != torch.float32 else g
        dist.all_reduce(acc, op=dist.ReduceOp.SUM, group=group)
        if acc is not g:
            g.copy_(acc)


__all__ = ["allreduce_weight_grads"]
