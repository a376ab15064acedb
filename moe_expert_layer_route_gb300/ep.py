"""Expert parallelism over G ranks: the MoE block with its experts sharded Shard(0).

"Halo's 2.8x over TRL is not a kernel, and its own benchmark proves it", Figure 3
("EP token routing") and section "Where the gap actually is": tokens are sorted by
expert, a dispatch all-to-all sends each row to the rank that owns its expert, the
owners run their experts, and a combine all-to-all returns the rows to be summed at
their token, weighted by the top-k probabilities. The TorchTurbo README's parallel plan
shards the fused expert tensors Shard(0) over ep_size ranks: rank g owns experts
[g E/G, (g+1) E/G).

Every step on the device is a library call (route, dispatch into the compact send
order, regroup, grouped GEMMs, unregroup, combine, and their backward); this module
only orders them around the two exchanges of each direction:

  counts   all-to-all of the per-expert row counts (rank r receives, from every
           source, the counts of r's experts) -- the receive splits of the rows;
  rows     all-to-all-v of bf16 rows (sent as int32 words: d is a multiple of 8).

`DistExchange` runs them as torch.distributed collectives (NCCL between GPUs; gloo
on CPU tensors). The stage functions are pluggable (`stages`): `CudaStages` calls the
library; a test may pass stand-ins that run the same steps elsewhere. No kernel ever
waits on another rank: the exchanges are host-ordered collectives between launches,
and a rank that never joins one surfaces as the collective's timeout error on the
host (the process group's timeout).
"""
from __future__ import annotations

import dataclasses

import torch

from . import (MoEShape, check_device_status, combine, ep_dispatch, ep_grad_scatter,
               ep_local_shape, ep_regroup, ep_unregroup, expert_ffn, expert_ffn_backward, route,
               shape)


# ------------------------------------------------------------------------ exchanges
class DistExchange:
    """The two exchanges as torch.distributed all-to-alls over `group`."""

    def __init__(self, group=None):
        import torch.distributed as dist
        self.dist = dist
        self.group = group
        self.G = dist.get_world_size(group)
        self.rank = dist.get_rank(group)

    def counts(self, send: torch.Tensor) -> torch.Tensor:
        """send [G, El] int32 (row r to rank r) -> recv [G, El] (row s from rank s)."""
        recv = torch.empty_like(send)
        self.dist.all_to_all_single(recv, send.contiguous(), group=self.group)
        return recv

    def rows(self, buf: torch.Tensor, send_splits: list[int], recv_splits: list[int]
             ) -> torch.Tensor:
        """All-to-all-v of the rows of buf [n, d] (split send_splits by destination) ->
        [sum(recv_splits), d], source-major. Rows travel as int32 words (a bf16 row of
        d, a multiple of 8, is d / 2 words), so any backend moves them bit for bit."""
        n, d = buf.shape
        words = buf.contiguous().view(torch.int32)
        out = torch.empty((sum(recv_splits), words.shape[1]), dtype=torch.int32,
                          device=buf.device)
        self.dist.all_to_all_single(out, words, recv_splits, send_splits, group=self.group)
        return out.view(buf.dtype)


# ---------------------------------------------------------------------------- stages
class CudaStages:
    """The library's CUDA calls for each stage (the default)."""
    route = staticmethod(lambda logits, k: route(logits, k))
    dispatch = staticmethod(lambda s, x, ids: ep_dispatch(s, x, ids))
    regroup = staticmethod(lambda s_loc, G, recv_counts, n, xr: ep_regroup(s_loc, G, recv_counts,
                                                                           n, xr))
    unregroup = staticmethod(lambda s_loc, n, o, dest_of: ep_unregroup(s_loc, n, o, dest_of))
    # raises if a regroup found received counts that do not add up (see moe_ep_regroup)
    check = staticmethod(lambda reg: check_device_status(reg["ws"]))
    combine = staticmethod(lambda s, ob, w, row_of: combine(s, ob, w, row_of))
    grad_scatter = staticmethod(
        lambda s, dy, w, ids, disp, ob, router_grad: ep_grad_scatter(s, dy, w, ids, disp, ob,
                                                                     router_grad))

    @staticmethod
    def expert_ffn(s_loc, xp, counts, w_gu, w_down, training):
        return expert_ffn(s_loc, xp, counts, w_gu, w_down, save_gu=training)

    @staticmethod
    def expert_backward(s_loc, g, xp, gu, h, counts, w_gu, w_down):
        return expert_ffn_backward(s_loc, g, xp, gu, h, counts, w_gu, w_down)


@dataclasses.dataclass
class EPContext:
    """What one rank's forward keeps for its backward."""
    s: MoEShape
    s_loc: MoEShape
    G: int
    ids: torch.Tensor
    w: torch.Tensor
    disp: dict
    recv_counts: torch.Tensor
    send_splits: list
    recv_splits: list
    reg: dict
    h: torch.Tensor
    gu: torch.Tensor | None
    ob: torch.Tensor


def ep_forward(x: torch.Tensor, logits: torch.Tensor, w_gu_loc: torch.Tensor,
               w_down_loc: torch.Tensor, k: int, E: int, exchange, training: bool = False,
               stages=CudaStages) -> tuple[torch.Tensor, EPContext]:
    """One rank's forward. x [T, d] bf16 and logits [T, E] fp32 are this rank's tokens;
    w_gu_loc [El, d, 2f] and w_down_loc [El, f, d] its experts (El = E / G). Returns
    y [T, d] bf16 and the context for ep_backward."""
    G = exchange.G
    T, d = x.shape
    El = w_gu_loc.shape[0]
    if El * G != E:
        raise ValueError(f"{E} experts cannot be split evenly over {G} ranks as {El} each")
    f = w_gu_loc.shape[2] // 2
    s = shape(T, d, E, k, f)
    s_loc = ep_local_shape(s, G)
    ids, w = stages.route(logits, k)
    disp = stages.dispatch(s, x, ids)                    # rows sorted by expert = by owner
    send_counts = disp["counts"].view(G, El)
    recv_counts = exchange.counts(send_counts)
    send_splits = [int(v) for v in send_counts.sum(dim=1).tolist()]
    recv_splits = [int(v) for v in recv_counts.sum(dim=1).tolist()]
    n_recv = sum(recv_splits)
    xr = exchange.rows(disp["xs"], send_splits, recv_splits)
    reg = stages.regroup(s_loc, G, recv_counts, n_recv, xr)
    h, gu, o = stages.expert_ffn(s_loc, reg["xp"], reg["counts"], w_gu_loc, w_down_loc, training)
    orr = stages.unregroup(s_loc, n_recv, o, reg["dest_of"])
    ob = exchange.rows(orr, recv_splits, send_splits)   # back in the send order
    y = stages.combine(s, ob, w, disp["row_of"])
    stages.check(reg)
    ctx = EPContext(s, s_loc, G, ids, w, disp, recv_counts, send_splits, recv_splits, reg, h, gu,
                    ob)
    return y, ctx


def ep_backward(ctx: EPContext, dy: torch.Tensor, w_gu_loc: torch.Tensor,
                w_down_loc: torch.Tensor, exchange, router_grad: bool = False,
                stages=CudaStages):
    """One rank's backward: (dx [T, d], dw_gu_loc, dw_down_loc) and, with router_grad,
    dlogits [T, E]. The weight gradients are complete for this rank's experts: every row
    routed to them from every rank passed through them."""
    n_recv = sum(ctx.recv_splits)
    gs, dl = stages.grad_scatter(ctx.s, dy, ctx.w, ctx.ids, ctx.disp, ctx.ob, router_grad)
    gr = exchange.rows(gs, ctx.send_splits, ctx.recv_splits)
    greg = stages.regroup(ctx.s_loc, ctx.G, ctx.recv_counts, n_recv, gr)
    g_loc = greg["xp"]
    dxp, dw_gu, dw_down = stages.expert_backward(ctx.s_loc, g_loc, ctx.reg["xp"], ctx.gu, ctx.h,
                                                 ctx.reg["counts"], w_gu_loc, w_down_loc)
    dxr = stages.unregroup(ctx.s_loc, n_recv, dxp, ctx.reg["dest_of"])
    dxs = exchange.rows(dxr, ctx.recv_splits, ctx.send_splits)
    dx = stages.combine(ctx.s, dxs, None, ctx.disp["row_of"])
    stages.check(greg)
    return (dx, dw_gu, dw_down, dl) if router_grad else (dx, dw_gu, dw_down)


__all__ = ["DistExchange", "CudaStages", "EPContext", "ep_forward", "ep_backward"]
