"""CPU oracle of the MoE expert block. Test infrastructure: see moe_oracle's header."""
from .moe_oracle import (route, router_logits, router_weight_backward, aux_stats, aux_loss_grad, dispatch, permute_rows, swiglu_expert, expert_ffn, combine,
                         forward, swiglu_backward, backward, router_backward, router_backward_token,
                         forward_token, backward_token,
                         expert_members, dw_down_rows, dw_gu_cols)

__all__ = ["route", "router_logits", "router_weight_backward", "aux_stats", "aux_loss_grad", "dispatch", "permute_rows", "swiglu_expert", "expert_ffn", "combine",
           "forward", "swiglu_backward", "backward", "router_backward", "router_backward_token",
           "forward_token", "backward_token",
           "expert_members", "dw_down_rows", "dw_gu_cols"]
