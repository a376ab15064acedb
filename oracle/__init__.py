"""CPU oracle of the MoE expert block. Test infrastructure: see moe_oracle's header."""
from .moe_oracle import (route, dispatch, permute_rows, swiglu_expert, expert_ffn, combine,
                         forward, swiglu_backward, backward, router_backward, router_backward_token,
                         forward_token, backward_token,
                         expert_members, dw_down_rows, dw_gu_cols)

__all__ = ["route", "dispatch", "permute_rows", "swiglu_expert", "expert_ffn", "combine",
           "forward", "swiglu_backward", "backward", "router_backward", "router_backward_token",
           "forward_token", "backward_token",
           "expert_members", "dw_down_rows", "dw_gu_cols"]
