"""CPU oracle of the routed MXFP4 MoE block (test infrastructure only)."""
from .moe_oracle import *  # noqa: F401,F403
from .moe_oracle import (bf16_to_f64, dense, dequant_mxfp4, e2m1_value, e8m0_value, experts_combine,
                         expert_ffn, latent_forward, moe_forward, parity_error, post_expert_norm, route,
                         router_logits, routing_scores, score_gap, shared_expert, sigmoid, silu)
