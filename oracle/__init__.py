"""CPU fp64 oracle of the MoE FFN layer (test infrastructure only).

Only the tests, the package smoke check and the benchmark's CPU-baseline leg
use this package; the library never imports it.
"""
from .moe_oracle import *  # noqa: F401,F403
from .moe_oracle import (E2M1_TABLE, E4M3_TABLE, decode_bf16, decode_e2m1_packed,  # noqa: F401
                         decode_e4m3, dequant, expert_weights, gates, layer_forward,
                         layer_forward_tokens, near_ties, permute, route, router_logits,
                         shared_weights, silu, swiglu_ffn, topk_ids, x_values,
                         encode_e4m3, act_scale, quantize_act_rows, round_bf16,
                         encode_e2m1, nvfp4_row_scale, nvfp4_block_scale, quantize_nvfp4_act_rows)
from . import qk_rope_oracle  # noqa: F401,E402
