"""fp64 CPU oracle of the expert-parallel MoE layer forward.

TEST INFRASTRUCTURE: only the tests, the smoke check and the benchmark's CPU-baseline
leg import this package. The product path (the CUDA library and its Python binding)
never calls it, and it shares no code, table or helper with that path.
"""
from .moe import (  # noqa: F401
    router_logits, top_k_experts, routing_weights, route,
    expert_partition, load_counts, expert_capacity, dispatch_layout, permute,
    silu, swiglu_expert, expert_outputs, combine_dispatch, combine_mask_sum,
    layer_forward, token_outputs, selection_scores, group_limited_top_k, route_variant,
    update_selection_bias, silu_grad, layer_backward, balance_stats, tp_slices,
    tp_row_split_forward, token_input_grads, expert_weight_grads,
)
