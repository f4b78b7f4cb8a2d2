"""Single-GPU expert-parallel MoE layer forward for B300 (sm_103a).

route -> dispatch into a send layout grouped by expert / logical EP partition ->
tcgen05 grouped-GEMM SwiGLU experts -> weighted combine (or mask-and-sum), all in
hand-written CUDA behind the C ABI of include/moe.h. This package is the thin Python
binding of that library (see binding.py) plus its build script (build.py).
"""
from .binding import (  # noqa: F401
    MOE_DEV_BAD_EXPERT_ID, MOE_DEV_TIMEOUT, MOE_DTYPE_BF16, MOE_DTYPE_FP32, MOE_MODE_DISPATCH,
    MOE_MODE_MASK_SUM, MoeConfig, MoeDiagnostics, MoeError, alloc_workspace, config, lib,
    MOE_PRIORITY_SLOT, MOE_PRIORITY_TOKEN, moe_balance_stats, moe_check_wait_timeout, moe_combine, moe_dispatch,
    moe_dispatch_noalloc, moe_expert_ffn, moe_layer_backward, moe_layer_forward, moe_pack_weights,
    moe_packed_gate_up_size, moe_read_device_status, moe_route, moe_tp_reduce, moe_tp_slice,
    moe_update_selection_bias, moe_workspace_size,
)
