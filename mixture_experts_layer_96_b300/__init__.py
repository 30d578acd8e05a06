"""Single-GPU MoE FFN layer for B300 (sm_103a), forward and backward: Python binding of the C ABI
in include/moe.h. The compute path is the CUDA library libmoe.so built from csrc/."""
from .moe import (  # noqa: F401
    BackwardWorkspace, ForwardOutputs, Grads, LayerWeights, MoEConfig, MoEError, Workspace, capacity,
    launch_count, load_library, make_config, moe_backward, moe_combine, moe_dispatch, moe_dispatch_sharded, moe_expert_ffn,
    moe_forward, moe_forward_hash, moe_forward_profiled, moe_forward_train, moe_get_status, moe_route, moe_route_hash, moe_route_logits, saved_gu_size, set_expert_gemm,
    workspace_size,
)
