"""Single-GPU MoE FFN layer forward for B300 (sm_103a): Python binding of the C ABI in
include/moe.h. The compute path is the CUDA library libmoe.so built from csrc/."""
from .moe import (  # noqa: F401
    ForwardOutputs, LayerWeights, MoEConfig, MoEError, Workspace, capacity, launch_count, load_library,
    make_config, moe_combine, moe_dispatch, moe_expert_ffn, moe_forward, moe_get_status, moe_route,
    moe_route_logits, workspace_size,
)
