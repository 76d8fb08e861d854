"""Fine-grained MoE layer (forward and backward) with aux-loss-free bias balancing on GB300 (sm_103a).

The computation lives in ``libmoe_gb300.so`` (CUDA kernels behind the C ABI declared
in ``include/moe_gb300.h``); this package is its thin ctypes binding.  Build the
library with ``python -m aux_loss_free_gb300.build``.
"""
from ._lib import (  # noqa: F401
    LIB_PATH,
    MOE_W_BF16,
    MOE_W_INT4_G32,
    MOE_X_BF16,
    MOE_X_F32,
    SIGNATURES,
    MoEDebug,
    MoEGrads,
    MoEError,
    MoEShape,
    MoEWeights,
    load_library,
    make_debug,
    make_grads,
    make_shape,
    make_weights,
    moe_abi_version,
    moe_bias_update,
    moe_combine,
    moe_device_status,
    moe_expert_ffn,
    moe_expert_ffn_workspace_size,
    moe_gate_up_block,
    moe_layer_bwd,
    moe_layer_bwd_workspace_size,
    moe_layer_fwd,
    moe_layer_workspace_size,
    moe_pack_gate_up,
    moe_permute,
    moe_permute_noalloc,
    moe_permute_workspace_size,
    moe_profile_start,
    moe_profile_stop,
    moe_quantize_int4,
    moe_route,
    moe_route_workspace_size,
)
