"""GB300 (sm_103a) MoE-layer forward: router, top-k softmax gating, stable expert
routing, tcgen05 grouped GEMMs with fused SwiGLU, and finalize -- hand-written CUDA
behind a C ABI (``include/moe_gb300.h``), with this package as a thin binding.

The ops are loaded lazily from the in-tree ``_lib/libmoe_gb300.so``; importing the
package does not need a GPU, calling an op does (there is no CPU fallback).
"""
from ._binding import (  # noqa: F401
    DEV_BAD_EXPERT_ID,
    DEV_WAIT_TIMEOUT,
    GraphedMoELayer,
    MoEError,
    MoELayer,
    MoELayerMX,
    MoELayerV2,
    MoELayerW4A8,
    add_rmsnorm_cast,
    finalize_routing_v2,
    init_routing_v2,
    re_routing,
    add_rmsnorm_mxquant,
    mx_quantize,
    pack_weights_mx,
    pack_weights_mx4,
    clear_device_status,
    compute_expert_tokens,
    exported_symbols,
    finalize_routing,
    forward,
    forward_workspace_bytes,
    gating_topk_softmax,
    get_device_status,
    grouped_matmul,
    grouped_matmul_swiglu,
    grouped_matmul_mx,
    grouped_matmul_swiglu_mx,
    init_routing,
    lib,
    library_path,
    pack_weights,
    router_logits,
    set_gemm_events,
    debug_set_gemm_stall,
    debug_set_pair_light,
)
from .workloads import CONFIGS, MoEConfig, make_inputs  # noqa: F401
