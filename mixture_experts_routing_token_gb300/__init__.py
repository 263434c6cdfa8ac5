"""GB300 (sm_103a) Mixture-of-Experts layer forward path (and the backward of its
grouped FFN).

The compute lives in ``libmoe_gb300.so`` (hand-written CUDA for sm_103a behind
the C ABI of ``include/moe.h``); this package is its thin Python binding with
the same entry-point names. Build the library with :func:`build`.
``expert_parallel`` runs the layer with its experts split over the ranks of a
process group (one GPU each).
"""
from ._binding import (  # noqa: F401
    MOE_BF16, MOE_F32, MOE_GROUP_TOPK_GREEDY, MOE_GROUP_TOPK_NOAUX_TC, MOE_MAX_EXPERTS, MOE_MAX_TOPK, MOE_STATUS_BAD_INDEX, MOE_STATUS_TIMEOUT,
    MoeError, SIGNATURES, LIB_PATH, MOE_ALIGN_NOALLOC_SCRATCH_INTS, lib, moe_align_by_expert,
    moe_align_by_expert_noalloc, moe_align_workspace_size,
    moe_gating_softmax_topk, moe_gating_softmax_topk_bf16, moe_group_limited_topk,
    moe_grouped_ffn_backward, moe_grouped_ffn_backward_workspace_size, moe_grouped_ffn, moe_grouped_ffn_workspace_size,
    moe_indices_to_multihot, moe_layer_forward, moe_layer_workspace_size, moe_multihot_to_indices,
    moe_gather_rows, moe_ep_receive_index, moe_ep_combine,
    profiler_enable, profiler_report, set_wait_limit_ns, version,
)


def build(force: bool = False) -> str:
    """Compile the CUDA library in-tree (nvcc, sm_103a) and return its path."""
    from .build import build as _build
    return _build(force=force)
