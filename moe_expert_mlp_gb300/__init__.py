"""Routed-expert MLP (grouped GEMM over ragged expert groups, forward and
backward) for one NVIDIA GB300, as a C-ABI CUDA library with a thin Python
binding.  See include/moe.h for the boundary."""
from ._lib import (  # noqa: F401
    EXPORTS,
    MoeError,
    lib,
    make_desc,
    moe_fc1_padded_width,
    moe_group_offsets,
    moe_mlp_bwd,
    moe_mlp_fwd,
    moe_mlp_desc_t,
    moe_permute_bwd,
    moe_read_device_status,
    moe_repack_fc1,
    moe_route_bwd,
    moe_route_permute,
    moe_unpack_fc1,
    moe_unpermute_combine,
    moe_unpermute_combine_bwd,
    moe_workspace_size,
)
from .layer import MoEExpertMLP  # noqa: F401
