"""GB300-native NVFP4 routed-expert MoE layer (libnvfp4moe + a thin binding).

The compute path is the CUDA library under ``csrc/`` (built in-tree by
``build.py``); this package only marshals torch tensors into its C ABI
(``include/nvfp4moe.h``).  ``synth`` draws the seeded synthetic inputs.
"""
from ._lib import (MoEWeights, NVFP4Tensor, Nvfp4Error, launch_count, load, moe_combine_rows,  # noqa: F401
                   moe_gather_rows, moe_route_permute,
                   moe_router_logits, moe_shared_expert,
                   moe_workspace, moe_workspace_intermediates, moe_workspace_size, moe_workspace_views,
                   nvfp4_linear, nvfp4_moe_w4a4, nvfp4_moe_w4a16, nvfp4_quantize_act, nvfp4_quantize_weights,
                   profile_collect, profile_enable, selftest_bounded_wait, set_kernel_choice, status_string)
