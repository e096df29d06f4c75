"""B300 (sm_103a) forward pass of the sparsely-gated noisy top-k MoE layer.

The compute lives in libmoe_b300.so (C ABI: include/moe.h), built from
csrc/ by ``python -m sparsely_gated_mixture_03_b300.build``.  ``binding``
exposes its entry points to Python with the same names; ``synthetic`` draws
seeded inputs shaped like the pages' workloads.
"""
from .binding import (FLAG_DEVICE_NOISE, FLAG_FFN_ROW_TILES, FLAG_FFN_SIZED_TILES, FLAG_SWITCH_GATE, MoeConfig, MoeError, MoeHierConfig, alloc_hier_workspace, alloc_workspace,
                      alloc_backward_workspace, alloc_batchwise_workspace,
                      backward_workspace_size, batchwise_workspace_size, expert_rows_dtype,
                      hier_workspace_size, lib, make_config, make_hier_config, moe_backward,
                      moe_backward_timed, moe_batchwise_forward, moe_batchwise_threshold_forward,
                      moe_balance_losses, moe_combine, moe_dispatch, moe_dispatch_noalloc,
                      moe_draw_noise, ep_plan_size, moe_ep_plan, moe_ep_regroup, moe_losses_from_sums,
                      moe_expert_ffn, moe_forward, moe_forward_timed, moe_gate,
                      moe_get_device_error, moe_hier_forward, moe_launch_counter,
                      moe_selftest_timeout, workspace_size)

__all__ = ["FLAG_DEVICE_NOISE", "FLAG_FFN_ROW_TILES", "FLAG_FFN_SIZED_TILES", "FLAG_SWITCH_GATE", "MoeConfig", "MoeError", "MoeHierConfig", "alloc_hier_workspace", "alloc_workspace",
           "alloc_backward_workspace", "alloc_batchwise_workspace", "backward_workspace_size",
           "batchwise_workspace_size", "expert_rows_dtype",
           "hier_workspace_size", "lib", "make_config", "make_hier_config", "moe_backward",
           "moe_backward_timed", "moe_batchwise_forward", "moe_batchwise_threshold_forward",
           "moe_balance_losses", "moe_combine", "moe_dispatch", "moe_dispatch_noalloc",
           "moe_draw_noise", "ep_plan_size", "moe_ep_plan", "moe_ep_regroup", "moe_losses_from_sums",
           "moe_expert_ffn", "moe_forward", "moe_forward_timed", "moe_gate",
           "moe_get_device_error", "moe_hier_forward", "moe_launch_counter",
           "moe_selftest_timeout", "workspace_size"]
