"""GB300-native neuron-aware sparse FFN decode path.

The compute lives in ``libpi.so`` (hand-written CUDA for sm_103a behind the C
ABI of ``include/pi.h``); :mod:`.binding` marshals torch CUDA tensors into it,
and :mod:`.runtime` holds layers and workspaces for whole decode steps.
"""
from .binding import (PiError, desc_of, layer_desc, lib, library_path, pi_compact,  # noqa: F401
                      pi_debug_set_wait_timeout, pi_debug_wait_timeout, pi_ffn_layer, pi_ffn_stack, pi_last_device_status,
                      pi_launches_per_layer, pi_predict, pi_rmsnorm_half, pi_sparse_fc1, pi_sparse_fc2,
                      pi_sparse_fc2_noalloc, pi_stack_plan, pi_stack_plan_for, cold_tier, pi_sparse_fc1_tiered,
                      pi_sparse_fc2_tiered, pi_ffn_layer_tiered,
                      pi_status_string, pi_workspace_bytes, pi_workspace_layout, ranks_array,
                      weights_array, weights_struct, attn_desc, attn_desc_of, attn_weights_struct,
                      pi_attn_heads, pi_attn_workspace_bytes)
