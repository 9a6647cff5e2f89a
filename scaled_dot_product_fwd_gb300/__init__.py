"""GB300-native fused scaled-dot-product attention forward (sm_103a).

    from scaled_dot_product_fwd_gb300 import sdpa_forward
    o, lse = sdpa_forward(q, k, v, scale=None, causal=False, mask=None, sinks=None)
    o, lse = sdpa_forward_host(q_pinned, k_pinned, v_pinned)   # host buffers, transfers overlapped

The work runs in the CUDA kernels of ``libsdpa_gb300.so`` (C ABI in
``include/sdpa.h``); this package only marshals arguments.
"""
from ._binding import (EXPORTS, KERNELS, LIB_PATH, SDPA_BF16, SDPA_F16, SDPA_F32,
                       SDPA_FLAG_BOOL_MASK, SDPA_FLAG_SHARED_GPU, SDPA_FLAG_STRIDES, STATUS,
                       SdpaError, SdpaParams, dtype_code, load_library, make_params,
                       DEBUG_OPTIONS, sdpa_abi_version, sdpa_debug_set_option,
                       sdpa_debug_set_wait_limit_ns, sdpa_device_status,
                       sdpa_last_launch_count, sdpa_backward, sdpa_backward_workspace_size,
                       sdpa_forward, sdpa_forward_host, sdpa_forward_raw, sdpa_host_staging_size,
                       sdpa_select_kernel,
                       sdpa_status_string,
                       sdpa_workspace_size)

__all__ = ["sdpa_forward", "sdpa_forward_host", "sdpa_host_staging_size", "sdpa_forward_raw", "sdpa_workspace_size", "sdpa_select_kernel",
           "sdpa_status_string", "sdpa_device_status", "sdpa_debug_set_wait_limit_ns",
           "sdpa_debug_set_option", "DEBUG_OPTIONS",
           "sdpa_abi_version", "sdpa_last_launch_count", "sdpa_backward",
           "sdpa_backward_workspace_size", "make_params", "SdpaParams", "SdpaError",
           "load_library",
           "EXPORTS", "KERNELS", "STATUS", "LIB_PATH", "SDPA_F32", "SDPA_F16", "SDPA_BF16",
           "SDPA_FLAG_SHARED_GPU", "SDPA_FLAG_BOOL_MASK", "SDPA_FLAG_STRIDES",
           "dtype_code"]
