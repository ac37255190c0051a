"""B300-native (sm_103a) Mixture-of-Grouped-Experts layer forward.

A thin ctypes binding over the C ABI in ``include/moge.h`` (``libmoge.so``).
Every function here only marshals arguments: torch tensors give device
pointers and the current CUDA stream; all work runs in the library's CUDA
kernels.  There is no fallback: if ``libmoge.so`` is missing or fails to load,
importing the binding's entry points raises.
"""
from .binding import (  # noqa: F401
    MOGE_F32, MOGE_BF16, MOGE_ROUTE_GROUPED, MOGE_ROUTE_GLOBAL_TOPK, MoGEError, Config, Aux,
    make_config, moge_workspace_bytes, alloc_workspace, moge_reset_device_status,
    moge_query_device_status, moge_route, moge_permute, moge_expert_ffn, moge_combine,
    moge_imbalance_score, moge_layer_forward, moge_abi_version, moge_status_string, library_path, load,
    moge_set_stage_events, moge_kernel_launch_count, MOGE_NUM_STAGES, STAGE_NAMES, moge_permute_noalloc,
    moge_imbalance_study, moge_workspace_bytes_shared, moge_layer_forward_shared, moge_selftest_bounded_wait,
    moge_layer_forward_residual,
)
