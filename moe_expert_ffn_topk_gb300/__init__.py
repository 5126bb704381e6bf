"""GB300-native fused MoE expert feed-forward with top-k combine.

The computation runs in the CUDA library ``_lib/libmoe_gb300.so`` (sources in ``csrc/``,
C ABI in ``include/moe_ffn.h``); this package is its thin Python binding. Importing it
without the built library raises ImportError: there is no fallback path.
"""
import torch

from ._binding import (MOE_ERR_BAD_ROUTE, MOE_ERR_BAD_SCALE, MOE_ERR_BOUNDS, MOE_ERR_CUDA,  # noqa: F401
                       MOE_ERR_INVALID_ARG, MOE_ERR_TIMEOUT, MOE_ERR_UNSUPPORTED, MOE_ERR_WORKSPACE, MOE_OK)
from ._binding import (ABI_FUNCTIONS, MODES, MOE_FLAG_FUSED, MOE_FLAG_NONE, MOE_FLAG_PAIR_L1,  # noqa: F401
                       MOE_FLAG_PREPARED_WEIGHTS,
                       MOE_FLAG_QUANTIZE_X, MOE_FLAG_SIMT, MOE_FLAG_SINGLE_CTA, MOE_FLAG_TOKEN_MAJOR,
                       MOE_FLAG_WEIGHT_MAJOR, MoeDims, MoeError, MoeOptions, dims, moe_check_device_error,
                       moe_combine, moe_debug_bounded_wait, moe_dispatch, moe_dispatch_quantize, moe_expert_l1,
                       moe_expert_l1_ex, moe_expert_l2, moe_expert_ffn, moe_forward, moe_forward_ex, moe_plan, moe_plan_noalloc,
                       moe_prepare_weights, moe_prepared_weights_bytes, moe_status_string,
                       moe_tensor_peak_probe, moe_workspace_bytes, moe_workspace_layout)
from ._binding import PEAK_KINDS  # noqa: F401


def alloc_workspace(d: MoeDims, mode, device="cuda") -> torch.Tensor:
    """A device byte buffer of moe_workspace_bytes(d, mode) bytes (torch allocations are
    at least 256-byte aligned)."""
    n = moe_workspace_bytes(d, mode)
    if n == 0:
        raise ValueError("dimensions outside the library's limits")
    return torch.empty(n, dtype=torch.uint8, device=device)
