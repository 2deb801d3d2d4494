"""GB300 (sm_103a) implementation of the Mixture-of-Top-k Attention (MiTA)
forward pass: a C-ABI library of hand-written CUDA kernels (csrc/, declared in
include/mita.h) with a thin Python binding of the same entry points."""
from ._lib import (MITA_ERR_ALLOC, MITA_ERR_CUDA, MITA_ERR_INVALID_ARG, MITA_ERR_TIMEOUT, MITA_ERR_UNSUPPORTED,
                   MITA_OK, MitaError, declared_functions, load, mita_forward, mita_forward_aux, mita_forward_host, mita_forward_noalloc,
                   mita_forward_routed, mita_forward_split, mita_forward_multi, mita_backward, mita_last_error, mita_profile_enable, mita_profile_read, mita_release_workspace,
                   mita_plan_info, mita_selftest_wait, mita_stage_name, mita_sync_status, mita_workspace_bytes)
from .build_lib import build

__all__ = [
    "MITA_OK", "MITA_ERR_INVALID_ARG", "MITA_ERR_UNSUPPORTED", "MITA_ERR_ALLOC", "MITA_ERR_CUDA",
    "MITA_ERR_TIMEOUT", "MitaError", "build", "load", "declared_functions", "mita_forward", "mita_forward_aux",
    "mita_forward_host", "mita_forward_noalloc", "mita_forward_routed", "mita_forward_split", "mita_forward_multi", "mita_backward", "mita_workspace_bytes", "mita_sync_status", "mita_last_error", "mita_release_workspace",
    "mita_profile_enable", "mita_profile_read", "mita_stage_name", "mita_selftest_wait", "mita_plan_info",
]
