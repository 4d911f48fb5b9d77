"""tp_reduce_moe_gb300: the fused decode-layer boundary op for one GB300 GPU.

MoE finalize (weighted gather of permuted expert rows) + shared-expert add +
the arithmetic of the post-experts tensor-parallel all-reduce over R rank
partials in this GPU's memory + residual add + RMSNorm, in one sm_103a launch,
behind the C ABI of ``libarfuse`` (``include/arfuse.h``).  This package is the
Python binding of that library (argument marshalling only) and its build step.
"""
from .binding import (  # noqa: F401
    AR_DEVERR_PERM_RANGE, AR_DEVERR_TIMEOUT, AR_ERR_ALIGNMENT, AR_ERR_CAPACITY, AR_ERR_CUDA,
    AR_ERR_DEVICE_CHECK, AR_ERR_INVALID_ARG, AR_ERR_UNSUPPORTED, AR_MAX_HIDDEN, AR_MAX_RANKS,
    AR_MAX_TOP_K, AR_OK, AR_REGIME_AUTO, AR_REGIME_CLUSTER, AR_REGIME_ONESHOT, AR_REGIME_SPLIT, AR_REGIME_STREAM,
    AR_VALIDATED,
    AR_WS_DRY_RUN, AR_WS_NORM_BF16_H, AR_WS_PDL, LIB_PATH, ArfuseError, Workspace, ar_finalize_rmsnorm, ar_rmsnorm,
    ar_status_string, ar_workspace_create, ar_workspace_destroy, ar_workspace_device_error,
    ar_workspace_last_regime, ar_workspace_last_grid, ar_workspace_last_plan, PlanInfo,
    ar_workspace_set_cluster_size, ar_workspace_set_regime,
    ar_workspace_set_producer_warps, ar_workspace_set_stage_bytes, load_library,
    AR_MAX_REGIME_RULES, RegimeRule, ar_workspace_get_regime_table, ar_workspace_set_regime_table,
    AR_MAX_HC_STREAMS, ar_mhc_post, AR_MAX_SPLIT_PARTS, ar_workspace_set_split_rows,
    ar_workspace_set_split_column_groups, ar_workspace_inject_wait_timeout)
