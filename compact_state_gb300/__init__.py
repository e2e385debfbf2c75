"""compact_state_gb300: one fused multi-tensor AdamW step on GB300 (sm_103a).

The optimizer step runs in ``libcompact_state.so`` (hand-written CUDA, C ABI
declared in ``include/compact_state.h``). This package is its thin binding:
``adamw_plan_create``, ``adamw_step``, ``adamw_plan_set_grads``,
``adamw_grad_prologue``, ``adamw_plan_info``, ``adamw_plan_error``,
``adamw_plan_set_debug``,
``adamw_plan_destroy``, ``adamw_state_bytes``, ``adamw_build_units``,
``adamw_build_queue``, ``adamw_shard_ranges``,
``adamw_step_noalloc``, ``adamw_noalloc_error``, ``adamw_noalloc_set_debug``
and ``adamw_strerror`` keep the C names and only
marshal arguments. ``torch_adapter`` builds descriptors from torch tensors.
"""
from ._binding import (  # noqa: F401
    CS_DTYPE_BF16, CS_DTYPE_F16, CS_DTYPE_F32, CS_INT8_BLOCK, CS_MAX_GROUPS,
    CS_MAX_TENSORS, CS_NOALLOC_MAX_TENSORS, CS_NOALLOC_MAX_UNITS, CS_NOALLOC_UNIT, CS_OK,
    CS_STATE_BF16, CS_STATE_DYN8, CS_STATE_F32, CS_STATE_INT8, CS_STATE_INT8_UV,
    CS_TENSOR_STATE_F32, DTYPE_CODES, EIGHT_BIT,
    EXPORTS, STATE_CODES, CompactStateError, Plan, adamw_build_queue, adamw_build_units,
    adamw_grad_prologue,
    adamw_group_t, adamw_noalloc_error, adamw_noalloc_set_debug,
    adamw_plan_create, adamw_plan_destroy, adamw_plan_error, adamw_plan_info,
    adamw_plan_info_t, adamw_plan_set_debug,
    adamw_plan_set_grads, adamw_shard_ranges, adamw_state_bytes, adamw_step,
    adamw_step_noalloc, adamw_strerror,
    adamw_tensor_t, groups_array, lib, pack_present, tensor_desc)
