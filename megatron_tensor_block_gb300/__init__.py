"""Megatron column/row tensor-parallel block with N logical shards on one
GB300 (sm_103a): a C-ABI CUDA library (``include/tp_block.h``) and its thin
Python binding. The binding's functions carry the C names."""
from .binding import (  # noqa: F401
    TP_BF16, TP_F32, TP_MAX_SHARDS, TP_MODE_DECODE, TP_MODE_MOE_FFN, TP_MODE_PREFILL, TP_OK,
    TP_PARAM_COLWISE, TP_PARAM_FUSED_GATE_UP, TP_PARAM_FUSED_QKV, TP_PARAM_PACKED_COLWISE,
    TP_PARAM_REPLICATED, TP_PARAM_ROWWISE, TP_PARAM_VOCAB_PARALLEL, Plan, TpError, load, tp_block_forward, tp_block_forward_noalloc,
    tp_gather_param, tp_noalloc_status, tp_debug_withhold_arrival, tp_gemm_bf16, tp_gemm_bf16_kn, tp_get_device_status, tp_last_error, tp_plan, tp_plan_describe, tp_plan_get_info, tp_profile_phase_stamps, tp_profile_phases, tp_profile_stages,
    tp_reduce_partials, tp_shard_kv, tp_shard_param, tp_shard_weights, tp_version, tp_workspace_init, tp_lm_head_forward,
    Stack, tp_stack_create, tp_stack_decode, tp_stack_ctas, tp_stack_set_stamps)
from . import binding  # noqa: F401
