"""Nyström self-attention forward pass for GB300 (sm_103a).

A thin binding of the C-ABI library libnystrom.so (include/nystrom.h); all
compute runs in the library's CUDA kernels.
"""
from ._binding import (  # noqa: F401
    LIB_PATH, NYS_BF16, NYS_CONV_PER_CHANNEL, NYS_CSTAGE_ASSIGN, NYS_CSTAGE_CENTROIDS,
    NYS_CSTAGE_CENTROIDS_PREV, NYS_CSTAGE_G, NYS_CONV_PER_HEAD, NYS_ERR_ALIGN, NYS_ERR_ARG, NYS_ERR_CUDA, NYS_ERR_NOMEM, NYS_ERR_SHAPE,
    NYS_ERR_TIMEOUT, NYS_ERR_UNSUPPORTED, NYS_FP32, NYS_OK, NYS_STAGE_A_S, NYS_STAGE_G,
    NYS_STAGE_K_TILDE, NYS_STAGE_Q_TILDE, NYS_STAGE_W, NYS_STAGE_Z, NystromError, load_library,
    nystrom_attention, nystrom_attn_fwd, nystrom_clustered_attn_fwd, nystrom_clustered_stage_offset,
    nystrom_clustered_workspace_bytes, nystrom_debug_stall_pinv, nystrom_attn_fwd_ex, nystrom_attn_fwd_host, nystrom_attn_fwd_noalloc, nystrom_attn_fwd_ws,
    nystrom_attn_stage_offset, nystrom_attn_workspace_bytes, nystrom_get_status,
    nystrom_last_error_string, nystrom_launch_count, nystrom_mha_fwd, nystrom_mha_workspace_bytes, nystrom_plan_describe, nystrom_profile_enable,
    nystrom_profile_read, nystrom_strerror,
)
