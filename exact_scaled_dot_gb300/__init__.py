"""Masked scaled dot-product attention, forward and backward, for GB300 (sm_103a).

The computation runs in the CUDA library built from ``csrc/`` (see
``include/attn.h`` for the C ABI); this package only marshals arguments.
"""
from ._binding import (  # noqa: F401
    ATTN_ERR_ALIGN, ATTN_ERR_CUDA, ATTN_ERR_DEVICE, ATTN_ERR_EMPTY_ROW, ATTN_ERR_NULL, ATTN_ERR_RANGE, ATTN_ERR_SCALE,
    ATTN_ERR_SHAPE, ATTN_ERR_TIMEOUT, ATTN_ERR_UNSUPPORTED, ATTN_ERR_WORKSPACE, ATTN_MAX_BATCH, ATTN_OK,
    AttnError, AttnRotary, AttnShape, AttnStrides, Rotary, attn_abi_version, attn_bwd, attn_bwd_finalize,
    attn_bwd_head_split, attn_bwd_main, attn_bwd_persistent, attn_bwd_noalloc,
    attn_bwd_noalloc_max_scratch_bytes, attn_bwd_preprocess, attn_bwd_workspace_bytes, attn_clear_status, attn_fwd,
    attn_fwd_decode, attn_fwd_decode_workspace_bytes, attn_fwd_workspace_bytes, attn_fwd_varlen_workspace_bytes,
    attn_get_status, attn_selftest_wait_timeout, attn_visible_pairs, load, make_shape, strerror,
    AttnVarlen, attn_bwd_varlen, attn_bwd_varlen_workspace_bytes, attn_fwd_varlen, attn_varlen_visible_pairs,
    attn_proj_bwd_input, attn_proj_bwd_weight, attn_proj_fwd, attn_rope, attn_rope_qk,
)
