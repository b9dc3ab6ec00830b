"""GB300-native Engram hot path: n-gram hash -> table gather/dequant -> wkv projection -> gate.

The compute lives in ``libengram.so`` (hand-written sm_103a CUDA behind a C ABI declared in
``include/engram.h``); this package is its thin Python binding.
"""
from .binding import (  # noqa: F401
    ERR_PIPE_TIMEOUT,
    ERR_RAW_ID,
    ERR_ROW_ID,
    TABLE_FORMATS,
    ProjectPlan,
    EngramDims,
    EngramError,
    ForwardPlan,
    HashTables,
    LayerWeights,
    engram_forward,
    engram_gate,
    engram_gather_dequant,
    engram_gather_fp8_codes,
    engram_hash,
    engram_layout,
    engram_project,
    engram_project_mxfp8,
    forward_workspace_bytes,
    hash_multipliers,
    lib,
    make_dims,
    mx_scale_shape,
    project_plan,
    project_workspace_bytes,
    quantize_mxfp8,
    set_gate_form,
    set_gate_fusion,
    set_gemm_mx_tile,
    set_gemm_schedule,
    set_gemm_tile,
    sync_status,
)
