"""Seeded synthetic inputs for the Engram hot path.

This module only draws random inputs: token ids, token maps, document cuts,
masks, lookback ids, tables, projection weights, norm weights and the fp32
highway.  It computes none of the method's own arithmetic (no hashing, no
dequantisation, no projection, no gate).  Both the CUDA path's tests and the
CPU oracle take their inputs from here, so this is the only module they share.

Small integer inputs are drawn with numpy's PCG64 (identical on every
platform).  Large float tables are drawn with torch on the device that will
hold them, seeded per tensor, so a 6-50 GB table never crosses the host.
"""
from .workloads import WORKLOADS, Workload, get_workload  # noqa: F401
from .gen import (  # noqa: F401
    batch_inputs,
    bf16_table,
    encode_fp8_e8m0,
    fp8_table,
    gate_weights,
    q2k_table,
    streams,
    token_map,
    wkv_weight,
    zipf_ids,
)
