"""GPU parity of the FP8 variant's operand gather (engram_set_operand_gather(1)): the projection
reads its token rows straight from the FP8 table into its operand tiles (cp.async into the
swizzled layout by four gather warps) instead of from a gathered copy in HBM.

The kv and the streams must be bit-identical to the path through the gathered copy (the tensor
cores see the same codes and scales), and the streams within tolerance of the oracle. Cases: the
decode step (256-row tiles), short token tiles (1 and 64 tokens), a tail row block (129 tokens),
a forced 48-column tile width, two layers, a layer mix with a Q2_K layer, ids outside the table
(zero rows and the row-id error bit, as the gathered copy gives), and a larger batch.
"""
from dataclasses import replace

import numpy as np
import pytest
import torch

from engram_synth import get_workload
from tests import _helpers as H

pytestmark = pytest.mark.gpu


def E():
    import engram_gram_hash_02_gb300 as mod
    return mod


def _forward(w, case, setup, gather, mx, tile=0):
    E().set_operand_gather(gather)
    E().set_gemm_mx_tile(tile)
    try:
        return H.gpu_forward(w, case, setup, mx=mx)
    finally:
        E().set_operand_gather(False)
        E().set_gemm_mx_tile(0)


@pytest.mark.parametrize("name,seq_lens,mx,tile", [
    ("decode_fp8_t256", None, True, 0),
    ("decode_fp8_t256", (1,) * 64, True, 0),           # one short token tile of 64 rows
    ("decode_fp8_t256", (1,), True, 0),                # of 16 rows, one of them real
    ("decode_fp8_t256", (1,) * 129, True, 0),          # a second row block with one row
    ("decode_fp8_t256", None, True, 48),
    ("decode_fp8_t256_2layer", None, True, 0),
    ("decode_fp8_t256_2layer", None, (True, False), 0),  # an FP8-variant layer, then a bf16-wkv layer
    ("prefill_fp8_t32768", (1500, 548), True, 0),      # documents, masked tokens, several row blocks
])
def test_operand_gather_matches_the_gathered_copy(name, seq_lens, mx, tile):
    w, case, setup = H.build(name, seq_lens=seq_lens)
    ref = _forward(w, case, setup, False, mx, tile)
    got = _forward(w, case, setup, True, mx, tile)
    assert got["err"] == ref["err"] == 0
    assert torch.equal(got["ids"], ref["ids"])
    assert torch.equal(got["kv_last"], ref["kv_last"])
    for l in range(w.layers):
        assert torch.equal(got["streams"][l], ref["streams"][l]), f"{name} layer {l}"
        if got["A_scales"][l] is not None:
            assert np.array_equal(got["A_scales"][l], ref["A_scales"][l])
    if w.tokens <= 512:
        oref = H.oracle_forward(w, case, mx=mx)
        for l, lref in enumerate(oref["layers"]):
            H.check_streams(got["streams"][l].cpu().numpy(), lref["streams"], lref["streams_in"], f"{name} {l}")
    del case
    torch.cuda.empty_cache()


def test_operand_gather_layer_mix_with_q2k():
    w = replace(get_workload("decode_fp8_t256_2layer"), name="mix_q2k", extra={"layer_formats": ("q2k", "fp8")})
    w, case, setup = H.build(w)
    ref = _forward(w, case, setup, False, (False, True))
    got = _forward(w, case, setup, True, (False, True))
    assert got["err"] == 0
    for l in range(w.layers):
        assert torch.equal(got["streams"][l], ref["streams"][l])


def test_operand_gather_ids_outside_the_table():
    """A table shorter than the layout: ids past its end read zero rows and set the row-id bit."""
    w, case, setup = H.build("decode_fp8_t256")
    short = dict(case.tables[0])
    short["num_rows"] = int(short["num_rows"]) // 2        # about half the ids now fall outside
    case.tables[0] = short
    ref = _forward(w, case, setup, False, True)
    got = _forward(w, case, setup, True, True)
    assert ref["err"] & E().ERR_ROW_ID and got["err"] & E().ERR_ROW_ID
    assert torch.equal(got["kv_last"], ref["kv_last"])
    assert torch.equal(got["streams"][0], ref["streams"][0])
    oref = H.oracle_forward(w, case, mx=True)
    H.check_streams(got["streams"][0].cpu().numpy(), oref["layers"][0]["streams"],
                    oref["layers"][0]["streams_in"], "ids outside the table")
