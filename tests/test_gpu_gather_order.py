"""Table-order gathers (engram_set_gather_order(1)): each layer's rows grouped by table region
before the gather, every row written at its own place. The results must be bit-identical to the
token-order path: ids, gathered rows (or FP8 codes and scale words), kv and streams."""
import numpy as np
import pytest
import torch

from tests import _helpers as H

pytestmark = pytest.mark.gpu


def E():
    import engram_gram_hash_02_gb300 as m
    return m


def _forward(w, case, setup, order, mx=False, side=False):
    E().set_gather_order(order)
    try:
        return H.gpu_forward(w, case, setup, mx=mx, side=side)
    finally:
        E().set_gather_order(0)


def _same(a, b, w, what):
    assert a["err"] == b["err"] == 0, what
    assert torch.equal(a["ids"], b["ids"]), what
    assert torch.equal(a["kv_last"], b["kv_last"]), what
    for l in range(w.layers):
        assert torch.equal(a["streams"][l], b["streams"][l]), f"{what} layer {l}"
        if a["A"][l] is not None:
            assert torch.equal(a["A"][l], b["A"][l]), f"{what} rows {l}"
        if a["A_codes"][l] is not None:
            assert torch.equal(a["A_codes"][l], b["A_codes"][l]), f"{what} codes {l}"
            assert np.array_equal(a["A_scales"][l], b["A_scales"][l]), f"{what} scale words {l}"


@pytest.mark.parametrize("name,seq_lens,mx,side", [
    ("decode_fp8_t256", None, False, False),       # FP8 rows (token order: fetched by the hash launch)
    ("decode_fp8_t256", None, True, False),        # FP8 codes and scale words (the FP8 variant)
    ("decode_fp8_t256", (1,) * 77, False, False),  # a ragged batch
    ("tiny_bf16", None, False, False),             # bf16 rows
    ("q2k_t8192", (300, 212), False, False),       # two Q2_K layers
    ("q2k_t8192", (300, 212), False, True),        # the second layer's order and gather on the side stream
    ("prefill_fp8_t32768", (700, 324), False, False),   # documents and masked tokens
])
def test_table_order_matches_token_order(name, seq_lens, mx, side):
    w, case, setup = H.build(name, seq_lens=seq_lens)
    ref = _forward(w, case, setup, 0, mx=mx, side=side)
    got = _forward(w, case, setup, 1, mx=mx, side=side)
    _same(got, ref, w, f"{name} {seq_lens} mx={mx} side={side}")
    del case
    torch.cuda.empty_cache()


def test_table_order_large_t16384():
    """The 53 GB table with 16384 tokens of uniform ids: 393k rows over 12k regions."""
    w, case, setup = H.build("large_fp8_t16384")
    ref = _forward(w, case, setup, 0)
    got = _forward(w, case, setup, 1)
    _same(got, ref, w, "large_fp8_t16384")
    del case, ref, got
    torch.cuda.empty_cache()
