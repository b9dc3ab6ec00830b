"""GPU parity of the gate joined to the projection (engram_set_gate_fusion).

Mode 1: the projection never stores the key columns of kv; its epilogue reduces them to per-tile
partial sums (sum key^2 and sum h*q*key*k per stream the tile covers) and a finishing pass applies
the gate. Mode 2: eight more warps of the projection kernel apply the gate to each row block's
tokens once every tile of the block is stored, overlapped with the tensor-core work. The streams must match the fp64 oracle within the stream tolerance, match
the unfused path to fp32 summation order, and masked tokens must stay bit-unchanged. The cases
put tile boundaries inside streams (split tiles of 288 columns at the decode size, forced tile
widths of 48 and 144 columns, whose 16-column pieces sit off the 32-column grid), run tiles across
the key/value boundary, two layers, the FP8 operand variant, short token tiles and a masked
multi-document batch.
"""
from dataclasses import replace

import numpy as np
import pytest
import torch

from engram_synth import get_workload
from tests import _helpers as H
from tests.test_gpu_forward import _sample

pytestmark = pytest.mark.gpu


def E():
    import engram_gram_hash_02_gb300 as mod
    return mod


def _forward(w, case, setup, mode, mx=False, tile=0):
    E().set_gate_fusion(mode)
    (E().set_gemm_mx_tile if mx else E().set_gemm_tile)(tile)
    try:
        return H.gpu_forward(w, case, setup, mx=mx)
    finally:
        E().set_gate_fusion(0)
        E().set_gemm_tile(0)
        E().set_gemm_mx_tile(0)


def _check(w, case, got, ref_unfused, sample, mx, mode=1):
    assert got["err"] == 0
    toks = _sample(w, case, sample) if sample else None
    ref = H.oracle_forward(w, case, toks, mx=mx)
    sel_t = torch.from_numpy(ref["tokens"]).to(got["ids"].device)
    for l, lref in enumerate(ref["layers"]):
        h = got["streams"][l].index_select(0, sel_t).cpu().numpy()
        H.check_streams(h, lref["streams"], lref["streams_in"], f"{w.name} fused layer {l}")
        # against the unfused path: the same kv, the gate's sums in another order
        d = (got["streams"][l] - ref_unfused["streams"][l]).abs().max().item()
        assert d <= 1e-4, f"{w.name} layer {l}: fused vs unfused max|d| {d:.3g}"
    # the value columns are still stored (mode 2: the keys too)
    hcH = w.hc * w.hidden
    assert torch.equal(got["kv_last"][:, hcH:], ref_unfused["kv_last"][:, hcH:])
    if mode == 2:
        assert torch.equal(got["kv_last"], ref_unfused["kv_last"])
    mask = case.batch.get("token_mask")
    if mask is not None:
        keep = torch.from_numpy(mask == 0).to(got["ids"].device)
        for l in range(w.layers):
            assert torch.equal(got["streams"][l][keep], case.streams[l][keep]), "masked tokens changed"


@pytest.mark.parametrize("name,seq_lens,mx,tile,sample", [
    ("decode_fp8_t256", None, False, 0, 0),            # split tiles of 288: boundaries inside streams
    ("decode_fp8_t256", None, False, 48, 0),           # 48-wide tiles: pieces off the 32-column grid
    ("decode_fp8_t256", None, False, 144, 0),
    ("decode_fp8_t256", None, True, 0, 0),             # FP8 operand variant
    ("decode_fp8_t256", None, True, 48, 0),
    ("decode_fp8_t256_2layer", None, False, 0, 0),     # two layers
    ("decode_fp8_t256", (1,) * 112, False, 0, 0),      # a single short token tile
    ("decode_fp8_t256", (1,) * 129, False, 0, 0),      # a second row block of one token
    ("prefill_fp8_t32768", (700, 324), False, 0, 0),   # documents and masked tokens, 256-row tiles
    ("prefill_fp8_t32768", (1500, 548), True, 0, 256),  # FP8 variant, several 256-row blocks
    ("q2k_t8192", (300,), False, 0, 0),
    ("tiny_fp8", None, False, 0, 0),                   # H 256 with 256-wide tiles: one stream each
])
@pytest.mark.parametrize("mode", [1, 2])
def test_fused_gate_matches_oracle_and_unfused(name, seq_lens, mx, tile, sample, mode):
    w, case, setup = H.build(name, seq_lens=seq_lens)
    ref_unfused = _forward(w, case, setup, 0, mx, tile)
    got = _forward(w, case, setup, mode, mx, tile)
    _check(w, case, got, ref_unfused, sample, mx, mode)
    del case
    torch.cuda.empty_cache()


@pytest.mark.parametrize("mode", [1, 2])
def test_fused_gate_large_t16384_sampled(mode):
    w, case, setup = H.build("large_fp8_t16384")
    ref_unfused = _forward(w, case, setup, 0)
    got = _forward(w, case, setup, mode)
    _check(w, case, got, ref_unfused, 96, False, mode)
    del case, got, ref_unfused
    torch.cuda.empty_cache()


@pytest.mark.parametrize("mode", [1, 2])
def test_fused_gate_is_repeatable(mode):
    w, case, setup = H.build("prefill_fp8_t32768", seq_lens=(1024,))
    a = _forward(w, case, setup, mode)
    b = _forward(w, case, setup, mode)
    assert torch.equal(a["streams"][0], b["streams"][0])
    del case
    torch.cuda.empty_cache()


@pytest.mark.parametrize("tile", [256, 64])
def test_fused_gate_hidden_128(tile):
    """hidden 128: 64-wide tiles are fused (two per stream); 256-wide tiles would cover three
    streams, so that layer runs unfused (bit-identical to the fusion off)."""
    w = replace(get_workload("tiny_fp8"), name="tiny_fp8_h128", hidden=128)
    w, case, setup = H.build(w)
    ref_unfused = _forward(w, case, setup, 0, tile=tile)
    got = _forward(w, case, setup, 1, tile=tile)
    if tile == 256:
        assert got["err"] == 0 and torch.equal(got["streams"][0], ref_unfused["streams"][0])
    else:
        _check(w, case, got, ref_unfused, 0, False)


def test_overlapped_gate_two_layer_q2k():
    w, case, setup = H.build("q2k_t8192", seq_lens=(700, 0, 324))
    ref = _forward(w, case, setup, 0)
    got = _forward(w, case, setup, 2)
    _check(w, case, got, ref, 0, False, 2)
