"""GPU parity of the whole path (engram_forward through the C ABI) against the oracle.

Every workload runs at its full size in the launch configuration the bench uses; the oracle
checks all tokens where it finishes in seconds and a seeded sample (always including masked,
document-start and sequence-start tokens) elsewhere.  Hash ids are compared for every token.
"""
from dataclasses import replace

import numpy as np
import pytest
import torch

from engram_synth import get_workload
from oracle import engram_oracle as O
from tests import _helpers as H

pytestmark = pytest.mark.gpu


def _sample(w, case, n):
    T = w.tokens
    if T <= n:
        return None
    rng = np.random.default_rng(1234)
    pick = set(rng.choice(T, size=n, replace=False).tolist())
    cu = case.batch["cu_seqlens"]
    pick.update(int(x) for x in cu[:-1] if x < T)                      # sequence starts
    sid = case.batch.get("sequence_ids")
    if sid is not None:
        pick.update(np.nonzero(np.diff(sid) != 0)[0][:64].tolist())
    mask = case.batch.get("token_mask")
    if mask is not None:
        pick.update(np.nonzero(mask == 0)[0][:64].tolist())
    pick.update([T - 1])
    return np.array(sorted(pick), dtype=np.int64)


@pytest.mark.parametrize("name,sample", [
    ("tiny_bf16", 0), ("decode_fp8_t256", 0), ("decode_fp8_t256_deadlb", 0),
    ("prefill_fp8_t32768", 384), ("q2k_t8192", 384), ("large_fp8_t1", 0), ("large_fp8_t64", 0),
    ("large_fp8_t1024", 256),
])
def test_forward_matches_oracle(name, sample):
    w, case, setup = H.build(name)
    got = H.gpu_forward(w, case, setup)
    toks = _sample(w, case, sample) if sample else None
    ref = H.oracle_forward(w, case, toks)
    assert got["err"] == 0
    assert np.array_equal(got["ids"].cpu().numpy(), ref["ids"].astype(np.int32))
    sel = ref["tokens"]
    sel_t = torch.from_numpy(sel).to(got["ids"].device)
    for l, lref in enumerate(ref["layers"]):
        h = got["streams"][l].index_select(0, sel_t).cpu().numpy()
        H.check_streams(h, lref["streams"], lref["streams_in"], f"{name} layer {l}")
    # every layer's rows, and the last layer's kv, are still in the workspace
    for l, lref in enumerate(ref["layers"]):
        assert np.array_equal(H.bits16(got["A"][l].index_select(0, sel_t)), lref["a_bits"]), f"{name} rows {l}"
    last = ref["layers"][-1]
    H.check_kv(got["kv_last"].index_select(0, sel_t).cpu().numpy(), last["kv"], f"{name} kv")
    mask = case.batch.get("token_mask")
    if mask is not None:
        keep = mask[sel] == 0
        for l in range(w.layers):
            h = got["streams"][l].index_select(0, sel_t).cpu().numpy()
            h0 = case.streams[l].index_select(0, sel_t).cpu().numpy()
            assert np.array_equal(h[keep], h0[keep])
    del case, got
    torch.cuda.empty_cache()


def test_forward_repeatable():
    # two runs on the same inputs give bit-identical streams (no races, no stale workspace)
    w, case, setup = H.build("decode_fp8_t256")
    a = H.gpu_forward(w, case, setup)
    b = H.gpu_forward(w, case, setup)
    for l in range(w.layers):
        assert torch.equal(a["streams"][l], b["streams"][l])
    assert torch.equal(a["ids"], b["ids"])
    del case
    torch.cuda.empty_cache()


def test_forward_large_t16384_sampled():
    w, case, setup = H.build("large_fp8_t16384")
    got = H.gpu_forward(w, case, setup)
    toks = _sample(w, case, 128)
    ref = H.oracle_forward(w, case, toks)
    assert np.array_equal(got["ids"].cpu().numpy(), ref["ids"].astype(np.int32))
    sel_t = torch.from_numpy(ref["tokens"]).to(got["ids"].device)
    h = got["streams"][0].index_select(0, sel_t).cpu().numpy()
    H.check_streams(h, ref["layers"][0]["streams"], ref["layers"][0]["streams_in"], "large t16384")
    assert got["err"] == 0
    del case, got
    torch.cuda.empty_cache()
    assert O is not None


# engram_forward gathers every layer's rows before the first projection: the hash kernel fetches
# the leading run of FP8 layers (at most 8), then one gather launch per run of layers with the
# same table format and operand kind (at most 8). These mixes reach each branch of that plan.
@pytest.mark.parametrize("base,layer_ids,fmts,mx,sample", [
    ("q2k_t8192", None, ("q2k", "fp8"), False, 384),           # no leading FP8 layer: two gather launches
    ("decode_fp8_t256_2layer", None, ("fp8", "q2k"), False, 0),  # FP8 rows from the hash kernel, Q2_K after
    ("decode_fp8_t256_2layer", None, None, (False, True), 0),    # one fused launch: bf16 rows, then codes
    ("tiny_fp8", tuple(range(1, 11)), None, tuple(l % 2 == 1 for l in range(10)), 0),   # 8 fused + 2
    ("tiny_fp8", tuple(range(1, 11)), ("q2k",) * 10, False, 0),  # gather launches of 8 and 2 layers
])
def test_forward_layer_mixes(base, layer_ids, fmts, mx, sample):
    w = get_workload(base)
    kw = {"name": f"{base}_mix"}
    if layer_ids is not None:
        kw["layer_ids"] = layer_ids
    if fmts is not None:
        kw["extra"] = {"layer_formats": fmts}
    w = replace(w, **kw)
    w, case, setup = H.build(w)
    got = H.gpu_forward(w, case, setup, mx=mx)
    toks = _sample(w, case, sample) if sample else None
    ref = H.oracle_forward(w, case, toks, mx=mx)
    assert got["err"] == 0
    assert np.array_equal(got["ids"].cpu().numpy(), ref["ids"].astype(np.int32))
    sel = ref["tokens"]
    sel_t = torch.from_numpy(sel).to(got["ids"].device)
    for l, lref in enumerate(ref["layers"]):
        what = f"{w.name} layer {l}"
        if got["A"][l] is not None:
            assert np.array_equal(H.bits16(got["A"][l].index_select(0, sel_t)), lref["a_bits"]), what
        else:
            assert np.array_equal(got["A_codes"][l].index_select(0, sel_t).cpu().numpy(), lref["a_bits"][0]), what
            assert np.array_equal(got["A_scales"][l][sel], lref["a_bits"][1]), what
        h = got["streams"][l].index_select(0, sel_t).cpu().numpy()
        H.check_streams(h, lref["streams"], lref["streams_in"], what)
    H.check_kv(got["kv_last"].index_select(0, sel_t).cpu().numpy(), ref["layers"][-1]["kv"], f"{w.name} kv")


@pytest.mark.parametrize("name,seq_lens", [
    ("tiny_bf16", (0, 5, 0, 3, 1)),          # empty sequences between ragged ones
    ("decode_fp8_t256", (1,) * 129),         # 129 tokens: split tiles whose second row block has one row
    ("decode_fp8_t256", (1,) * 112),         # the largest short token tile
    ("q2k_t8192", (7, 0, 120)),              # two Q2_K layers on a ragged batch of 127 tokens
])
def test_forward_ragged_and_boundary_sizes(name, seq_lens):
    w, case, setup = H.build(name, seq_lens=seq_lens)
    got = H.gpu_forward(w, case, setup)
    ref = H.oracle_forward(w, case)
    assert got["err"] == 0
    assert np.array_equal(got["ids"].cpu().numpy(), ref["ids"].astype(np.int32))
    for l, lref in enumerate(ref["layers"]):
        what = f"{name} T={w.tokens} layer {l}"
        assert np.array_equal(H.bits16(got["A"][l]), lref["a_bits"]), what
        H.check_streams(got["streams"][l].cpu().numpy(), lref["streams"], lref["streams_in"], what)
    H.check_kv(got["kv_last"].cpu().numpy(), ref["layers"][-1]["kv"], f"{name} T={w.tokens} kv")


def test_forward_zero_tokens_is_a_no_op():
    w, case, setup = H.build("tiny_bf16", seq_lens=(0,))
    got = H.gpu_forward(w, case, setup)
    assert got["err"] == 0 and got["ids"].numel() == 0 and got["streams"][0].numel() == 0


# engram_forward2: the gathers of the layers after the first run on a caller side stream, joined
# back by events before each projection. The streams must be bit-identical to engram_forward's (the
# same kernels on the same data), over the plans of the layer mixes above.
@pytest.mark.parametrize("base,layer_ids,fmts,mx", [
    ("q2k_t8192", None, None, False),                            # layer 0 gathered on the main stream
    ("q2k_t8192", None, ("q2k", "fp8"), False),
    ("decode_fp8_t256_2layer", None, ("fp8", "q2k"), False),      # FP8 rows from the hash, Q2_K on the side
    ("decode_fp8_t256_2layer", None, None, (False, True)),
    ("tiny_fp8", tuple(range(1, 11)), ("q2k",) * 10, False),     # runs of 8 and 1 on the side stream
    ("tiny_fp8", tuple(range(1, 11)), tuple(("q2k", "bf16")[l % 2] for l in range(10)), False),
    ("tiny_bf16", None, None, False),                            # one layer: nothing to move
])
def test_forward2_side_stream_matches_forward(base, layer_ids, fmts, mx):
    w = get_workload(base)
    kw = {"name": f"{base}_side"}
    if layer_ids is not None:
        kw["layer_ids"] = layer_ids
    if fmts is not None:
        kw["extra"] = {"layer_formats": fmts}
    w = replace(w, **kw)
    if fmts is not None and "bf16" in fmts:
        w = replace(w, head_dim=256)
    w, case, setup = H.build(w)
    ref = H.gpu_forward(w, case, setup, mx=mx)
    for _ in range(2):                                           # twice: the events are reused
        got = H.gpu_forward(w, case, setup, mx=mx, side=True)
        assert got["err"] == 0
        assert torch.equal(got["ids"], ref["ids"])
        for l in range(w.layers):
            assert torch.equal(got["streams"][l], ref["streams"][l]), f"{w.name} layer {l}"
    del case
    torch.cuda.empty_cache()


def test_forward2_q2k_matches_oracle():
    w, case, setup = H.build("q2k_t8192")
    got = H.gpu_forward(w, case, setup, side=True)
    toks = _sample(w, case, 256)
    ref = H.oracle_forward(w, case, toks)
    assert got["err"] == 0
    sel_t = torch.from_numpy(ref["tokens"]).to(got["ids"].device)
    for l, lref in enumerate(ref["layers"]):
        assert np.array_equal(H.bits16(got["A"][l].index_select(0, sel_t)), lref["a_bits"])
        h = got["streams"][l].index_select(0, sel_t).cpu().numpy()
        H.check_streams(h, lref["streams"], lref["streams_in"], f"q2k side stream layer {l}")
    del case
    torch.cuda.empty_cache()


def _forward_plan(w, case, setup):
    """An engram_forward plan over its own copies of the streams (and its own workspace)."""
    import engram_gram_hash_02_gb300 as E
    from engram_synth.case import to_device
    primes, offsets, rows, mult = setup
    b = case.batch
    dims = H.dims_for(w, H.pad_id_of(w, b["token_map"]))
    tables = E.HashTables(to_device(b["token_map"], "cuda"), to_device(mult, "cuda"), to_device(primes, "cuda"),
                          to_device(offsets, "cuda"))
    layers = [E.LayerWeights(t["fmt"], t["table"], t["scales"], t["num_rows"], case.wkv[l], case.q_weight[l],
                             case.k_weight[l]) for l, t in enumerate(case.tables)]
    streams = [s.clone() for s in case.streams]
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    plan = E.ForwardPlan(dims, tables, layers, to_device(b["input_ids"], "cuda"), streams,
                         cu_seqlens=to_device(b["cu_seqlens"], "cuda"),
                         sequence_ids=to_device(b["sequence_ids"], "cuda"),
                         token_mask=to_device(b["token_mask"], "cuda"),
                         lookback_ids=to_device(b["lookback_ids"], "cuda"), err=err)
    return plan, streams, err


def test_forward2_from_two_host_threads():
    """engram_forward2 called from two host threads at once, each with its own main and side
    streams and its own buffers (ctypes releases the interpreter lock during the call, so the calls
    overlap on the host): two Q2_K layers, so the second layer's rows are gathered on the side
    stream and joined back by the library's events. After n in-place updates each thread's streams
    equal those of n updates on one thread, bit for bit."""
    import threading
    w, case, setup = H.build("q2k_t8192", seq_lens=(300, 212))
    n = 8
    ref_plan, ref_streams, ref_err = _forward_plan(w, case, setup)
    side = torch.cuda.Stream()
    for _ in range(n):
        ref_plan.run(side_stream=side)
    torch.cuda.synchronize()
    plans = [_forward_plan(w, case, setup) for _ in range(2)]
    errors = []

    def worker(i):
        try:
            plan = plans[i][0]
            main, side_i = torch.cuda.Stream(), torch.cuda.Stream()
            for _ in range(n):
                plan.run(stream=main, side_stream=side_i)
            main.synchronize()
        except Exception as e:                                   # reported below
            errors.append(e)

    threads = [threading.Thread(target=worker, args=(i,)) for i in range(2)]
    for t in threads:
        t.start()
    for t in threads:
        t.join(timeout=300)
    torch.cuda.synchronize()
    assert not errors, errors
    assert int(ref_err.item()) == 0
    for i, (_, streams, err) in enumerate(plans):
        assert int(err.item()) == 0
        for l in range(w.layers):
            assert torch.equal(streams[l], ref_streams[l]), f"thread {i} layer {l}"
    del case
    torch.cuda.empty_cache()
