"""GPU test of engram_forward_noalloc, the entry point for callers that may not allocate device
memory (an engine whose pool owns all device memory and lends a plugin only its own tensors, or
a real-time loop that cannot take cudaMalloc's implicit synchronisation).  It keeps its scratch
in a static device array instead of a caller workspace.

Checked through the C ABI against engram_forward (caller workspace) on the decode workload (one
and two layers, each layer's rows in its own slot of the array), on two calls in a row, so leftovers in the shared static array cannot leak into a result.  This
file is collected last, so a run that stops at the first failure has run every other test.
"""
import ctypes

import pytest
import torch

from engram_synth.case import to_device
from tests import _helpers as H

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _plan(w, case, setup, streams, out_ids, err, workspace=None):
    import engram_gram_hash_02_gb300 as E
    primes, offsets, rows, mult = setup
    b = case.batch
    dims = H.dims_for(w, H.pad_id_of(w, b["token_map"]))
    tables = E.HashTables(to_device(b["token_map"], DEV), to_device(mult, DEV), to_device(primes, DEV),
                          to_device(offsets, DEV))
    layers = [E.LayerWeights(t["fmt"], t["table"], t["scales"], t["num_rows"], case.wkv[l], case.q_weight[l],
                             case.k_weight[l]) for l, t in enumerate(case.tables)]
    return E.ForwardPlan(dims, tables, layers, to_device(b["input_ids"], DEV), streams,
                         cu_seqlens=to_device(b["cu_seqlens"], DEV), sequence_ids=to_device(b["sequence_ids"], DEV),
                         token_mask=to_device(b["token_mask"], DEV), lookback_ids=to_device(b["lookback_ids"], DEV),
                         workspace=workspace, out_ids=out_ids, err=err)


@pytest.mark.parametrize("name", ["decode_fp8_t256", "decode_fp8_t256_2layer"])
def test_noalloc_matches_workspace_entry_point_twice(name):
    w, case, setup = H.build(name)
    shape = (w.tokens, w.layers, w.cols)
    ref_streams = [s.clone() for s in case.streams]
    ref_ids = torch.empty(shape, dtype=torch.int32, device=DEV)
    ref_err = torch.zeros(1, dtype=torch.int32, device=DEV)
    _plan(w, case, setup, ref_streams, ref_ids, ref_err).run()
    torch.cuda.synchronize()
    assert int(ref_err.item()) == 0

    unused = torch.empty(256, dtype=torch.uint8, device=DEV)   # the no-alloc call takes no workspace
    for call in range(2):
        streams = [s.clone() for s in case.streams]
        ids = torch.full(shape, -1, dtype=torch.int32, device=DEV)
        err = torch.zeros(1, dtype=torch.int32, device=DEV)
        _plan(w, case, setup, streams, ids, err, workspace=unused).run_noalloc()
        torch.cuda.synchronize()
        assert int(err.item()) == 0, f"call {call}: device error flag {int(err.item())}"
        assert torch.equal(ids, ref_ids), f"call {call}: hash ids differ"
        for l in range(w.layers):
            got = streams[l].double()
            ref = ref_streams[l].double()
            max_abs = float((got - ref).abs().max())
            rel = float((got - ref).norm() / ref.norm())
            assert max_abs <= H.STREAM_MAX_ABS and rel <= H.STREAM_REL_L2, (call, max_abs, rel)
    del case
    torch.cuda.empty_cache()


def test_noalloc_rejects_calls_beyond_its_scratch():
    import engram_gram_hash_02_gb300 as E
    from engram_gram_hash_02_gb300 import binding as B
    dims = E.make_dims(1, 4, 8, 256, 4096, 4, 163840, 131072, 0)
    T = 32768                                   # the prefill batch needs ~3.2 GB of scratch
    assert E.forward_workspace_bytes(dims, T) > B.NOALLOC_SCRATCH_BYTES
    tokens = B._Tokens(None, T, None, 1, None, None, None)
    rc = B.lib().engram_forward_noalloc(ctypes.byref(dims), None, None, ctypes.byref(tokens), None, None, None,
                                        torch.cuda.current_stream().cuda_stream)
    assert rc == -1
    msg = B.lib().engram_last_error().decode()
    assert "scratch" in msg and str(E.forward_workspace_bytes(dims, T)) in msg
