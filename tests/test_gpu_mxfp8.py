"""GPU parity of the FP8 (MXFP8) operand variant through the C ABI: the weight encoder and the
raw FP8 gather bit-exact against the oracle, the block-scaled tcgen05 projection within the fp32
summation bound of the oracle's fp64 product of the dequantised operands, and the whole forward
pass with MXFP8 wkv within the stream tolerance."""
import numpy as np
import pytest
import torch

from oracle import engram_oracle as O
from tests import _helpers as H

pytestmark = pytest.mark.gpu
DEV = "cuda"


def E():
    import engram_gram_hash_02_gb300 as m
    return m


def _random_bf16(N, K, seed):
    g = torch.Generator(device=DEV).manual_seed(seed)
    w = torch.randn(N, K, generator=g, device=DEV) * 0.02
    w *= torch.exp2(torch.randint(-8, 9, (N, 1), generator=g, device=DEV).float())   # per-row magnitudes
    w[:, 64:96] = 0                                                                   # an all-zero block per row
    w[0, 5] = 448.0                                                                   # boundary blocks
    w[1, min(40, K - 1)] = -450.0
    return w.to(torch.bfloat16)


@pytest.mark.parametrize("N,K", [(512, 6144), (37, 256), (3, 32)])
def test_quantize_bit_exact(N, K):
    w = _random_bf16(N, K, N + K)
    codes, sc = E().quantize_mxfp8(w)
    torch.cuda.synchronize()
    rc, rs = O.mxfp8_quantize(H.bits16(w))
    assert tuple(sc.shape) == E().mx_scale_shape(N, K)
    assert np.array_equal(H.mx_words_to_rows(sc, N, K // 32), rs)
    assert np.array_equal(codes.cpu().numpy(), rc)


def test_quantize_decode_wkv_sampled_rows():
    w, case, _ = H.build("decode_fp8_t256")
    codes, sc = E().quantize_mxfp8(case.wkv[0])
    torch.cuda.synchronize()
    rows = np.random.default_rng(0).choice(w.N, 1024, replace=False)
    rows_t = torch.from_numpy(rows).to(DEV)
    rc, rs = O.mxfp8_quantize(H.bits16(case.wkv[0].index_select(0, rows_t)))
    assert np.array_equal(codes.index_select(0, rows_t).cpu().numpy(), rc)
    assert np.array_equal(H.mx_words_to_rows(sc, w.N, w.K // 32)[rows], rs)


def test_gather_fp8_codes_bit_exact_with_out_of_range_ids():
    w, case, setup = H.build("decode_fp8_t256")
    tab = case.tables[0]
    g = torch.Generator(device=DEV).manual_seed(9)
    T, C = 300, w.cols
    ids = torch.randint(0, tab["num_rows"], (T, C), generator=g, device=DEV, dtype=torch.int32)
    ids[3, 5] = -1
    ids[7, 0] = tab["num_rows"]
    ids[299, C - 1] = 2 ** 31 - 1
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    codes, sc = E().engram_gather_fp8_codes(ids, tab["table"], tab["scales"], tab["num_rows"], w.head_dim, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == E().ERR_ROW_ID
    t_np, s_np, remap, nrows = H.compact_table(tab, ids.cpu().numpy().astype(np.int64))
    rc, rs, bad = O.gather_fp8_raw(t_np, s_np, remap, nrows)
    assert bad == 3
    assert np.array_equal(codes.cpu().numpy(), rc)
    assert np.array_equal(H.mx_words_to_rows(sc, T, C * w.head_dim // 32), rs)


def _random_mx(T, K, N, seed):
    g = torch.Generator(device=DEV).manual_seed(seed)
    a = torch.randint(0, 256, (T, K), generator=g, device=DEV, dtype=torch.uint8)
    b = torch.randint(0, 256, (N, K), generator=g, device=DEV, dtype=torch.uint8)
    a[(a & 0x7F) == 0x7F] = 0x38                                  # no NaN codes
    b[(b & 0x7F) == 0x7F] = 0x30
    sa = torch.randint(118, 132, (T, K // 32), generator=g, device=DEV, dtype=torch.uint8)
    sb = torch.randint(118, 132, (N, K // 32), generator=g, device=DEV, dtype=torch.uint8)
    return a, sa, b, sb


def _words(sc_rows: torch.Tensor) -> torch.Tensor:
    return torch.from_numpy(H.mx_rows_to_words(sc_rows.cpu().numpy())).to(DEV)


@pytest.mark.parametrize("T,K,N,bn", [(200, 512, 1280, 0), (64, 1024, 2048, 0), (300, 2048, 3072, 0),
                                      (1, 6144, 35840, 0), (64, 6144, 35840, 0), (256, 6144, 20480, 0),
                                      (129, 768, 400, 0), (256, 1024, 2048, 128), (100, 1024, 2048, 208),
                                      (2200, 1024, 2048, 0)])     # several row blocks, a ragged last one
def test_project_mxfp8_vs_oracle(T, K, N, bn):
    a, sa, b, sb = _random_mx(T, K, N, T + K + N)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    E().set_gemm_mx_tile(bn)
    try:
        kv = E().engram_project_mxfp8(a, _words(sa), b, _words(sb), err=err)
        kv2 = E().engram_project_mxfp8(a, _words(sa), b, _words(sb))
        torch.cuda.synchronize()
    finally:
        E().set_gemm_mx_tile(0)
    assert int(err.item()) == 0
    assert torch.equal(kv, kv2)                                   # deterministic
    ref = O.project_mxfp8(a.cpu().numpy(), sa.cpu().numpy(), b.cpu().numpy(), sb.cpu().numpy())
    H.check_kv(kv.cpu().numpy(), ref, f"mxfp8 T={T} K={K} N={N}")


def test_project_mxfp8_rejects_bad_shapes():
    a, sa, b, sb = _random_mx(8, 96, 32, 1)                       # K not a multiple of 128
    with pytest.raises(E().EngramError) as ei:
        E().engram_project_mxfp8(a, _words(sa), b, _words(sb))
    assert ei.value.code == -1


def _sample(w, case, n):
    """All tokens up to n, else a seeded sample plus sequence starts, document starts and masked."""
    T = w.tokens
    if T <= n:
        return None
    rng = np.random.default_rng(77)
    pick = set(rng.choice(T, size=n, replace=False).tolist())
    pick.update(int(x) for x in case.batch["cu_seqlens"][:-1] if x < T)
    sid = case.batch.get("sequence_ids")
    if sid is not None:
        pick.update(np.nonzero(np.diff(sid) != 0)[0][:64].tolist())
    mask = case.batch.get("token_mask")
    if mask is not None:
        pick.update(np.nonzero(mask == 0)[0][:64].tolist())
    pick.add(T - 1)
    return np.array(sorted(pick), dtype=np.int64)


@pytest.mark.parametrize("name,sample", [("tiny_fp8", 0), ("decode_fp8_t256", 0), ("decode_fp8_t256_2layer", 0),
                                         ("large_fp8_t1", 0), ("large_fp8_t64", 0), ("large_fp8_t1024", 256),
                                         ("prefill_fp8_t32768", 384)])
def test_forward_mxfp8_matches_oracle(name, sample):
    w, case, setup = H.build(name)
    got = H.gpu_forward(w, case, setup, mx=True)
    toks = _sample(w, case, sample) if sample else None
    ref = H.oracle_forward(w, case, toks, mx=True)
    assert got["err"] == 0
    assert np.array_equal(got["ids"].cpu().numpy(), ref["ids"].astype(np.int32))
    sel = ref["tokens"]
    sel_t = torch.from_numpy(sel).to(DEV)
    last = ref["layers"][-1]
    assert np.array_equal(got["A_codes_last"].index_select(0, sel_t).cpu().numpy(), last["a_bits"][0])
    assert np.array_equal(got["A_scales_last"][sel], last["a_bits"][1])
    H.check_kv(got["kv_last"].index_select(0, sel_t).cpu().numpy(), last["kv"], f"{name} mx kv")
    for l, lref in enumerate(ref["layers"]):
        h = got["streams"][l].index_select(0, sel_t).cpu().numpy()
        H.check_streams(h, lref["streams"], lref["streams_in"], f"{name} mx layer {l}")
    mask = case.batch.get("token_mask")
    if mask is not None:                                   # masked tokens bit-unchanged
        keep = mask[sel] == 0
        for l in range(w.layers):
            h = got["streams"][l].index_select(0, sel_t).cpu().numpy()
            assert np.array_equal(h[keep], case.streams[l].index_select(0, sel_t).cpu().numpy()[keep])


def test_noalloc_forward_with_mxfp8_matches_workspace_forward():
    import engram_gram_hash_02_gb300 as Em
    from engram_synth.case import to_device
    w, case, setup = H.build("decode_fp8_t256")
    primes, offsets, rows, mult = setup
    b = case.batch
    dims = H.dims_for(w, H.pad_id_of(w, b["token_map"]))
    tables = Em.HashTables(to_device(b["token_map"], DEV), to_device(mult, DEV), to_device(primes, DEV),
                           to_device(offsets, DEV))
    layers = []
    for l, t in enumerate(case.tables):
        codes, sc = Em.quantize_mxfp8(case.wkv[l])
        layers.append(Em.LayerWeights(t["fmt"], t["table"], t["scales"], t["num_rows"], codes, case.q_weight[l],
                                      case.k_weight[l], wkv_scales=sc))
    outs = []
    for noalloc in (False, True, True):
        streams = [s.clone() for s in case.streams]
        err = torch.zeros(1, dtype=torch.int32, device=DEV)
        plan = Em.ForwardPlan(dims, tables, layers, to_device(b["input_ids"], DEV), streams,
                              cu_seqlens=to_device(b["cu_seqlens"], DEV), lookback_ids=to_device(b["lookback_ids"], DEV),
                              err=err)
        plan.run_noalloc() if noalloc else plan.run()
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        outs.append(streams[0])
    assert torch.equal(outs[0], outs[1]) and torch.equal(outs[0], outs[2])   # same kernels, same order


def test_forward_mxfp8_needs_an_fp8_table():
    w, case, setup = H.build("tiny_bf16")
    with pytest.raises(E().EngramError) as ei:
        H.gpu_forward(w, case, setup, mx=True)
    assert ei.value.code == -1 and "FP8" in str(ei.value)
