"""GPU parity of each stage through the C ABI against the oracle, on seeded inputs.

Hash ids and dequantised rows must be bit-exact; the projection within bf16 output rounding of
the fp64 product; the gate within the stream tolerance.  Sizes span several tiles with ragged
tails; edge cases cover empty, single-token, out-of-range and masked inputs.
"""
import numpy as np
import pytest
import torch

from engram_synth import gen, get_workload
from engram_synth.case import to_device
from oracle import engram_oracle as O
from tests import _helpers as H

pytestmark = pytest.mark.gpu
DEV = "cuda"


def E():
    import engram_gram_hash_02_gb300 as mod
    return mod


# ------------------------------------------------------------------------------------------- hash

def _hash_both(w, batch, layout=None):
    primes, offsets, rows, mult = layout or H.product_setup(w)
    pad = H.pad_id_of(w, batch["token_map"])
    dims = H.dims_for(w, pad)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    got = E().engram_hash(dims, to_device(batch["input_ids"], DEV), to_device(batch["token_map"], DEV),
                          to_device(mult, DEV), to_device(primes, DEV), to_device(offsets, DEV),
                          cu_seqlens=to_device(batch["cu_seqlens"], DEV),
                          sequence_ids=to_device(batch.get("sequence_ids"), DEV),
                          token_mask=to_device(batch.get("token_mask"), DEV),
                          lookback_ids=to_device(batch.get("lookback_ids"), DEV), err=err)
    op, oo, _, om = H.oracle_setup(w)
    win, bad = O.windows(batch["input_ids"], batch["token_map"], pad, w.max_ngram, batch["cu_seqlens"],
                         batch.get("sequence_ids"), batch.get("token_mask"), batch.get("lookback_ids"))
    ref = O.hash_ids(win, om, op, oo, w.compressed_vocab)
    return got.cpu().numpy(), ref, int(err.item()), int(bad.sum())


@pytest.mark.parametrize("name", ["tiny_bf16", "decode_fp8_t256", "decode_fp8_t256_deadlb",
                                  "prefill_fp8_t32768", "q2k_t8192", "large_fp8_t16384"])
def test_hash_bit_exact(name):
    w = get_workload(name)
    batch = gen.batch_inputs(w)
    got, ref, err, bad = _hash_both(w, batch)
    assert got.shape == ref.shape
    assert np.array_equal(got, ref.astype(np.int32))
    assert err == 0 and bad == 0


def test_hash_edge_cases():
    w = get_workload("decode_fp8_t256")
    rng = np.random.default_rng(0)
    # ragged sequences incl. empty ones, bad raw ids, masked runs, document cuts, dead lookback
    lens = [0, 1, 5, 0, 37, 2, 3, 0, 64]
    T = sum(lens)
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    ids = rng.integers(0, w.raw_vocab, size=T).astype(np.int32)
    ids[[3, 10]] = [w.raw_vocab, -5]                         # outside the map: pad + flag
    mask = (rng.random(T) > 0.25).astype(np.uint8)
    sid = np.ones(T, dtype=np.int32)
    sid[20:40] = 2
    sid[45] = 0
    lb = rng.integers(0, w.compressed_vocab, size=(len(lens), 3)).astype(np.int32)
    lb[rng.random(lb.shape) < 0.3] = -1
    tmap = gen.token_map(w.raw_vocab, w.compressed_vocab, "surjection", 1)
    batch = {"input_ids": ids, "cu_seqlens": cu, "sequence_ids": sid, "token_mask": mask,
             "lookback_ids": lb, "token_map": tmap}
    got, ref, err, bad = _hash_both(w, batch)
    assert np.array_equal(got, ref.astype(np.int32))
    assert bad == 2 and err == E().ERR_RAW_ID
    # T = 0 is a no-op
    batch0 = dict(batch, input_ids=np.zeros(0, np.int32), cu_seqlens=np.zeros(2, np.int32),
                  sequence_ids=None, token_mask=None, lookback_ids=None)
    got0, ref0, err0, _ = _hash_both(w, batch0)
    assert got0.shape == (0, 1, 24) and err0 == 0


def test_hash_all_masked_is_all_pad_window():
    w = get_workload("tiny_bf16")
    batch = gen.batch_inputs(w)
    batch["token_mask"] = np.zeros(w.tokens, dtype=np.uint8)
    got, ref, _, _ = _hash_both(w, batch)
    assert np.array_equal(got, ref.astype(np.int32))
    assert np.all(got == got[0])


# ------------------------------------------------------------------------------------------ gather

def _gather_case(fmt, rows, T, C, D, seed):
    g = torch.Generator().manual_seed(seed)
    if fmt == "fp8":
        table, scales = gen.fp8_table(rows, D, 0.02, seed, DEV)
        # exercise the scale range, incl. byte 0 (+0.0) and large exponents
        scales[: rows // 8] = torch.randint(0, 255, (rows // 8, D // 32), generator=g).to(torch.uint8).to(DEV)
    elif fmt == "q2k":
        table, scales = gen.q2k_table(rows, seed, DEV), None
    else:
        table, scales = gen.bf16_table(rows, D, 0.02, seed, DEV), None
    ids = torch.randint(0, rows, (T, C), generator=g, dtype=torch.int32)
    ids[0, 0] = rows                # out of range -> zero row
    ids[T // 2, C - 1] = -7
    ids[(T - 1) // 2, 1] = rows - 1   # last and first rows of the table
    ids[T - 1, C // 2] = 0
    return table, scales, ids


def _oracle_rows(fmt, table, scales, ids_np, rows, D):
    t_np = table.cpu().view(torch.int16).numpy().view(np.uint16) if fmt == "bf16" else table.cpu().numpy()
    s_np = None if scales is None else scales.cpu().numpy()
    return O.gather(fmt, t_np, s_np, ids_np, rows, D)


@pytest.mark.parametrize("fmt,D,C,T,rows", [
    ("fp8", 256, 24, 300, 5000), ("fp8", 64, 3, 17, 100), ("fp8", 256, 24, 1, 77),
    ("q2k", 256, 24, 300, 5000), ("q2k", 256, 5, 9, 40),
    ("bf16", 64, 8, 64, 32140), ("bf16", 24, 3, 13, 50),
])
def test_gather_bit_exact(fmt, D, C, T, rows):
    table, scales, ids = _gather_case(fmt, rows, T, C, D, seed=D + C + T)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    got = E().engram_gather_dequant(fmt, ids.to(DEV), table, scales, rows, D, err=err)
    ref, n_oob = _oracle_rows(fmt, table, scales, ids.numpy(), rows, D)
    torch.cuda.synchronize()
    assert np.array_equal(H.bits16(got), ref)
    assert n_oob == 2 and int(err.item()) == E().ERR_ROW_ID


def test_gather_strided_ids_view():
    # ids given as the per-layer slice of a [T, L, C] hash output
    table, scales, ids = _gather_case("fp8", 3000, 50, 24 * 2, 256, seed=5)
    ids3 = ids.view(50, 2, 24).to(DEV)
    got = E().engram_gather_dequant("fp8", ids3[:, 1], table, scales, 3000, 256)
    ref, _ = _oracle_rows("fp8", table, scales, ids.view(50, 2, 24)[:, 1].numpy(), 3000, 256)
    assert np.array_equal(H.bits16(got), ref)


# ---------------------------------------------------------------------------------------- project

@pytest.mark.parametrize("T,K,N", [
    (64, 512, 1280), (1, 512, 1280), (129, 576, 400), (300, 6144, 1296), (256, 1024, 4096),
    (77, 520, 272), (513, 256, 512),
])
def test_project_vs_fp64(T, K, N):
    g = torch.Generator(device=DEV).manual_seed(T * 7 + K + N)
    A = (torch.randn(T, K, generator=g, device=DEV) * 0.02).to(torch.bfloat16)
    W = (torch.randn(N, K, generator=g, device=DEV) * 0.02).to(torch.bfloat16)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    kv = E().engram_project(A, W, err=err)
    ref = O.project(H.bits16(A), H.bits16(W))
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    H.check_kv(kv.cpu().numpy(), ref, f"T={T} K={K} N={N}")
    # the library GEMM and torch's fp32 matmul of the same bf16 values agree to fp32 summation order
    tm = (A.float() @ W.float().t())
    assert torch.allclose(kv, tm, rtol=1e-4, atol=1e-4 * float(tm.pow(2).mean().sqrt()))


@pytest.mark.parametrize("bn", [16, 48, 128, 144, 256, 96])
@pytest.mark.parametrize("T", [260, 100])
def test_project_tile_widths_data_parallel(bn, T):
    # N = 1440 is 90, 30, 12, 10, 6 or 15 column tiles; T 260 is two 256-row blocks, T 100 one
    # 128-row block split into even / odd k-step chains
    K, N = 640, 1440
    g = torch.Generator(device=DEV).manual_seed(bn * 10 + T)
    A = (torch.randn(T, K, generator=g, device=DEV) * 0.02).to(torch.bfloat16)
    W = (torch.randn(N, K, generator=g, device=DEV) * 0.02).to(torch.bfloat16)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    try:
        E().set_gemm_tile(bn)
        E().set_gemm_schedule(1)
        kv = E().engram_project(A, W, err=err)
        torch.cuda.synchronize()
    finally:
        E().set_gemm_tile(0)
        E().set_gemm_schedule(0)
    assert int(err.item()) == 0
    H.check_kv(kv.cpu().numpy(), O.project(H.bits16(A), H.bits16(W)), f"bn={bn} T={T}")


@pytest.mark.parametrize("T,K,N", [
    (64, 512, 1280),       # 5 tiles x 8 k-blocks over 40 CTAs: every tile cut 8 ways
    (256, 1024, 4096),     # 16 tiles x 16 k-blocks: tiles cut across ~10 CTAs
    (300, 6144, 1296),     # 2 row blocks (ragged), ragged last column tile
    (1, 6144, 2560),
    (256, 6144, 20480),    # the decode projection
])
def test_project_stream_k_matches_fp64_and_is_deterministic(T, K, N):
    g = torch.Generator(device=DEV).manual_seed(T + K + N)
    A = (torch.randn(T, K, generator=g, device=DEV) * 0.02).to(torch.bfloat16)
    W = (torch.randn(N, K, generator=g, device=DEV) * 0.02).to(torch.bfloat16)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    nbytes = E().project_workspace_bytes(T, K, N)
    assert nbytes > 0, "this shape should qualify for stream-K"
    ws = torch.full((nbytes,), 0xAB, dtype=torch.uint8, device=DEV)      # stale contents must not matter
    try:
        E().set_gemm_schedule(2)
        kv1 = E().engram_project(A, W, err=err, workspace=ws)
        kv2 = E().engram_project(A, W, err=err, workspace=ws)
        E().set_gemm_schedule(1)
        kv_dp = E().engram_project(A, W, err=err, workspace=None)
        torch.cuda.synchronize()
    finally:
        E().set_gemm_schedule(0)
    assert int(err.item()) == 0
    assert torch.equal(kv1, kv2)                     # fixed summation order
    rows = np.arange(T) if T <= 300 else np.random.default_rng(0).choice(T, 64, replace=False)
    ref = O.project(H.bits16(A)[rows], H.bits16(W))
    H.check_kv(kv1.cpu().numpy()[rows], ref, f"stream-K T={T} K={K} N={N}")
    H.check_kv(kv_dp.cpu().numpy()[rows], ref, f"data-parallel T={T} K={K} N={N}")


@pytest.mark.parametrize("T,K,N", [
    (256, 6144, 20480),    # the decode projection: 2 x 72 CTAs of 128 x 288 (halves of 144)
    (200, 640, 20480),     # ragged second row block
    (129, 256, 20480),     # a one-row second row block
    (160, 512, 19008),     # halves of 128; the last column block reaches only into its first half
])
def test_project_split_tiles_match_unsplit_and_fp64(T, K, N):
    # 129..256 tokens with wide wkv run as pairs of 128-row CTAs on 2*BN-column tiles; forcing the
    # tile width (engram_set_gemm_tile) runs the 256-row tiles instead. Each output element sums
    # the same k steps in the same order either way.
    g = torch.Generator(device=DEV).manual_seed(T + K + N)
    A = (torch.randn(T, K, generator=g, device=DEV) * 0.02).to(torch.bfloat16)
    W = (torch.randn(N, K, generator=g, device=DEV) * 0.02).to(torch.bfloat16)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    try:
        E().set_gemm_schedule(1)
        split = E().engram_project(A, W, err=err)
        E().set_gemm_tile(144)
        whole = E().engram_project(A, W, err=err)
        torch.cuda.synchronize()
    finally:
        E().set_gemm_tile(0)
        E().set_gemm_schedule(0)
    assert int(err.item()) == 0
    assert torch.equal(split, whole)
    H.check_kv(split.cpu().numpy(), O.project(H.bits16(A), H.bits16(W)), f"split T={T} K={K} N={N}")


@pytest.mark.parametrize("T,bn", [(40, 64), (1, 16), (112, 128)])
def test_project_short_token_tiles_over_several_waves(T, bn):
    # one block of at most 112 tokens loads only its rows (rounded up to 16); with narrow tiles
    # every CTA runs several tiles in a row over the same ring
    K, N = 256, 35840
    g = torch.Generator(device=DEV).manual_seed(T + bn)
    A = (torch.randn(T, K, generator=g, device=DEV) * 0.02).to(torch.bfloat16)
    W = (torch.randn(N, K, generator=g, device=DEV) * 0.02).to(torch.bfloat16)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    try:
        E().set_gemm_tile(bn)
        kv = E().engram_project(A, W, err=err)
        torch.cuda.synchronize()
    finally:
        E().set_gemm_tile(0)
    assert int(err.item()) == 0
    H.check_kv(kv.cpu().numpy(), O.project(H.bits16(A), H.bits16(W)), f"short T={T} bn={bn}")


def test_project_integer_exact():
    # small integers: every product and partial sum is exact in fp32
    g = torch.Generator(device=DEV).manual_seed(3)
    A = torch.randint(-3, 4, (200, 256), generator=g, device=DEV).to(torch.bfloat16)
    W = torch.randint(-3, 4, (320, 256), generator=g, device=DEV).to(torch.bfloat16)
    ref = O.project(H.bits16(A), H.bits16(W))
    kv = E().engram_project(A, W)
    assert np.array_equal(kv.cpu().numpy().astype(np.float64), ref)


# ------------------------------------------------------------------------------------------- gate

# The gate kernel is persistent (a few CTAs per SM, two shared-memory buffers each): the larger
# cases give every CTA many items, so the buffers are reused across several phases.
@pytest.mark.parametrize("T,hc,H_,masked", [(64, 4, 256, False), (37, 4, 4096, True), (5, 4, 7168, True),
                                            (9, 2, 1000, False), (3, 1, 8, True), (16, 8, 512, False),
                                            (700, 4, 4096, True), (120, 4, 8192, False), (90, 4, 7168, True),
                                            (3000, 8, 64, True)])
@pytest.mark.parametrize("form", [1, 2])
def test_gate_vs_oracle(T, hc, H_, masked, form):
    """Both gate kernels (1 persistent, 2 one CTA per item) at every shape."""
    E().set_gate_form(form)
    try:
        _gate_vs_oracle(T, hc, H_, masked)
    finally:
        E().set_gate_form(0)


def _gate_vs_oracle(T, hc, H_, masked):
    g = torch.Generator(device=DEV).manual_seed(T + hc + H_)
    h = torch.randn(T, hc, H_, generator=g, device=DEV)
    kv = torch.randn(T, (hc + 1) * H_, generator=g, device=DEV) * 0.03
    q = (1 + 0.1 * torch.randn(hc, H_, generator=g, device=DEV)).to(torch.bfloat16)
    k = (1 + 0.1 * torch.randn(hc, H_, generator=g, device=DEV)).to(torch.bfloat16)
    mask = None
    if masked:
        mask = (torch.rand(T, generator=g, device=DEV) > 0.3).to(torch.uint8)
    h0 = h.cpu().numpy().astype(np.float64)
    dims = E().make_dims(1, 3, 4, 64, H_, hc, 10, 10, 0, 1e-6, 1e-6)
    E().engram_gate(dims, h, kv, q, k, token_mask=mask)
    ref, _ = O.gate(h0, kv.cpu().numpy().astype(np.float64), H.bits16(q), H.bits16(k), 1e-6, 1e-6,
                    None if mask is None else mask.cpu().numpy())
    got = h.cpu().numpy()
    if mask is not None:
        keep = mask.cpu().numpy() == 0
        assert np.array_equal(got[keep], h0[keep].astype(np.float32))   # bit-unchanged
    H.check_streams(got, ref, h0, f"gate T={T} hc={hc} H={H_}")


@pytest.fixture(params=[1, 2], ids=["persistent", "per_item"])
def gate_form(request):
    E().set_gate_form(request.param)
    yield request.param
    E().set_gate_form(0)


def test_gate_all_masked_leaves_streams_bit_unchanged(gate_form):
    T, hc, H_ = 500, 4, 4096
    h = torch.randn(T, hc, H_, device=DEV)
    before = h.clone()
    kv = torch.randn(T, (hc + 1) * H_, device=DEV)
    q = torch.ones(hc, H_, device=DEV, dtype=torch.bfloat16)
    mask = torch.zeros(T, dtype=torch.uint8, device=DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    dims = E().make_dims(1, 3, 4, 64, H_, hc, 10, 10, 0)
    E().engram_gate(dims, h, kv, q, q, token_mask=mask, err=err)
    assert torch.equal(h, before) and int(err.item()) == 0


def test_gate_zero_value_bit_unchanged(gate_form):
    T, hc, H_ = 8, 4, 512
    h = torch.randn(T, hc, H_, device=DEV)
    before = h.clone()
    kv = torch.zeros(T, (hc + 1) * H_, device=DEV)
    kv[:, : hc * H_] = torch.randn(T, hc * H_, device=DEV)
    q = torch.ones(hc, H_, device=DEV, dtype=torch.bfloat16)
    dims = E().make_dims(1, 3, 4, 64, H_, hc, 10, 10, 0)
    E().engram_gate(dims, h, kv, q, q)
    assert torch.equal(h, before)


# --------------------------------------------------------------------------------------- errors

def test_bad_arguments_return_einval():
    dims = E().make_dims(1, 3, 4, 64, 256, 4, 10, 10, 0)
    A = torch.zeros(4, 100, dtype=torch.bfloat16, device=DEV)   # K % 8 != 0
    W = torch.zeros(16, 100, dtype=torch.bfloat16, device=DEV)
    with pytest.raises(E().EngramError) as ei:
        E().engram_project(A, W)
    assert ei.value.code == -1
    h = torch.zeros(2, 4, 256, device=DEV)
    kv = torch.zeros(2, 5 * 256, device=DEV)
    q = torch.zeros(4, 256, device=DEV, dtype=torch.bfloat16)
    bad = E().make_dims(1, 3, 4, 64, 256, 9, 10, 10, 0)          # hc > 8: refused by the library
    h9 = torch.zeros(2, 9, 256, device=DEV)
    kv9 = torch.zeros(2, 10 * 256, device=DEV)
    q9 = torch.zeros(9, 256, device=DEV, dtype=torch.bfloat16)
    with pytest.raises(E().EngramError) as ei:
        E().engram_gate(bad, h9, kv9, q9, q9)
    assert ei.value.code == -1
    with pytest.raises(ValueError):                              # streams shape disagrees with dims
        E().engram_gate(dims, h9, kv9, q9, q9)
    E().engram_gate(dims, h[:0], kv[:0], q, q)                   # T = 0: no-op


def test_sync_status_reports_substituted_ids():
    """engram_sync_status (through the C ABI): 0 on clean inputs; ENGRAM_EDATA (-3) once a row id
    outside the table was read as a zero row, or a raw id outside the token map hashed as pad_id.
    The ids are set on the host; nothing faults."""
    rows, T, C, D = 3000, 40, 24, 256
    table, scales, ids = _gather_case("fp8", rows, T, C, D, seed=11)
    ok_ids = ids.clamp(0, rows - 1).to(DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    E().engram_gather_dequant("fp8", ok_ids, table, scales, rows, D, err=err)
    assert E().sync_status(err) == 0
    E().engram_gather_dequant("fp8", ids.to(DEV), table, scales, rows, D, err=err)   # ids[0, 0] == rows
    assert E().sync_status(err) == -3
    assert "row id" in E().lib().engram_last_error().decode()

    w = get_workload("decode_fp8_t256")
    batch = gen.batch_inputs(w)
    primes, offsets, _, mult = H.product_setup(w)
    dims = H.dims_for(w, H.pad_id_of(w, batch["token_map"]))
    args = (to_device(batch["token_map"], DEV), to_device(mult, DEV), to_device(primes, DEV), to_device(offsets, DEV))
    err.zero_()
    E().engram_hash(dims, to_device(batch["input_ids"], DEV), *args, cu_seqlens=to_device(batch["cu_seqlens"], DEV),
                    lookback_ids=to_device(batch["lookback_ids"], DEV), err=err)
    assert E().sync_status(err) == 0
    bad = batch["input_ids"].copy()
    bad[17] = w.raw_vocab                          # outside the token map
    E().engram_hash(dims, to_device(bad, DEV), *args, cu_seqlens=to_device(batch["cu_seqlens"], DEV),
                    lookback_ids=to_device(batch["lookback_ids"], DEV), err=err)
    assert E().sync_status(err) == -3
    assert "raw id" in E().lib().engram_last_error().decode()
