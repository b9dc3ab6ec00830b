"""The Python binding refuses tensors whose shapes disagree with the dimensions the library will
index them by (the C side sees only pointers). Every check fires on the host, before any device
check, so these run on CPU tensors and launch nothing."""
import pytest
import torch


@pytest.fixture(scope="module")
def E():
    from engram_gram_hash_02_gb300 import build as B
    B.build()
    import engram_gram_hash_02_gb300 as E
    return E


L_, NG, HH, D, H, HC, RAW, V, T = 2, 3, 4, 64, 256, 4, 4096, 1024, 16
C_ = (NG - 1) * HH
K_, N_ = C_ * D, H * (HC + 1)
ROWS = 500


def _good(E, fmt="fp8", mx=False):
    dims = E.make_dims(L_, NG, HH, D, H, HC, RAW, V, 0)
    tables = E.HashTables(torch.zeros(RAW, dtype=torch.int32), torch.ones(L_, NG, dtype=torch.int64),
                          torch.ones(L_, C_, dtype=torch.int64), torch.zeros(L_, C_, dtype=torch.int64))
    layers = []
    for _ in range(L_):
        if fmt == "fp8":
            tab, sc = torch.zeros(ROWS, D, dtype=torch.uint8), torch.zeros(ROWS, D // 32, dtype=torch.uint8)
        elif fmt == "q2k":
            tab, sc = torch.zeros(ROWS, 84, dtype=torch.uint8), None
        else:
            tab, sc = torch.zeros(ROWS, D, dtype=torch.bfloat16), None
        if mx:
            wkv, wsc = torch.zeros(N_, K_, dtype=torch.uint8), torch.zeros(E.mx_scale_shape(N_, K_), dtype=torch.uint8)
        else:
            wkv, wsc = torch.zeros(N_, K_, dtype=torch.bfloat16), None
        layers.append(E.LayerWeights(fmt, tab, sc, ROWS, wkv, torch.ones(HC, H, dtype=torch.bfloat16),
                                     torch.ones(HC, H, dtype=torch.bfloat16), wkv_scales=wsc))
    streams = [torch.zeros(T, HC, H) for _ in range(L_)]
    kw = dict(cu_seqlens=torch.tensor([0, 10, T], dtype=torch.int32), sequence_ids=torch.ones(T, dtype=torch.int32),
              token_mask=torch.ones(T, dtype=torch.uint8), lookback_ids=torch.zeros(2, NG - 1, dtype=torch.int32),
              out_ids=torch.zeros(T, L_, C_, dtype=torch.int32), err=torch.zeros(1, dtype=torch.int32))
    return dims, tables, layers, torch.zeros(T, dtype=torch.int32), streams, kw


def _plan_error(E, dims, tables, layers, ids, streams, kw):
    with pytest.raises(ValueError) as ei:
        E.ForwardPlan(dims, tables, layers, ids, streams, **kw)
    return str(ei.value)


@pytest.mark.parametrize("fmt,mx", [("fp8", False), ("fp8", True), ("q2k", False), ("bf16", False)])
def test_well_formed_arguments_pass_the_shape_checks(E, fmt, mx):
    # the only complaint left for CPU tensors is the device check
    msg = _plan_error(E, *_good(E, fmt, mx))
    assert "CUDA" in msg, msg


def _mutations(E):
    """(what, function mutating the good argument set) -> each must be refused by a shape check."""
    def m(fn):
        return fn
    return {
        "short layer list": m(lambda a: a[2].pop()),
        "short stream list": m(lambda a: a[4].pop()),
        "stream rows": m(lambda a: a[4].__setitem__(1, torch.zeros(T - 1, HC, H))),
        "stream width": m(lambda a: a[4].__setitem__(0, torch.zeros(T, HC, H // 2))),
        "streams of another hc": m(lambda a: a[4].__setitem__(0, torch.zeros(T, HC - 1, H))),
        "lookback width": m(lambda a: a[5].__setitem__("lookback_ids", torch.zeros(2, NG, dtype=torch.int32))),
        "lookback rows": m(lambda a: a[5].__setitem__("lookback_ids", torch.zeros(3, NG - 1, dtype=torch.int32))),
        "mask length": m(lambda a: a[5].__setitem__("token_mask", torch.ones(T + 1, dtype=torch.uint8))),
        "sequence ids length": m(lambda a: a[5].__setitem__("sequence_ids", torch.ones(T - 1, dtype=torch.int32))),
        "out_ids shape": m(lambda a: a[5].__setitem__("out_ids", torch.zeros(T, 1, C_, dtype=torch.int32))),
        "cu_seqlens empty": m(lambda a: a[5].__setitem__("cu_seqlens", torch.zeros(1, dtype=torch.int32))),
        "q weight": m(lambda a: setattr(a[2][0], "q_weight", torch.ones(HC, H - 8, dtype=torch.bfloat16))),
        "k weight": m(lambda a: setattr(a[2][1], "k_weight", torch.ones(HC + 1, H, dtype=torch.bfloat16))),
        "wkv": m(lambda a: setattr(a[2][0], "wkv", torch.zeros(N_ - 16, K_, dtype=torch.bfloat16))),
        "table too small": m(lambda a: setattr(a[2][0], "num_rows", ROWS + 1)),
        "scales too small": m(lambda a: setattr(a[2][1], "scales", torch.zeros(ROWS - 1, D // 32, dtype=torch.uint8))),
        "token map": m(lambda a: setattr(a[1], "token_map", torch.zeros(RAW - 1, dtype=torch.int32))),
        "multipliers": m(lambda a: setattr(a[1], "multipliers", torch.ones(L_, NG - 1, dtype=torch.int64))),
        "primes": m(lambda a: setattr(a[1], "primes", torch.ones(1, C_, dtype=torch.int64))),
        "empty err": m(lambda a: a[5].__setitem__("err", torch.zeros(0, dtype=torch.int32))),
        "2-D input ids": m(lambda a: a.__setitem__(3, torch.zeros(T, 1, dtype=torch.int32))),
    }


@pytest.mark.parametrize("what", list(_mutations(__import__("types").SimpleNamespace()).keys()))
def test_each_shape_disagreement_is_refused(E, what):
    args = list(_good(E))
    _mutations(E)[what](args)
    msg = _plan_error(E, *args)
    assert "CUDA" not in msg, f"{what}: got to the device check: {msg}"


def test_mxfp8_weight_scales_shape(E):
    args = list(_good(E, "fp8", True))
    args[2][0].wkv_scales = torch.zeros(N_, K_ // 32, dtype=torch.uint8)    # the row layout, not the word layout
    assert "wkv_scales" in _plan_error(E, *args)


def test_stage_wrappers_check_shapes(E):
    dims = E.make_dims(1, NG, HH, D, H, HC, RAW, V, 0)
    h = torch.zeros(T, HC, H)
    with pytest.raises(ValueError, match="kv"):
        E.engram_gate(dims, h, torch.zeros(T, N_ - 4), torch.ones(HC, H, dtype=torch.bfloat16),
                      torch.ones(HC, H, dtype=torch.bfloat16))
    with pytest.raises(ValueError, match="q_weight"):
        E.engram_gate(dims, h, torch.zeros(T, N_), torch.ones(HC - 1, H, dtype=torch.bfloat16),
                      torch.ones(HC, H, dtype=torch.bfloat16))
    with pytest.raises(ValueError, match="out"):
        E.engram_project(torch.zeros(T, K_, dtype=torch.bfloat16), torch.zeros(N_, K_, dtype=torch.bfloat16),
                         out=torch.zeros(T, N_ - 16))
    ids = torch.zeros(T, C_, dtype=torch.int32)
    with pytest.raises(ValueError, match="table"):
        E.engram_gather_dequant("fp8", ids, torch.zeros(10, D, dtype=torch.uint8),
                                torch.zeros(10, D // 32, dtype=torch.uint8), 11, D)
    with pytest.raises(ValueError, match="out"):
        E.engram_gather_dequant("bf16", ids, torch.zeros(10, D, dtype=torch.bfloat16), None, 10, D,
                                out=torch.zeros(T, K_ - 8, dtype=torch.bfloat16))
    with pytest.raises(ValueError, match="lookback"):
        E.engram_hash(E.make_dims(1, NG, HH, D, H, HC, RAW, V, 0), torch.zeros(T, dtype=torch.int32),
                      torch.zeros(RAW, dtype=torch.int32), torch.ones(1, NG, dtype=torch.int64),
                      torch.ones(1, C_, dtype=torch.int64), torch.zeros(1, C_, dtype=torch.int64),
                      lookback_ids=torch.zeros(1, NG, dtype=torch.int32))
