"""The C-ABI library on a machine without a GPU: it builds, loads, exports every function the
header declares, and its host-only parts behave (layout, argument checks that fire before any
CUDA call).  No kernel is launched here."""
import ctypes
import re
from pathlib import Path

import numpy as np
import pytest

from oracle import engram_oracle as O

ROOT = Path(__file__).resolve().parents[1]
HEADER = ROOT / "include" / "engram.h"


@pytest.fixture(scope="module")
def lib():
    from engram_gram_hash_02_gb300 import build as B
    from engram_gram_hash_02_gb300 import binding
    B.build()
    return binding.lib()


def declared_functions():
    text = HEADER.read_text()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)          # drop comments
    names = re.findall(r"^[A-Za-z_][\w\s\*]*?\b(engram_\w+)\s*\(", text, flags=re.M)
    return sorted(set(names))


def test_header_declares_the_boundary_calls():
    names = declared_functions()
    for want in ("engram_hash", "engram_gather_dequant", "engram_project", "engram_gate", "engram_forward",
                 "engram_forward_workspace_bytes", "engram_forward_noalloc", "engram_layout",
                 "engram_last_error"):
        assert want in names, want


def test_library_exports_every_declared_function(lib):
    missing = [n for n in declared_functions() if not hasattr(lib, n)]
    assert not missing, f"declared in engram.h but not exported: {missing}"


def test_version_string(lib):
    v = lib.engram_version().decode()
    assert "sm_103a" in v


def _c_layout(lib, vocab, L, ng, hh):
    C = (ng - 1) * hh
    p = np.zeros(L * C, np.int64)
    o = np.zeros(L * C, np.int64)
    r = np.zeros(L, np.int64)
    rc = lib.engram_layout(vocab, L, ng, hh, p.ctypes.data, o.ctypes.data, r.ctypes.data)
    return rc, p.reshape(L, C), o.reshape(L, C), r


@pytest.mark.parametrize("vocab,L,ng,hh", [(4001, 1, 3, 4), (1 << 20, 1, 4, 8), (1 << 19, 2, 4, 8), (97, 3, 5, 2)])
def test_host_layout_equals_oracle(lib, vocab, L, ng, hh):
    rc, p, o, r = _c_layout(lib, vocab, L, ng, hh)
    assert rc == 0
    op, oo, orows = O.layout(vocab, L, ng, hh)               # oracle: [L, orders, heads]
    assert np.array_equal(p, np.asarray(op).reshape(L, -1))
    assert np.array_equal(o, np.asarray(oo).reshape(L, -1))
    assert np.array_equal(r, np.asarray(orows).reshape(L))


def test_host_layout_rejects_bad_arguments(lib):
    rc, *_ = _c_layout(lib, 0, 1, 3, 4)
    assert rc == -1
    assert "engram_layout" in lib.engram_last_error().decode()


def test_argument_checks_fire_before_any_cuda_call(lib):
    from engram_gram_hash_02_gb300 import binding as Bd
    stream = None
    # projection: NULL operands
    rc = lib.engram_project(None, None, None, 4, 64, 64, None, 0, None, stream)
    assert rc == -1 and "non-NULL" in lib.engram_last_error().decode()
    # projection: K not a multiple of 8
    rc = lib.engram_project(None, None, None, 4, 60, 64, None, 0, None, stream)
    assert rc == -1 and "K must be" in lib.engram_last_error().decode()
    # gather: unknown table format
    buf = (ctypes.c_uint8 * 4096)()
    addr = (ctypes.addressof(buf) + 15) & ~15
    rc = lib.engram_gather_dequant(7, addr, 8, 1, 8, 64, addr, addr, 10, addr, None, stream)
    assert rc == -1 and "unknown table format" in lib.engram_last_error().decode()
    # gate: hidden not a multiple of 8
    dims = Bd.EngramDims(1, 3, 4, 64, 7, 4, 16, 16, 0, 1e-6, 1e-6)
    rc = lib.engram_gate(ctypes.byref(dims), addr, addr, addr, addr, None, 1, None, stream)
    assert rc == -1 and "hidden" in lib.engram_last_error().decode()
    # hash: pad id outside the compressed vocabulary
    dims = Bd.EngramDims(1, 3, 4, 64, 256, 4, 16, 16, 99, 1e-6, 1e-6)
    rc = lib.engram_hash(ctypes.byref(dims), addr, 1, addr, 1, None, None, None, addr, addr, addr, addr, addr,
                         None, stream)
    assert rc == -1 and "pad_id" in lib.engram_last_error().decode()


def test_forward_workspace_covers_ids_rows_and_kv(lib):
    from engram_gram_hash_02_gb300 import binding as Bd
    dims = Bd.EngramDims(1, 4, 8, 256, 4096, 4, 163840, 131072, 0, 1e-6, 1e-6)
    T = 256
    C, K, N = 24, 24 * 256, 4096 * 5
    need = lib.engram_forward_workspace_bytes(ctypes.byref(dims), T)
    assert need >= 4 * T * C + 2 * T * K + 4 * T * N
    assert need % 256 == 0


def test_fp8_variant_argument_checks_fire_before_any_cuda_call(lib):
    buf = (ctypes.c_uint8 * 4096)()
    addr = (ctypes.addressof(buf) + 15) & ~15
    stream = None
    # encoder: K not a multiple of 32
    rc = lib.engram_quantize_mxfp8(addr, 4, 33, addr, addr, stream)
    assert rc == -1 and "multiple of 32" in lib.engram_last_error().decode()
    # projection: K not a multiple of 128
    rc = lib.engram_project_mxfp8(addr, addr, addr, addr, addr, 4, 96, 32, None, stream)
    assert rc == -1 and "multiple of 128" in lib.engram_last_error().decode()
    # projection: scales must be 16-byte aligned (the stage's scale words are bulk-copied)
    rc = lib.engram_project_mxfp8(addr, addr + 4, addr, addr, addr, 4, 128, 32, None, stream)
    assert rc == -1 and "16-byte aligned" in lib.engram_last_error().decode()
    # raw FP8 gather: head_dim not a multiple of 32
    rc = lib.engram_gather_fp8_codes(addr, 8, 1, 8, 48, addr, addr, 10, addr, addr, None, stream)
    assert rc == -1 and "multiple of 32" in lib.engram_last_error().decode()
    # T = 0 and N = 0 are no-ops
    assert lib.engram_project_mxfp8(None, None, None, None, None, 0, 128, 32, None, stream) == 0
    assert lib.engram_quantize_mxfp8(None, 0, 64, None, None, stream) == 0


def test_mx_scale_shape():
    from engram_gram_hash_02_gb300 import binding as Bd
    assert Bd.mx_scale_shape(256, 6144) == (48, 256, 4)
    assert Bd.mx_scale_shape(1, 6144) == (48, 4, 4)          # rows padded to a multiple of 4
    assert Bd.mx_scale_shape(5, 96) == (1, 8, 4)             # 3 blocks of 32 -> one word per row


def test_forward_host_checks_fire_before_any_cuda_call(lib):
    from engram_gram_hash_02_gb300 import binding as Bd
    buf = (ctypes.c_uint8 * 8192)()
    addr = (ctypes.addressof(buf) + 255) & ~255
    stream = None
    tables = Bd._HashTables(addr, addr, addr, addr)
    tok = Bd._Tokens(addr, 256, addr, 256, None, None, None)
    streams = (ctypes.c_void_p * 2)(addr, addr)

    def layer(fmt, wkv_fmt):
        return Bd._LayerWeights(Bd.TABLE_FORMATS[fmt], addr, addr, 1000, addr, addr, addr, wkv_fmt,
                                addr if wkv_fmt == Bd.WKV_MXFP8 else None)

    # more than 256 (layer, column) pairs
    dims = Bd.EngramDims(11, 4, 8, 256, 4096, 4, 163840, 131072, 0, 1e-6, 1e-6)
    layers = (Bd._LayerWeights * 11)(*[layer("fp8", Bd.WKV_BF16)] * 11)
    rc = lib.engram_forward(ctypes.byref(dims), ctypes.byref(tables), layers, ctypes.byref(tok), streams, addr,
                            1 << 40, None, None, stream)
    assert rc == -1 and "256" in lib.engram_last_error().decode()
    # a workspace below engram_forward_workspace_bytes
    dims = Bd.EngramDims(2, 4, 8, 256, 4096, 4, 163840, 131072, 0, 1e-6, 1e-6)
    need = lib.engram_forward_workspace_bytes(ctypes.byref(dims), 256)
    layers = (Bd._LayerWeights * 2)(layer("fp8", Bd.WKV_BF16), layer("q2k", Bd.WKV_MXFP8))
    rc = lib.engram_forward(ctypes.byref(dims), ctypes.byref(tables), layers, ctypes.byref(tok), streams, addr,
                            need - 256, None, None, stream)
    assert rc == -1 and str(need) in lib.engram_last_error().decode()
    # an MXFP8 wkv needs an FP8 table (its rows are the A operand): rejected before any launch
    rc = lib.engram_forward(ctypes.byref(dims), ctypes.byref(tables), layers, ctypes.byref(tok), streams, addr,
                            need, None, None, stream)
    assert rc == -1 and "MXFP8 wkv needs an FP8" in lib.engram_last_error().decode()
    # zero tokens: nothing to do
    tok0 = Bd._Tokens(addr, 0, addr, 1, None, None, None)
    assert lib.engram_forward(ctypes.byref(dims), ctypes.byref(tables), layers, ctypes.byref(tok0), streams, None,
                              0, None, None, stream) == 0


def test_forward_workspace_holds_one_operand_slot_per_layer(lib):
    from engram_gram_hash_02_gb300 import binding as Bd
    r256 = lambda x: (x + 255) // 256 * 256
    for T in (1, 7, 256, 4096):
        one = Bd.EngramDims(1, 4, 8, 256, 4096, 4, 163840, 131072, 0, 1e-6, 1e-6)
        two = Bd.EngramDims(2, 4, 8, 256, 4096, 4, 163840, 131072, 0, 1e-6, 1e-6)
        C, K, N = 24, 24 * 256, 4096 * 5
        w1 = lib.engram_forward_workspace_bytes(ctypes.byref(one), T)
        w2 = lib.engram_forward_workspace_bytes(ctypes.byref(two), T)
        done = lambda L: r256((T + 127) // 128 * L * 4)       # the overlapped gate's row-block counters
        slot = w2 - w1 - (r256(4 * T * 2 * C) - r256(4 * T * C)) - (done(2) - done(1))
        # a slot holds the bf16 rows, or the FP8 codes and then their scale words
        assert slot >= 2 * T * K and slot >= r256(T * K) + (K // 128) * ((T + 3) // 4 * 4) * 4
        assert w1 == r256(4 * T * C) + slot + r256(4 * T * N) + done(1)


def test_sync_status_rejects_a_null_word(lib):
    assert lib.engram_sync_status(None, None) == -1
    assert "err_flag" in lib.engram_last_error().decode()


def _plan(lib, T, K, N, fmt, sms):
    from engram_gram_hash_02_gb300.binding import ProjectPlan
    out = ProjectPlan()
    rc = lib.engram_project_plan(T, K, N, fmt, sms, ctypes.byref(out))
    return rc, out.as_dict()


def _check_plan(p, T, fmt, sms, forced=0):
    where = f"T={T} fmt={fmt} sms={sms} forced={forced}: {p}"
    # the tensor cores read a full 128-row token tile from the last stage: inside the allocation
    assert p["mma_read_end"] <= p["smem_avail"], where
    assert p["smem_avail"] + 1024 == p["smem_bytes"] <= 232448, where
    assert p["stages"] >= 2, where
    assert 1 <= p["grid"] <= sms, where
    assert p["tile_rows"] in (128, 256), where
    assert p["tile_cols"] % 16 == 0 and 16 <= p["tile_cols"] <= (512 if p["split"] == 2 else 256), where
    assert p["tmem_cols"] in (32, 64, 128, 256, 512), where
    rows = p["token_rows_loaded"]
    assert rows % 16 == 0 and 16 <= rows <= 128, where
    if rows < 128:                       # short token tiles only for one block of at most 112 tokens
        assert T <= 112 and p["tile_rows"] == 128 and not p["stream_k"], where
    if forced and p["split"] == 1:
        assert p["tile_cols"] == forced, where


@pytest.mark.parametrize("K,N", [(6144, 20480), (6144, 35840), (512, 1280), (2048, 1280), (128, 16), (6144, 112)])
def test_projection_plans_keep_the_mma_reads_inside_shared_memory(lib, K, N):
    """Every plan the two projection planners make (T 1..512 and a few large T, automatic and
    forced tile widths) keeps the last stage's 128-row token-tile reads inside the CTA's shared
    memory, and its other sizes within what the kernels assume."""
    Ts = list(range(1, 513)) + [1000, 4096, 32768]
    try:
        for fmt in (0, 1):
            if fmt == 1 and K % 128:
                continue
            setter = lib.engram_set_gemm_tile if fmt == 0 else lib.engram_set_gemm_mx_tile
            for forced in (0, 16, 48, 112, 128, 144, 224, 256):
                setter(forced)
                for T in Ts:
                    for sms in (148, 152):
                        rc, p = _plan(lib, T, K, N, fmt, sms)
                        if rc != 0:
                            # only a forced width the MXFP8 tensor memory cannot hold may be refused
                            assert fmt == 1 and forced >= 224 and T > 128, (T, K, N, forced,
                                                                            lib.engram_last_error().decode())
                            continue
                        _check_plan(p, T, fmt, sms, forced)
    finally:
        lib.engram_set_gemm_tile(0)
        lib.engram_set_gemm_mx_tile(0)


def test_projection_plan_rejects_bad_shapes(lib):
    assert _plan(lib, 0, 6144, 20480, 0, 152)[0] == -1
    assert _plan(lib, 256, 6144, 20481, 0, 152)[0] == -1
    assert _plan(lib, 256, 6100, 20480, 1, 152)[0] == -1      # MXFP8 needs K % 128 == 0
    assert _plan(lib, 256, 6144, 20480, 7, 152)[0] == -1


def test_decode_plan_is_the_split_tile():
    """The decode shape (256 tokens, wide wkv) runs split tiles: pairs of 128-row CTAs."""
    import engram_gram_hash_02_gb300 as E
    p = E.project_plan(256, 6144, 20480, "bf16", 148)
    assert p["split"] == 2 and p["tile_rows"] == 128 and p["grid"] <= 148
