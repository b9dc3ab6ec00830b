"""ctypes binding of libengram: argument marshalling only.

Every stage runs in the CUDA library; these wrappers check tensor dtypes and
devices, pass raw pointers, sizes and the current CUDA stream, and turn a
non-zero return code into ``EngramError``.  There is no fallback: if the
library is missing, ``lib()`` raises.
"""
from __future__ import annotations

import ctypes as C
import os
from dataclasses import dataclass

import numpy as np
import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libengram.so")

TABLE_BF16, TABLE_FP8_E8M0, TABLE_Q2K = 0, 1, 2
WKV_BF16, WKV_MXFP8 = 0, 1
TABLE_FORMATS = {"bf16": TABLE_BF16, "fp8": TABLE_FP8_E8M0, "q2k": TABLE_Q2K}
ERR_RAW_ID, ERR_ROW_ID, ERR_PIPE_TIMEOUT = 1, 2, 4
NOALLOC_SCRATCH_BYTES = 32 << 20   # ENGRAM_NOALLOC_SCRATCH_BYTES
INT64_MAX = (1 << 63) - 1


class EngramError(RuntimeError):
    def __init__(self, fn: str, code: int, msg: str):
        super().__init__(f"{fn} failed ({code}): {msg}")
        self.code = code


class EngramDims(C.Structure):
    _fields_ = [("layers", C.c_int32), ("max_ngram", C.c_int32), ("n_heads", C.c_int32),
                ("head_dim", C.c_int32), ("hidden", C.c_int32), ("hc", C.c_int32),
                ("raw_vocab", C.c_int32), ("compressed_vocab", C.c_int32), ("pad_id", C.c_int32),
                ("eps", C.c_float), ("clamp", C.c_float)]

    @property
    def cols(self) -> int:
        return (self.max_ngram - 1) * self.n_heads


class _LayerWeights(C.Structure):
    _fields_ = [("table_format", C.c_int32), ("table", C.c_void_p), ("table_scales", C.c_void_p),
                ("table_rows", C.c_int64), ("wkv", C.c_void_p), ("q_weight", C.c_void_p),
                ("k_weight", C.c_void_p), ("wkv_format", C.c_int32), ("wkv_scales", C.c_void_p)]


class _HashTables(C.Structure):
    _fields_ = [("token_map", C.c_void_p), ("multipliers", C.c_void_p), ("primes", C.c_void_p),
                ("offsets", C.c_void_p)]


class ProjectPlan(C.Structure):
    """engram_project_plan's answer (see include/engram.h, EngramProjectPlan)."""
    _fields_ = [(n, C.c_int32) for n in ("grid", "threads", "smem_bytes", "tile_rows", "tile_cols", "split",
                                          "token_rows_loaded", "stages", "stage_bytes", "tmem_cols", "stream_k",
                                          "mma_read_end", "smem_avail")]

    def as_dict(self) -> dict:
        return {n: getattr(self, n) for n, _ in self._fields_}


class _Tokens(C.Structure):
    _fields_ = [("input_ids", C.c_void_p), ("T", C.c_int64), ("cu_seqlens", C.c_void_p),
                ("num_seqs", C.c_int32), ("sequence_ids", C.c_void_p), ("token_mask", C.c_void_p),
                ("lookback_ids", C.c_void_p)]


_lib = None
P, I32, I64, SZ = C.c_void_p, C.c_int32, C.c_int64, C.c_size_t


def lib() -> C.CDLL:
    """The loaded CUDA library.  Raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"libengram.so not built ({LIB_PATH}); run "
                               "`python -m engram_gram_hash_02_gb300.build`")
        L = C.CDLL(LIB_PATH)
        L.engram_last_error.restype = C.c_char_p
        L.engram_version.restype = C.c_char_p
        L.engram_layout.argtypes = [I64, I32, I32, I32, P, P, P]
        L.engram_hash.argtypes = [P, P, I64, P, I32, P, P, P, P, P, P, P, P, P, P]
        L.engram_gather_dequant.argtypes = [I32, P, I64, I64, I32, I32, P, P, I64, P, P, P]
        L.engram_project.argtypes = [P, P, P, I64, I32, I32, P, SZ, P, P]
        L.engram_gate.argtypes = [P, P, P, P, P, P, I64, P, P]
        L.engram_forward_workspace_bytes.argtypes = [P, I64]
        L.engram_forward_workspace_bytes.restype = SZ
        L.engram_forward.argtypes = [P, P, P, P, P, P, SZ, P, P, P]
        L.engram_forward_noalloc.argtypes = [P, P, P, P, P, P, P, P]
        L.engram_forward2.argtypes = [P, P, P, P, P, P, SZ, P, P, P, P]
        L.engram_set_gemm_tile.argtypes = [I32]
        L.engram_set_gemm_tile.restype = None
        L.engram_set_gemm_schedule.argtypes = [I32]
        L.engram_set_gemm_schedule.restype = None
        L.engram_project_workspace_bytes.argtypes = [I64, I32, I32]
        L.engram_project_workspace_bytes.restype = SZ
        L.engram_quantize_mxfp8.argtypes = [P, I64, I32, P, P, P]
        L.engram_gather_fp8_codes.argtypes = [P, I64, I64, I32, I32, P, P, I64, P, P, P, P]
        L.engram_project_mxfp8.argtypes = [P, P, P, P, P, I64, I32, I32, P, P]
        L.engram_set_gemm_mx_tile.argtypes = [I32]
        L.engram_set_gemm_mx_tile.restype = None
        L.engram_sync_status.argtypes = [P, P]
        L.engram_set_gate_form.argtypes = [I32]
        L.engram_set_gate_form.restype = None
        L.engram_set_gate_fusion.argtypes = [I32]
        L.engram_set_gate_fusion.restype = None
        L.engram_set_operand_gather.argtypes = [I32]
        L.engram_set_operand_gather.restype = None
        L.engram_set_gather_order.argtypes = [I32]
        L.engram_set_gather_order.restype = None
        L.engram_project_plan.argtypes = [I64, I32, I32, I32, I32, P]
        _lib = L
    return _lib


def _check(fn: str, rc: int):
    if rc != 0:
        raise EngramError(fn, rc, lib().engram_last_error().decode())


def _ptr(t) -> int | None:
    return None if t is None else t.data_ptr()


def _dev(t: torch.Tensor, dtype, name: str) -> torch.Tensor:
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype} (got {t.dtype})")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t


def _opt(t, dtype, name):
    return None if t is None else _dev(t, dtype, name)


def _stream(stream) -> int | None:
    s = torch.cuda.current_stream() if stream is None else stream
    return s.cuda_stream


def _u16(t: torch.Tensor, name: str) -> torch.Tensor:
    """bf16 tensors cross the C boundary as their bit patterns."""
    return _dev(t, torch.bfloat16, name)


def _shape(t, shape, name: str):
    """The kernels index every tensor by the sizes they are given: a tensor of another shape is
    read or written past its end, so shapes are checked here (before any device check)."""
    if t is None:
        return
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if tuple(t.shape) != tuple(int(x) for x in shape):
        raise ValueError(f"{name} must have shape {tuple(int(x) for x in shape)} (got {tuple(t.shape)})")


def _numel_at_least(t, n: int, name: str):
    if t is not None and t.numel() * t.element_size() < n:
        raise ValueError(f"{name} holds {t.numel() * t.element_size()} bytes, needs at least {n}")


def _table_shape_check(fmt: str, table, scales, num_rows: int, head_dim: int, where: str):
    if int(num_rows) < 0:
        raise ValueError(f"{where}: num_rows must be >= 0")
    row_bytes = {"fp8": head_dim, "q2k": 84, "bf16": 2 * head_dim}[fmt]
    _numel_at_least(table, int(num_rows) * row_bytes, f"{where}: table")
    if fmt == "fp8":
        if scales is None:
            raise ValueError(f"{where}: an FP8 table needs its scales")
        _numel_at_least(scales, int(num_rows) * (head_dim // 32), f"{where}: table scales")


# ---------------------------------------------------------------------------------------------
# host-side setup
# ---------------------------------------------------------------------------------------------

def engram_layout(vocab_size: int, layers: int, max_ngram: int, n_heads: int):
    """Prime bucket sizes, offsets and rows per layer (computed by the library on the host)."""
    cols = (max_ngram - 1) * n_heads
    primes = np.zeros((layers, cols), dtype=np.int64)
    offsets = np.zeros((layers, cols), dtype=np.int64)
    rows = np.zeros(layers, dtype=np.int64)
    _check("engram_layout", lib().engram_layout(vocab_size, layers, max_ngram, n_heads,
                                                 primes.ctypes.data, offsets.ctypes.data, rows.ctypes.data))
    return primes, offsets, rows


def hash_multipliers(layer_ids, max_ngram: int, compressed_vocab: int) -> np.ndarray:
    """Odd multiplier per (layer, window slot): 2x+1 with x drawn by numpy's default_rng
    seeded 10007*layer_id in [0, max(1, (INT64_MAX // V) // 2)), as the vLLM page's
    compute_hash_multipliers defines them (host setup, once per model)."""
    bound = max(1, (INT64_MAX // int(compressed_vocab)) // 2)
    out = np.empty((len(layer_ids), max_ngram), dtype=np.int64)
    for i, layer_id in enumerate(layer_ids):
        x = np.random.default_rng(10007 * int(layer_id)).integers(0, bound, size=(max_ngram,), dtype=np.int64)
        out[i] = x * 2 + 1
    return out


def make_dims(layers, max_ngram, n_heads, head_dim, hidden, hc, raw_vocab, compressed_vocab,
              pad_id, eps=1e-6, clamp=1e-6) -> EngramDims:
    return EngramDims(layers, max_ngram, n_heads, head_dim, hidden, hc, raw_vocab,
                      compressed_vocab, pad_id, eps, clamp)


# ---------------------------------------------------------------------------------------------
# stages
# ---------------------------------------------------------------------------------------------

def engram_hash(dims: EngramDims, input_ids, token_map, multipliers, primes, offsets, cu_seqlens=None,
                sequence_ids=None, token_mask=None, lookback_ids=None, out=None, err=None, stream=None):
    T = input_ids.numel()
    S = 1 if cu_seqlens is None else cu_seqlens.numel() - 1
    _shape(token_map, (dims.raw_vocab,), "token_map")
    _shape(multipliers, (dims.layers, dims.max_ngram), "multipliers")
    _shape(primes, (dims.layers, dims.cols), "primes")
    _shape(offsets, (dims.layers, dims.cols), "offsets")
    _shape(sequence_ids, (T,), "sequence_ids")
    _shape(token_mask, (T,), "token_mask")
    _shape(lookback_ids, (S, dims.max_ngram - 1), "lookback_ids")
    _shape(out, (T, dims.layers, dims.cols), "out")
    _dev(input_ids, torch.int32, "input_ids")
    _dev(token_map, torch.int32, "token_map")
    _dev(multipliers, torch.int64, "multipliers")
    _dev(primes, torch.int64, "primes")
    _dev(offsets, torch.int64, "offsets")
    _opt(cu_seqlens, torch.int32, "cu_seqlens")
    _opt(sequence_ids, torch.int32, "sequence_ids")
    _opt(token_mask, torch.uint8, "token_mask")
    _opt(lookback_ids, torch.int32, "lookback_ids")
    _opt(err, torch.int32, "err")
    if out is None:
        out = torch.empty((T, dims.layers, dims.cols), dtype=torch.int32, device=input_ids.device)
    _dev(out, torch.int32, "out")
    _check("engram_hash", lib().engram_hash(
        C.byref(dims), _ptr(input_ids), T, _ptr(cu_seqlens), S, _ptr(sequence_ids), _ptr(token_mask),
        _ptr(lookback_ids), _ptr(token_map), _ptr(multipliers), _ptr(primes), _ptr(offsets), _ptr(out),
        _ptr(err), _stream(stream)))
    return out


def engram_gather_dequant(fmt: str, ids, table, scales, num_rows: int, head_dim: int, out=None, err=None,
                          stream=None):
    """ids: int32 [T, C] (a strided view [T, L, C][:, l] is fine: rows must have unit column stride)."""
    if not (isinstance(ids, torch.Tensor) and ids.dim() == 2):
        raise ValueError("ids must be a [T, C] tensor")
    T, Cc = ids.shape
    code = TABLE_FORMATS[fmt]
    _table_shape_check(fmt, table, scales, num_rows, head_dim, "engram_gather_dequant")
    _shape(out, (T, Cc * head_dim), "out")
    if not (ids.is_cuda and ids.dtype == torch.int32 and ids.stride(1) == 1):
        raise ValueError("ids must be a CUDA int32 [T, C] tensor with unit column stride")
    if not (table.is_cuda and table.is_contiguous()):
        raise ValueError("table must be a contiguous CUDA tensor")
    if scales is not None:
        _dev(scales, torch.uint8, "scales")
    if out is None:
        out = torch.empty((T, Cc * head_dim), dtype=torch.bfloat16, device=ids.device)
    _u16(out, "out")
    _opt(err, torch.int32, "err")
    _check("engram_gather_dequant", lib().engram_gather_dequant(
        code, _ptr(ids), ids.stride(0), T, Cc, head_dim, _ptr(table), _ptr(scales), int(num_rows), _ptr(out),
        _ptr(err), _stream(stream)))
    return out


def engram_project(A, wkv, out=None, err=None, workspace="auto", stream=None):
    """workspace: a uint8 CUDA tensor, None (no workspace), or "auto" (allocated at the size
    engram_project_workspace_bytes asks for)."""
    if A.dim() != 2 or wkv.dim() != 2:
        raise ValueError("A and wkv must be 2-D")
    T, K = A.shape
    N, K2 = wkv.shape
    if K != K2:
        raise ValueError(f"A is [T, {K}] but wkv is [{N}, {K2}]")
    _shape(out, (T, N), "out")
    _u16(A, "A")
    _u16(wkv, "wkv")
    if out is None:
        out = torch.empty((T, N), dtype=torch.float32, device=A.device)
    _dev(out, torch.float32, "out")
    _opt(err, torch.int32, "err")
    if isinstance(workspace, str):
        nbytes = project_workspace_bytes(T, K, N) if T > 0 else 0
        workspace = torch.empty(nbytes, dtype=torch.uint8, device=A.device) if nbytes else None
    ws_bytes = 0 if workspace is None else workspace.numel()
    _check("engram_project", lib().engram_project(_ptr(A), _ptr(wkv), _ptr(out), T, K, N, _ptr(workspace), ws_bytes,
                                                   _ptr(err), _stream(stream)))
    return out


def engram_gate(dims: EngramDims, streams, kv, q_weight, k_weight, token_mask=None, err=None, stream=None):
    """Updates ``streams`` (fp32 [T, hc, H]) in place and returns it."""
    if not isinstance(streams, torch.Tensor) or streams.dim() != 3:
        raise ValueError("streams must be a [T, hc, H] tensor")
    T = streams.shape[0]
    _shape(streams, (T, dims.hc, dims.hidden), "streams")
    _shape(kv, (T, dims.hidden * (dims.hc + 1)), "kv")
    _shape(q_weight, (dims.hc, dims.hidden), "q_weight")
    _shape(k_weight, (dims.hc, dims.hidden), "k_weight")
    _shape(token_mask, (T,), "token_mask")
    _dev(streams, torch.float32, "streams")
    _dev(kv, torch.float32, "kv")
    _u16(q_weight, "q_weight")
    _u16(k_weight, "k_weight")
    _opt(token_mask, torch.uint8, "token_mask")
    _opt(err, torch.int32, "err")
    _check("engram_gate", lib().engram_gate(C.byref(dims), _ptr(streams), _ptr(kv), _ptr(q_weight),
                                             _ptr(k_weight), _ptr(token_mask), T, _ptr(err), _stream(stream)))
    return streams


def set_gemm_tile(bn: int = 0):
    lib().engram_set_gemm_tile(int(bn))


def set_gemm_schedule(s: int = 0):
    """0 automatic, 1 data-parallel tiles, 2 stream-K (when the workspace allows)."""
    lib().engram_set_gemm_schedule(int(s))


def mx_scale_shape(rows: int, K: int):
    """Shape of an MXFP8 scale array: [ceil(K/128), rows rounded up to 4, 4] bytes; byte
    (kb, r, j) is the scale of row r's block of 32 columns 4*kb + j."""
    return ((K // 32 + 3) // 4, (rows + 3) // 4 * 4, 4)


def quantize_mxfp8(w: torch.Tensor, codes=None, scales=None, stream=None):
    """bf16 [N, K] -> (e4m3 codes uint8 [N, K], scales uint8 ``mx_scale_shape(N, K)``)
    (engram_quantize_mxfp8)."""
    _u16(w, "w")
    N, K = w.shape
    _shape(codes, (N, K), "codes")
    _shape(scales, mx_scale_shape(N, K), "scales")
    codes = torch.empty(N, K, dtype=torch.uint8, device=w.device) if codes is None else _dev(codes, torch.uint8, "codes")
    scales = (torch.empty(mx_scale_shape(N, K), dtype=torch.uint8, device=w.device) if scales is None
              else _dev(scales, torch.uint8, "scales"))
    _check("engram_quantize_mxfp8", lib().engram_quantize_mxfp8(_ptr(w), N, K, _ptr(codes), _ptr(scales),
                                                               _stream(stream)))
    return codes, scales


def engram_gather_fp8_codes(ids, table, table_scales, num_rows: int, head_dim: int, codes=None, scales=None,
                            err=None, stream=None):
    """FP8 rows by id without dequantisation. ids int32 [T, C] (or a [T, L*C] slice: the row
    stride is ids.stride(0)) -> (codes uint8 [T, C*head_dim], scales ``mx_scale_shape(T, C*head_dim)``)."""
    if not (isinstance(ids, torch.Tensor) and ids.dim() == 2):
        raise ValueError("ids must be a [T, C] tensor")
    T, Cc = ids.shape
    _table_shape_check("fp8", table, table_scales, num_rows, head_dim, "engram_gather_fp8_codes")
    _shape(codes, (T, Cc * head_dim), "codes")
    _shape(scales, mx_scale_shape(T, Cc * head_dim), "scales")
    if ids.dtype != torch.int32 or not ids.is_cuda or ids.stride(1) != 1:
        raise ValueError("ids must be a CUDA int32 tensor with unit column stride")
    _dev(table, torch.uint8, "table")
    _dev(table_scales, torch.uint8, "table_scales")
    _opt(err, torch.int32, "err")
    codes = (torch.empty(T, Cc * head_dim, dtype=torch.uint8, device=ids.device) if codes is None
             else _dev(codes, torch.uint8, "codes"))
    scales = (torch.empty(mx_scale_shape(T, Cc * head_dim), dtype=torch.uint8, device=ids.device) if scales is None
              else _dev(scales, torch.uint8, "scales"))
    _check("engram_gather_fp8_codes", lib().engram_gather_fp8_codes(
        _ptr(ids), ids.stride(0), T, Cc, head_dim, _ptr(table), _ptr(table_scales), int(num_rows), _ptr(codes),
        _ptr(scales), _ptr(err), _stream(stream)))
    return codes, scales


def engram_project_mxfp8(a_codes, a_scales, w_codes, w_scales, out=None, err=None, stream=None):
    """kv fp32 [T, N] = A * W^T from MXFP8 operands (engram_project_mxfp8)."""
    for t, n in ((a_codes, "a_codes"), (a_scales, "a_scales"), (w_codes, "w_codes"), (w_scales, "w_scales")):
        _dev(t, torch.uint8, n)
    T, K = a_codes.shape
    N = w_codes.shape[0]
    _shape(w_codes, (N, K), "w_codes")
    _shape(a_scales, mx_scale_shape(T, K), "a_scales")
    _shape(w_scales, mx_scale_shape(N, K), "w_scales")
    _shape(out, (T, N), "out")
    out = torch.empty(T, N, dtype=torch.float32, device=a_codes.device) if out is None else _dev(out, torch.float32, "out")
    _opt(err, torch.int32, "err")
    _check("engram_project_mxfp8", lib().engram_project_mxfp8(_ptr(a_codes), _ptr(a_scales), _ptr(w_codes),
                                                             _ptr(w_scales), _ptr(out), T, K, N, _ptr(err),
                                                             _stream(stream)))
    return out


def set_gate_form(form: int = 0):
    """0 automatic, 1 persistent gate kernel, 2 one CTA per (token, stream) item."""
    lib().engram_set_gate_form(int(form))


def set_gate_fusion(mode=0):
    """How engram_forward joins the gate to the projection: 0 (or False) a separate gate kernel,
    1 (or True) the key reductions in the projection's epilogue, 2 the gate inside the projection
    kernel, overlapped with it."""
    lib().engram_set_gate_fusion(int(mode))


def set_operand_gather(on: bool = False):
    """engram_forward with the FP8 variant's projection gathering its token rows from the table."""
    lib().engram_set_operand_gather(1 if on else 0)


def set_gather_order(mode: int = 0):
    """engram_forward's gathers: 0 token order, 1 table order (rows grouped by table region)."""
    lib().engram_set_gather_order(int(mode))


def set_gemm_mx_tile(bn: int = 0):
    lib().engram_set_gemm_mx_tile(int(bn))


def project_workspace_bytes(T: int, K: int, N: int) -> int:
    return int(lib().engram_project_workspace_bytes(T, K, N))


def project_plan(T: int, K: int, N: int, wkv_format: str = "bf16", num_sms: int = 152) -> dict:
    """The tile plan the projection would launch for this shape (engram_project_plan; host
    only)."""
    out = ProjectPlan()
    fmt = {"bf16": WKV_BF16, "mxfp8": WKV_MXFP8}[wkv_format]
    _check("engram_project_plan", lib().engram_project_plan(int(T), int(K), int(N), fmt, int(num_sms), C.byref(out)))
    return out.as_dict()


def sync_status(err: torch.Tensor, stream=None) -> int:
    """engram_sync_status: waits for the stream, then 0 (err word clear), ENGRAM_EDATA (-3, an
    id out of range was substituted) or ENGRAM_ECUDA (-2).  Returns the code; the message is
    engram_last_error()."""
    _dev(err, torch.int32, "err")
    return int(lib().engram_sync_status(_ptr(err), _stream(stream)))


# ---------------------------------------------------------------------------------------------
# whole path
# ---------------------------------------------------------------------------------------------

@dataclass
class LayerWeights:
    """One layer's resident weights. ``wkv`` is bf16 [N, K], or e4m3 codes (uint8 [N, K]) with
    ``wkv_scales`` (uint8 [N, K/32]) for the FP8 variant (see ``quantize_mxfp8``)."""
    fmt: str
    table: torch.Tensor
    scales: torch.Tensor | None
    num_rows: int
    wkv: torch.Tensor
    q_weight: torch.Tensor
    k_weight: torch.Tensor
    wkv_scales: torch.Tensor | None = None


@dataclass
class HashTables:
    token_map: torch.Tensor
    multipliers: torch.Tensor
    primes: torch.Tensor
    offsets: torch.Tensor


def forward_workspace_bytes(dims: EngramDims, T: int) -> int:
    return int(lib().engram_forward_workspace_bytes(C.byref(dims), T))


def _check_forward_shapes(dims, tables, layers, input_ids, streams, cu_seqlens, sequence_ids, token_mask,
                          lookback_ids, workspace, out_ids, err):
    """Every size engram_forward reads from dims, checked against the tensors (the C side can see
    only pointers: a short list or an undersized tensor would be read or written past its end)."""
    L = int(dims.layers)
    if len(layers) != L or len(streams) != L:
        raise ValueError(f"dims.layers is {L} but {len(layers)} layer weights and {len(streams)} stream tensors "
                         "were given")
    if not isinstance(input_ids, torch.Tensor) or input_ids.dim() != 1:
        raise ValueError("input_ids must be a 1-D tensor [T]")
    T = input_ids.numel()
    H, hc, D, Cc = int(dims.hidden), int(dims.hc), int(dims.head_dim), dims.cols
    K, N = Cc * D, H * (hc + 1)
    if cu_seqlens is not None and (cu_seqlens.dim() != 1 or cu_seqlens.numel() < 2):
        raise ValueError("cu_seqlens must be a 1-D tensor [S + 1] with S >= 1")
    S = 1 if cu_seqlens is None else cu_seqlens.numel() - 1
    _shape(sequence_ids, (T,), "sequence_ids")
    _shape(token_mask, (T,), "token_mask")
    _shape(lookback_ids, (S, dims.max_ngram - 1), "lookback_ids")
    _shape(out_ids, (T, L, Cc), "out_ids")
    if err is not None and err.numel() < 1:
        raise ValueError("err must hold one int32")
    _shape(tables.token_map, (dims.raw_vocab,), "token_map")
    _shape(tables.multipliers, (L, dims.max_ngram), "multipliers")
    _shape(tables.primes, (L, Cc), "primes")
    _shape(tables.offsets, (L, Cc), "offsets")
    for i, (w, st) in enumerate(zip(layers, streams)):
        _shape(st, (T, hc, H), f"streams[{i}]")
        _shape(w.q_weight, (hc, H), f"layers[{i}].q_weight")
        _shape(w.k_weight, (hc, H), f"layers[{i}].k_weight")
        _shape(w.wkv, (N, K), f"layers[{i}].wkv")
        if w.wkv_scales is not None:
            _shape(w.wkv_scales, mx_scale_shape(N, K), f"layers[{i}].wkv_scales")
        if w.fmt not in TABLE_FORMATS:
            raise ValueError(f"layers[{i}]: unknown table format {w.fmt!r}")
        _table_shape_check(w.fmt, w.table, w.scales, w.num_rows, D, f"layers[{i}]")
    # the workspace's size reaches the library with its pointer, which refuses one that is too small


class ForwardPlan:
    """Marshalled arguments of engram_forward for fixed tensors, so a hot loop pays one
    ctypes call per step."""

    def __init__(self, dims: EngramDims, tables: HashTables, layers: list, input_ids, streams: list,
                 cu_seqlens=None, sequence_ids=None, token_mask=None, lookback_ids=None, workspace=None,
                 out_ids=None, err=None):
        self.dims = dims
        T = input_ids.numel()
        _check_forward_shapes(dims, tables, layers, input_ids, streams, cu_seqlens, sequence_ids, token_mask,
                              lookback_ids, workspace, out_ids, err)
        _dev(input_ids, torch.int32, "input_ids")
        for name, t, dt in (("cu_seqlens", cu_seqlens, torch.int32), ("sequence_ids", sequence_ids, torch.int32),
                            ("token_mask", token_mask, torch.uint8), ("lookback_ids", lookback_ids, torch.int32),
                            ("out_ids", out_ids, torch.int32), ("err", err, torch.int32)):
            _opt(t, dt, name)
        self._tables = _HashTables(_ptr(tables.token_map), _ptr(tables.multipliers), _ptr(tables.primes),
                                   _ptr(tables.offsets))
        arr = (_LayerWeights * len(layers))()
        for i, w in enumerate(layers):
            mx = w.wkv_scales is not None
            if mx:
                _dev(w.wkv, torch.uint8, "wkv (MXFP8 codes)")
                _dev(w.wkv_scales, torch.uint8, "wkv_scales")
            arr[i] = _LayerWeights(TABLE_FORMATS[w.fmt], _ptr(w.table), _ptr(w.scales), int(w.num_rows),
                                   _ptr(w.wkv), _ptr(w.q_weight), _ptr(w.k_weight), WKV_MXFP8 if mx else WKV_BF16,
                                   _ptr(w.wkv_scales))
            _dev(streams[i], torch.float32, f"streams[{i}]")
        self._layers = arr
        S = 1 if cu_seqlens is None else cu_seqlens.numel() - 1
        self._tokens = _Tokens(_ptr(input_ids), T, _ptr(cu_seqlens), S, _ptr(sequence_ids), _ptr(token_mask),
                               _ptr(lookback_ids))
        self._streams = (C.c_void_p * len(streams))(*[s.data_ptr() for s in streams])
        need = forward_workspace_bytes(dims, T)
        if workspace is None:
            # the minimum plus the projection's stream-K scratch
            K, N = dims.cols * dims.head_dim, dims.hidden * (dims.hc + 1)
            need += project_workspace_bytes(T, K, N) if T > 0 else 0
            workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=input_ids.device)
        self.workspace = workspace
        self._ws_bytes = workspace.numel() * workspace.element_size()
        self._out_ids = out_ids
        self._err = err
        self._keep = (tables, layers, input_ids, streams, cu_seqlens, sequence_ids, token_mask, lookback_ids)

    def run(self, stream=None, side_stream=None):
        """engram_forward on `stream` (default: the current stream); with `side_stream`,
        engram_forward2 (the later layers' gathers on the side stream)."""
        if side_stream is not None:
            _check("engram_forward2", lib().engram_forward2(
                C.byref(self.dims), C.byref(self._tables), self._layers, C.byref(self._tokens), self._streams,
                _ptr(self.workspace), self._ws_bytes, _ptr(self._out_ids), _ptr(self._err), _stream(stream),
                side_stream.cuda_stream))
            return
        _check("engram_forward", lib().engram_forward(
            C.byref(self.dims), C.byref(self._tables), self._layers, C.byref(self._tokens), self._streams,
            _ptr(self.workspace), self._ws_bytes, _ptr(self._out_ids), _ptr(self._err), _stream(stream)))


    def run_noalloc(self, stream=None):
        """The same pass through engram_forward_noalloc: scratch in the library's static device
        array instead of self.workspace (for callers that may not allocate)."""
        _check("engram_forward_noalloc", lib().engram_forward_noalloc(
            C.byref(self.dims), C.byref(self._tables), self._layers, C.byref(self._tokens), self._streams,
            _ptr(self._out_ids), _ptr(self._err), _stream(stream)))


def engram_forward(dims: EngramDims, tables: HashTables, layers: list, input_ids, streams: list, **kw):
    """Hash once, then per layer gather -> project -> gate (streams updated in place)."""
    stream = kw.pop("stream", None)
    plan = ForwardPlan(dims, tables, layers, input_ids, streams, **kw)
    plan.run(stream)
    return plan
