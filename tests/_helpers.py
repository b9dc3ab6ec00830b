"""Shared test plumbing: build a workload on both sides (CUDA path via the product binding,
oracle via oracle/), run them, and compare."""
from __future__ import annotations

import numpy as np
import torch

from engram_synth import get_workload
from engram_synth.case import make_case, to_device
from oracle import engram_oracle as O

# Gated-stream tolerance against the fp64 oracle fed the same bf16 operands.
STREAM_MAX_ABS = 2e-3
STREAM_REL_L2 = 1e-3
UPDATE_REL_L2 = 1e-2


def bits16(t: torch.Tensor) -> np.ndarray:
    """bf16 tensor -> numpy uint16 bit patterns (host)."""
    return t.detach().contiguous().cpu().view(torch.int16).numpy().view(np.uint16)


def oracle_setup(w):
    primes, offsets, rows = O.layout(w.vocab_size, w.layers, w.max_ngram, w.n_heads)
    mult = O.hash_multipliers(w.layer_ids, w.max_ngram, w.compressed_vocab)
    return primes, offsets, rows, mult


def product_setup(w):
    import engram_gram_hash_02_gb300 as E
    primes, offsets, rows = E.engram_layout(w.vocab_size, w.layers, w.max_ngram, w.n_heads)
    mult = E.hash_multipliers(w.layer_ids, w.max_ngram, w.compressed_vocab)
    return primes, offsets, rows, mult


def pad_id_of(w, token_map):
    return int(token_map[w.pad_token_id])


def dims_for(w, pad_id):
    import engram_gram_hash_02_gb300 as E
    return E.make_dims(w.layers, w.max_ngram, w.n_heads, w.head_dim, w.hidden, w.hc, w.raw_vocab,
                       w.compressed_vocab, pad_id, w.eps, w.clamp)


def oracle_dims(w, pad_id):
    return {"max_ngram": w.max_ngram, "n_heads": w.n_heads, "head_dim": w.head_dim, "hidden": w.hidden,
            "hc": w.hc, "compressed_vocab": w.compressed_vocab, "pad_id": pad_id, "eps": w.eps,
            "clamp": w.clamp}


def build(name_or_w, device="cuda", seq_lens=None, seed=None):
    w = get_workload(name_or_w) if isinstance(name_or_w, str) else name_or_w
    if seq_lens is not None:
        w = w.with_tokens(seq_lens)
    primes, offsets, rows, mult = product_setup(w)
    case = make_case(w, rows, device, seed)
    return w, case, (primes, offsets, rows, mult)


def _per_layer(flag, layers: int) -> list:
    return [bool(f) for f in flag] if isinstance(flag, (list, tuple)) else [bool(flag)] * layers


def a_slot_bytes(T: int, K: int) -> int:
    """One layer's operand slot in the engram_forward workspace: bf16 rows [T, K], or the FP8
    variant's codes [T, K] then (256-byte aligned) scale words [ceil(K/128), T4, 4]."""
    r256 = lambda x: (x + 255) // 256 * 256
    return r256(max(T * K * 2, r256(T * K) + (K + 127) // 128 * ((T + 3) // 4 * 4) * 4))


def gpu_forward(w, case, setup, device="cuda", with_err=True, mx=False, side=False):
    """Run engram_forward on the device; returns ids, per-layer streams, the workspace views.
    With ``mx`` (a bool, or one per layer) the layers carry MXFP8 wkv (quantised on the device)
    and the FP8 variant runs for them."""
    import engram_gram_hash_02_gb300 as E
    primes, offsets, rows, mult = setup
    b = case.batch
    pad = pad_id_of(w, b["token_map"])
    dims = dims_for(w, pad)
    tables = E.HashTables(to_device(b["token_map"], device), to_device(mult, device),
                          to_device(primes, device), to_device(offsets, device))
    mxl = _per_layer(mx, w.layers)
    layers = []
    for l, t in enumerate(case.tables):
        wkv, wsc = case.wkv[l], None
        if mxl[l]:
            wkv, wsc = E.quantize_mxfp8(case.wkv[l])
        layers.append(E.LayerWeights(t["fmt"], t["table"], t["scales"], t["num_rows"], wkv, case.q_weight[l],
                                     case.k_weight[l], wkv_scales=wsc))
    streams = [s.clone() for s in case.streams]
    err = torch.zeros(1, dtype=torch.int32, device=device) if with_err else None
    out_ids = torch.empty((w.tokens, w.layers, w.cols), dtype=torch.int32, device=device)
    plan = E.ForwardPlan(dims, tables, layers, to_device(b["input_ids"], device), streams,
                         cu_seqlens=to_device(b["cu_seqlens"], device),
                         sequence_ids=to_device(b["sequence_ids"], device),
                         token_mask=to_device(b["token_mask"], device),
                         lookback_ids=to_device(b["lookback_ids"], device), out_ids=out_ids, err=err)
    # with `side`, engram_forward2: the later layers' gathers on a second stream
    plan.run(side_stream=torch.cuda.Stream(device) if side else None)
    torch.cuda.synchronize()
    ws = plan.workspace
    T, K, N, L = w.tokens, w.K, w.N, w.layers
    id_bytes = ((T * L * w.cols * 4 + 255) // 256) * 256
    slot = a_slot_bytes(T, K)
    kv0 = id_bytes + L * slot
    kv_last = ws[kv0:kv0 + T * N * 4].view(torch.float32).view(T, N)
    out = {"ids": out_ids, "streams": streams, "kv_last": kv_last, "err": int(err.item()) if err is not None else 0,
           "dims": dims, "A": [], "A_codes": [], "A_scales": []}
    # every layer's gathered operand stays in its slot
    code_bytes = ((T * K + 255) // 256) * 256
    shp = E.mx_scale_shape(T, K)
    for l in range(L):
        a0 = id_bytes + l * slot
        if mxl[l]:
            out["A"].append(None)
            out["A_codes"].append(ws[a0:a0 + T * K].view(T, K))
            sc = ws[a0 + code_bytes:a0 + code_bytes + shp[0] * shp[1] * shp[2]].view(shp)
            out["A_scales"].append(mx_words_to_rows(sc, T, K // 32))
        else:
            out["A"].append(ws[a0:a0 + T * K * 2].view(torch.bfloat16).view(T, K))
            out["A_codes"].append(None)
            out["A_scales"].append(None)
    if mxl[-1]:
        out["A_codes_last"], out["A_scales_last"] = out["A_codes"][-1], out["A_scales"][-1]
    else:
        out["A_last"] = out["A"][-1]
    return out


def mx_words_to_rows(sc: torch.Tensor, rows: int, nblk: int) -> np.ndarray:
    """MXFP8 scales in the projection's word layout [ceil(nblk/4), rows4, 4] -> bytes [rows, nblk]
    (the oracle's layout)."""
    a = sc.detach().cpu().numpy()
    return a.transpose(1, 0, 2).reshape(a.shape[1], -1)[:rows, :nblk]


def mx_rows_to_words(sc_rows: np.ndarray) -> np.ndarray:
    """Bytes [rows, nblk] -> the word layout [ceil(nblk/4), rows4, 4] (pad entries 127)."""
    R, nb = sc_rows.shape
    R4, nb4 = (R + 3) // 4 * 4, (nb + 3) // 4 * 4
    pad = np.full((R4, nb4), 127, dtype=np.uint8)
    pad[:R, :nb] = sc_rows
    return np.ascontiguousarray(pad.reshape(R4, nb4 // 4, 4).transpose(1, 0, 2))


def oracle_mxfp8_quantize(wkv: torch.Tensor, rows: int = 2048):
    """The oracle's MXFP8 encoding of a bf16 weight, a block of rows at a time (rows are
    independent; this bounds the fp64 temporaries)."""
    bits = bits16(wkv)
    parts = [O.mxfp8_quantize(bits[i:i + rows]) for i in range(0, bits.shape[0], rows)]
    return np.concatenate([p[0] for p in parts]), np.concatenate([p[1] for p in parts])


def compact_table(tab: dict, ids: np.ndarray):
    """Fetch only the rows ``ids`` touch from a device table; remap ids into the compact copy
    (out-of-range ids stay out of range).  Returns (table_np, scales_np, remapped, num_rows)."""
    flat = ids.reshape(-1)
    ok = (flat >= 0) & (flat < tab["num_rows"])
    uniq, inv = np.unique(flat[ok], return_inverse=True)
    idx = torch.from_numpy(uniq.astype(np.int64)).to(tab["table"].device)
    t = tab["table"].index_select(0, idx).cpu()
    if tab["fmt"] == "bf16":
        t_np = t.view(torch.int16).numpy().view(np.uint16)
    else:
        t_np = t.numpy()
    s_np = tab["scales"].index_select(0, idx).cpu().numpy() if tab["scales"] is not None else None
    remap = np.full(flat.shape, -1, dtype=np.int64)
    remap[ok] = inv
    return t_np, s_np, remap.reshape(ids.shape), len(uniq)


def oracle_forward(w, case, tokens=None, mx=False):
    """The oracle's whole path on the selected tokens (all if None), from its own layout. With
    ``mx`` (a bool, or one per layer), the FP8 variant: raw FP8 rows and the oracle's own MXFP8
    encoding of wkv."""
    primes, offsets, rows, mult = oracle_setup(w)
    b = case.batch
    pad = pad_id_of(w, b["token_map"])
    win, bad = O.windows(b["input_ids"], b["token_map"], pad, w.max_ngram, b["cu_seqlens"], b["sequence_ids"],
                         b["token_mask"], b["lookback_ids"])
    ids = O.hash_ids(win, mult, primes, offsets, w.compressed_vocab)
    T = ids.shape[0]
    sel = np.arange(T) if tokens is None else np.asarray(tokens, dtype=np.int64)
    mask = b["token_mask"]
    mxl = _per_layer(mx, w.layers)
    layers = []
    for l, tab in enumerate(case.tables):
        t_np, s_np, remap, nrows = compact_table(tab, ids[sel, l, :])
        if mxl[l]:
            codes, sc, n_oob = O.gather_fp8_raw(t_np, s_np, remap, nrows)
            wc, ws_ = oracle_mxfp8_quantize(case.wkv[l])
            kv = O.project_mxfp8(codes, sc, wc, ws_)
            a_bits = (codes, sc)
        else:
            a_bits, n_oob = O.gather(tab["fmt"], t_np, s_np, remap, nrows, w.head_dim)
            kv = O.project(a_bits, bits16(case.wkv[l]))
        h0 = case.streams[l][torch.from_numpy(sel).to(case.streams[l].device)].cpu().numpy()
        out, g = O.gate(h0, kv, bits16(case.q_weight[l]), bits16(case.k_weight[l]), w.eps, w.clamp,
                        None if mask is None else mask[sel])
        layers.append({"a_bits": a_bits, "kv": kv, "streams": out, "streams_in": h0, "gate": g})
    return {"ids": ids, "bad_raw": int(bad.sum()), "tokens": sel, "layers": layers}


def check_streams(got: np.ndarray, ref: np.ndarray, h0: np.ndarray, what=""):
    d = got.astype(np.float64) - ref
    max_abs = float(np.abs(d).max()) if d.size else 0.0
    rel = float(np.linalg.norm(d) / max(np.linalg.norm(ref), 1e-30))
    upd_ref = ref - h0
    upd_rel = float(np.linalg.norm((got - h0) - upd_ref) / max(np.linalg.norm(upd_ref), 1e-30))
    assert max_abs <= STREAM_MAX_ABS, f"{what}: max|d| {max_abs:.3g}"
    assert rel <= STREAM_REL_L2, f"{what}: rel-L2 {rel:.3g}"
    if np.linalg.norm(upd_ref) > 0:
        assert upd_rel <= UPDATE_REL_L2, f"{what}: update rel-L2 {upd_rel:.3g}"
    return max_abs, rel, upd_rel


def check_kv(got, ref: np.ndarray, what=""):
    """fp32 kv from the tensor cores against the fp64 product of the same bf16 operands.
    Products of bf16 values are exact in fp32; what remains is fp32 summation over K terms:
    a random walk of about sqrt(K) * 2^-24 * rms (~5e-6 rms at K = 6144). The bound allows
    20x that plus 2^-14 relative."""
    g = np.asarray(got, dtype=np.float64)
    rms = float(np.sqrt(np.mean(ref * ref))) if ref.size else 0.0
    tol = 2.0 ** -14 * np.abs(ref) + 1e-4 * rms
    bad = np.abs(g - ref) > tol
    assert not bad.any(), f"{what}: {int(bad.sum())} of {bad.size} kv outside tolerance; worst {float(np.abs(g - ref).max()):.3g}"
