"""Seeded generators for every input of the Engram hot path.

Every function takes an explicit seed.  Sub-streams are keyed by a small tag so
two tensors of one workload never share random numbers.
"""
from __future__ import annotations

import numpy as np
import torch

# per-tensor sub-stream tags
_T_IDS, _T_MAP, _T_DOCS, _T_MASK, _T_LOOKBACK = 1, 2, 3, 4, 5
_T_TABLE, _T_WKV, _T_QK, _T_STREAMS = 10, 20, 30, 40


def _np_rng(seed: int, tag: int) -> np.random.Generator:
    return np.random.default_rng([int(seed), int(tag)])


def _torch_gen(seed: int, tag: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed) * 1_000_003 + int(tag))
    return g


# --------------------------------------------------------------------------
# token ids, maps, documents, masks, lookback
# --------------------------------------------------------------------------

def token_map(raw_vocab: int, compressed_vocab: int, kind: str, seed: int) -> np.ndarray:
    """A seeded map raw id -> compressed id, standing in for the tokenizer
    normalisation map.  'permutation' needs raw_vocab == compressed_vocab;
    'surjection' permutes the first compressed_vocab raw ids onto every
    compressed id and sends the rest to uniform compressed ids."""
    rng = _np_rng(seed, _T_MAP)
    if kind == "permutation":
        if raw_vocab != compressed_vocab:
            raise ValueError("a permutation map needs raw_vocab == compressed_vocab")
        return rng.permutation(compressed_vocab).astype(np.int32)
    if kind != "surjection" or raw_vocab < compressed_vocab:
        raise ValueError(f"bad token map kind {kind!r} for {raw_vocab}->{compressed_vocab}")
    head = rng.permutation(compressed_vocab)
    tail = rng.integers(0, compressed_vocab, size=raw_vocab - compressed_vocab)
    return np.concatenate([head, tail]).astype(np.int32)


def zipf_ids(n: int, vocab: int, alpha: float, rng: np.random.Generator) -> np.ndarray:
    """n raw ids with P(rank r) proportional to r**-alpha on ranks 1..vocab;
    ranks are sent to ids through a seeded permutation."""
    ranks = np.arange(1, vocab + 1, dtype=np.float64)
    cdf = np.cumsum(ranks ** (-alpha))
    cdf /= cdf[-1]
    r = np.searchsorted(cdf, rng.random(n), side="right")
    r = np.minimum(r, vocab - 1)
    perm = rng.permutation(vocab)
    return perm[r].astype(np.int32)


def batch_inputs(w, seed: int | None = None) -> dict:
    """Per-call token inputs of a workload, as numpy arrays (host)."""
    seed = w.seed if seed is None else seed
    T = w.tokens
    S = len(w.seq_lens)
    O = w.max_ngram - 1
    rng = _np_rng(seed, _T_IDS)
    if w.id_dist == "zipf":
        ids = zipf_ids(T, w.raw_vocab, w.zipf_alpha, rng)
    else:
        ids = rng.integers(0, w.raw_vocab, size=T).astype(np.int32)
    cu = np.zeros(S + 1, dtype=np.int32)
    cu[1:] = np.cumsum(np.asarray(w.seq_lens, dtype=np.int64))
    out = {"input_ids": ids, "cu_seqlens": cu, "sequence_ids": None,
           "token_mask": None, "lookback_ids": None,
           "token_map": token_map(w.raw_vocab, w.compressed_vocab, w.map_kind, seed)}
    if w.docs_per_seq is not None:
        drng = _np_rng(seed, _T_DOCS)
        sid = np.zeros(T, dtype=np.int32)
        lo, hi = w.docs_per_seq
        for s in range(S):
            a, b = int(cu[s]), int(cu[s + 1])
            L = b - a
            nd = int(drng.integers(lo, hi + 1))
            nd = max(1, min(nd, L))
            cuts = np.sort(drng.choice(np.arange(1, L), size=nd - 1, replace=False)) if nd > 1 else []
            doc = np.zeros(L, dtype=np.int32)
            for c in cuts:
                doc[c:] += 1
            sid[a:b] = doc + 1
        out["sequence_ids"] = sid
    if w.mask_frac > 0:
        mrng = _np_rng(seed, _T_MASK)
        out["token_mask"] = (mrng.random(T) >= w.mask_frac).astype(np.uint8)
    if w.lookback:
        lrng = _np_rng(seed, _T_LOOKBACK)
        lb = lrng.integers(0, w.compressed_vocab, size=(S, O)).astype(np.int32)
        if w.lookback_dead_frac > 0:
            dead = lrng.random((S, O)) < w.lookback_dead_frac
            lb[dead] = -1
        out["lookback_ids"] = lb
    return out


# --------------------------------------------------------------------------
# tables (drawn on the device that will hold them)
# --------------------------------------------------------------------------

def bf16_table(rows: int, dim: int, std: float, seed: int, device="cpu") -> torch.Tensor:
    g = _torch_gen(seed, _T_TABLE, device)
    t = torch.randn(rows, dim, generator=g, device=device, dtype=torch.float32)
    return (t * std).to(torch.bfloat16)


def encode_fp8_e8m0(x: torch.Tensor, block: int = 32):
    """Encode fp32 rows x [R, D] as e4m3 bytes [R, D] plus one power-of-two
    scale byte per block of 32 [R, D/32] (byte 127 = 1.0).  The scale is the
    smallest power of two that brings the block's largest magnitude to <= 448;
    values are rounded to nearest-even by torch's float8_e4m3fn cast."""
    R, D = x.shape
    xb = x.view(R, D // block, block)
    amax = xb.abs().amax(dim=-1)
    e = torch.ceil(torch.log2(torch.clamp(amax, min=1e-30) / 448.0))
    e = torch.clamp(e, -126, 127).to(torch.int32)
    scaled = torch.ldexp(xb, (-e).unsqueeze(-1).to(x.dtype))
    q = scaled.reshape(R, D).to(torch.float8_e4m3fn).view(torch.uint8)
    return q, (e + 127).to(torch.uint8)


def fp8_table(rows: int, dim: int, std: float, seed: int, device="cpu", chunk_rows: int = 1 << 20):
    """FP8-E4M3 table [rows, dim] with E8M0 scales [rows, dim/32], values
    ~N(0, std) before encoding.  Drawn in chunks to bound temporaries."""
    g = _torch_gen(seed, _T_TABLE, device)
    weight = torch.empty(rows, dim, dtype=torch.uint8, device=device)
    scales = torch.empty(rows, dim // 32, dtype=torch.uint8, device=device)
    for a in range(0, rows, chunk_rows):
        b = min(rows, a + chunk_rows)
        x = torch.randn(b - a, dim, generator=g, device=device, dtype=torch.float32) * std
        q, s = encode_fp8_e8m0(x)
        weight[a:b] = q
        scales[a:b] = s
        del x, q, s
    return weight, scales


Q2K_ROW_BYTES = 84


def q2k_table(rows: int, seed: int, device="cpu", chunk_rows: int = 1 << 21) -> torch.Tensor:
    """Q2_K rows [rows, 84]: 16 bytes of 4-bit scale/min pairs and 64 bytes of
    2-bit quants (uniform bytes), then fp16 d ~ 0.003*U(0.5,1.5) and fp16
    dmin ~ 0.002*U(0.5,1.5), little-endian."""
    g = _torch_gen(seed, _T_TABLE, device)
    out = torch.empty(rows, Q2K_ROW_BYTES, dtype=torch.uint8, device=device)
    for a in range(0, rows, chunk_rows):
        b = min(rows, a + chunk_rows)
        n = b - a
        out[a:b, :80] = torch.randint(0, 256, (n, 80), generator=g, device=device, dtype=torch.uint8)
        u = torch.rand(n, 2, generator=g, device=device, dtype=torch.float32) + 0.5
        dd = (u * torch.tensor([0.003, 0.002], device=device)).to(torch.float16)
        out[a:b, 80:84] = dd.contiguous().view(torch.uint8).view(n, 4)
    return out


def wkv_weight(N: int, K: int, std: float, seed: int, device="cpu") -> torch.Tensor:
    g = _torch_gen(seed, _T_WKV, device)
    return (torch.randn(N, K, generator=g, device=device, dtype=torch.float32) * std).to(torch.bfloat16)


def gate_weights(hc: int, H: int, std: float, seed: int, device="cpu"):
    g = _torch_gen(seed, _T_QK, device)
    q = 1.0 + std * torch.randn(hc, H, generator=g, device=device, dtype=torch.float32)
    k = 1.0 + std * torch.randn(hc, H, generator=g, device=device, dtype=torch.float32)
    return q.to(torch.bfloat16), k.to(torch.bfloat16)


def streams(T: int, hc: int, H: int, seed: int, device="cpu") -> torch.Tensor:
    g = _torch_gen(seed, _T_STREAMS, device)
    return torch.randn(T, hc, H, generator=g, device=device, dtype=torch.float32)
