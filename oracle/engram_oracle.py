"""CPU oracle of the Engram hot path (hash -> gather/dequant -> wkv -> gate).

TEST INFRASTRUCTURE ONLY.  Only the tests, ``__graft_entry__.smoke()`` and the
CPU-baseline / reference legs of ``bench.py`` may import this module.  It shares
no code with the CUDA library and never imports it; the product path does not
route through it.

Plain numpy, fp64 for floating point, written to be checked by eye against the
pages it cites:

* [Atlas] "spark_model::layers::engram_v41" rustdoc, module overview (stages 1-4).
* [NeMo]  "nemo_automodel.components.models.deepseek_v41.engram" API page.
* [vLLM]  "vllm.models.deepseek_v41.common.engram" API page (PR 59747 docs).

Readings where the pages are silent (each is stated at the function):
  - the n-gram mix is the XOR of (id * multiplier) over the window, reduced
    modulo each head's prime (the pages only say multipliers are odd and bounded
    so each product fits int64);
  - unavailable window slots (before the sequence, across a document change,
    through a masked or padding position) hold ``pad_id``;
  - the Q2_K row is the public GGML Q2_K super-block;
  - the gate's dot product is divided by sqrt(hidden).
Pins for every function live in tests/test_oracle_*.py (brute force, closed
forms, hand-built blocks, library routines).  Parity with DeepSeek's released
tables and hash is unpinned: neither is available.
"""
from __future__ import annotations

import numpy as np

INT64_MAX = (1 << 63) - 1
E8M0_BLOCK = 32
Q2K_ROW_BYTES = 84
Q2K_ROW_ELEMS = 256

# ---------------------------------------------------------------------------
# Layout: primes, offsets, multipliers
# ---------------------------------------------------------------------------


def is_prime(n: int) -> bool:
    """Deterministic Miller-Rabin for n < 2**32: trial division by the primes up
    to 37, then witnesses 2, 7 and 61.  [vLLM] ``_is_prime``.  A witness that
    is a multiple of n is skipped, so 61 itself is prime (a literal reading
    of the page's routine would call 61 composite; no table size is near it)."""
    n = int(n)
    if n < 2:
        return False
    for p in (2, 3, 5, 7, 11, 13, 17, 19, 23, 29, 31, 37):
        if n % p == 0:
            return n == p
    if n >= 1 << 32:
        raise ValueError("witness set 2, 7, 61 is only proven below 2**32")
    d, r = n - 1, 0
    while d % 2 == 0:
        d //= 2
        r += 1
    for a in (2, 7, 61):
        if a % n == 0:
            continue                  # a witness equal to n says nothing (n = 61)
        x = pow(a, d, n)
        if x == 1 or x == n - 1:
            continue
        composite = True
        for _ in range(r - 1):
            x = (x * x) % n
            if x == n - 1:
                composite = False
                break
        if composite:
            return False
    return True


def next_unused_prime(start: int, seen: set) -> int:
    """Smallest prime strictly above ``start`` not in ``seen``.
    [vLLM] ``find_next_prime``; [NeMo] ``_next_prime``."""
    c = int(start) + 1
    while not (is_prime(c) and c not in seen):
        c += 1
    return c


def layout(vocab_size: int, n_layers: int, max_ngram: int, n_heads: int):
    """Bucket layout of the hash tables.  [vLLM] ``EngramLayout.__init__``.

    For each layer, for each n-gram size 2..max_ngram, the search restarts at
    vocab_size - 1 and draws n_heads successive unused primes; no prime is used
    twice in the whole model.  Columns are ordered n-gram size major, head minor.
    Offsets are the exclusive running sum of the layer's primes, restarting at 0
    per layer.  Returns primes int64 [L, O, Hh], offsets int64 [L, O*Hh] and the
    rows each layer's table needs (the sum of its primes)."""
    O = max_ngram - 1
    primes = np.zeros((n_layers, O, n_heads), dtype=np.int64)
    seen: set = set()
    for layer in range(n_layers):
        for o in range(O):
            current = vocab_size - 1
            for h in range(n_heads):
                current = next_unused_prime(current, seen)
                seen.add(current)
                primes[layer, o, h] = current
    flat = primes.reshape(n_layers, O * n_heads)
    offsets = np.zeros_like(flat)
    offsets[:, 1:] = np.cumsum(flat, axis=1)[:, :-1]
    rows = flat.sum(axis=1)
    return primes, offsets, rows


def hash_multipliers(layer_ids, max_ngram: int, compressed_vocab: int) -> np.ndarray:
    """One odd multiplier per (layer, window slot), int64 [L, max_ngram].
    [vLLM] ``compute_hash_multipliers``: draw x uniformly in
    [0, max(1, (INT64_MAX // V) // 2)) from numpy's default_rng seeded with
    10007 * layer_id, and return 2x + 1, so id * multiplier < 2**63 for any
    compressed id below V."""
    bound = max(1, (INT64_MAX // int(compressed_vocab)) // 2)
    rows = []
    for layer_id in layer_ids:
        rng = np.random.default_rng(10007 * int(layer_id))
        x = rng.integers(0, bound, size=(max_ngram,), dtype=np.int64)
        rows.append(2 * x + 1)
    return np.stack(rows).astype(np.int64)


# ---------------------------------------------------------------------------
# Stage 1: n-gram windows and hash ids
# ---------------------------------------------------------------------------


def compressed_ids(input_ids, token_map, pad_id: int):
    """Raw tokenizer id -> compressed id through token_map.  Raw ids outside
    the map are reported and replaced by pad_id.  [vLLM] module docstring
    (token_map); [NeMo] ``DeepseekV41NgramHash`` (pad_id)."""
    ids = np.asarray(input_ids, dtype=np.int64)
    tm = np.asarray(token_map, dtype=np.int64)
    bad = (ids < 0) | (ids >= tm.shape[0])
    c = np.where(bad, pad_id, tm[np.clip(ids, 0, tm.shape[0] - 1)])
    return c, bad


def windows(input_ids, token_map, pad_id: int, max_ngram: int, cu_seqlens=None,
            sequence_ids=None, token_mask=None, lookback_ids=None):
    """Compressed ids of the window ending at each position: w[t, k] is the id
    k positions back (k = 0 is t itself), or pad_id where that slot is not
    available.  Returns (w int64 [T, max_ngram], bad_raw bool [T]).

    Reading of [NeMo] ``DeepseekV41NgramHash.forward`` ("without crossing
    document, image, or padding boundaries"; token_mask false "blocks all
    lookback through those positions"; sequence_ids zero marks padding) and of
    [vLLM] ``NgramHashState`` (lookback_token_ids precede each chunk;
    lookback_dead_mask).  Walking back from t, the walk stops at the first
    position that is dead (mask false or sequence id 0), at a change of
    sequence id between neighbours, at the start of the sequence
    (cu_seqlens), or in the lookback row at an entry < 0.  Slot k holds the id
    only while the walk is still open; a dead t gives an all-pad window.
    lookback_ids[s, i] is the compressed id at position
    cu_seqlens[s] - (max_ngram-1) + i and counts as the same document as the
    chunk's first position."""
    c, bad = compressed_ids(input_ids, token_map, pad_id)
    T = c.shape[0]
    O = max_ngram - 1
    cu = np.array([0, T] if cu_seqlens is None else cu_seqlens, dtype=np.int64)
    t = np.arange(T, dtype=np.int64)
    seq = np.searchsorted(cu, t, side="right") - 1
    start = cu[seq]
    alive = np.ones(T, dtype=bool)
    if token_mask is not None:
        alive &= np.asarray(token_mask) != 0
    sid = None
    if sequence_ids is not None:
        sid = np.asarray(sequence_ids, dtype=np.int64)
        alive &= sid != 0
    lb = None if lookback_ids is None else np.asarray(lookback_ids, dtype=np.int64).reshape(-1, O)

    w = np.full((T, max_ngram), pad_id, dtype=np.int64)
    open_ = alive.copy()
    w[:, 0] = np.where(open_, c, pad_id)
    for k in range(1, max_ngram):
        p = t - k
        in_chunk = p >= start
        pc = np.clip(p, 0, max(T - 1, 0))
        ok_chunk = in_chunk & alive[pc]
        if sid is not None:
            ok_chunk &= sid[pc] == sid[np.clip(p + 1, 0, max(T - 1, 0))]
        i = p - start + O
        if lb is not None:
            ic = np.clip(i, 0, O - 1)
            lbv = lb[seq, ic]
            ok_lb = (~in_chunk) & (i >= 0) & (lbv >= 0)
        else:
            lbv = np.zeros(T, dtype=np.int64)
            ok_lb = np.zeros(T, dtype=bool)
        open_ &= np.where(in_chunk, ok_chunk, ok_lb)
        w[:, k] = np.where(open_, np.where(in_chunk, c[pc], lbv), pad_id)
    return w, bad


def hash_ids(w, multipliers, primes, offsets, compressed_vocab: int):
    """Row ids [T, L, C] from windows w [T, max_ngram].

    [vLLM] ``EngramLayout`` / ``NgramHashState.forward`` / ``compute_hash_multipliers``;
    [Atlas] stage 1.  For layer l, n-gram size n and head h (column
    c = (n-2)*n_heads + h):
        mix = XOR over k < n of (w[t, k] * multipliers[l, k])   (int64, no overflow)
        id  = offsets[l, c] + mix mod primes[l, n-2, h]
    The XOR mix is a reading: the pages only fix that each product fits int64."""
    w = np.asarray(w, dtype=np.int64)
    if w.size and (w.min() < 0 or w.max() >= compressed_vocab):
        raise ValueError("window ids must be compressed ids in [0, V)")
    m = np.asarray(multipliers, dtype=np.int64)
    pr = np.asarray(primes, dtype=np.int64)
    off = np.asarray(offsets, dtype=np.int64)
    L, O, Hh = pr.shape
    if m.max() > INT64_MAX // max(1, compressed_vocab - 1):
        raise ValueError("multiplier too large: id * multiplier could overflow int64")
    T = w.shape[0]
    out = np.zeros((T, L, O * Hh), dtype=np.int64)
    for layer in range(L):
        for o in range(O):
            n = o + 2
            mix = np.zeros(T, dtype=np.int64)
            for k in range(n):
                mix ^= w[:, k] * m[layer, k]
            for h in range(Hh):
                col = o * Hh + h
                out[:, layer, col] = off[layer, col] + mix % pr[layer, o, h]
    return out


# ---------------------------------------------------------------------------
# Stage 2: table rows -> bf16
# ---------------------------------------------------------------------------


def e4m3_to_float(b):
    """OCP FP8 E4M3 (the 'fn' variant torch calls float8_e4m3fn): sign, 4
    exponent bits (bias 7), 3 mantissa bits; exponent 0 is subnormal
    (m * 2**-9); 0x7F/0xFF are NaN; no infinities.  Returns fp64."""
    b = np.asarray(b, dtype=np.int64)
    sign = np.where((b >> 7) & 1, -1.0, 1.0)
    e = (b >> 3) & 0xF
    m = b & 0x7
    mag = np.where(e == 0, m * 2.0 ** -9, (1.0 + m / 8.0) * np.exp2(e.astype(np.float64) - 7.0))
    val = sign * mag
    return np.where((e == 0xF) & (m == 0x7), np.nan, val)


def e8m0_to_float(b):
    """The E8M0 scale byte read as the exponent field of an fp32:
    float(bits = byte << 23).  Byte 127 is 1.0, byte 0 is +0.0, byte 255 is
    +inf.  [vLLM] ``_engram_lookup_kernel`` (ue8m0 byte is the fp32 exponent)."""
    b = np.asarray(b, dtype=np.uint32)
    return (b << np.uint32(23)).astype(np.uint32).view(np.float32).astype(np.float64)


def f32_to_bf16_bits(x):
    """Round fp32 values to bf16 (round to nearest, ties to even) and return
    the 16-bit patterns.  NaN -> 0x7FC0 with the sign kept."""
    x = np.ascontiguousarray(np.asarray(x, dtype=np.float32))
    u = x.view(np.uint32).astype(np.uint64)
    lsb = (u >> np.uint64(16)) & np.uint64(1)
    r = ((u + np.uint64(0x7FFF) + lsb) >> np.uint64(16)).astype(np.uint16)
    nan = np.isnan(x)
    if nan.any():
        r = np.where(nan, ((u >> np.uint64(16)).astype(np.uint16) & np.uint16(0x8000)) | np.uint16(0x7FC0), r)
    return r.astype(np.uint16)


def bf16_bits_to_f64(bits):
    b = np.ascontiguousarray(np.asarray(bits, dtype=np.uint16)).astype(np.uint32) << np.uint32(16)
    return b.view(np.float32).astype(np.float64)


def dequant_fp8_rows(weight, scales, rows):
    """bf16 bits [n, D] of table rows ``rows`` of an FP8-E4M3 table with one
    E8M0 scale per 32 values.  [vLLM] ``_engram_lookup_kernel``: value times
    scale in fp32, then rounded to bf16.  The fp64 product of a 4-bit
    significand and a power of two is exact, and equals the fp32 product
    after one rounding to fp32."""
    weight = np.asarray(weight, dtype=np.uint8)
    scales = np.asarray(scales, dtype=np.uint8)
    rows = np.asarray(rows, dtype=np.int64)
    v = e4m3_to_float(weight[rows])                               # [n, D]
    s = e8m0_to_float(scales[rows])                               # [n, D/32]
    s = np.repeat(s, E8M0_BLOCK, axis=1)
    with np.errstate(over="ignore", invalid="ignore"):
        prod = (v * s).astype(np.float32)
    return f32_to_bf16_bits(prod)


def dequant_q2k_rows(table, rows):
    """bf16 bits [n, 256] of Q2_K rows (one 84-byte super-block per row).
    [Atlas] stage 2 and ENGRAM_ROW_BYTES fix only the 84-byte, 256-wide row;
    the reading is the public GGML Q2_K block: bytes 0-15 hold sixteen
    (scale | min << 4) nibble pairs, one per 16 elements; bytes 16-79 hold
    2-bit quants; bytes 80-81 and 82-83 are fp16 d and dmin.  Element e:
        half = e // 128, j = (e % 128) // 32, l = e % 32, b = e // 16
        q = (qs[32*half + l] >> 2j) & 3
        y = d * (scales[b] & 15) * q - dmin * (scales[b] >> 4)
    d*sc*q and dmin*m are exact, so y is their exact difference rounded once
    to fp32 (fp64 holds the difference exactly: fp16 exponents span < 53 bits),
    then rounded to bf16."""
    t = np.asarray(table, dtype=np.uint8)[np.asarray(rows, dtype=np.int64)]   # [n, 84]
    n = t.shape[0]
    sc = t[:, 0:16].astype(np.int64)
    qs = t[:, 16:80].astype(np.int64)
    d = t[:, 80:82].copy().view(np.float16).astype(np.float64)[:, 0]
    dmin = t[:, 82:84].copy().view(np.float16).astype(np.float64)[:, 0]
    e = np.arange(Q2K_ROW_ELEMS)
    half, j, l, b = e // 128, (e % 128) // 32, e % 32, e // 16
    q = (qs[:, 32 * half + l] >> (2 * j)) & 3                  # [n, 256]
    scale = (sc[:, b] & 15).astype(np.float64)
    mn = (sc[:, b] >> 4).astype(np.float64)
    with np.errstate(over="ignore", invalid="ignore"):
        y = (d[:, None] * scale) * q - dmin[:, None] * mn
        y32 = y.astype(np.float32)
    assert y32.shape == (n, Q2K_ROW_ELEMS)
    return f32_to_bf16_bits(y32)


def gather(fmt: str, table, scales, ids, num_rows: int, head_dim: int):
    """Stage 2 for one layer: ids [T, C] -> bf16 bits [T, C*head_dim], the
    rows concatenated in column order.  Ids outside [0, num_rows) give zero
    rows ([vLLM] ``_engram_lookup_kernel``: rows it does not own read 0).
    Returns (bits, n_out_of_range)."""
    ids = np.asarray(ids, dtype=np.int64)
    T, C = ids.shape
    flat = ids.reshape(-1)
    ok = (flat >= 0) & (flat < num_rows)
    safe = np.where(ok, flat, 0)
    if fmt == "fp8":
        bits = dequant_fp8_rows(table, scales, safe)
    elif fmt == "q2k":
        bits = dequant_q2k_rows(table, safe)
    elif fmt == "bf16":
        bits = np.asarray(table, dtype=np.uint16)[safe]
    else:
        raise ValueError(fmt)
    bits = np.where(ok[:, None], bits, np.uint16(0)).astype(np.uint16)
    return bits.reshape(T, C * head_dim), int((~ok).sum())


# ---------------------------------------------------------------------------
# Stage 3: wkv projection
# ---------------------------------------------------------------------------


def project(a_bits, wkv_bits):
    """kv[t, n] = sum_k A[t, k] * wkv[n, k] in fp64 from bf16 operands.
    [vLLM] ``Engram.__init__`` (wkv: n_hash_cols*head_dim -> dim*(hc+1)) and
    ``Engram.forward``; [Atlas] stage 3.  Columns [j*H, (j+1)*H) are stream j's
    key, the last H the shared value."""
    a = bf16_bits_to_f64(a_bits)
    w = bf16_bits_to_f64(wkv_bits)
    return a @ w.T


# ---------------------------------------------------------------------------
# Stage 3, FP8 operand variant: MXFP8 operands
#
# The FP8 table rows already are e4m3 codes with one power-of-two (E8M0) scale
# per 32 values ([vLLM] ``ParallelEngramEmbedding``: weight float8_e4m3fn plus a
# ue8m0 scale per 32-element block).  The variant feeds those codes and scales
# to the projection as they are, and stores wkv the same way: per row and per
# block of 32 along K, one scale byte and 32 e4m3 codes.  The pages do not
# print a weight encoder; the reading is the rule the table's scale convention
# implies: the scale is the smallest power of two 2**e with
# max|w| / 2**e <= 448 (so no value saturates), byte = 127 + e, and each code
# is w / 2**e rounded to nearest, ties to even.  An all-zero block gets byte 127
# and zero codes.  Dequantised values are exact in bf16 and fp32.
# ---------------------------------------------------------------------------

E4M3_MAX = 448.0


def float_to_e4m3(x):
    """fp64 values -> OCP E4M3 (fn) codes, round to nearest, ties to even.
    Magnitudes above 448 saturate to 448 (the format has no infinities); NaN
    becomes 0x7F.  Subnormals are multiples of 2**-9 below 2**-6."""
    x = np.asarray(x, dtype=np.float64)
    sign = np.signbit(x).astype(np.int64) << 7
    a = np.abs(x)
    nan = np.isnan(x)
    a = np.where(nan, 0.0, a)
    code = np.zeros(a.shape, dtype=np.int64)
    sub = a < 2.0 ** -6
    # subnormal range: q = rint(a / 2**-9) in 0..8; code 8 is 2**-6, the first normal
    code = np.where(sub, np.rint(a * 2.0 ** 9).astype(np.int64), code)
    mant, ex = np.frexp(np.where(sub, 1.0, a))                 # a = mant * 2**ex, mant in [0.5, 1)
    E = ex.astype(np.int64) - 1                                # a = (2 * mant) * 2**E
    q = np.rint((2.0 * mant - 1.0) * 8.0).astype(np.int64)     # 3 mantissa bits, ties to even
    E = np.where(q == 8, E + 1, E)
    q = np.where(q == 8, 0, q)
    normal = (E + 7) << 3 | q
    over = (E + 7 > 15) | ((E + 7 == 15) & (q == 7))
    normal = np.where(over, 0x7E, normal)
    code = np.where(sub, code, normal)
    code = np.where(nan, 0x7F, code | sign)
    return code.astype(np.uint8)


def mxfp8_quantize(w_bits, block: int = E8M0_BLOCK):
    """bf16 bits [N, K] -> (e4m3 codes uint8 [N, K], scale bytes uint8 [N, K/32])
    under the reading stated above.  K must be a multiple of 32."""
    w = bf16_bits_to_f64(w_bits)
    N, K = w.shape
    assert K % block == 0
    wb = w.reshape(N, K // block, block)
    amax = np.abs(wb).max(axis=2)                              # [N, K/32]
    e = np.zeros(amax.shape, dtype=np.int64)
    nz = amax > 0
    # smallest e with amax / 2**e <= 448: start from the binary exponent and correct
    _, ex = np.frexp(np.where(nz, amax / E4M3_MAX, 1.0))       # amax/448 = m * 2**ex, m in [0.5, 1)
    e = np.where(nz, ex.astype(np.int64), 0)                   # 2**ex >= amax/448 > 2**(ex-1)
    e = np.where(nz & (np.ldexp(E4M3_MAX, (e - 1)) >= amax), e - 1, e)
    e = np.clip(e, -127, 127)
    codes = float_to_e4m3(wb / np.exp2(e.astype(np.float64))[:, :, None]).reshape(N, K)
    return codes, (e + 127).astype(np.uint8)


def mxfp8_dequant(codes, scale_bytes, block: int = E8M0_BLOCK):
    """fp64 values of MXFP8 data: e4m3 value times 2**(byte - 127), per block of
    32 along the last axis."""
    v = e4m3_to_float(codes)
    s = np.exp2(np.asarray(scale_bytes, dtype=np.float64) - 127.0)
    return v * np.repeat(s, block, axis=-1)


def gather_fp8_raw(weight, scales, ids, num_rows: int):
    """FP8 variant of stage 2: ids [T, C] -> (codes [T, C*D], scales [T, C*D/32]),
    the table's bytes copied without dequantisation; ids outside [0, num_rows)
    give a zero row (codes 0, scale byte 127)."""
    ids = np.asarray(ids, dtype=np.int64)
    T, C = ids.shape
    weight = np.asarray(weight, dtype=np.uint8)
    scales = np.asarray(scales, dtype=np.uint8)
    flat = ids.reshape(-1)
    ok = (flat >= 0) & (flat < num_rows)
    safe = np.where(ok, flat, 0)
    codes = np.where(ok[:, None], weight[safe], np.uint8(0)).astype(np.uint8)
    sc = np.where(ok[:, None], scales[safe], np.uint8(127)).astype(np.uint8)
    return codes.reshape(T, -1), sc.reshape(T, -1), int((~ok).sum())


def project_mxfp8(a_codes, a_scales, w_codes, w_scales):
    """kv[t, n] = sum_k A[t, k] * W[n, k] in fp64 from MXFP8 operands (each value
    its code times its block's power-of-two scale)."""
    return mxfp8_dequant(a_codes, a_scales) @ mxfp8_dequant(w_codes, w_scales).T


# ---------------------------------------------------------------------------
# Stage 4: gate
# ---------------------------------------------------------------------------


def gate(streams, kv, q_weight_bits, k_weight_bits, eps: float, clamp: float, token_mask=None):
    """New fp32-highway values (fp64) after the gated update.

    [NeMo] ``_engram_gate_core``; [vLLM] ``Engram`` docstring and ``forward``
    (clamp 1e-6, masked tokens pass through); [Atlas] stage 4 (in place on the
    fp32 highway [T, hc, H]).  For token t and stream j:
        hn  = h_j * (mean(h_j^2) + eps)^-1/2 * q_weight[j]
        kn  = key_j * (mean(key_j^2) + eps)^-1/2 * k_weight[j]
        s   = <hn, kn> / sqrt(H)              (the 1/sqrt(H) is a reading)
        s'  = sign(s) * sqrt(max(|s|, clamp))
        h_j = h_j + sigmoid(s') * value
    with key_j = kv[t, j*H:(j+1)*H] and value = kv[t, hc*H:].  Tokens whose
    mask is 0 keep their streams."""
    h = np.asarray(streams, dtype=np.float64)
    T, hc, H = h.shape
    kv = np.asarray(kv, dtype=np.float64).reshape(T, hc + 1, H)
    key, value = kv[:, :hc, :], kv[:, hc, :]
    qw = bf16_bits_to_f64(q_weight_bits).reshape(hc, H)
    kw = bf16_bits_to_f64(k_weight_bits).reshape(hc, H)
    hn = h / np.sqrt(np.mean(h * h, axis=-1, keepdims=True) + eps) * qw
    kn = key / np.sqrt(np.mean(key * key, axis=-1, keepdims=True) + eps) * kw
    s = np.sum(hn * kn, axis=-1) / np.sqrt(H)                     # [T, hc]
    s2 = np.sign(s) * np.sqrt(np.maximum(np.abs(s), clamp))
    g = 1.0 / (1.0 + np.exp(-s2))
    out = h + g[:, :, None] * value[:, None, :]
    if token_mask is not None:
        keep = np.asarray(token_mask) == 0
        out[keep] = h[keep]
    return out, g


# ---------------------------------------------------------------------------
# Whole path
# ---------------------------------------------------------------------------


def forward(dims: dict, batch: dict, hash_tables: dict, layers: list, streams_in: list, tokens=None):
    """Hash once for all layers, then per layer gather -> project -> gate.

    dims: max_ngram, n_heads, head_dim, hidden, hc, compressed_vocab, pad_id,
    eps, clamp.  batch: input_ids, cu_seqlens, sequence_ids, token_mask,
    lookback_ids.  hash_tables: token_map, multipliers, primes, offsets.
    layers[l]: fmt, table, scales, num_rows, wkv_bits, q_bits, k_bits.
    streams_in[l]: fp32 [T, hc, H].  ``tokens`` restricts stages 2-4 to a
    subset of positions (the hash always covers every token, since windows
    reach back).  Returns dict with ids [T, L, C], and per layer the A bits,
    kv (fp64) and new streams (fp64) of the selected tokens."""
    w, bad = windows(batch["input_ids"], hash_tables["token_map"], dims["pad_id"], dims["max_ngram"],
                     batch.get("cu_seqlens"), batch.get("sequence_ids"), batch.get("token_mask"),
                     batch.get("lookback_ids"))
    ids = hash_ids(w, hash_tables["multipliers"], hash_tables["primes"], hash_tables["offsets"],
                   dims["compressed_vocab"])
    T = ids.shape[0]
    sel = np.arange(T) if tokens is None else np.asarray(tokens, dtype=np.int64)
    mask = batch.get("token_mask")
    res = {"ids": ids, "bad_raw": int(bad.sum()), "tokens": sel, "layers": []}
    for layer, lw in enumerate(layers):
        a_bits, n_oob = gather(lw["fmt"], lw["table"], lw.get("scales"), ids[sel, layer, :],
                               lw["num_rows"], dims["head_dim"])
        kv = project(a_bits, lw["wkv_bits"])
        out, g = gate(np.asarray(streams_in[layer])[sel], kv, lw["q_bits"], lw["k_bits"],
                      dims["eps"], dims["clamp"], None if mask is None else np.asarray(mask)[sel])
        res["layers"].append({"a_bits": a_bits, "kv": kv, "streams": out, "gate": g, "oob": n_oob})
    return res
