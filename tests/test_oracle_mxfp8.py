"""Pins of the oracle's MXFP8 functions (the FP8 operand variant of the projection).

The encoder is pinned to the OCP E4M3 definition through independent routes: every code's
value round-trips, torch's float8_e4m3fn cast (a library routine) agrees on random values and
on exact midpoints (ties to even), saturation and NaN are hand-checked. The scale rule is pinned
by hand-built blocks at its boundary and by its defining property (the smallest power of two
that keeps every value at or below 448), the error by the half-ulp bound, and the projection by
an exact integer case.
"""
import numpy as np
import pytest
import torch

from oracle import engram_oracle as O


def _bf16(x):
    return O.f32_to_bf16_bits(np.asarray(x, dtype=np.float32))


def test_every_code_round_trips():
    codes = np.arange(256, dtype=np.uint8)
    v = O.e4m3_to_float(codes)
    ok = ~np.isnan(v)
    assert np.array_equal(O.float_to_e4m3(v[ok]), codes[ok])


def test_encoder_matches_torch_cast_on_random_values():
    rng = np.random.default_rng(7)
    x = np.concatenate([rng.normal(0, s, 50000) for s in (1e-3, 0.05, 1.0, 30.0, 200.0)])
    x = x[np.abs(x) <= 448.0]
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(O.float_to_e4m3(x), ref)


def test_midpoints_round_to_even_code():
    codes = np.arange(0, 0x7E, dtype=np.uint8)              # positive, non-NaN, below the max
    v = O.e4m3_to_float(codes)
    mid = (v[:-1] + v[1:]) / 2.0                             # exactly between neighbours
    got = O.float_to_e4m3(mid)
    even = np.where(codes[:-1] % 2 == 0, codes[:-1], codes[1:])
    assert np.array_equal(got, even)
    ref = torch.from_numpy(mid).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(got, ref)


def test_saturation_sign_and_nan():
    got = O.float_to_e4m3(np.array([448.0, 460.0, 1e9, -500.0, -0.0, np.nan, 2.0 ** -10, 3 * 2.0 ** -10]))
    # 2^-10 is half of the smallest subnormal: ties to even -> 0; 3 * 2^-10 -> 2 * 2^-9 (even)
    assert list(got) == [0x7E, 0x7E, 0x7E, 0xFE, 0x80, 0x7F, 0x00, 0x02]


def test_scale_at_the_448_boundary():
    w = np.zeros((4, 64), dtype=np.float32)
    w[0, 0] = 448.0                     # fits exactly: scale 1
    w[1, 5] = -450.0                    # just above: scale 2
    w[2, 40] = 0.001                    # block 1 of row 2 only; block 0 stays all-zero
    w[3, :32] = 3.0 * 2.0 ** -20        # small block
    codes, sc = O.mxfp8_quantize(_bf16(w))
    assert sc[0, 0] == 127 and codes[0, 0] == 0x7E
    assert sc[1, 0] == 128 and O.e4m3_to_float(codes[1, 5]) == -224.0   # -225 rounds to -224
    assert sc[2, 0] == 127 and not codes[2, :32].any()       # all-zero block
    e = int(sc[2, 1]) - 127                                  # 0.001 / 2^e <= 448 with e minimal
    assert 0.001 / 2.0 ** e <= 448.0 < 0.001 / 2.0 ** (e - 1)
    assert sc[3, 0] == 127 - 27                              # 1.5 * 2^-19 / 2^-27 = 384 <= 448 < 768
    assert np.all(np.abs(O.mxfp8_dequant(codes[3:4, :32], sc[3:4, :1]) - 3.0 * 2.0 ** -20) == 0)


def test_scale_is_minimal_and_error_within_half_ulp():
    rng = np.random.default_rng(3)
    w = (rng.normal(0, 0.02, (96, 512)) * np.exp2(rng.integers(-6, 7, (96, 1)))).astype(np.float32)
    bits = _bf16(w)
    wv = O.bf16_bits_to_f64(bits)
    codes, sc = O.mxfp8_quantize(bits)
    e = sc.astype(np.int64) - 127
    amax = np.abs(wv.reshape(96, 16, 32)).max(axis=2)
    assert np.all(amax / np.exp2(e) <= 448.0)
    assert np.all(amax / np.exp2(e - 1) > 448.0)             # one less would saturate
    scaled = wv / np.repeat(np.exp2(e.astype(float)), 32, axis=1)
    back = O.e4m3_to_float(codes)
    mag = np.maximum(np.abs(scaled), 2.0 ** -6)
    half_ulp = np.exp2(np.floor(np.log2(mag)) - 4)           # 3 mantissa bits
    assert np.all(np.abs(back - scaled) <= half_ulp * (1 + 1e-12))


def test_quantize_agrees_with_the_generators_encoder():
    # the seeded generator encodes the FP8 tables with the same rule (torch ops); the two agree
    from engram_synth import gen
    rng = np.random.default_rng(11)
    w = rng.normal(0, 0.02, (40, 256)).astype(np.float32)
    bits = _bf16(w)
    codes, sc = O.mxfp8_quantize(bits)
    q, s = gen.encode_fp8_e8m0(torch.from_numpy(O.bf16_bits_to_f64(bits).astype(np.float32)))
    assert np.array_equal(codes, q.numpy()) and np.array_equal(sc, s.numpy())


def test_raw_gather_matches_the_dequantising_gather():
    rng = np.random.default_rng(5)
    R, D = 50, 64
    weight = rng.integers(0, 256, (R, D)).astype(np.uint8)
    weight[(weight & 0x7F) == 0x7F] = 0x38                   # no NaN codes
    scales = rng.integers(115, 135, (R, D // 32)).astype(np.uint8)
    ids = rng.integers(-3, R + 3, (7, 4))
    codes, sc, bad = O.gather_fp8_raw(weight, scales, ids, R)
    bits, bad2 = O.gather("fp8", weight, scales, ids, R, D)
    assert bad == bad2 == int(((ids < 0) | (ids >= R)).sum())
    assert np.array_equal(O.mxfp8_dequant(codes, sc), O.bf16_bits_to_f64(bits))


def test_project_mxfp8_exact_integer_case():
    rng = np.random.default_rng(2)
    ints = np.array([0, 1, 2, 3, 4, 5, 6, 7, 8, -1, -2, -3, -4, -8])
    T, N, K = 5, 6, 64
    a = rng.choice(ints, (T, K))
    w = rng.choice(ints, (N, K))
    sa = rng.integers(126, 129, (T, K // 32))               # scales 1/2, 1, 2
    sw = rng.integers(126, 129, (N, K // 32))
    ac = O.float_to_e4m3(a.astype(float))
    wc = O.float_to_e4m3(w.astype(float))
    got = O.project_mxfp8(ac, sa.astype(np.uint8), wc, sw.astype(np.uint8))
    for t in range(T):
        for n in range(N):
            num = 0
            for k in range(K):
                num += int(a[t, k]) * int(w[n, k]) * 2 ** (int(sa[t, k // 32]) - 127 + int(sw[n, k // 32]) - 127 + 2)
            assert got[t, n] == num / 4
