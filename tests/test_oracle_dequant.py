"""Pins of the oracle's table decoding: E4M3 values, E8M0 scales, bf16
rounding, FP8 rows and Q2_K rows.

E4M3/E8M0 are pinned to the OFP8 specification points and the page's scale
rule (tests/golden/e4m3_e8m0_points.txt) and to torch's float8_e4m3fn decoder
for all 256 bytes; bf16 rounding to torch's float32 -> bfloat16 cast; FP8 and
Q2_K rows to hand-built blocks whose values follow from the format by hand.
"""
import os

import numpy as np
import pytest
import torch

from engram_synth import encode_fp8_e8m0
from oracle import engram_oracle as O

GOLD = os.path.join(os.path.dirname(__file__), "golden", "e4m3_e8m0_points.txt")


def _golden():
    out = []
    for line in open(GOLD):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        fmt, b, v = line.split()
        out.append((fmt, int(b, 16), float(v)))
    return out


@pytest.mark.parametrize("fmt,b,v", _golden())
def test_golden_points(fmt, b, v):
    got = float((O.e4m3_to_float if fmt == "e4m3" else O.e8m0_to_float)(np.array([b]))[0])
    if np.isnan(v):
        assert np.isnan(got)
    else:
        assert got == v
        assert np.signbit(got) == np.signbit(v)


def test_e4m3_all_bytes_match_torch():
    b = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(b).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = O.e4m3_to_float(b)
    both_nan = np.isnan(ref) & np.isnan(got)
    assert np.all(both_nan | (ref == got))
    assert np.array_equal(np.signbit(ref[~both_nan]), np.signbit(got[~both_nan]))


def test_e8m0_powers_of_two():
    b = np.arange(1, 255)
    assert np.array_equal(O.e8m0_to_float(b), np.ldexp(1.0, b - 127))


def test_bf16_rounding_matches_torch():
    rng = np.random.default_rng(3)
    x = np.concatenate([
        rng.standard_normal(20000).astype(np.float32),
        (rng.standard_normal(5000) * 1e-39).astype(np.float32),       # fp32 subnormals
        rng.integers(0, 1 << 32, size=20000, dtype=np.uint64).astype(np.uint32).view(np.float32),
        # exact ties: low 16 bits 0x8000 with odd and even upper halves
        (np.arange(1000, dtype=np.uint32) << 16 | 0x8000).view(np.float32),
        np.array([0.0, -0.0, np.inf, -np.inf, 3.4e38, -3.4e38], dtype=np.float32),
    ])
    x = x[~np.isnan(x)]
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(O.f32_to_bf16_bits(x), ref)


def _fp8_row(values_byte, scale_bytes, D=64):
    w = np.full((1, D), values_byte, dtype=np.uint8)
    s = np.array([scale_bytes], dtype=np.uint8)
    return w, s


def test_fp8_rows_hand_built():
    # 1.0 (0x38) everywhere, scales 1.0 / 2.0 for the two 32-blocks of a 64-wide row
    w, s = _fp8_row(0x38, [127, 128])
    bits = O.dequant_fp8_rows(w, s, [0])
    assert bits[0, :32].tolist() == [0x3F80] * 32      # bf16 1.0
    assert bits[0, 32:].tolist() == [0x4000] * 32      # bf16 2.0
    # scale byte 0 is +0.0: products are zeros carrying the value's sign
    w, s = _fp8_row(0xB8, [0, 0])                       # -1.0
    assert O.dequant_fp8_rows(w, s, [0])[0].tolist() == [0x8000] * 64
    # 448 * 2^-10 = 0.4375 = bf16 0x3EE0; 2^-9 * 2^3 = 2^-6 = bf16 0x3C80
    w = np.zeros((2, 32), dtype=np.uint8)
    w[0], w[1] = 0x7E, 0x01
    s = np.array([[117], [130]], dtype=np.uint8)
    bits = O.dequant_fp8_rows(w, s, [0, 1, 0])
    assert bits[0].tolist() == [0x3EE0] * 32
    assert bits[1].tolist() == [0x3C80] * 32
    assert bits[2].tolist() == [0x3EE0] * 32


def test_fp8_encoder_round_trip_within_half_ulp():
    g = torch.Generator().manual_seed(0)
    x = torch.randn(64, 256, generator=g) * 0.02
    q, s = encode_fp8_e8m0(x)
    back = O.bf16_bits_to_f64(O.dequant_fp8_rows(q.numpy(), s.numpy(), np.arange(64)))
    xs = x.numpy().astype(np.float64)
    # e4m3 has 3 fraction bits: relative error <= 2^-4 above the subnormal range,
    # plus bf16 rounding of the exact product (none: 4 significant bits fit).
    scale = O.e8m0_to_float(s.numpy()).repeat(32, axis=1)
    tol = np.maximum(np.abs(xs) * 2.0 ** -4, scale * 2.0 ** -10)
    assert np.all(np.abs(back - xs) <= tol)


def _q2k_block(scales, qs, d, dmin):
    b = np.zeros(84, dtype=np.uint8)
    b[0:16] = scales
    b[16:80] = qs
    b[80:82] = np.array([d], dtype=np.float16).view(np.uint8)
    b[82:84] = np.array([dmin], dtype=np.float16).view(np.uint8)
    return b


def test_q2k_all_threes():
    blk = _q2k_block([0x01] * 16, [0xFF] * 64, 1.0, 0.0)
    y = O.bf16_bits_to_f64(O.dequant_q2k_rows(blk[None], [0]))
    assert np.all(y == 3.0)


def test_q2k_min_term_alone():
    # q = 0 everywhere: y = -dmin * m, m = high nibble of the sub-block byte
    sc = [(m << 4) | 0x7 for m in range(16)]
    blk = _q2k_block(sc, [0] * 64, 0.25, 0.5)
    y = O.bf16_bits_to_f64(O.dequant_q2k_rows(blk[None], [0]))[0]
    for e in range(256):
        assert y[e] == -0.5 * (e // 16), e


def test_q2k_element_order_one_hot():
    # a single 2-bit field set to 1 lights exactly one element:
    # qs byte 32*half + l, bit pair j  ->  element 128*half + 32*j + l
    sc = [0x01] * 16
    for half in range(2):
        for j in range(4):
            for l in (0, 5, 16, 31):
                qs = np.zeros(64, dtype=np.uint8)
                qs[32 * half + l] = 1 << (2 * j)
                y = O.bf16_bits_to_f64(O.dequant_q2k_rows(_q2k_block(sc, qs, 1.0, 0.0)[None], [0]))[0]
                nz = np.nonzero(y)[0].tolist()
                assert nz == [128 * half + 32 * j + l], (half, j, l, nz)
                assert y[nz[0]] == 1.0


def test_q2k_subblock_scale_index():
    # sub-block b (16 elements) uses scales[b]: scale b+1 times q = 3
    sc = [(b % 15) + 1 for b in range(16)]
    blk = _q2k_block(sc, [0xFF] * 64, 0.5, 0.0)
    y = O.bf16_bits_to_f64(O.dequant_q2k_rows(blk[None], [0]))[0]
    for e in range(256):
        assert y[e] == 0.5 * sc[e // 16] * 3


def test_q2k_single_rounding_of_difference():
    # d*sc*q - dmin*m with a result that needs rounding to fp32 then bf16:
    # compare with exact rational arithmetic rounded once to fp32, then to bf16.
    from fractions import Fraction
    rng = np.random.default_rng(5)
    for trial in range(50):
        d = np.float16(rng.uniform(-2, 2) * 2.0 ** rng.integers(-14, 6))
        dmin = np.float16(rng.uniform(-2, 2) * 2.0 ** rng.integers(-14, 6))
        sc = rng.integers(0, 256, size=16)
        qs = rng.integers(0, 256, size=64)
        blk = _q2k_block(sc, qs, float(d), float(dmin))
        got = O.dequant_q2k_rows(blk[None], [0])[0]
        for e in (0, 17, 100, 129, 255):
            half, j, l, b = e // 128, (e % 128) // 32, e % 32, e // 16
            q = (int(qs[32 * half + l]) >> (2 * j)) & 3
            exact = Fraction(float(d)) * (int(sc[b]) & 15) * q - Fraction(float(dmin)) * (int(sc[b]) >> 4)
            f32 = np.float32(float(exact))   # exact fits fp64 (< 53 bits), one rounding to fp32
            assert Fraction(float(exact)) == exact
            ref = torch.tensor([float(f32)], dtype=torch.float32).to(torch.bfloat16).view(torch.int16).item() & 0xFFFF
            assert int(got[e]) == ref, (trial, e)


def test_gather_zero_rows_for_out_of_range_ids():
    table = np.arange(4 * 8, dtype=np.uint16).reshape(4, 8) + 1
    bits, n_oob = O.gather("bf16", table, None, np.array([[0, 3], [-1, 4]]), 4, 8)
    assert n_oob == 2
    assert bits[0].tolist() == table[0].tolist() + table[3].tolist()
    assert bits[1].tolist() == [0] * 16
