"""Pins of the oracle's projection and gate.

The projection is pinned to exact integer arithmetic (small integers are exact
in bf16 and in fp64); the gate to closed forms of the normalised dot, the
signed square root and the sigmoid, and to the pass-through rules for masked
tokens and a zero value.
"""
import math

import numpy as np
import torch

from oracle import engram_oracle as O


def _bf16_bits(x):
    return torch.tensor(np.asarray(x, dtype=np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def test_project_exact_integers():
    rng = np.random.default_rng(0)
    T, K, N = 7, 96, 40
    a = rng.integers(-8, 9, size=(T, K))
    w = rng.integers(-8, 9, size=(N, K))
    kv = O.project(_bf16_bits(a), _bf16_bits(w))
    exact = [[sum(int(a[t, k]) * int(w[n, k]) for k in range(K)) for n in range(N)] for t in range(T)]
    assert np.array_equal(kv, np.array(exact, dtype=np.float64))


def _gate_case(h, key, value, qw=None, kw=None, eps=1e-6, clamp=1e-6, mask=None):
    T, hc, H = h.shape
    kv = np.concatenate([key.reshape(T, hc * H), value.reshape(T, H)], axis=1)
    qw = np.ones((hc, H)) if qw is None else qw
    kw = np.ones((hc, H)) if kw is None else kw
    return O.gate(h, kv, _bf16_bits(qw), _bf16_bits(kw), eps, clamp, mask)


def _sig(x):
    return 1.0 / (1.0 + math.exp(-x))


def test_gate_zero_value_leaves_streams():
    rng = np.random.default_rng(1)
    h = rng.standard_normal((3, 4, 64))
    out, _ = _gate_case(h, rng.standard_normal((3, 4, 64)), np.zeros((3, 64)))
    assert np.array_equal(out, h)


def test_gate_masked_tokens_untouched():
    rng = np.random.default_rng(2)
    h = rng.standard_normal((4, 2, 32))
    mask = np.array([1, 0, 1, 0], dtype=np.uint8)
    out, _ = _gate_case(h, rng.standard_normal((4, 2, 32)), rng.standard_normal((4, 32)), mask=mask)
    assert np.array_equal(out[1], h[1]) and np.array_equal(out[3], h[3])
    assert not np.array_equal(out[0], h[0])


def test_gate_identical_stream_and_key():
    # hn = kn, so <hn, kn> = H * m2 / (m2 + eps) and s = sqrt(H) * m2 / (m2 + eps)
    rng = np.random.default_rng(3)
    H = 256
    h = rng.standard_normal((2, 4, H))
    v = rng.standard_normal((2, H))
    eps = 1e-6
    out, g = _gate_case(h, h.copy(), v, eps=eps)
    for t in range(2):
        for j in range(4):
            m2 = float(np.mean(h[t, j] ** 2))
            s = math.sqrt(H) * m2 / (m2 + eps)
            assert abs(g[t, j] - _sig(math.sqrt(s))) < 1e-12
            assert np.allclose(out[t, j], h[t, j] + g[t, j] * v[t], rtol=0, atol=1e-12)
    assert abs(_sig(4.0) - 0.9820137900379085) < 1e-15
    assert np.all(np.abs(g - 0.9820137900379085) < 1e-6)


def test_gate_opposite_key():
    rng = np.random.default_rng(4)
    H = 256
    h = rng.standard_normal((1, 3, H))
    _, g = _gate_case(h, -h, rng.standard_normal((1, H)))
    assert np.all(np.abs(g - _sig(-4.0)) < 1e-6)


def test_gate_orthogonal_and_zero_weight_give_half():
    H = 64
    h = np.zeros((1, 2, H))
    key = np.zeros((1, 2, H))
    h[0, :, : H // 2] = 1.0
    key[0, :, H // 2:] = 1.0                 # orthogonal: s = 0, sign(0) = 0
    _, g = _gate_case(h, key, np.ones((1, H)))
    assert np.all(g == 0.5)
    rng = np.random.default_rng(5)
    h = rng.standard_normal((2, 2, H))
    _, g = _gate_case(h, rng.standard_normal((2, 2, H)), np.ones((2, H)), qw=np.zeros((2, H)))
    assert np.all(g == 0.5)


def test_gate_clamp_and_sign():
    # a tiny positive score is lifted to sqrt(clamp); negative scores mirror
    H = 4
    h = np.array([[[1.0, 0.0, 0.0, 0.0]]])
    key = np.array([[[1.0, 1e4, 0.0, 0.0]]])
    clamp = 0.25
    _, g = _gate_case(h, key, np.zeros((1, H)), clamp=clamp)
    rh = 1.0 / math.sqrt(0.25 + 1e-6)
    rk = 1.0 / math.sqrt((1.0 + 1e8) / 4 + 1e-6)
    s = rh * rk / 2.0                        # <hn, kn> / sqrt(4)
    assert s < clamp
    assert abs(g[0, 0] - _sig(math.sqrt(clamp))) < 1e-12
    _, g2 = _gate_case(h, -key, np.zeros((1, H)), clamp=clamp)
    assert abs(g2[0, 0] - _sig(-math.sqrt(clamp))) < 1e-12


def test_gate_scale_invariance_of_key():
    # RMS normalisation: scaling the key by a positive constant does not move the gate
    rng = np.random.default_rng(6)
    h = rng.standard_normal((3, 4, 128))
    key = rng.standard_normal((3, 4, 128))
    v = rng.standard_normal((3, 128))
    _, g1 = _gate_case(h, key, v, eps=0.0)
    _, g2 = _gate_case(h, 37.0 * key, v, eps=0.0)
    assert np.allclose(g1, g2, rtol=0, atol=1e-12)


def test_gate_weights_enter_per_stream_and_element():
    # q_weight on the stream, k_weight on the key: only their product matters
    rng = np.random.default_rng(7)
    H = 32
    h = rng.standard_normal((2, 2, H))
    key = rng.standard_normal((2, 2, H))
    v = rng.standard_normal((2, H))
    qw = np.full((2, H), 2.0)
    kw = np.full((2, H), 0.5)
    _, g1 = _gate_case(h, key, v, qw=qw, kw=kw)
    _, g2 = _gate_case(h, key, v)
    assert np.allclose(g1, g2, rtol=0, atol=1e-15)
    qw2 = np.ones((2, H))
    qw2[1] = 0.0
    _, g3 = _gate_case(h, key, v, qw=qw2)
    assert np.allclose(g3[:, 0], g2[:, 0]) and np.all(g3[:, 1] == 0.5)
