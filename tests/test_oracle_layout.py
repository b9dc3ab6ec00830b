"""Pins of the oracle's layout: primality, prime drawing, offsets, multipliers.

The primality test is pinned to trial division and to known pseudoprimes; the
prime layout to the rules of the vLLM ``EngramLayout`` class (each prime is the
smallest unused prime above the previous one, restarting above
vocab_size - 1 per n-gram size); the multipliers to the bounds stated by
``compute_hash_multipliers`` (odd, and id * multiplier < 2**63).
"""
import math

import numpy as np
import pytest

from oracle import engram_oracle as O


def _trial_prime(n: int) -> bool:
    if n < 2:
        return False
    if n % 2 == 0:
        return n == 2
    r = math.isqrt(n)
    f = 3
    while f <= r:
        if n % f == 0:
            return False
        f += 2
    return True


def test_is_prime_matches_trial_division_small():
    for n in range(0, 20000):
        assert O.is_prime(n) == _trial_prime(n), n


@pytest.mark.parametrize("base", [1 << 19, 1 << 20, 1 << 23, (1 << 31) - 50])
def test_is_prime_matches_trial_division_near_table_sizes(base):
    for n in range(base - 300, base + 300):
        assert O.is_prime(n) == _trial_prime(n), n


def test_is_prime_known_hard_cases():
    # strong pseudoprimes to small bases and Carmichael numbers are composite
    for n in (561, 1105, 1729, 2047, 3277, 4033, 4681, 8321, 25326001, 3215031751,
              2152302898747 % (1 << 32) | 1):
        if n < (1 << 32):
            assert O.is_prime(n) == _trial_prime(n), n
    for n in (25326001, 3215031751):
        assert not O.is_prime(n)
    for p in (2, 3, 37, 41, 2147483647, 4294967291, 1048583, 524309, 8388617):
        assert O.is_prime(p), p


def test_is_prime_refuses_beyond_proven_range():
    with pytest.raises(ValueError):
        O.is_prime((1 << 32) + 15)


def test_tiny_layout_is_the_eight_primes_after_4000():
    # one layer, sizes 2..3, 4 heads: the 8 primes drawn are the 8 smallest
    # primes above 4000, in order, by trial division.
    primes, offsets, rows = O.layout(4001, 1, 3, 4)
    expect = [p for p in range(4001, 4100) if _trial_prime(p)][:8]
    assert primes.reshape(-1).tolist() == expect
    assert offsets[0].tolist() == [0] + list(np.cumsum(expect)[:-1])
    assert rows.tolist() == [sum(expect)]


@pytest.mark.parametrize("vocab,L,ng,hh", [(1 << 20, 1, 4, 8), (1 << 19, 2, 4, 8), (4001, 3, 3, 4)])
def test_layout_rules(vocab, L, ng, hh):
    primes, offsets, rows = O.layout(vocab, L, ng, hh)
    flat = primes.reshape(-1)
    assert len(set(flat.tolist())) == flat.size          # never reused
    assert all(_trial_prime(int(p)) for p in flat)
    used = set()
    for layer in range(L):
        for o in range(ng - 1):
            prev = vocab - 1
            for h in range(hh):
                p = int(primes[layer, o, h])
                # p is the smallest unused prime above prev
                for q in range(prev + 1, p):
                    assert not (_trial_prime(q) and q not in used), (q, p)
                assert p > prev
                used.add(p)
                prev = p
        # bucket ranges of one layer are disjoint and tile [0, rows)
        lf = primes[layer].reshape(-1)
        assert offsets[layer, 0] == 0
        assert np.all(offsets[layer, 1:] == offsets[layer, :-1] + lf[:-1])
        assert rows[layer] == lf.sum()


def test_layout_against_sympy_nextprime():
    sympy = pytest.importorskip("sympy")
    primes, _, _ = O.layout(1 << 20, 1, 4, 8)
    # order 0 takes 8 consecutive primes above 2^20-1; order 1 restarts but
    # skips them, so the whole layer is 24 consecutive primes.
    p, expect = (1 << 20) - 1, []
    for _ in range(24):
        p = sympy.nextprime(p)
        expect.append(p)
    assert primes.reshape(-1).tolist() == expect


@pytest.mark.parametrize("V", [1024, 131072, 163840])
def test_multipliers_odd_bounded(V):
    m = O.hash_multipliers((1, 14), 4, V)
    assert m.shape == (2, 4) and m.dtype == np.int64
    bound = max(1, (O.INT64_MAX // V) // 2)
    assert np.all(m % 2 == 1)
    assert np.all(m >= 1) and np.all(m <= 2 * bound - 1)
    # id * multiplier fits int64 for every compressed id
    assert all(int(x) * (V - 1) <= O.INT64_MAX for x in m.reshape(-1))
    # layers hash differently; a layer's row is reproducible
    assert not np.array_equal(m[0], m[1])
    assert np.array_equal(O.hash_multipliers((14,), 4, V)[0], m[1])
