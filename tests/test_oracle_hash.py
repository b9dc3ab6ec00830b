"""Pins of the oracle's n-gram windows and hash ids.

The windows are checked against a literal walk back written independently here
(pure Python, one position at a time), on many tiny random batches with
sequence cuts, documents, masks and lookback rows.  The hash is checked
against Python big-int arithmetic of the stated mix, plus invariants: every id
falls in its head's bucket, equal windows give equal ids, tokens behind a
boundary do not matter, and a decode step with lookback equals hashing the
whole sequence.
"""
import numpy as np
import pytest

from oracle import engram_oracle as O


def _walk(t, cu, c, alive, sid, lb, pad, max_ngram):
    """Literal walk back from t: the list of window ids, k = 0..max_ngram-1."""
    s = max(i for i in range(len(cu) - 1) if cu[i] <= t < cu[i + 1])
    start = cu[s]
    depth = max_ngram - 1
    out = []
    blocked = not alive[t]
    for k in range(max_ngram):
        p = t - k
        if k > 0 and not blocked:
            if p >= start:
                if not alive[p]:
                    blocked = True
                elif sid is not None and sid[p] != sid[p + 1]:
                    blocked = True
            else:
                i = p - start + depth          # index into the lookback row
                if lb is None or i < 0 or lb[s][i] < 0:
                    blocked = True
        if blocked:
            out.append(pad)
        elif p >= start:
            out.append(c[p])
        else:
            out.append(lb[s][p - start + depth])
    return out


def _random_batch(rng, max_ngram, V_raw, V_c):
    S = int(rng.integers(1, 4))
    lens = rng.integers(0, 9, size=S)
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int64)
    T = int(cu[-1])
    ids = rng.integers(0, V_raw, size=T)
    tmap = rng.integers(0, V_c, size=V_raw)
    mask = (rng.random(T) > 0.2).astype(np.uint8) if rng.random() < 0.7 else None
    sid = None
    if rng.random() < 0.6:
        sid = np.zeros(T, dtype=np.int64)
        for s in range(S):
            a, b = cu[s], cu[s + 1]
            doc = 1
            for p in range(a, b):
                if p > a and rng.random() < 0.3:
                    doc += 1
                sid[p] = 0 if rng.random() < 0.1 else doc
    lb = None
    if rng.random() < 0.6:
        lb = rng.integers(0, V_c, size=(S, max_ngram - 1))
        lb[rng.random(lb.shape) < 0.2] = -1
    return ids, tmap, cu, mask, sid, lb


@pytest.mark.parametrize("max_ngram", [2, 3, 4, 5])
def test_windows_match_literal_walk(max_ngram):
    rng = np.random.default_rng(100 + max_ngram)
    V_raw, V_c = 16, 12
    for trial in range(300):
        ids, tmap, cu, mask, sid, lb = _random_batch(rng, max_ngram, V_raw, V_c)
        pad = int(rng.integers(0, V_c))
        w, bad = O.windows(ids, tmap, pad, max_ngram, cu, sid, mask, lb)
        T = len(ids)
        c = [int(tmap[i]) for i in ids]
        alive = [(mask is None or mask[p] != 0) and (sid is None or sid[p] != 0) for p in range(T)]
        for t in range(T):
            assert w[t].tolist() == _walk(t, cu.tolist(), c, alive, sid, lb, pad, max_ngram), (trial, t)
        assert not bad.any()


def test_out_of_map_raw_ids_are_padded_and_reported():
    tmap = np.array([5, 6, 7])
    w, bad = O.windows([0, 3, -1, 2], tmap, 9, 2)
    assert bad.tolist() == [False, True, True, False]
    assert w[:, 0].tolist() == [5, 9, 9, 7]


def _bigint_hash(w_row, m, primes, offsets, layer):
    L, Oo, Hh = primes.shape
    out = []
    for o in range(Oo):
        n = o + 2
        mix = 0
        for k in range(n):
            prod = int(w_row[k]) * int(m[layer, k])
            assert 0 <= prod < (1 << 63)
            mix ^= prod
        for h in range(Hh):
            out.append(int(offsets[layer, o * Hh + h]) + mix % int(primes[layer, o, h]))
    return out


def test_hash_matches_bigint_arithmetic():
    rng = np.random.default_rng(7)
    V = 131072
    primes, offsets, _ = O.layout(1 << 20, 2, 4, 8)
    m = O.hash_multipliers((1, 14), 4, V)
    w = rng.integers(0, V, size=(200, 4))
    w[:5] = V - 1          # largest products
    w[5:8] = 0
    ids = O.hash_ids(w, m, primes, offsets, V)
    for t in range(w.shape[0]):
        for layer in range(2):
            assert ids[t, layer].tolist() == _bigint_hash(w[t], m, primes, offsets, layer)


def test_hash_ids_fall_in_their_buckets_and_equal_windows_agree():
    rng = np.random.default_rng(8)
    V = 1024
    primes, offsets, rows = O.layout(4001, 1, 3, 4)
    m = O.hash_multipliers((1,), 3, V)
    w = rng.integers(0, V, size=(500, 3))
    w[100:200] = w[0]
    ids = O.hash_ids(w, m, primes, offsets, V)
    lo = offsets[0][None, :]
    hi = lo + primes[0].reshape(-1)[None, :]
    assert np.all(ids[:, 0] >= lo) and np.all(ids[:, 0] < hi)
    assert np.all(ids[100:200] == ids[0])
    # the 2-gram columns see only slots 0..1
    w2 = w.copy()
    w2[:, 2] = (w2[:, 2] + 1) % V
    ids2 = O.hash_ids(w2, m, primes, offsets, V)
    assert np.array_equal(ids2[:, 0, :4], ids[:, 0, :4])
    assert not np.array_equal(ids2[:, 0, 4:], ids[:, 0, 4:])


def test_boundaries_hide_tokens_and_masked_is_all_pad():
    V_raw = V_c = 64
    tmap = np.arange(64)
    pad = 3
    ids = np.array([10, 11, 12, 13, 14, 15, 16, 17])
    sid = np.array([1, 1, 1, 2, 2, 2, 2, 2])
    mask = np.array([1, 1, 1, 1, 1, 0, 1, 1], dtype=np.uint8)
    w, _ = O.windows(ids, tmap, pad, 4, None, sid, mask, None)
    # document 2 starts at 3: its windows never see 10..12
    assert w[3].tolist() == [13, pad, pad, pad]
    assert w[4].tolist() == [14, 13, pad, pad]
    # position 5 is masked: all pad; 6 and 7 cannot look through it
    assert w[5].tolist() == [pad] * 4
    assert w[6].tolist() == [16, pad, pad, pad]
    assert w[7].tolist() == [17, 16, pad, pad]
    # changing a token before the document start changes nothing after it
    ids2 = ids.copy()
    ids2[:3] = [40, 41, 42]
    w2, _ = O.windows(ids2, tmap, pad, 4, None, sid, mask, None)
    assert np.array_equal(w2[3:], w[3:])
    del V_raw, V_c


def test_decode_with_lookback_equals_whole_sequence():
    rng = np.random.default_rng(9)
    V_raw, V_c = 300, 200
    tmap = rng.integers(0, V_c, size=V_raw)
    pad = int(tmap[0])
    primes, offsets, _ = O.layout(1 << 20, 1, 4, 8)
    m = O.hash_multipliers((1,), 4, V_c)
    seqs = [rng.integers(0, V_raw, size=int(n)) for n in (1, 2, 3, 4, 9)]
    # whole sequences
    whole = []
    for s in seqs:
        w, _ = O.windows(s, tmap, pad, 4)
        whole.append(O.hash_ids(w, m, primes, offsets, V_c)[-1])
    # decode: last token of each sequence, previous 3 compressed ids as lookback (-1 = none)
    last = np.array([s[-1] for s in seqs])
    lb = np.full((len(seqs), 3), -1, dtype=np.int64)
    for i, s in enumerate(seqs):
        prev = [int(tmap[x]) for x in s[:-1]][-3:]
        if prev:
            lb[i, 3 - len(prev):] = prev
    cu = np.arange(len(seqs) + 1)
    w, _ = O.windows(last, tmap, pad, 4, cu, None, None, lb)
    dec = O.hash_ids(w, m, primes, offsets, V_c)
    for i in range(len(seqs)):
        assert np.array_equal(dec[i], whole[i]), i
