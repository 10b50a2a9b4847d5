"""Pins of the oracle's router: top-k order and ties, weights, permutation (no GPU)."""
import itertools

import numpy as np
import scipy.special

from oracle import moe


def _brute_topk(l, k):
    """The unique k-subset S with (l_i, -i) > (l_j, -j) for all i in S, j not in S,
    found by enumerating every subset; returned in rank order."""
    E = len(l)
    key = lambda i: (l[i], -i)
    winners = [S for S in itertools.combinations(range(E), k)
               if all(key(i) > key(j) for i in S for j in range(E) if j not in S)]
    assert len(winners) == 1
    return sorted(winners[0], key=key, reverse=True)


def test_topk_brute_force_with_ties(rng):
    for trial in range(60):
        E, k = 8, 3
        l = rng.integers(-3, 4, size=E).astype(np.float64)   # many exact ties
        if trial % 3 == 0:
            l = rng.standard_normal(E)
        got = moe.top_k(l[None, :], k)[0].tolist()
        assert got == _brute_topk(l.tolist(), k), (l, got)


def test_topk_all_equal_takes_lowest_indices():
    assert moe.top_k(np.zeros((1, 512)), 10)[0].tolist() == list(range(10))


def test_weights_sum_to_one_and_order(rng):
    l = rng.standard_normal((32, 512)) * 3
    idx = moe.top_k(l, 10)
    w = moe.routing_weights(l, idx)
    assert np.all(np.abs(w.sum(axis=1) - 1.0) < 1e-12)
    assert np.all(np.diff(w, axis=1) <= 0)          # ranked by logit => weights descend


def test_weights_full_k_is_plain_softmax(rng):
    l = rng.standard_normal((5, 16)) * 4
    idx = moe.top_k(l, 16)
    w = moe.routing_weights(l, idx)
    ref = np.take_along_axis(scipy.special.softmax(l, axis=1), idx.astype(np.int64), axis=1)
    assert np.allclose(w, ref, rtol=1e-13, atol=0)


def test_weights_are_renormalised_full_softmax(rng):
    l = rng.standard_normal((7, 512)) * 2 + rng.standard_normal((7, 1)) * 50
    idx = moe.top_k(l, 10)
    p = scipy.special.softmax(l, axis=1)
    sel = np.take_along_axis(p, idx.astype(np.int64), axis=1)
    ref = sel / sel.sum(axis=1, keepdims=True)
    assert np.allclose(moe.routing_weights(l, idx), ref, rtol=1e-12, atol=0)


def test_permutation_brute_force(rng):
    T, k, E = 37, 4, 11
    idx = np.stack([rng.choice(E, size=k, replace=False) for _ in range(T)]).astype(np.int32)
    counts, offsets, perm, pos = moe.permutation(idx, E)
    # brute force: walk experts in order, and slots in (t, j) order inside each
    expect = []
    for e in range(E):
        for t in range(T):
            for j in range(k):
                if idx[t, j] == e:
                    expect.append(t * k + j)
    assert perm.tolist() == expect
    assert counts.tolist() == [int((idx == e).sum()) for e in range(E)]
    assert offsets[0] == 0 and offsets[-1] == T * k
    assert all(offsets[e + 1] - offsets[e] == counts[e] for e in range(E))
    for t in range(T):
        for j in range(k):
            assert perm[pos[t, j]] == t * k + j


def test_permutation_degenerate_cases():
    # every token on the same experts; and T = 0
    idx = np.tile(np.arange(3, dtype=np.int32), (5, 1))
    counts, offsets, perm, pos = moe.permutation(idx, 8)
    assert counts.tolist() == [5, 5, 5, 0, 0, 0, 0, 0]
    assert perm.tolist() == [0, 3, 6, 9, 12, 1, 4, 7, 10, 13, 2, 5, 8, 11, 14]
    c0, o0, p0, q0 = moe.permutation(np.zeros((0, 3), np.int32), 8)
    assert c0.sum() == 0 and o0.tolist() == [0] * 9 and p0.size == 0
