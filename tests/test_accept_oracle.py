"""Pins of the greedy accept-length oracle (oracle.accept_prefix), without a GPU.

The hand fixture is worked from the rule itself; the other pins tie the
oracle to statements that do not share its loop: the accepted prefix agrees
position by position and the next position (if any) disagrees; the length is
the index of the first disagreement, found with numpy; equal arrays accept
every token and disagreement everywhere accepts none.
"""
import os

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "accept_prefix_hand.txt")


def load_hand():
    rows = [l.split() for l in open(GOLDEN) if l.strip() and not l.startswith("#")]
    cu, draft, target, want = (np.array([int(x) for x in r], dtype=np.int64) for r in rows)
    return cu, draft, target, want


def test_hand_fixture():
    cu, draft, target, want = load_hand()
    assert oracle.accept_prefix(draft, target, cu).tolist() == want.tolist()


def random_case(seed, batch=40, max_T=40, p_mismatch=0.15, vocab=7):
    rng = np.random.default_rng(seed)
    lens = rng.integers(0, max_T + 1, size=batch)
    cu = np.concatenate([[0], np.cumsum(lens)])
    draft = rng.integers(0, vocab, size=int(cu[-1]))
    target = np.where(rng.random(int(cu[-1])) < p_mismatch, rng.integers(0, vocab, size=int(cu[-1])),
                      draft)
    return cu, draft, target


@pytest.mark.parametrize("seed", range(5))
def test_prefix_property_and_first_mismatch(seed):
    cu, draft, target = random_case(seed)
    a = oracle.accept_prefix(draft, target, cu)
    for r in range(len(cu) - 1):
        d, g = draft[cu[r]:cu[r + 1]], target[cu[r]:cu[r + 1]]
        T = len(d)
        assert 0 <= a[r] <= T
        assert np.array_equal(d[:a[r]], g[:a[r]])
        if a[r] < T:
            assert d[a[r]] != g[a[r]]
        neq = np.flatnonzero(d != g)
        assert a[r] == (neq[0] if neq.size else T)


def test_all_equal_and_all_different():
    cu = np.array([0, 3, 3, 20])
    x = np.arange(20)
    assert oracle.accept_prefix(x, x, cu).tolist() == [3, 0, 17]
    assert oracle.accept_prefix(x, x + 1, cu).tolist() == [0, 0, 0]


def test_empty_batch():
    assert oracle.accept_prefix([], [], [0]).size == 0
