"""Pins for the oracle's shared-prefix length (blink.py `_shared_prefix_len`), CPU only.

The oracle follows the page (common prefix of the lexicographic minimum and maximum); the pins
use the definition itself (the longest p on which every sequence agrees, clipped so each keeps a
token) by brute force, and hand-worked cases.
"""
import itertools

import numpy as np
import pytest

from oracle import oracle


def _definition(seqs):
    if len(seqs) < 2:
        return 0
    p = 0
    while all(len(s) > p for s in seqs) and len({s[p] for s in seqs}) == 1:
        p += 1
    return min(p, min(len(s) for s in seqs) - 1)


@pytest.mark.parametrize("seqs,expect", [
    ([[1, 2, 3, 4], [1, 2, 3, 5], [1, 2, 9]], 2),
    ([[5, 5, 5], [5, 5, 5]], 2),          # identical: each keeps its last token
    ([[7, 8], [7, 8, 9, 10]], 1),          # one is a prefix of the other: clipped to 2 - 1
    ([[3, 1], [4, 1]], 0),
    ([[1, 2, 3]], 0),                       # a single sequence shares nothing
])
def test_shared_prefix_hand_worked(seqs, expect):
    assert oracle.shared_prefix_len(seqs) == expect


def test_shared_prefix_brute_force():
    rng = np.random.default_rng(0)
    for n in range(1, 5):
        for _ in range(300):
            base = rng.integers(0, 3, size=int(rng.integers(0, 6))).tolist()
            seqs = [base[: int(rng.integers(0, len(base) + 1))] + rng.integers(0, 3, size=int(rng.integers(1, 4))).tolist()
                    for _ in range(n)]
            assert oracle.shared_prefix_len(seqs) == _definition(seqs), seqs
    for seqs in itertools.product([[0], [1], [0, 0], [0, 1], [1, 0], [0, 0, 1]], repeat=3):
        assert oracle.shared_prefix_len(list(seqs)) == _definition(list(seqs))
