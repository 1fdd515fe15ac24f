"""Pins for the oracle's pack plan (blink.py `_batches` / `_padded`), CPU only.

The oracle is checked against (1) hand-worked cases of the pages' rule and (2) a
characterisation of the greedy partition that does not retrace the oracle's loop: the slots
are Python's stable sort of the lengths; every forward is feasible (one row, or width x rows
within the budget and the row cap); every forward but the last is maximal (the next slot would
make it infeasible).  Feasible + maximal-from-its-start determines the greedy partition
uniquely, so a wrong comparison, an off-by-one in the count or a wrong tie order fails here.
"""
import itertools
import json
import os

import numpy as np
import pytest

from oracle import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "plan_cases.json")


def _cases():
    with open(GOLDEN) as f:
        return json.load(f)["cases"]


@pytest.mark.parametrize("case", _cases(), ids=lambda c: c["name"])
def test_plan_matches_hand_worked_cases(case):
    got = oracle.pack_plan(case["lengths"], case["budget"], case["max_rows"])
    assert got["n_forwards"] == case["n_forwards"]
    for key in ("order", "fwd_of_slot", "fwd_slot_start", "fwd_width", "cu_seqlens", "last_varlen",
                "last_padded"):
        assert got[key].tolist() == case[key], key


def _check_characterisation(lengths, budget, max_rows):
    plan = oracle.pack_plan(lengths, budget, max_rows)
    n = len(lengths)
    order = plan["order"].tolist()
    assert order == sorted(range(n), key=lambda i: lengths[i])
    nf = plan["n_forwards"]
    starts = plan["fwd_slot_start"].tolist()
    assert starts[0] == 0 and starts[nf] == n and all(s == n for s in starts[nf:])
    for f in range(nf):
        lo, hi = starts[f], starts[f + 1]
        assert hi > lo
        rows = hi - lo
        lens = [lengths[order[s]] for s in range(lo, hi)]
        width = max(lens)
        assert plan["fwd_width"][f] == width
        assert all(plan["fwd_of_slot"][s] == f for s in range(lo, hi))
        feasible = rows == 1 or (width * rows <= budget and (max_rows == 0 or rows <= max_rows))
        assert feasible
        if f + 1 < nf:
            nxt = lengths[order[hi]]
            grown = max(width, nxt) * (rows + 1) > budget or (max_rows > 0 and rows + 1 > max_rows)
            assert grown, "a forward closed early"
        for r, s in enumerate(range(lo, hi)):
            assert plan["last_padded"][s] == r * width + lengths[order[s]] - 1
    assert all(w == 0 for w in plan["fwd_width"][nf:].tolist())
    cu = np.concatenate([[0], np.cumsum([lengths[i] for i in order])])
    assert plan["cu_seqlens"].tolist() == cu.tolist()
    assert plan["last_varlen"].tolist() == (cu[1:] - 1).tolist()


def test_plan_exhaustive_small():
    """Every length vector with n <= 4 and lengths 1..5, several budgets and row caps."""
    for n in range(1, 5):
        for lengths in itertools.product(range(1, 6), repeat=n):
            for budget in (1, 3, 5, 6, 8, 10, 12, 25):
                for max_rows in (0, 1, 2, 3):
                    _check_characterisation(list(lengths), budget, max_rows)


def test_plan_random_large():
    rng = np.random.default_rng(7)
    for trial in range(40):
        n = int(rng.integers(1, 2000))
        lengths = rng.integers(1, 1200, size=n).tolist()
        budget = int(rng.choice([500, 4096, 32768]))
        max_rows = int(rng.choice([0, 0, 1, 7, 64]))
        _check_characterisation(lengths, budget, max_rows)


def test_plan_rejects_bad_arguments():
    with pytest.raises(oracle.OracleError):
        oracle.pack_plan([3, 0, 2], 10)
    with pytest.raises(oracle.OracleError):
        oracle.pack_plan([3, 2], 0)


def test_plan_page_row_cap_example():
    """blink.py `_forward_shared`: rows_cap = max(1, PREFIX_KV_TOKENS // (prefix + longest tail)).
    With an 18432-token prefix and a 256-token tail that is 7 rows per forward."""
    rows_cap = max(1, 131072 // (18432 + 256))
    assert rows_cap == 7
    lengths = [256] * 64
    plan = oracle.pack_plan(lengths, 32768, rows_cap)
    assert plan["n_forwards"] == 10
    assert np.diff(plan["fwd_slot_start"][:11]).tolist() == [7] * 9 + [1]
