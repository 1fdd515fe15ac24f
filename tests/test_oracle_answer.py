"""Pins for the oracle's answer assembly (blink.py `answer_for`), CPU only: hand-worked cases."""
import json
import math
import os

import pytest

from oracle import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "answer_cases.json")


def _cases():
    with open(GOLDEN) as f:
        return json.load(f)["cases"]


@pytest.mark.parametrize("case", _cases(), ids=lambda c: c["name"])
def test_answer_hand_worked(case):
    got = oracle.answer(case["qtype"], case["probs"])
    assert got["index"] == case["index"]
    assert abs(got["value"] - case["value"]) < 1e-12
    if case["confidence"] is None:
        assert math.isnan(got["confidence"])
    else:
        assert abs(got["confidence"] - case["confidence"]) < 1e-12


def test_answer_rejects_unknown_type():
    with pytest.raises(oracle.OracleError):
        oracle.answer(7, [0.5, 0.5])
