"""Pins for the oracle's label readout (blink.py `_read`, `_read_batched`, `softmax`), CPU only.

Pins: hand-worked values (tests/golden/readout_cases.json), the logits against numpy's float64
matmul of the gathered label rows, the probabilities against scipy's softmax of z / T, and the
closed-form special cases (one label gives 1, equal logits give 1/K, probabilities sum to 1).
"""
import json
import os

import numpy as np
import pytest
from scipy.special import softmax as scipy_softmax

from oracle import oracle
from shared_prefix_question_gb300 import workloads as wl

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "readout_cases.json")


def _golden():
    with open(GOLDEN) as f:
        return json.load(f)


@pytest.mark.parametrize("case", _golden()["cases"], ids=lambda c: c["name"])
def test_readout_hand_worked(case):
    g = _golden()
    hidden = wl.bf16_bits(np.array(g["hidden"], dtype=np.float32))
    unembed = wl.bf16_bits(np.array(g["unembed"], dtype=np.float32))
    z, p, st = oracle.label_readout(hidden, case["last_idx"], unembed, case["label_off"], case["label_ids"],
                                    case["temperature"])
    assert st == 0
    np.testing.assert_allclose(z, case["logits"], rtol=0, atol=0)
    np.testing.assert_allclose(p, case["probs"], rtol=0, atol=2e-16)


@pytest.mark.parametrize("name", ["tiny", "2k"])
def test_readout_against_library_matmul_and_softmax(name):
    w = wl.WORKLOADS[name]
    if name == "2k":  # keep the CPU suite quick: a narrower vocabulary, same hidden size and labels
        w = wl.Workload("2k-narrow", w.index, w.P, w.n, w.tail_lo, w.tail_hi, w.Hq, w.Hkv, w.d, w.H, 4096,
                        w.k_lo, w.k_hi, 0.7, "table")
    ins = wl.readout_inputs(w)
    z, p, st = oracle.label_readout(ins.hidden, ins.last_idx, ins.unembed, ins.label_off, ins.label_ids,
                                    ins.temperature)
    assert st == 0
    hf = wl.bits_to_f32(ins.hidden).astype(np.float64)
    wf = wl.bits_to_f32(ins.unembed).astype(np.float64)
    for b in range(len(ins.last_idx)):
        lo, hi = ins.label_off[b], ins.label_off[b + 1]
        ids = ins.label_ids[lo:hi]
        ref_z = wf[ids] @ hf[ins.last_idx[b]]
        np.testing.assert_allclose(z[lo:hi], ref_z, rtol=1e-12, atol=1e-12)
        ref_p = scipy_softmax(ref_z / ins.temperature)
        np.testing.assert_allclose(p[lo:hi], ref_p, rtol=0, atol=1e-14)
        assert abs(p[lo:hi].sum() - 1.0) < 1e-12


def test_readout_special_cases():
    rng = np.random.default_rng(3)
    H, V = 32, 64
    hidden = wl.normal_bf16(rng, (3, H))
    unembed = wl.normal_bf16(rng, (V, H))
    # one label gives probability 1; the same id offered 4 times gives 1/4 each
    z, p, st = oracle.label_readout(hidden, [0, 2], unembed, [0, 1, 5], [9, 4, 4, 4, 4], 0.3)
    assert st == 0
    assert p[0] == 1.0
    np.testing.assert_allclose(p[1:], 0.25, rtol=0, atol=1e-16)
    # T = 1 is the plain softmax; smaller T sharpens towards the argmax, order preserved
    z1, p1, _ = oracle.label_readout(hidden, [1], unembed, [0, 6], [1, 2, 3, 4, 5, 6], 1.0)
    np.testing.assert_allclose(p1, scipy_softmax(z1), rtol=0, atol=1e-15)
    _, p2, _ = oracle.label_readout(hidden, [1], unembed, [0, 6], [1, 2, 3, 4, 5, 6], 0.25)
    assert np.argmax(p2) == np.argmax(p1)
    assert p2.max() > p1.max()
    assert (np.argsort(p1) == np.argsort(p2)).all()


def test_readout_bad_label_marks_only_its_question():
    rng = np.random.default_rng(4)
    hidden = wl.normal_bf16(rng, (2, 16))
    unembed = wl.normal_bf16(rng, (10, 16))
    z, p, st = oracle.label_readout(hidden, [0, 1], unembed, [0, 2, 4], [1, 2, 3, 10], 1.0)
    assert st == 5
    assert np.isfinite(p[:2]).all() and np.isnan(p[2:]).all()


def test_readout_rejects_bad_temperature():
    hidden = np.zeros((1, 4), dtype=np.uint16)
    unembed = np.zeros((4, 4), dtype=np.uint16)
    for t in (0.0, -1.0, float("inf"), float("nan")):
        with pytest.raises(oracle.OracleError):
            oracle.label_readout(hidden, [0], unembed, [0, 1], [0], t)
