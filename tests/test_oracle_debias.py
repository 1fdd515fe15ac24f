"""Pins for the oracle's log-space readout (ruling engine.py `_score_plain`, `_prior`, `answer`),
CPU only.

- One pass, no prior: softmax(log_softmax(z) / T) is softmax(z / T) (scipy's softmax).
- Hand-worked: two options, shown in both orders, logits [0, ln 3] then [ln 3, 0].
- Full rotation: when every option appears once at every position, a prior that depends only on
  the position shifts every option's mean by the same amount and cancels in the softmax.
- Shift invariance: adding a constant to one pass's logits changes nothing.
"""
import math

import numpy as np
from scipy.special import log_softmax, softmax

from oracle import oracle


def test_single_pass_no_prior_is_plain_softmax():
    rng = np.random.default_rng(0)
    for K in (1, 2, 5, 26, 255):
        z = rng.normal(size=K) * 3
        raws, probs = oracle.rotation_debias([z], [list(range(K))], [[0]], None, 0.7)
        np.testing.assert_allclose(probs[0], softmax(z / 0.7), rtol=0, atol=1e-14)
        np.testing.assert_allclose(raws[0], log_softmax(z), rtol=0, atol=1e-13)


def test_hand_worked_two_orders():
    z0 = [0.0, math.log(3.0)]          # order (option 0, option 1)
    z1 = [math.log(3.0), 0.0]          # order (option 1, option 0): position 0 shows option 1
    raws, probs = oracle.rotation_debias([z0, z1], [[0, 1], [1, 0]], [[0, 1]], None, 1.0)
    np.testing.assert_allclose(raws[0], [math.log(0.25), math.log(0.75)], rtol=0, atol=1e-15)
    np.testing.assert_allclose(probs[0], [0.25, 0.75], rtol=0, atol=1e-15)
    prior = {2: [math.log(0.6), math.log(0.4)]}
    raws_p, probs_p = oracle.rotation_debias([z0, z1], [[0, 1], [1, 0]], [[0, 1]], lambda K: prior[K], 1.0)
    np.testing.assert_allclose(probs_p[0], [0.25, 0.75], rtol=0, atol=1e-15)       # cancels (full rotation)
    np.testing.assert_allclose(raws_p[0] - raws[0], -(math.log(0.6) + math.log(0.4)) / 2, rtol=0, atol=1e-15)


def test_full_rotation_cancels_any_positional_prior():
    rng = np.random.default_rng(1)
    K = 7
    passes = [rng.normal(size=K) for _ in range(K)]
    keys = [[(pos + r) % K for pos in range(K)] for r in range(K)]
    pri = log_softmax(rng.normal(size=K))
    _, with_prior = oracle.rotation_debias(passes, keys, [list(range(K))], lambda k: pri, 0.5)
    _, without = oracle.rotation_debias(passes, keys, [list(range(K))], None, 0.5)
    np.testing.assert_allclose(with_prior[0], without[0], rtol=0, atol=1e-14)
    # a partial rotation does not cancel it
    _, part_p = oracle.rotation_debias(passes[:2], keys[:2], [[0, 1]], lambda k: pri, 0.5)
    _, part = oracle.rotation_debias(passes[:2], keys[:2], [[0, 1]], None, 0.5)
    assert np.abs(part_p[0] - part[0]).max() > 1e-3


def test_logit_shift_invariance():
    rng = np.random.default_rng(2)
    z = [rng.normal(size=4) for _ in range(3)]
    keys = [[0, 1, 2, 3], [3, 0, 1, 2], [2, 3, 0, 1]]
    _, a = oracle.rotation_debias(z, keys, [[0, 1, 2]], None, 1.3)
    z2 = [z[0] + 5.0, z[1] - 2.0, z[2]]
    _, b = oracle.rotation_debias(z2, keys, [[0, 1, 2]], None, 1.3)
    np.testing.assert_allclose(a[0], b[0], rtol=0, atol=1e-14)
