"""The log-space readout on the device (ruling engine.py `_score_plain`, `_prior`, `answer`)
against the FP64 oracle: debiased mean log-probabilities within 1e-4, probabilities within 1e-3,
answers as for the label readout.  Orders: cyclic shifts of the options for a choice (all K or
the first few), the forward and reversed level order for a score."""
import numpy as np
import pytest
import torch

from oracle import oracle
from shared_prefix_question_gb300 import blink
from shared_prefix_question_gb300 import workloads as wl
from tests.helpers import dev_i32

pytestmark = pytest.mark.gpu


def _case(seed, B, max_k, max_rot):
    rng = np.random.default_rng(seed)
    pass_logits, pass_keys, q_passes, qtypes, counts = [], [], [], [], []
    for q in range(B):
        qt = int(rng.integers(0, 3))
        K = 2 if qt == wl.QTYPE_NOUL else int(rng.integers(2, 11)) if qt == wl.QTYPE_SCORE else int(rng.integers(1, max_k + 1))
        if qt == wl.QTYPE_SCORE:
            orders = [list(range(K)), list(range(K))[::-1]]
        else:
            R = min(K, max_rot)
            orders = [[(pos + r) % K for pos in range(K)] for r in range(R)]
        q_passes.append(list(range(len(pass_logits), len(pass_logits) + len(orders))))
        for o in orders:
            pass_logits.append(rng.normal(size=K) * 2)
            pass_keys.append(o)
        qtypes.append(qt)
        counts.append(K)
    prior_tab = np.zeros((255, 255), dtype=np.float32)
    for K in range(1, 256):
        x = rng.normal(size=K) * 0.5
        prior_tab[K - 1, :K] = x - (x.max() + np.log(np.exp(x - x.max()).sum()))
    return pass_logits, pass_keys, q_passes, np.array(qtypes, dtype=np.int32), np.array(counts), prior_tab


@pytest.mark.parametrize("seed,B,max_k,max_rot,use_prior,T", [(0, 64, 26, 4, True, 0.7), (1, 300, 255, 3, True, 1.0),
                                                              (2, 17, 8, 8, False, 1.0)])
def test_rotation_debias_matches_oracle(seed, B, max_k, max_rot, use_prior, T):
    pl, pk, qp, qt, counts, prior_tab = _case(seed, B, max_k, max_rot)
    pass_off = np.concatenate([[0], np.cumsum([len(z) for z in pl])]).astype(np.int32)
    raw_off = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    q_pass = np.array([p[0] for p in qp] + [qp[-1][-1] + 1], dtype=np.int32)
    logits = torch.from_numpy(np.concatenate(pl).astype(np.float32)).cuda()
    keys = dev_i32(np.concatenate(pk))
    prior = torch.from_numpy(prior_tab.reshape(-1)).cuda() if use_prior else None
    hp = torch.empty(int(raw_off[-1]), dtype=torch.float32, pin_memory=True)
    ha = torch.empty(B, 3, dtype=torch.float32, pin_memory=True)
    probs, raw, answers = blink.blink_rotation_debias(logits, dev_i32(pass_off), keys, dev_i32(q_pass), dev_i32(raw_off),
                                                      T, prior=prior, host_probs=hp, qtype=dev_i32(qt),
                                                      host_answers=ha)
    torch.cuda.synchronize()
    # the oracle sees the same fp32 logits and prior the device saw
    pl32 = [np.asarray(z, dtype=np.float32).astype(np.float64) for z in pl]
    prior_fn = (lambda K: prior_tab[K - 1, :K].astype(np.float64)) if use_prior else None
    raws_ref, probs_ref = oracle.rotation_debias(pl32, pk, qp, prior_fn, T)
    raw = raw.cpu().numpy().astype(np.float64)
    got = hp.numpy().astype(np.float64)
    for q in range(B):
        lo, hi = raw_off[q], raw_off[q + 1]
        np.testing.assert_allclose(raw[lo:hi], raws_ref[q], rtol=0, atol=1e-4)
        np.testing.assert_allclose(got[lo:hi], probs_ref[q], rtol=0, atol=1e-3)
        ref = oracle.answer(int(qt[q]), probs_ref[q])
        srt = np.sort(probs_ref[q])[::-1]
        if len(srt) < 2 or srt[0] - srt[1] > 1e-4:
            assert int(ha[q, 0]) == ref["index"]


def test_rotation_debias_flags_bad_order():
    logits = torch.zeros(4, dtype=torch.float32, device="cuda")
    with pytest.raises(blink.BlinkError) as e:
        blink.blink_rotation_debias(logits, dev_i32([0, 2, 4]), dev_i32([0, 1, 0, 2]), dev_i32([0, 2]),
                                    dev_i32([0, 2]), 1.0, host_probs=torch.empty(2, pin_memory=True))
    assert e.value.status == blink.BLINK_DEVICE_FLAG
