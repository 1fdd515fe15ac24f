"""Fused label readout vs the FP64 oracle (blink.py `_read` / `_read_batched`, `softmax`).

Probabilities within 1e-3 absolute and the same argmax (ties to the first label in request
order, as blink.py's answer assembly breaks them); a near-tie (oracle logit gap < 1e-4)
accepts either of the two.
"""
import numpy as np
import pytest
import torch

from shared_prefix_question_gb300 import blink
from shared_prefix_question_gb300 import workloads as wl
from tests.helpers import compare_readout, dev_bf16, dev_i32

pytestmark = pytest.mark.gpu

_UNEMBED = {}


def _unembed(w):
    key = (w.V, w.H)
    if key not in _UNEMBED:
        rng = np.random.default_rng(7000 + w.H)
        _UNEMBED.clear()
        _UNEMBED[key] = wl.normal_bf16(rng, (w.V, w.H), std=0.02)
    return _UNEMBED[key]


def _run(ins, host=True, logits=False):
    hidden = dev_bf16(ins.hidden)
    W = dev_bf16(ins.unembed)
    sum_k = len(ins.label_ids)
    hp = torch.empty(sum_k, dtype=torch.float32, pin_memory=True) if host else None
    lg = torch.empty(sum_k, dtype=torch.float32, device="cuda") if logits else None
    probs, ws = blink.blink_label_readout(hidden, dev_i32(ins.last_idx), W, dev_i32(ins.label_off),
                                          dev_i32(ins.label_ids), ins.temperature, host_probs=hp, logits=lg)
    torch.cuda.synchronize()
    out = hp.numpy().astype(np.float64) if host else probs.cpu().numpy().astype(np.float64)
    return out, (lg.cpu().numpy() if logits else None), ws


@pytest.mark.parametrize("name", ["tiny", "2k", "18k", "plain", "max", "readout_stress"])
def test_readout_workloads(name):
    w = wl.WORKLOADS[name]
    ins = wl.readout_inputs(w, unembed=None if name == "tiny" else _unembed(w))
    probs, _, _ = _run(ins)
    compare_readout(probs, ins)


def test_readout_device_copy_and_logits():
    w = wl.WORKLOADS["tiny"]
    ins = wl.readout_inputs(w)
    probs, logits, _ = _run(ins, host=False, logits=True)
    compare_readout(probs, ins)
    from oracle import oracle
    z, _, _ = oracle.label_readout(ins.hidden, ins.last_idx, ins.unembed, ins.label_off, ins.label_ids, 1.0)
    assert np.abs(logits - z).max() < 1e-4


def test_readout_special_cases():
    rng = np.random.default_rng(11)
    H, V = 264, 500
    hidden = wl.normal_bf16(rng, (5, H))
    W = wl.normal_bf16(rng, (V, H), std=0.05)
    # one label -> 1; a repeated id -> uniform; 255 labels (the maximum)
    off = np.array([0, 1, 5, 5 + 255], dtype=np.int32)
    ids = np.concatenate([[3], [7, 7, 7, 7], rng.choice(V, 255, replace=False)]).astype(np.int32)
    ins = wl.ReadoutInputs(hidden, np.array([4, 0, 2], dtype=np.int32), W, off, ids, 0.37)
    probs, _, _ = _run(ins)
    assert probs[0] == 1.0
    np.testing.assert_allclose(probs[1:5], 0.25, atol=1e-7)
    compare_readout(probs, ins)


def test_readout_bad_label_flagged():
    rng = np.random.default_rng(12)
    H, V = 64, 100
    hidden = wl.normal_bf16(rng, (2, H))
    W = wl.normal_bf16(rng, (V, H))
    off = np.array([0, 2, 4], dtype=np.int32)
    ids = np.array([1, 2, 3, V], dtype=np.int32)  # the last id is out of range
    hp = torch.empty(4, dtype=torch.float32, pin_memory=True)
    with pytest.raises(blink.BlinkError) as e:
        blink.blink_label_readout(dev_bf16(hidden), dev_i32([0, 1]), dev_bf16(W), dev_i32(off), dev_i32(ids), 1.0,
                                  host_probs=hp)
    assert e.value.status == blink.BLINK_DEVICE_FLAG
    p = hp.numpy()
    assert np.isfinite(p[:2]).all() and abs(p[:2].sum() - 1) < 1e-6
    assert np.isnan(p[2:]).all()


def test_readout_repeated_calls_reuse_workspace():
    w = wl.WORKLOADS["tiny"]
    ins = wl.readout_inputs(w)
    hidden, W = dev_bf16(ins.hidden), dev_bf16(ins.unembed)
    last, off, ids = dev_i32(ins.last_idx), dev_i32(ins.label_off), dev_i32(ins.label_ids)
    ws = None
    for _ in range(3):
        probs, ws = blink.blink_label_readout(hidden, last, W, off, ids, 1.0, ws=ws)
        torch.cuda.synchronize()
        compare_readout(probs.cpu().numpy().astype(np.float64), ins)


@pytest.mark.parametrize("name", ["tiny", "18k", "max"])
def test_readout_answers(name):
    """blink.py `answer_for` on the device, fused into the readout, against the oracle's answers
    computed from the oracle's probabilities."""
    from oracle import oracle
    from tests.helpers import ARGMAX_TIE_GAP
    w = wl.WORKLOADS[name]
    ins = wl.readout_inputs(w, unembed=None if name == "tiny" else _unembed(w))
    qt = wl.question_types(w, ins.label_off)
    hidden = dev_bf16(ins.hidden)
    W = dev_bf16(ins.unembed)
    hp = torch.empty(len(ins.label_ids), dtype=torch.float32, pin_memory=True)
    ha = torch.empty(len(ins.last_idx), 3, dtype=torch.float32, pin_memory=True)
    probs, ws, answers = blink.blink_label_readout(hidden, dev_i32(ins.last_idx), W, dev_i32(ins.label_off),
                                                   dev_i32(ins.label_ids), ins.temperature, host_probs=hp,
                                                   qtype=dev_i32(qt), host_answers=ha)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(answers.cpu().numpy(), ha.numpy())
    z, p_ref, st = oracle.label_readout(ins.hidden, ins.last_idx, ins.unembed, ins.label_off, ins.label_ids,
                                        ins.temperature)
    got = ha.numpy().astype(np.float64)
    for b in range(len(ins.last_idx)):
        lo, hi = ins.label_off[b], ins.label_off[b + 1]
        ref = oracle.answer(int(qt[b]), p_ref[lo:hi])
        zb = z[lo:hi]
        top = np.argsort(-zb, kind="stable")
        near_tie = hi - lo >= 2 and zb[top[0]] - zb[top[1]] < ARGMAX_TIE_GAP
        if near_tie:
            assert int(got[b, 0]) in (int(top[0]), int(top[1]))
        else:
            assert int(got[b, 0]) == ref["index"], b
            K = hi - lo
            tol = 1e-3 * max(1, K) if qt[b] == wl.QTYPE_SCORE else 1e-3
            if np.isnan(ref["confidence"]):
                assert np.isnan(got[b, 1])
            else:
                assert abs(got[b, 1] - ref["confidence"]) <= 2e-3
            assert abs(got[b, 2] - ref["value"]) <= tol


@pytest.mark.parametrize("with_slots", [False, True])
def test_readout_two_launch_path_matches_fused(with_slots):
    """From 8192 labels on, the readout writes every logit first and runs the softmaxes (and
    answers) in a second launch, one warp per question; below that, the warp that completes a
    question runs its softmax.  Both compute each label's FP32 dot and each softmax the same way,
    so the workspace entry (two launches here) equals the no-alloc entry (fused) bit for bit, and
    both match the oracle.  Questions share a pool of ids, some repeat an id inside one question,
    and H = 5128 leaves a ragged last batch of chunks."""
    rng = np.random.default_rng(31 + with_slots)
    H, V, B = 5128, 4000, 500
    pool = rng.choice(V, 40, replace=False)
    ks = rng.integers(1, 41, size=B)
    parts = []
    for b, k in enumerate(ks):
        if b % 7 == 0:
            parts.append(rng.choice(V, k))  # repeats inside one question too
        elif b % 2:
            parts.append(pool[:k])
        else:
            parts.append(rng.permutation(pool)[:k])
    off = np.concatenate([[0], np.cumsum(ks)]).astype(np.int32)
    ids = np.concatenate(parts).astype(np.int32)
    assert len(ids) >= 8192  # the two-launch path
    rows = B + 5
    hidden = wl.normal_bf16(rng, (rows, H))
    W = wl.normal_bf16(rng, (V, H), std=0.02)
    last = rng.permutation(rows)[:B].astype(np.int32)
    slot_of = rng.permutation(B).astype(np.int32) if with_slots else None
    per_slot = np.empty(B, dtype=np.int32)
    if with_slots:
        per_slot[slot_of] = last  # question b reads last_by_slot[slot_of[b]] == last[b]
    ins = wl.ReadoutInputs(hidden, last, W, off, ids, 0.7)
    d_hidden, d_W, d_off, d_ids = dev_bf16(hidden), dev_bf16(W), dev_i32(off), dev_i32(ids)
    d_last = dev_i32(per_slot if with_slots else last)
    d_slot = dev_i32(slot_of) if with_slots else None
    lg_two = torch.empty(len(ids), dtype=torch.float32, device="cuda")
    lg_fused = torch.empty_like(lg_two)
    p_two, ws = blink.blink_label_readout(d_hidden, d_last, d_W, d_off, d_ids, 0.7, logits=lg_two, slot_of=d_slot)
    p_fused = blink.blink_label_readout_noalloc(d_hidden, d_last, d_W, d_off, d_ids, 0.7, logits=lg_fused,
                                                slot_of=d_slot)
    torch.cuda.synchronize()
    assert blink.blink_read_device_status(ws) == blink.BLINK_OK
    assert torch.equal(lg_two, lg_fused)
    assert torch.equal(p_two, p_fused)
    compare_readout(p_two.cpu().numpy().astype(np.float64), ins)


@pytest.mark.parametrize("with_slots", [False, True])
def test_readout_ragged_rows_and_shared_ids(with_slots):
    """Full-size rows whose last batch of 16-byte chunks is ragged (H = 5128: two batches of 256
    chunks, then 129), label ids shared across questions (blink.py `render` offers the first K
    labels of one pool) and repeated inside some questions, hidden rows reached through a slot
    map: the probabilities match the oracle."""
    rng = np.random.default_rng(31 + with_slots)
    H, V, B = 5128, 4000, 120
    pool = rng.choice(V, 40, replace=False)
    ks = rng.integers(1, 41, size=B)
    parts = []
    for b, k in enumerate(ks):
        if b % 7 == 0:
            parts.append(rng.choice(V, k))  # repeats inside one question too
        elif b % 2:
            parts.append(pool[:k])
        else:
            parts.append(rng.permutation(pool)[:k])
    off = np.concatenate([[0], np.cumsum(ks)]).astype(np.int32)
    ids = np.concatenate(parts).astype(np.int32)
    rows = B + 5
    hidden = wl.normal_bf16(rng, (rows, H))
    W = wl.normal_bf16(rng, (V, H), std=0.02)
    last = rng.permutation(rows)[:B].astype(np.int32)
    slot_of = rng.permutation(B).astype(np.int32) if with_slots else None
    per_slot = np.empty(B, dtype=np.int32)
    if with_slots:
        per_slot[slot_of] = last  # question b reads last_by_slot[slot_of[b]] == last[b]
    ins = wl.ReadoutInputs(hidden, last, W, off, ids, 0.7)
    probs, ws = blink.blink_label_readout(dev_bf16(hidden), dev_i32(per_slot if with_slots else last), dev_bf16(W),
                                          dev_i32(off), dev_i32(ids), 0.7,
                                          slot_of=dev_i32(slot_of) if with_slots else None)
    torch.cuda.synchronize()
    assert blink.blink_read_device_status(ws) == blink.BLINK_OK
    compare_readout(probs.cpu().numpy().astype(np.float64), ins)
