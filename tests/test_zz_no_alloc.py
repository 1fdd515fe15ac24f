"""The readout entry point that allocates nothing (blink_label_readout_noalloc).

Some callers cannot allocate device memory: a host that gives this code only its input and
output buffers and owns the rest of the device memory, or a latency-critical loop that must not
call cudaMalloc (it can synchronise the whole device).  For them the library keeps the readout's
scratch in a static device array.  This test calls that entry point through the C ABI and checks
it against the workspace entry point on two calls in a row, on a small and on a large label
count (the large one takes the two-launch form that needs no tickets), and checks that a call
which failed on the device (a label id outside the vocabulary, flagged in the shared array's error
word) leaves nothing behind that disturbs the next call.  It is collected last so that a run that
stops at the first failure has already run every other test.
"""
import ctypes

import numpy as np
import pytest
import torch

from shared_prefix_question_gb300 import blink
from shared_prefix_question_gb300 import workloads as wl
from tests.helpers import PROB_ABS_TOL, dev_bf16, dev_i32

pytestmark = pytest.mark.gpu


def _vp(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else None


def _inputs(name):
    w = wl.WORKLOADS[name]
    rng = np.random.default_rng(99)
    unembed = None if name == "tiny" else wl.normal_bf16(rng, (w.V, w.H), std=0.02)
    ins = wl.readout_inputs(w, unembed=unembed)
    dev = {"hidden": dev_bf16(ins.hidden), "W": dev_bf16(ins.unembed), "last": dev_i32(ins.last_idx),
           "off": dev_i32(ins.label_off), "ids": dev_i32(ins.label_ids)}
    return ins, dev


def _noalloc(dev, ids, B, sum_k, temperature):
    """One call through the C ABI with a host copy; returns (status, host probs, device probs)."""
    L = blink.lib()
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    probs = torch.full((sum_k,), float("nan"), dtype=torch.float32, device="cuda")
    host = torch.empty(sum_k, dtype=torch.float32, pin_memory=True)
    hidden, W = dev["hidden"], dev["W"]
    st = L.blink_label_readout_noalloc(_vp(hidden), hidden.stride(0), hidden.shape[0], _vp(dev["last"]), None,
                                       _vp(W), W.shape[0], W.shape[1], _vp(dev["off"]), _vp(ids), B, sum_k,
                                       ctypes.c_float(temperature), _vp(probs), _vp(host), None, stream)
    return st, host.numpy().copy(), probs.cpu().numpy()


@pytest.mark.parametrize("name", ["tiny", "18k", "max"])
def test_noalloc_matches_workspace_readout_twice(name):
    ins, dev = _inputs(name)
    B, sum_k = len(ins.last_idx), len(ins.label_ids)
    ref, _ = blink.blink_label_readout(dev["hidden"], dev["last"], dev["W"], dev["off"], dev["ids"], ins.temperature)
    torch.cuda.synchronize()
    ref = ref.cpu().numpy()
    for call in range(2):
        st, got, on_device = _noalloc(dev, dev["ids"], B, sum_k, ins.temperature)
        assert st == blink.BLINK_OK, f"call {call}: status {st}"
        assert np.isfinite(got).all()
        assert np.abs(got - ref).max() <= PROB_ABS_TOL, f"call {call}"
        np.testing.assert_array_equal(on_device, got)


@pytest.mark.parametrize("name", ["tiny", "max"])
def test_noalloc_call_after_a_flagged_call(name):
    """A label id past the vocabulary is caught on the device (its row is not read; the question's
    probabilities become NaN and the error word is set).  The next call, on the same stream with
    valid ids, starts from a cleared word: BLINK_OK and the workspace readout's probabilities."""
    ins, dev = _inputs(name)
    B, sum_k = len(ins.last_idx), len(ins.label_ids)
    bad_ids = ins.label_ids.copy()
    bad_ids[ins.label_off[1]] = ins.unembed.shape[0] + 5  # first label of question 1
    st, got, _ = _noalloc(dev, dev_i32(bad_ids), B, sum_k, ins.temperature)
    assert st == blink.BLINK_DEVICE_FLAG
    assert np.isnan(got[ins.label_off[1]:ins.label_off[2]]).all()
    ref, _ = blink.blink_label_readout(dev["hidden"], dev["last"], dev["W"], dev["off"], dev["ids"], ins.temperature)
    torch.cuda.synchronize()
    st, got, _ = _noalloc(dev, dev["ids"], B, sum_k, ins.temperature)
    assert st == blink.BLINK_OK
    assert np.abs(got - ref.cpu().numpy()).max() <= PROB_ABS_TOL


def test_noalloc_rejects_more_questions_than_its_scratch():
    L = blink.lib()
    fake = ctypes.c_void_p(0x1000)  # refused on the host before any use
    st = L.blink_label_readout_noalloc(fake, 256, 4, fake, None, fake, 1024, 256, fake, fake,
                                       blink.STATIC_SCRATCH_QUESTIONS + 1, blink.STATIC_SCRATCH_QUESTIONS + 1,
                                       ctypes.c_float(1.0), fake, None, None, None)
    assert st == blink.BLINK_OUT_OF_RANGE
