"""The readout entry point that allocates nothing (blink_label_readout_noalloc).

Some callers cannot allocate device memory: a host that gives this code only its input and
output buffers and owns the rest of the device memory, or a latency-critical loop that must not
call cudaMalloc (it can synchronise the whole device).  For them the library keeps the readout's
scratch in a static device array.  This test calls that entry point through the C ABI and checks
it against the workspace entry point on two calls in a row (the second call must not be
disturbed by what the first left in the shared array).  It is collected last so that a run that
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


@pytest.mark.parametrize("name", ["tiny", "18k"])
def test_noalloc_matches_workspace_readout_twice(name):
    w = wl.WORKLOADS[name]
    rng = np.random.default_rng(99)
    unembed = None if name == "tiny" else wl.normal_bf16(rng, (w.V, w.H), std=0.02)
    ins = wl.readout_inputs(w, unembed=unembed)
    hidden, W = dev_bf16(ins.hidden), dev_bf16(ins.unembed)
    last, off, ids = dev_i32(ins.last_idx), dev_i32(ins.label_off), dev_i32(ins.label_ids)
    B, sum_k = len(ins.last_idx), len(ins.label_ids)
    L = blink.lib()
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    ref, _ = blink.blink_label_readout(hidden, last, W, off, ids, ins.temperature)
    torch.cuda.synchronize()
    ref = ref.cpu().numpy()
    for call in range(2):
        probs = torch.full((sum_k,), float("nan"), dtype=torch.float32, device="cuda")
        host = torch.empty(sum_k, dtype=torch.float32, pin_memory=True)
        st = L.blink_label_readout_noalloc(_vp(hidden), hidden.stride(0), hidden.shape[0], _vp(last), None, _vp(W),
                                           W.shape[0], W.shape[1], _vp(off), _vp(ids), B, sum_k,
                                           ctypes.c_float(ins.temperature), _vp(probs), _vp(host), None, stream)
        assert st == blink.BLINK_OK, f"call {call}: status {st}"
        got = host.numpy()
        assert np.isfinite(got).all()
        assert np.abs(got - ref).max() <= PROB_ABS_TOL, f"call {call}"
        np.testing.assert_array_equal(probs.cpu().numpy(), got)


def test_noalloc_rejects_more_questions_than_its_scratch():
    L = blink.lib()
    fake = ctypes.c_void_p(0x1000)  # refused on the host before any use
    st = L.blink_label_readout_noalloc(fake, 256, 4, fake, None, fake, 1024, 256, fake, fake,
                                       blink.STATIC_SCRATCH_QUESTIONS + 1, blink.STATIC_SCRATCH_QUESTIONS + 1,
                                       ctypes.c_float(1.0), fake, None, None, None)
    assert st == blink.BLINK_OUT_OF_RANGE
