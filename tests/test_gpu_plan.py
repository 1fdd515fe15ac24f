"""Device pack plan vs the oracle's sequential rule (blink.py `_batches` / `_padded`): bit-exact."""
import numpy as np
import pytest
import torch

from oracle import oracle
from shared_prefix_question_gb300 import blink
from shared_prefix_question_gb300 import workloads as wl
from tests.helpers import dev_i32

pytestmark = pytest.mark.gpu

KEYS = ("order", "fwd_of_slot", "fwd_slot_start", "fwd_width", "cu_seqlens", "last_varlen", "last_padded")


def _check(lengths, budget, max_rows):
    d = blink.blink_pack_plan(dev_i32(lengths), budget, max_rows, sync=True)
    ref = oracle.pack_plan(lengths, budget, max_rows)
    assert d["n_forwards"] == ref["n_forwards"]
    for k in KEYS:
        np.testing.assert_array_equal(d[k].cpu().numpy(), ref[k], err_msg=k)
    inv = np.empty_like(ref["order"])
    inv[ref["order"]] = np.arange(len(lengths), dtype=np.int32)
    np.testing.assert_array_equal(d["slot_of"].cpu().numpy(), inv)


# 2049 and up: the keys are sorted over the whole GPU (block-sorted runs of 1024, then merge
# rounds), including a short last run (2049, 5000, 17000) and an unpaired one (9000)
@pytest.mark.parametrize("n", [1, 2, 3, 64, 255, 256, 1000, 2048, 2049, 4096, 5000, 9000, 17000, 32768])
def test_plan_random(n):
    rng = np.random.default_rng(n)
    for budget, max_rows, hi in ((32768, 0, 1000), (32768, 7, 256), (100, 0, 60), (1, 0, 5), (10 ** 9, 0, 131072),
                                 (5000, 64, 131072)):
        lengths = rng.integers(1, hi + 1, size=n).astype(np.int32)
        _check(lengths, budget, max_rows)


def test_plan_ties_and_edges():
    _check(np.full(300, 17, dtype=np.int32), 17 * 10, 0)          # all equal: request order, 10 per forward
    _check(np.full(300, 17, dtype=np.int32), 17 * 10, 1)          # row cap 1: one forward per slot
    _check(np.array([131072, 1, 131072], dtype=np.int32), 32768, 0)  # longer than the budget runs alone
    _check(np.arange(1, 2049, dtype=np.int32)[::-1].copy(), 32768, 0)
    _check(np.full(32768, 131072, dtype=np.int32), 32768, 0)      # every slot alone: 32768 forwards


@pytest.mark.parametrize("name", ["tiny", "2k", "18k", "plain", "max"])
def test_plan_workloads(name):
    w = wl.WORKLOADS[name]
    lengths = wl.tail_lengths(w)
    _check(lengths, wl.TOKEN_BUDGET, 0)
    if w.P:
        rows_cap = max(1, wl.PREFIX_KV_TOKENS // (w.P + int(lengths.max())))  # blink.py `_forward_shared`
        _check(lengths, wl.TOKEN_BUDGET, rows_cap)


def test_plan_rejects_bad_length_on_device():
    for bad in (0, -3, 131073):
        lengths = np.array([5, bad, 7], dtype=np.int32)
        with pytest.raises(blink.BlinkError) as e:
            blink.blink_pack_plan(dev_i32(lengths), 100, 0, sync=True)
        assert e.value.status == blink.BLINK_DEVICE_FLAG
        big = np.full(6000, 9, dtype=np.int32)  # the whole-GPU sort path flags it the same way
        big[4321] = bad
        with pytest.raises(blink.BlinkError) as e:
            blink.blink_pack_plan(dev_i32(big), 100, 0, sync=True)
        assert e.value.status == blink.BLINK_DEVICE_FLAG
    d = blink.blink_pack_plan(dev_i32(np.array([5, 7], dtype=np.int32)), 100, 0, sync=False)
    torch.cuda.synchronize()
    assert int(d["n_forwards_dev"].item()) == 1
