"""The prefix-chunk plan (host logic, CPU only): which units of a one-request launch run whole and
how the others' prefix tiles are cut into chunks.  The kernel gives chunk j of a cut unit the
prefix tiles [j c, j c + max(0, min(n_pre - j c, c))) and the last chunk the tail tiles too, so a
plan is valid when every prefix tile lands in exactly one chunk and only the last chunk can come
out short or empty; the whole units and the chunks must fit the launch forms (a small grid of at
most four waves, or whole waves plus one wave of chunks)."""
import itertools

import pytest

from shared_prefix_question_gb300 import blink, build
from shared_prefix_question_gb300 import workloads as wl

BN = 128


@pytest.fixture(scope="module")
def lib():
    build.build()
    return blink.lib()


def _units(rows, Hq, Hkv):
    tpt = 128 // (Hq // Hkv)
    return (-(-rows // tpt) + 1) // 2 * Hkv


def _check_plan(rows, P, Hq, Hkv, d, sms):
    whole, S, c = blink.blink_attention_split_plan(rows, P, Hq, Hkv, d, sms)
    units, n_pre = _units(rows, Hq, Hkv), -(-P // BN)
    assert S >= 1
    if S == 1:
        assert whole == units and c == n_pre
        return whole, S, c
    assert P > 0 and n_pre >= 2 and c >= 1
    # the chunk ranges the kernel derives, brute force: a partition of [0, n_pre)
    covered = []
    for j in range(S):
        n = max(0, min(n_pre - j * c, c))
        if j < S - 1:
            assert n == c  # only the last chunk may be short or empty
        covered.extend(range(j * c, j * c + n))
    assert covered == list(range(n_pre))
    rest = units - whole
    if whole == 0:          # a small grid: every unit cut, chunks of >= 4 tiles, within four waves
        assert units * S <= 4 * sms and c >= 4
    else:                   # whole waves run whole, the last partial wave's units cut into one more wave
        assert whole % sms == 0 and 0 < rest and rest * S <= sms
    return whole, S, c


def test_split_plan_partitions_the_prefix_tiles(lib):
    shapes = [(4, 2), (8, 2), (10, 2), (16, 8), (32, 8), (40, 8), (8, 8)]
    for sms, d, (Hq, Hkv), P, rows in itertools.product(
            (132, 148, 152, 160), (64, 128), shapes,
            (0, 100, 128, 129, 1000, 2048, 4096, 18432, 131072),
            (1, 5, 40, 128, 300, 1306, 5000, 10627, 30000)):
        _check_plan(rows, P, Hq, Hkv, d, sms)


def test_split_plans_of_the_measured_workloads(lib):
    """The plans the timed rows run on a 152-SM GB300 (the model's choices, pinned so that a
    change to the model shows up here)."""
    rows_2k = int(wl.tail_lengths(wl.WORKLOADS["2k"]).sum())
    assert _check_plan(rows_2k, 2048, 32, 8, 128, 152) == (152, 6, 3)    # 168 units: 152 whole, 16 cut
    assert _check_plan(128, 18432, 32, 8, 128, 152) == (0, 9, 16)       # one question of 128 tokens
    assert _check_plan(64, 18432, 32, 8, 128, 152) == (0, 17, 9)        # one question of 64 tokens
    rows_18k = int(wl.tail_lengths(wl.WORKLOADS["18k"]).sum())
    assert _check_plan(rows_18k, 18432, 32, 8, 128, 152)[1] == 1         # 1336 units: nothing cut
    rows_max = int(wl.tail_lengths(wl.WORKLOADS["max"]).sum())
    assert _check_plan(rows_max, 131072, 40, 8, 128, 152)[1] == 1
    assert _check_plan(150000, 0, 32, 8, 128, 152)[1] == 1               # no prefix: nothing to cut


def test_split_plan_rejects_bad_arguments(lib):
    for args in [(0, 2048, 32, 8, 128, 152), (100, -1, 32, 8, 128, 152), (100, 2048, 30, 8, 128, 152),
                 (100, 2048, 32, 8, 96, 152), (100, 2048, 32, 8, 128, 0)]:
        with pytest.raises(blink.BlinkError) as e:
            blink.blink_attention_split_plan(*args)
        assert e.value.status == blink.BLINK_INVALID_ARG
