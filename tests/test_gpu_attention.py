"""tcgen05 prefix-tail attention vs the FP64 oracle (blink.py PREFIX_CACHE note, `_forward_shared`).

Every output row is compared, at the small sizes and at the full 2k, 18k and plain workloads;
the largest request on four whole questions, one whole kv-head group and sampled pairs.  Tolerance: max |O - O_ref| within
2e-2 of max |O_ref|; LSE within 2e-3 (absolute, natural log, scaled for large values).
"""
import numpy as np
import pytest
import torch

from shared_prefix_question_gb300 import blink
from shared_prefix_question_gb300 import workloads as wl
from tests.helpers import compare_attention, dev_bf16, owned_rows, run_attention, sample_pairs

pytestmark = pytest.mark.gpu


def _w(name, index, P, Hq, Hkv, d):
    return wl.Workload(name, index, P, 0, 1, 1, Hq, Hkv, d, 8, 8, 1, 1, 1.0, "letters")


SMALL = [
    # name, P, lengths, Hq, Hkv, d
    ("tiny", 64, [8, 12, 16, 24], 4, 2, 64),
    ("ragged-prefix-g4", 200, [1, 5, 37, 130, 3], 8, 2, 128),
    ("g5", 300, [10, 70, 25], 10, 2, 128),
    ("g1-d64", 129, [3, 200], 2, 2, 64),
    ("no-prefix", 0, [1, 17, 300, 64], 8, 2, 128),
    ("g8", 256, [33, 7], 16, 2, 128),
    ("many-short", 77, list(np.random.default_rng(3).integers(1, 5, size=40)), 8, 2, 128),
    ("single-row", 1, [1], 4, 4, 64),
    ("long-tail", 128, [700, 2], 4, 1, 128),
]


@pytest.mark.parametrize("case", SMALL, ids=lambda c: c[0])
def test_attention_small_all_rows(case):
    name, P, lengths, Hq, Hkv, d = case
    ins = wl.attention_inputs(_w(name, 300 + len(name), P, Hq, Hkv, d), lengths=np.array(lengths), P=P)
    out, lse, st = run_attention(ins)
    assert st == blink.BLINK_OK
    compare_attention(ins, out, lse)


def test_attention_padded_layout():
    P, lengths, width = 130, [5, 40, 1], 48
    ins = wl.attention_inputs(_w("pad", 400, P, 4, 1, 128), lengths=np.array(lengths), P=P, padded_width=width)
    out, lse, st = run_attention(ins, padded=True)
    assert st == blink.BLINK_OK
    compare_attention(ins, out, lse)
    owned = np.zeros(ins.rows, dtype=bool)
    for s, L in zip(ins.seq_start, ins.seq_len):
        owned[s:s + L] = True
    assert (out[~owned] == 0).all()
    assert np.isneginf(lse[:, ~owned]).all()


def test_attention_arena_slice():
    """The prefix is a region of a wider KV arena (simit engine.py: one arena, a region per
    request): rows start at an arena offset and are `stride` elements apart."""
    P, Hq, Hkv, d = 300, 8, 2, 128
    ins = wl.attention_inputs(_w("arena", 401, P, Hq, Hkv, d), lengths=np.array([20, 9]), P=P)
    stride = Hkv * d + 64
    kstart = 37
    arena_k = torch.zeros(kstart + P + 5, stride, dtype=torch.bfloat16, device="cuda")
    arena_v = torch.zeros_like(arena_k)
    arena_k[kstart:kstart + P, :Hkv * d] = dev_bf16(ins.k_pre).reshape(P, -1)
    arena_v[kstart:kstart + P, :Hkv * d] = dev_bf16(ins.v_pre).reshape(P, -1)
    out, lse, st = run_attention(ins, pre_row_stride=stride, k_pre_dev=arena_k[kstart], v_pre_dev=arena_v[kstart])
    assert st == blink.BLINK_OK
    compare_attention(ins, out, lse)


def test_attention_cu_slice_offsets():
    """A slice of a larger cu_seqlens array (cu[0] != 0) with pointers offset by cu[0] rows."""
    from tests.helpers import dev_i32, host_f64
    P, Hq, Hkv, d = 150, 4, 2, 64
    lengths = np.array([6, 9, 4, 11])
    ins = wl.attention_inputs(_w("slice", 402, P, Hq, Hkv, d), lengths=lengths, P=P)
    q, kt, vt = dev_bf16(ins.q), dev_bf16(ins.k_tail), dev_bf16(ins.v_tail)
    kp, vp = dev_bf16(ins.k_pre), dev_bf16(ins.v_pre)
    cu = dev_i32(ins.cu_seqlens)
    base = int(ins.cu_seqlens[2])
    out, lse, ws = blink.blink_prefix_tail_attention(q[base:], kp, vp, kt[base:], vt[base:], cu[2:], B=2, P=P,
                                                     max_tail=11, want_lse=True)
    torch.cuda.synchronize()
    assert blink.blink_read_device_status(ws) == blink.BLINK_OK
    full = np.full((ins.rows, Hq, d), np.nan)
    full[base:] = host_f64(out)
    full_lse = np.full((Hq, ins.rows), np.nan)
    full_lse[:, base:] = host_f64(lse)
    toks = np.arange(base, ins.rows, dtype=np.int32)
    for h in range(Hq):
        compare_attention(ins, full, full_lse, select=(toks, np.full_like(toks, h)))


def test_attention_device_flag_on_bad_length():
    """A question longer than max_tail is flagged on the device (no trap); other rows still run."""
    P = 64
    ins = wl.attention_inputs(_w("flag", 403, P, 4, 2, 64), lengths=np.array([8, 30]), P=P)
    out, lse, st = run_attention(ins, max_tail=16)
    assert st == blink.BLINK_DEVICE_FLAG


@pytest.mark.parametrize("name", ["2k", "18k", "plain"])
def test_attention_workloads_every_row(name):
    """Every output row of the full-size workloads against the oracle, in the launch shapes the
    benchmark times: the 18k tails packed in the plan's slot order (ascending length, as the step
    packs them), the 2k and plain workloads in request order (as the per-workload rows are timed)."""
    w = wl.WORKLOADS[name]
    lengths = wl.tail_lengths(w)
    if name == "18k":
        lengths = np.sort(lengths, kind="stable")
    ins = wl.attention_inputs(w, lengths=lengths)
    out, lse, st = run_attention(ins)
    assert st == blink.BLINK_OK
    compare_attention(ins, out, lse)


def test_attention_max_workload_whole_questions_and_kv_group():
    """The largest request (131072-token prefix, 512 tails, 40/8 heads).  Its every row would
    take the oracle about 40 minutes, so the comparison covers: four whole questions (every head,
    every tail row: the first, the last, the longest and one drawn at random), every row of the
    last kv head's group of five query heads over all 512 questions, and 256 sampled pairs that
    include every question's first and last tail row.  Every owned output is finite."""
    w = wl.WORKLOADS["max"]
    ins = wl.attention_inputs(w)
    out, lse, st = run_attention(ins)
    assert st == blink.BLINK_OK
    rng = np.random.default_rng(44)
    B, g = len(ins.seq_len), ins.Hq // ins.Hkv
    whole = sorted({0, B - 1, int(np.argmax(ins.seq_len)), int(rng.integers(1, B - 1))})
    toks, heads = [], []
    for b in whole:
        t = np.arange(ins.seq_start[b], ins.seq_start[b] + ins.seq_len[b])
        toks.append(np.repeat(t, ins.Hq))
        heads.append(np.tile(np.arange(ins.Hq), len(t)))
    rows = owned_rows(ins)
    group = np.arange((ins.Hkv - 1) * g, ins.Hkv * g)
    toks.append(np.repeat(rows, g))
    heads.append(np.tile(group, len(rows)))
    st_tok, st_head = sample_pairs(ins, 256, seed=w.index)
    toks.append(st_tok)
    heads.append(st_head)
    sel = (np.concatenate(toks).astype(np.int32), np.concatenate(heads).astype(np.int32))
    compare_attention(ins, out, lse, select=sel)
    assert np.isfinite(out[rows]).all()


@pytest.mark.parametrize("long_prefix", [False, True])
@pytest.mark.parametrize("Hq,Hkv,d", [(8, 2, 128), (10, 2, 128), (4, 2, 64)])
def test_attention_several_requests_one_launch(Hq, Hkv, d, long_prefix):
    """blink.py `logits_many` packs the questions of several requests into one forward; each
    request keeps its own prefix (a region of one KV arena, simit engine.py).  Every request's
    rows must equal the single-request oracle over that request's prefix."""
    from tests.helpers import dev_i32, host_f64
    rng = np.random.default_rng(Hq * 7 + d + 1000 * long_prefix)
    reqs = [  # (prefix length, tail lengths)
        (300, [17, 5, 40]),
        (0, [33, 2]),        # a request on the plain causal path
        (129, [1, 64, 9, 12]),
        (1000, [90]),
    ]
    if long_prefix:  # one request long enough that the launch uses the two-tile kernel
        reqs.append((3300, [30, 7]))
    stride = Hkv * d + 64
    starts, slot = [], 7
    for P, _ in reqs:
        starts.append(slot)
        slot += P + 13
    slots = slot
    arena_k = wl.normal_bf16(rng, (slots, stride))
    arena_v = wl.normal_bf16(rng, (slots, stride))
    lengths = [L for _, tails in reqs for L in tails]
    rows = int(sum(lengths))
    q = wl.normal_bf16(rng, (rows, Hq, d))
    kt = wl.normal_bf16(rng, (rows, Hkv, d))
    vt = wl.normal_bf16(rng, (rows, Hkv, d))
    cu = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32)
    req_rows = [0]
    for _, tails in reqs:
        req_rows.append(req_rows[-1] + sum(tails))
    out, lse, ws = blink.blink_prefix_tail_attention_multi(
        dev_bf16(q), dev_bf16(arena_k), dev_bf16(arena_v), dev_bf16(kt), dev_bf16(vt), dev_i32(cu), B=len(lengths),
        req_rows=req_rows, req_prefix_start=starts, req_prefix_len=[P for P, _ in reqs], max_tail=max(lengths),
        want_lse=True, arena_row_stride=stride)
    torch.cuda.synchronize()
    assert blink.blink_read_device_status(ws) == blink.BLINK_OK
    out, lse = host_f64(out), host_f64(lse)
    qi = 0
    for (P, tails), s0, r0, r1 in zip(reqs, starts, req_rows[:-1], req_rows[1:]):
        kp = arena_k[s0:s0 + P, :Hkv * d].reshape(P, Hkv, d).copy()
        vp = arena_v[s0:s0 + P, :Hkv * d].reshape(P, Hkv, d).copy()
        sub = wl.AttentionInputs(q[r0:r1], kp, vp, kt[r0:r1], vt[r0:r1],
                                 (cu[qi:qi + len(tails)] - r0).astype(np.int32), np.array(tails, dtype=np.int32),
                                 (cu[qi:qi + len(tails) + 1] - r0).astype(np.int32), r1 - r0, P, Hq, Hkv, d)
        compare_attention(sub, out[r0:r1], lse[:, r0:r1])
        qi += len(tails)


@pytest.mark.parametrize("case", [
    # name, P, lengths, Hq, Hkv, d, padded width (0: varlen)
    ("one-question", 4096, [40], 8, 2, 128, 0),
    ("three-padded-g5-d64", 3000, [5, 33, 17], 10, 2, 64, 48),
    ("one-question-18k-shape", 18432, [64], 32, 8, 128, 0),
], ids=lambda c: c[0])
def test_attention_split_prefix_small_grid(case):
    """A grid that fills a small part of the GPU (a single question against a long prefix) cuts
    the prefix into chunks run by separate blocks; their partial outputs are merged by LSE, the
    same merge as the prefix and tail parts.  Every row matches the oracle."""
    name, P, lengths, Hq, Hkv, d, width = case
    ins = wl.attention_inputs(_w(name, 500 + len(name), P, Hq, Hkv, d), lengths=np.array(lengths), P=P,
                              padded_width=width or None)
    rows = ins.rows
    assert blink.attention_workspace_bytes(rows, len(lengths), P, Hq, Hkv, d) > 256  # the split path
    out, lse, st = run_attention(ins, padded=bool(width))
    assert st == blink.BLINK_OK
    compare_attention(ins, out, lse)
    if width:
        owned = np.zeros(ins.rows, dtype=bool)
        for s, L in zip(ins.seq_start, ins.seq_len):
            owned[s:s + L] = True
        assert (out[~owned] == 0).all()
        assert np.isneginf(lse[:, ~owned]).all()


def test_bounded_wait_gives_up_and_the_context_stays_usable():
    """Every wait inside the kernels is bounded: one that never completes gives up, latches
    BLINK_DEVICE_TIMEOUT in the workspace's error word and returns, with nothing faulted.  The
    self-test waits on a barrier nothing arrives at (5 ms limit); afterwards the same workspace
    and context run an attention call that matches the oracle."""
    ws = blink.new_workspace(256, torch.device("cuda"))
    t0 = __import__("time").perf_counter()
    assert blink.blink_selftest_wait_timeout(5000, ws) == blink.BLINK_DEVICE_TIMEOUT
    assert __import__("time").perf_counter() - t0 < 5.0
    assert blink.blink_read_device_status(ws) == blink.BLINK_OK  # the self-test cleared the word
    ins = wl.attention_inputs(_w("after-timeout", 600, 64, 4, 2, 64), lengths=np.array([8, 12]), P=64)
    out, lse, st = run_attention(ins)
    assert st == blink.BLINK_OK
    compare_attention(ins, out, lse)


@pytest.mark.parametrize("case", [
    # name, P, n tails, Hq, Hkv, padded width (0: varlen)
    ("g2", 3072, 40, 16, 8, 0),
    ("g5-padded", 2500, 58, 10, 2, 64),
], ids=lambda c: c[0])
def test_attention_two_tile_kernel_all_rows(case):
    """A prefix of 20-24 key tiles with short tails runs the two-tile kernel (a block's estimated
    KV iterations exceed the single-tile limit) in one wave of at most 152 blocks (the prefix is not
    split: enough blocks for a small-grid split not to pay, no partial second wave to split);
    every row matches the oracle.  Both cases end a kv head's blocks on a row pair whose second
    tile starts past the last row; g = 5 leaves 3 of every 128 tile rows unused; the padded case
    checks that rows no question owns stay zero with LSE -inf.  (The small cases above, with a
    short prefix, run the single-tile kernel.)"""
    name, P, n, Hq, Hkv, width = case
    d = 128
    lengths = np.random.default_rng(41 + n).integers(20, 49, size=n)
    ins = wl.attention_inputs(_w("two-tile-" + name, 700 + n, P, Hq, Hkv, d), lengths=lengths, P=P,
                              padded_width=width or None)
    tpt = 128 // (Hq // Hkv)
    assert (ins.rows + tpt - 1) // tpt % 2 == 1  # an odd tile count: the last block has one tile
    assert blink.attention_workspace_bytes(ins.rows, len(lengths), P, Hq, Hkv, d) == 256  # unsplit
    out, lse, st = run_attention(ins, padded=bool(width))
    assert st == blink.BLINK_OK
    compare_attention(ins, out, lse)
    if width:
        owned = np.zeros(ins.rows, dtype=bool)
        for s, L in zip(ins.seq_start, ins.seq_len):
            owned[s:s + L] = True
        assert (out[~owned] == 0).all()
        assert np.isneginf(lse[:, ~owned]).all()


@pytest.mark.parametrize("case", [
    # name, P, Hq, Hkv, d, padded width (0: varlen)
    ("d128-g4", 1024, 32, 8, 128, 0),
    ("d64-g5-padded", 1000, 10, 2, 64, 64),
], ids=lambda c: c[0])
def test_attention_split_of_the_last_partial_wave(case):
    """A launch a few (row pair, kv head) units longer than the GPU has SMs (the 2k workload's
    shape: 160 units on 152 SMs) runs whole waves unsplit and cuts only the last partial wave's
    units into prefix chunks, merged by LSE.  Every row matches the oracle, whichever launch
    computed it; rows owned by no question stay zero with LSE -inf."""
    name, P, Hq, Hkv, d, width = case
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    tpt = 128 // (Hq // Hkv)
    pairs = -(-(sms + 8) // Hkv)                 # row pairs per kv head: units = sms + 8 or a few more
    n = pairs * 2 * tpt // (width or 40)         # questions of about 40 tokens (or padded rows)
    rng = np.random.default_rng(900 + d)
    lengths = rng.integers(30, 51, size=n)
    ins = wl.attention_inputs(_w("tail-wave-" + name, 800 + d, P, Hq, Hkv, d), lengths=lengths, P=P,
                              padded_width=width or None)
    units = ((ins.rows + tpt - 1) // tpt + 1) // 2 * Hkv
    assert sms < units < 2 * sms
    assert blink.attention_workspace_bytes(ins.rows, len(lengths), P, Hq, Hkv, d) > 256  # the split path
    out, lse, st = run_attention(ins, padded=bool(width))
    assert st == blink.BLINK_OK
    compare_attention(ins, out, lse)
    if width:
        owned = np.zeros(ins.rows, dtype=bool)
        for s0, L in zip(ins.seq_start, ins.seq_len):
            owned[s0:s0 + L] = True
        assert (out[~owned] == 0).all()
        assert np.isneginf(lse[:, ~owned]).all()


@pytest.mark.gpu
def test_workspace_query_holds_the_split_plan():
    """blink_attention_workspace sizes the fp32 partials of exactly the plan blink_attention_split_plan
    reports for this GPU's SM count (256-byte header, then LSE and O of every chunk of every cut
    unit, each region 256-byte aligned)."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    for rows, P, Hq, Hkv, d in [(1306, 2048, 32, 8, 128), (128, 18432, 32, 8, 128), (64, 18432, 32, 8, 128),
                                (40, 4096, 8, 2, 128), (144, 3000, 10, 2, 64), (10627, 18432, 32, 8, 128)]:
        whole, S, c = blink.blink_attention_split_plan(rows, P, Hq, Hkv, d, sms)
        ws = blink.attention_workspace_bytes(rows, 1, P, Hq, Hkv, d)
        if S == 1:
            assert ws == 256
            continue
        tpt = 128 // (Hq // Hkv)
        units = (-(-rows // tpt) + 1) // 2 * Hkv
        n = (units - whole) * S
        up = lambda x: -(-x // 256) * 256
        assert ws == 256 + up(n * 256 * 4) + up(n * 256 * d * 4)
