"""Pins for the oracle's prefix-tail attention, CPU only.

The pages' statement of the shared-prefix path (blink.py, PREFIX_CACHE note: "same tokens,
same positions; only floating-point order differs") says a tail run against the cached prefix
equals the same rows of one plain causal pass over [prefix ; tail].  The plain pass here is a
library routine, PyTorch's scaled_dot_product_attention in float64 with is_causal=True, run over
the concatenated sequence, so the oracle is pinned to something other than itself.  Closed
forms and special cases (constant values, a single key, identical keys) add pins that need no
library at all.
"""
import math

import numpy as np
import pytest
import torch

from oracle import oracle
from shared_prefix_question_gb300 import workloads as wl


def _f64(bits):
    return torch.from_numpy(wl.bits_to_f32(bits).astype(np.float64))


def _sdpa_reference(ins, b, prefix_q_bits):
    """Rows of question b from one causal SDPA pass over [prefix ; tail_b] (float64)."""
    P, Hq, Hkv, d = ins.P, ins.Hq, ins.Hkv, ins.d
    g = Hq // Hkv
    s, L = int(ins.seq_start[b]), int(ins.seq_len[b])
    q_tail = _f64(ins.q[s:s + L])                       # [L, Hq, d]
    q_pre = _f64(prefix_q_bits)                         # [P, Hq, d]
    q = torch.cat([q_pre, q_tail], 0).permute(1, 0, 2)  # [Hq, P+L, d]
    k = torch.cat([_f64(ins.k_pre), _f64(ins.k_tail[s:s + L])], 0).permute(1, 0, 2)
    v = torch.cat([_f64(ins.v_pre), _f64(ins.v_tail[s:s + L])], 0).permute(1, 0, 2)
    k = k.repeat_interleave(g, dim=0)                   # query head h reads kv head h // g
    v = v.repeat_interleave(g, dim=0)
    o = torch.nn.functional.scaled_dot_product_attention(q[None], k[None], v[None], is_causal=True)[0]
    scores = (q @ k.transpose(1, 2)) / math.sqrt(d)
    mask = torch.ones(P + L, P + L, dtype=torch.bool).tril()
    lse = torch.logsumexp(scores.masked_fill(~mask, float("-inf")), dim=-1)
    return o[:, P:].permute(1, 0, 2).numpy(), lse[:, P:].numpy()


@pytest.mark.parametrize("P,lengths,Hq,Hkv,d", [
    (64, [8, 12, 16, 24], 4, 2, 64),   # the tiny workload's shape
    (37, [1, 5, 9], 6, 3, 32),         # ragged sizes, group 2
    (0, [1, 7, 30], 4, 4, 16),         # no prefix: plain causal attention
    (50, [3, 11], 5, 1, 16),           # one kv head for five query heads
])
def test_attention_equals_causal_pass_over_concatenation(P, lengths, Hq, Hkv, d):
    w = wl.WORKLOADS["tiny"]
    w = wl.Workload("t", 90 + len(lengths) + P, P, len(lengths), 1, 1, Hq, Hkv, d, 8, 8, 1, 1, 1.0, "letters")
    ins = wl.attention_inputs(w, lengths=np.array(lengths), P=P)
    out, lse = oracle.prefix_tail_attention(ins.q, ins.k_pre, ins.v_pre, ins.k_tail, ins.v_tail,
                                            ins.seq_start, ins.seq_len, P, Hq, Hkv, d)
    rng = np.random.default_rng(5)
    prefix_q = wl.normal_bf16(rng, (P, Hq, d))
    for b in range(len(lengths)):
        s, L = int(ins.seq_start[b]), int(ins.seq_len[b])
        ref_o, ref_lse = _sdpa_reference(ins, b, prefix_q)
        np.testing.assert_allclose(out[s:s + L], ref_o, rtol=0, atol=1e-12)
        np.testing.assert_allclose(lse[:, s:s + L], ref_lse, rtol=0, atol=1e-12)


def test_padded_layout_equals_varlen():
    w = wl.WORKLOADS["tiny"]
    lengths = np.array([8, 12, 16, 24])
    var = wl.attention_inputs(w, lengths=lengths)
    width = 24
    rows = len(lengths) * width
    pad = {}
    for name in ("q", "k_tail", "v_tail"):
        src = getattr(var, name)
        dst = np.zeros((rows,) + src.shape[1:], dtype=np.uint16)
        for b, L in enumerate(lengths):
            dst[b * width:b * width + L] = src[var.seq_start[b]:var.seq_start[b] + L]
        pad[name] = dst
    starts = (np.arange(len(lengths)) * width).astype(np.int32)
    o1, l1 = oracle.prefix_tail_attention(var.q, var.k_pre, var.v_pre, var.k_tail, var.v_tail,
                                          var.seq_start, var.seq_len, w.P, w.Hq, w.Hkv, w.d)
    o2, l2 = oracle.prefix_tail_attention(pad["q"], var.k_pre, var.v_pre, pad["k_tail"], pad["v_tail"],
                                          starts, var.seq_len, w.P, w.Hq, w.Hkv, w.d)
    for b, L in enumerate(lengths):
        np.testing.assert_array_equal(o1[var.seq_start[b]:var.seq_start[b] + L], o2[b * width:b * width + L])
        np.testing.assert_array_equal(l1[:, var.seq_start[b]:var.seq_start[b] + L], l2[:, b * width:b * width + L])
    # padding rows are never computed
    assert np.isnan(o2[8:24]).all()


def test_constant_values_give_that_value():
    """If every visible value row is the same vector c, the output is c whatever the scores."""
    w = wl.WORKLOADS["tiny"]
    ins = wl.attention_inputs(w)
    c = wl.bf16_bits(np.linspace(-2, 2, w.d, dtype=np.float32))
    v_pre = np.broadcast_to(c, ins.v_pre.shape).copy()
    v_tail = np.broadcast_to(c, ins.v_tail.shape).copy()
    out, _ = oracle.prefix_tail_attention(ins.q, ins.k_pre, v_pre, ins.k_tail, v_tail, ins.seq_start,
                                          ins.seq_len, w.P, w.Hq, w.Hkv, w.d)
    ref = wl.bits_to_f32(c).astype(np.float64)
    np.testing.assert_allclose(out, np.broadcast_to(ref, out.shape), rtol=0, atol=1e-13)


def test_single_key_and_identical_keys():
    """With no prefix, a question's first row sees one key: O = v_0 and LSE = score.  With all keys
    equal, every score is the same s: O is the plain mean of the visible values and LSE = s + ln n."""
    Hq = Hkv = 2
    d = 16
    w = wl.Workload("k", 77, 0, 3, 1, 1, Hq, Hkv, d, 8, 8, 1, 1, 1.0, "letters")
    lengths = np.array([5, 1, 4])
    ins = wl.attention_inputs(w, lengths=lengths, P=0)
    out, lse = oracle.prefix_tail_attention(ins.q, ins.k_pre, ins.v_pre, ins.k_tail, ins.v_tail,
                                            ins.seq_start, ins.seq_len, 0, Hq, Hkv, d)
    qf = wl.bits_to_f32(ins.q).astype(np.float64)
    kf = wl.bits_to_f32(ins.k_tail).astype(np.float64)
    vf = wl.bits_to_f32(ins.v_tail).astype(np.float64)
    for b in range(3):
        t = int(ins.seq_start[b])
        np.testing.assert_allclose(out[t], vf[t], rtol=0, atol=1e-15)
        s = (qf[t] * kf[t]).sum(-1) / math.sqrt(d)
        np.testing.assert_allclose(lse[:, t], s, rtol=0, atol=1e-12)
    # identical keys along the tail and prefix
    P = 10
    w2 = wl.Workload("k2", 78, P, 2, 1, 1, Hq, Hkv, d, 8, 8, 1, 1, 1.0, "letters")
    ins = wl.attention_inputs(w2, lengths=np.array([3, 6]), P=P)
    key = ins.k_pre[0:1, :, :]
    k_pre = np.broadcast_to(key, ins.k_pre.shape).copy()
    k_tail = np.broadcast_to(key, ins.k_tail.shape).copy()
    out, lse = oracle.prefix_tail_attention(ins.q, k_pre, ins.v_pre, k_tail, ins.v_tail, ins.seq_start,
                                            ins.seq_len, P, Hq, Hkv, d)
    qf = wl.bits_to_f32(ins.q).astype(np.float64)
    kf = wl.bits_to_f32(key[0]).astype(np.float64)
    vp = wl.bits_to_f32(ins.v_pre).astype(np.float64)
    vt = wl.bits_to_f32(ins.v_tail).astype(np.float64)
    for b in range(2):
        for i in range(int(ins.seq_len[b])):
            t = int(ins.seq_start[b]) + i
            visible = np.concatenate([vp, vt[int(ins.seq_start[b]):t + 1]], 0)  # [n, Hkv, d]
            np.testing.assert_allclose(out[t], visible.mean(0), rtol=0, atol=1e-13)
            s = (qf[t] * kf).sum(-1) / math.sqrt(d)
            np.testing.assert_allclose(lse[:, t], s + math.log(visible.shape[0]), rtol=0, atol=1e-12)


def test_selected_rows_match_full_run():
    w = wl.WORKLOADS["tiny"]
    ins = wl.attention_inputs(w)
    full, lfull = oracle.prefix_tail_attention(ins.q, ins.k_pre, ins.v_pre, ins.k_tail, ins.v_tail,
                                               ins.seq_start, ins.seq_len, w.P, w.Hq, w.Hkv, w.d)
    tok = np.array([0, 7, 8, 33, 59], dtype=np.int32)
    head = np.array([0, 3, 1, 2, 3], dtype=np.int32)
    sel, lsel = oracle.prefix_tail_attention(ins.q, ins.k_pre, ins.v_pre, ins.k_tail, ins.v_tail,
                                             ins.seq_start, ins.seq_len, w.P, w.Hq, w.Hkv, w.d,
                                             select=(tok, head))
    for t, h in zip(tok, head):
        np.testing.assert_array_equal(sel[t, h], full[t, h])
        assert lsel[h, t] == lfull[h, t]


def test_arena_row_stride():
    """The prefix may be a slice of a wider KV arena row (simit engine.py keeps one arena with a
    region per request); a stride larger than Hkv*d must give the same result."""
    w = wl.WORKLOADS["tiny"]
    ins = wl.attention_inputs(w)
    stride = w.Hkv * w.d + 40
    def widen(x):
        y = np.zeros((x.shape[0], stride), dtype=np.uint16)
        y[:, : w.Hkv * w.d] = x.reshape(x.shape[0], -1)
        return y
    a, _ = oracle.prefix_tail_attention(ins.q, ins.k_pre, ins.v_pre, ins.k_tail, ins.v_tail, ins.seq_start,
                                        ins.seq_len, w.P, w.Hq, w.Hkv, w.d)
    b, _ = oracle.prefix_tail_attention(ins.q, widen(ins.k_pre), widen(ins.v_pre), ins.k_tail, ins.v_tail,
                                        ins.seq_start, ins.seq_len, w.P, w.Hq, w.Hkv, w.d,
                                        pre_row_stride=stride)
    np.testing.assert_array_equal(a, b)
