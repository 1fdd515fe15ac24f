"""Shared test helpers: move seeded numpy inputs to the device, compare against the oracle."""
from __future__ import annotations

import numpy as np
import torch

from oracle import oracle
from shared_prefix_question_gb300 import workloads as wl

ATTN_REL_TOL = 2e-2   # max |O - O_ref| / max |O_ref|, from the stated target
LSE_ABS_TOL = 2e-3    # natural-log LSE; fp32 (max, sum) over fp32 scores
PROB_ABS_TOL = 1e-3   # label probabilities, from the stated target
ARGMAX_TIE_GAP = 1e-4  # logit gap below which either argmax is accepted


def dev_bf16(a: np.ndarray, device="cuda") -> torch.Tensor:
    t = torch.from_numpy(np.ascontiguousarray(a, dtype=np.uint16).view(np.int16)).view(torch.bfloat16)
    return t.to(device)


def dev_i32(a, device="cuda") -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).to(device)


def host_f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().numpy().astype(np.float64)


def run_attention(ins: wl.AttentionInputs, padded: bool = False, want_lse: bool = True, max_tail=None,
                  pre_row_stride=None, k_pre_dev=None, v_pre_dev=None):
    from shared_prefix_question_gb300 import blink
    q = dev_bf16(ins.q)
    kt = dev_bf16(ins.k_tail)
    vt = dev_bf16(ins.v_tail)
    if ins.P > 0:
        kp = k_pre_dev if k_pre_dev is not None else dev_bf16(ins.k_pre)
        vp = v_pre_dev if v_pre_dev is not None else dev_bf16(ins.v_pre)
    else:
        kp = vp = None
    cu = dev_i32(ins.cu_seqlens)
    ss = dev_i32(ins.seq_start) if padded else None
    mt = int(ins.seq_len.max()) if max_tail is None else max_tail
    out, lse, ws = blink.blink_prefix_tail_attention(q, kp, vp, kt, vt, cu, B=len(ins.seq_len), P=ins.P, max_tail=mt,
                                                     seq_start=ss, want_lse=want_lse, pre_row_stride=pre_row_stride)
    torch.cuda.synchronize()
    st = blink.blink_read_device_status(ws)
    return host_f64(out), (host_f64(lse) if lse is not None else None), st


def owned_rows(ins: wl.AttentionInputs) -> np.ndarray:
    return np.concatenate([np.arange(s, s + L) for s, L in zip(ins.seq_start, ins.seq_len)]).astype(np.int64)


def compare_attention(ins: wl.AttentionInputs, out, lse, select=None, n_threads=0):
    """Oracle on all owned rows (or the selected (token, head) pairs); returns (err, scale)."""
    ref, ref_lse = oracle.prefix_tail_attention(ins.q, ins.k_pre, ins.v_pre, ins.k_tail, ins.v_tail, ins.seq_start,
                                                ins.seq_len, ins.P, ins.Hq, ins.Hkv, ins.d, select=select,
                                                n_threads=n_threads)
    if select is None:
        rows = owned_rows(ins)
        got, want = out[rows], ref[rows]
        gl = lse[:, rows] if lse is not None else None
        wlse = ref_lse[:, rows]
    else:
        tok, head = select
        got, want = out[tok, head], ref[tok, head]
        gl = lse[head, tok] if lse is not None else None
        wlse = ref_lse[head, tok]
    assert np.isfinite(got).all(), "non-finite attention output"
    err = float(np.abs(got - want).max())
    scale = float(np.abs(want).max())
    assert err <= ATTN_REL_TOL * scale, f"attention error {err:.3e} > {ATTN_REL_TOL} x scale {scale:.3e}"
    if gl is not None:
        lerr = float(np.abs(gl - wlse).max())
        assert lerr <= LSE_ABS_TOL * max(1.0, float(np.abs(wlse).max())), f"lse error {lerr:.3e}"
    return err, scale


def sample_pairs(ins: wl.AttentionInputs, n: int, seed: int = 0):
    """(token, head) pairs: every question's first and last tail row, plus random rows."""
    rng = np.random.default_rng(seed)
    toks = [int(s) for s in ins.seq_start] + [int(s + L - 1) for s, L in zip(ins.seq_start, ins.seq_len)]
    rows = owned_rows(ins)
    toks += rng.choice(rows, size=max(0, n - len(toks)), replace=True).tolist()
    toks = np.asarray(toks[:max(n, 1)], dtype=np.int32)
    heads = rng.integers(0, ins.Hq, size=toks.shape[0]).astype(np.int32)
    return toks, heads


def compare_readout(probs_gpu: np.ndarray, ins: wl.ReadoutInputs):
    z, p, st = oracle.label_readout(ins.hidden, ins.last_idx, ins.unembed, ins.label_off, ins.label_ids,
                                    ins.temperature)
    assert st == 0
    err = float(np.abs(probs_gpu - p).max())
    assert err <= PROB_ABS_TOL, f"probability error {err:.3e}"
    for b in range(len(ins.last_idx)):
        lo, hi = ins.label_off[b], ins.label_off[b + 1]
        zb = z[lo:hi]
        top = np.argsort(-zb, kind="stable")
        if hi - lo >= 2 and zb[top[0]] - zb[top[1]] < ARGMAX_TIE_GAP:
            assert int(np.argmax(probs_gpu[lo:hi])) in (top[0], top[1])
        else:
            assert int(np.argmax(probs_gpu[lo:hi])) == int(top[0]), f"argmax differs for question {b}"
    return err
