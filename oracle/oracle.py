"""Python face of the FP64 CPU oracle (oracle/blink_oracle.c).

TEST INFRASTRUCTURE, NOT PRODUCT CODE.  Only the tests, the smoke check and the benchmark's
CPU-baseline leg may import this module.  It does not import the product package and the
product package does not import it; both sides receive their inputs from the seeded input
generators.

What each function follows on the pages is stated in the C source beside it:
  pack_plan              blink.py, `_batches` / `_padded`
  prefix_tail_attention  blink.py, PREFIX_CACHE note and `_forward_shared`
  label_readout          blink.py, `_read` / `_read_batched`, `softmax`, `decide`
and, written here in Python because the pages keep them on the host:
  answer                 blink.py, `answer_for`
  shared_prefix_len      blink.py, `_shared_prefix_len`
  rotation_debias        ruling engine.py, `_score_plain` / `_prior` / `answer`
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "blink_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (plain C, -O2, no fast-math: IEEE double semantics kept)."""
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.run(
            ["gcc", "-O2", "-fno-fast-math", "-ffp-contract=off", "-fPIC", "-shared", "-pthread",
             "-o", tmp, _SRC, "-lm"],
            check=True,
        )
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB_PATH)
        i32p = ctypes.POINTER(ctypes.c_int32)
        u16p = ctypes.POINTER(ctypes.c_uint16)
        f64p = ctypes.POINTER(ctypes.c_double)
        lib.oracle_pack_plan.restype = ctypes.c_int32
        lib.oracle_pack_plan.argtypes = [i32p, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32] + [i32p] * 7
        lib.oracle_prefix_tail_attention.restype = ctypes.c_int
        lib.oracle_prefix_tail_attention.argtypes = [
            u16p, u16p, u16p, ctypes.c_int64, u16p, u16p, i32p, i32p, ctypes.c_int32, ctypes.c_int64,
            ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, ctypes.c_double,
            i32p, i32p, ctypes.c_int64, f64p, f64p, ctypes.c_int32]
        lib.oracle_label_readout.restype = ctypes.c_int
        lib.oracle_label_readout.argtypes = [
            u16p, ctypes.c_int64, i32p, u16p, ctypes.c_int32, ctypes.c_int32, i32p, i32p, ctypes.c_int32,
            ctypes.c_double, f64p, f64p]
        _lib = lib
    return _lib


def _ptr(a: np.ndarray | None, ctype):
    if a is None:
        return ctypes.cast(None, ctypes.POINTER(ctype))
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data_as(ctypes.POINTER(ctype))


def _bits(a: np.ndarray) -> np.ndarray:
    """bf16 data arrives as uint16 bit patterns."""
    a = np.ascontiguousarray(a)
    if a.dtype != np.uint16:
        raise TypeError("bf16 inputs are passed as uint16 bit patterns")
    return a


class OracleError(ValueError):
    pass


def pack_plan(lengths, budget: int, max_rows: int = 0) -> dict:
    """The sequential packing rule; returns every plan array plus n_forwards."""
    lib = _load()
    lengths = np.ascontiguousarray(lengths, dtype=np.int32)
    n = int(lengths.shape[0])
    out = {k: np.zeros(n + (1 if k in ("fwd_slot_start", "cu_seqlens") else 0), dtype=np.int32)
           for k in ("order", "fwd_of_slot", "fwd_slot_start", "fwd_width", "cu_seqlens",
                     "last_varlen", "last_padded")}
    nf = lib.oracle_pack_plan(
        _ptr(lengths, ctypes.c_int32), n, int(budget), int(max_rows),
        *(_ptr(out[k], ctypes.c_int32) for k in ("order", "fwd_of_slot", "fwd_slot_start", "fwd_width",
                                                 "cu_seqlens", "last_varlen", "last_padded")))
    if nf < 0:
        raise OracleError("bad plan arguments")
    out["n_forwards"] = int(nf)
    return out


def prefix_tail_attention(q, k_pre, v_pre, k_tail, v_tail, seq_start, seq_len, P: int, Hq: int, Hkv: int,
                          d: int, scale: float = 0.0, pre_row_stride: int | None = None,
                          select=None, n_threads: int = 0):
    """FP64 attention of every tail row over [shared prefix ; own tail, causal].

    q, k_tail, v_tail: uint16 arrays shaped [rows, H*, d]; k_pre, v_pre: uint16 [P, stride] rows.
    select: optional (tok[], head[]) pairs; only those outputs are computed.
    Returns (out [rows, Hq, d] float64, lse [Hq, rows] float64); rows not computed hold NaN.
    """
    lib = _load()
    q = _bits(q)
    k_tail = _bits(k_tail)
    v_tail = _bits(v_tail)
    rows = int(q.shape[0])
    seq_start = np.ascontiguousarray(seq_start, dtype=np.int32)
    seq_len = np.ascontiguousarray(seq_len, dtype=np.int32)
    B = int(seq_start.shape[0])
    if P > 0:
        k_pre = _bits(k_pre)
        v_pre = _bits(v_pre)
        if pre_row_stride is None:
            pre_row_stride = Hkv * d
    else:
        k_pre = np.zeros(1, dtype=np.uint16)
        v_pre = np.zeros(1, dtype=np.uint16)
        pre_row_stride = Hkv * d
    out = np.full((rows, Hq, d), np.nan, dtype=np.float64)
    lse = np.full((Hq, rows), np.nan, dtype=np.float64)
    if select is not None:
        sel_tok = np.ascontiguousarray(select[0], dtype=np.int32)
        sel_head = np.ascontiguousarray(select[1], dtype=np.int32)
        n_sel = int(sel_tok.shape[0])
    else:
        sel_tok = sel_head = None
        n_sel = 0
    st = lib.oracle_prefix_tail_attention(
        _ptr(q, ctypes.c_uint16), _ptr(k_pre, ctypes.c_uint16), _ptr(v_pre, ctypes.c_uint16),
        int(pre_row_stride), _ptr(k_tail, ctypes.c_uint16), _ptr(v_tail, ctypes.c_uint16),
        _ptr(seq_start, ctypes.c_int32), _ptr(seq_len, ctypes.c_int32), B, rows, int(P), int(Hq), int(Hkv),
        int(d), float(scale), _ptr(sel_tok, ctypes.c_int32), _ptr(sel_head, ctypes.c_int32), n_sel,
        _ptr(out, ctypes.c_double), _ptr(lse, ctypes.c_double), int(n_threads))
    if st != 0:
        raise OracleError(f"attention oracle rejected its arguments (status {st})")
    return out, lse


def label_readout(hidden, last_idx, unembed, label_off, label_ids, temperature: float,
                  hidden_row_stride: int | None = None):
    """FP64 label logits and temperature softmax.  Returns (logits, probs, status)."""
    lib = _load()
    hidden = _bits(hidden)
    unembed = _bits(unembed)
    V, H = int(unembed.shape[0]), int(unembed.shape[1])
    if hidden_row_stride is None:
        hidden_row_stride = int(hidden.shape[-1])
    last_idx = np.ascontiguousarray(last_idx, dtype=np.int32)
    label_off = np.ascontiguousarray(label_off, dtype=np.int32)
    label_ids = np.ascontiguousarray(label_ids, dtype=np.int32)
    B = int(last_idx.shape[0])
    n = int(label_ids.shape[0])
    logits = np.zeros(n, dtype=np.float64)
    probs = np.zeros(n, dtype=np.float64)
    st = lib.oracle_label_readout(
        _ptr(hidden, ctypes.c_uint16), int(hidden_row_stride), _ptr(last_idx, ctypes.c_int32),
        _ptr(unembed, ctypes.c_uint16), V, H, _ptr(label_off, ctypes.c_int32), _ptr(label_ids, ctypes.c_int32),
        B, float(temperature), _ptr(logits, ctypes.c_double), _ptr(probs, ctypes.c_double))
    if st == 1:
        raise OracleError("readout oracle rejected its arguments")
    return logits, probs, int(st)


QTYPE_CHOICE, QTYPE_NOUL, QTYPE_SCORE = 0, 1, 2


def answer(qtype: int, probs) -> dict:
    """blink.py `answer_for`, restated over one question's probabilities in request order.

    The probabilities are renormalised (divided by their sum, or by 1 if it is 0).  A choice
    answers the first label with the largest probability and a confidence of
    (p_best - 1/K) / (1 - 1/K) (1 when K = 1); a noul answers p of its first label ("yes"); a
    score answers the expected level sum_i i * p_i, the most probable level (ties to the lowest)
    and the same confidence clamped to [0, 1].
    Returns {"index", "confidence", "value"}: the chosen label, the confidence (NaN for a noul)
    and p_best / p_yes / the expected level.
    """
    p = [float(x) for x in probs]
    z = sum(p) or 1.0
    p = [x / z for x in p]
    K = len(p)
    best = max(range(K), key=lambda k: (p[k], -k))  # first in request order among equals
    if qtype == QTYPE_CHOICE:
        conf = (p[best] - 1 / K) / (1 - 1 / K) if K > 1 else 1.0
        return {"index": best, "confidence": conf, "value": p[best]}
    if qtype == QTYPE_NOUL:
        return {"index": best, "confidence": float("nan"), "value": p[0]}
    if qtype == QTYPE_SCORE:
        ev = sum(i * p[i] for i in range(K))
        conf = min(1.0, max(0.0, (p[best] - 1 / K) / (1 - 1 / K))) if K > 1 else 1.0
        return {"index": best, "confidence": conf, "value": ev}
    raise OracleError(f"unknown question type {qtype}")


def shared_prefix_len(seqs) -> int:
    """blink.py `_shared_prefix_len`, as the page states it: with fewer than two sequences, 0;
    otherwise the common prefix of the lexicographically smallest and largest sequences (which
    is the common prefix of all of them), clipped so every sequence keeps at least one token."""
    seqs = [list(map(int, s)) for s in seqs]
    if len(seqs) < 2:
        return 0
    lo, hi = min(seqs), max(seqs)
    n = min(len(lo), len(hi))
    p = 0
    while p < n and lo[p] == hi[p]:
        p += 1
    return min(p, min(len(s) for s in seqs) - 1)


def rotation_debias(pass_logits, pass_keys, question_passes, prior=None, temperature: float = 1.0):
    """The ruling engine's log-space readout, in float64.

    pass_logits[p]  the answer codes' logits of pass p (one per shown position)
    pass_keys[p]    the option index each position of pass p shows
    question_passes[q]  the passes of question q
    prior           None, or a function K -> the K content-free log-probabilities by position
    Per pass: log-softmax, minus the prior by position; per option: the mean of its values over
    the question's passes; then softmax(raw / T).  Returns (raw list, probs list) per question.
    """
    raws, probs = [], []
    for passes in question_passes:
        K = len(pass_logits[passes[0]])
        values = [[] for _ in range(K)]
        for p in passes:
            z = np.asarray(pass_logits[p], dtype=np.float64)
            if z.shape[0] != K:
                raise OracleError("passes of one question differ in size")
            m = z.max()
            lp = z - (m + np.log(np.exp(z - m).sum()))
            if prior is not None:
                lp = lp - np.asarray(prior(K), dtype=np.float64)
            for pos, key in enumerate(pass_keys[p]):
                values[int(key)].append(lp[pos])
        raw = np.array([np.mean(v) for v in values])
        t = raw / temperature
        e = np.exp(t - t.max())
        raws.append(raw)
        probs.append(e / e.sum())
    return raws, probs
