"""Thin Python binding of the C ABI in include/blink.h (libblink.so, built in-tree for sm_103a).

Argument marshalling only: every step of the path runs in the library's CUDA kernels.  Torch
tensors supply device memory and the current CUDA stream; outputs are allocated with torch when
the caller does not pass them.  There is no CPU fallback: without the built library or a CUDA
device every call raises.
"""
from __future__ import annotations

import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libblink.so")

BLINK_OK = 0
BLINK_INVALID_ARG = 1
BLINK_OUT_OF_RANGE = 2
BLINK_WORKSPACE_TOO_SMALL = 3
BLINK_CUDA_ERROR = 4
BLINK_DEVICE_FLAG = 5
BLINK_DEVICE_TIMEOUT = 6

MAX_OPTIONS = 255
MAX_QUESTIONS = 512
MAX_INPUT_TOKENS = 131072
MAX_PLAN_SEQUENCES = 32768


class BlinkError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {status_string(status)} (status {status})")


_lib = None

_vp = ctypes.c_void_p
_i32 = ctypes.c_int32
_i64 = ctypes.c_int64
_f32 = ctypes.c_float
_sz = ctypes.c_size_t

_SIGNATURES = {
    "blink_status_string": (ctypes.c_char_p, [_i32]),
    "blink_read_device_status": (_i32, [_vp, _i32, _vp]),
    "blink_selftest_wait_timeout": (_i32, [ctypes.c_uint32, _vp, _sz, _vp]),
    "blink_pack_plan_workspace": (_sz, [_i32]),
    "blink_pack_plan": (_i32, [_vp, _i32, _i32, _i32] + [_vp] * 10 + [_vp]),
    "blink_attention_workspace": (_sz, [_i32] * 6),
    "blink_attention_split_plan": (_i32, [_i32] * 6 + [_vp] * 3),
    "blink_prefix_tail_attention": (_i32, [_vp, _vp, _vp, _i64, _vp, _vp, _vp, _vp, _i32, _i32, _i32, _i32, _i32,
                                           _i32, _i32, _f32, _vp, _vp, _vp, _sz, _vp]),
    "blink_prefix_tail_attention_multi": (_i32, [_vp, _vp, _vp, _i64, _i64, _vp, _vp, _vp, _vp, _i32, _i32, _i32, _vp,
                                                 _vp, _vp, _i32, _i32, _i32, _i32, _f32, _vp, _vp, _vp, _sz, _vp]),
    "blink_shared_prefix_len_workspace": (_sz, []),
    "blink_shared_prefix_len": (_i32, [_vp, _i64, _vp, _i32, _vp, _vp, _vp, _sz, _vp]),
    "blink_kv_to_arena": (_i32, [_vp, _vp, _i64, _i64, _i32, _vp, _vp, _i64, _i64, _i64, _vp]),
    "blink_rotation_debias_workspace": (_sz, []),
    "blink_rotation_debias": (_i32, [_vp, _vp, _vp, _i32, _vp, _vp, _i32, _i32, _vp, _f32, _vp, _vp, _vp, _vp, _vp, _vp,
                                     _vp, _sz, _vp]),
    "blink_label_readout_workspace": (_sz, [_i32]),
    "blink_label_readout": (_i32, [_vp, _i64, _i32, _vp, _vp, _vp, _i32, _i32, _vp, _vp, _i32, _i32, _f32, _vp, _vp, _vp,
                                   _vp, _vp, _vp, _vp, _sz, _vp]),
    "blink_label_readout_noalloc": (_i32, [_vp, _i64, _i32, _vp, _vp, _vp, _i32, _i32, _vp, _vp, _i32, _i32, _f32, _vp,
                                           _vp, _vp, _vp]),
}


def lib():
    """Load libblink.so (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with __graft_entry__.build() or "
                               "python -m shared_prefix_question_gb300.build")
        L = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in _SIGNATURES.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _lib = L
    return _lib


def exported_symbols():
    return list(_SIGNATURES)


def status_string(status: int) -> str:
    try:
        return lib().blink_status_string(int(status)).decode()
    except Exception:  # library not loadable: still give a readable message
        return "status"


def _ptr(t: torch.Tensor | None):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream: torch.cuda.Stream | None):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _need_cuda(*ts):
    for t in ts:
        if t is not None and (not t.is_cuda or not t.is_contiguous()):
            raise ValueError("tensors passed to the library must be contiguous CUDA tensors")


def _check(status: int, what: str):
    if status != BLINK_OK:
        raise BlinkError(status, what)


# ------------------------------------------------------------------------------------------------ plan
def blink_pack_plan(lengths: torch.Tensor, budget: int, max_rows: int = 0, out: dict | None = None,
                    sync: bool = False, stream=None) -> dict:
    """Token-budget pack plan of int32 `lengths` (device).  Returns the plan tensors; with
    sync=True also `n_forwards` as a Python int (one pinned D2H copy, synchronising)."""
    _need_cuda(lengths)
    if lengths.dtype != torch.int32:
        raise ValueError("lengths must be int32")
    n = lengths.numel()
    dev = lengths.device
    if out is None:
        out = {k: torch.empty(n + (1 if k in ("fwd_slot_start", "cu_seqlens") else 0), dtype=torch.int32, device=dev)
               for k in ("order", "slot_of", "fwd_of_slot", "fwd_slot_start", "fwd_width", "cu_seqlens",
                         "last_varlen", "last_padded")}
        out["n_forwards_dev"] = torch.empty(1, dtype=torch.int32, device=dev)
    host = torch.empty(1, dtype=torch.int32, pin_memory=True) if sync else None
    st = lib().blink_pack_plan(_ptr(lengths), n, int(budget), int(max_rows), _ptr(out["order"]),
                               _ptr(out["slot_of"]), _ptr(out["fwd_of_slot"]), _ptr(out["fwd_slot_start"]), _ptr(out["fwd_width"]),
                               _ptr(out["cu_seqlens"]), _ptr(out["last_varlen"]), _ptr(out["last_padded"]),
                               _ptr(out["n_forwards_dev"]), _ptr(host), _stream(stream))
    _check(st, "blink_pack_plan")
    if sync:
        out["n_forwards"] = int(host.item())
    return out


# ------------------------------------------------------------------------------------------------ attention
def pack_plan_workspace_bytes(n: int) -> int:
    """0: the planner's scratch is its own output arrays."""
    return int(lib().blink_pack_plan_workspace(n))


def attention_workspace_bytes(rows, B, P, Hq, Hkv, d) -> int:
    return int(lib().blink_attention_workspace(rows, B, P, Hq, Hkv, d))


def blink_attention_split_plan(rows: int, P: int, Hq: int, Hkv: int, d: int, sms: int):
    """The prefix-chunk plan of one request on a GPU with `sms` SMs (host computation only):
    (whole_units, chunks, chunk_tiles) as include/blink.h describes them."""
    w, c, t = ctypes.c_int64(0), ctypes.c_int32(0), ctypes.c_int32(0)
    st = lib().blink_attention_split_plan(int(rows), int(P), int(Hq), int(Hkv), int(d), int(sms), ctypes.byref(w),
                                          ctypes.byref(c), ctypes.byref(t))
    _check(st, "blink_attention_split_plan")
    return int(w.value), int(c.value), int(t.value)


def new_workspace(nbytes: int, device) -> torch.Tensor:
    """A zero-filled device workspace (the first word is the device error word)."""
    return torch.zeros(max(256, (nbytes + 255) // 256 * 256), dtype=torch.uint8, device=device)


def blink_prefix_tail_attention(q, k_pre, v_pre, k_tail, v_tail, cu_seqlens, B: int, P: int, max_tail: int,
                                seq_start=None, scale: float = 0.0, out=None, lse=None, want_lse: bool = False,
                                ws=None, pre_row_stride: int | None = None, stream=None):
    """q [rows, Hq, d], k_tail/v_tail [rows, Hkv, d], k_pre/v_pre [P, Hkv, d] (or rows of an arena with
    `pre_row_stride` elements), all bf16 on the device.  Returns (out, lse, ws)."""
    _need_cuda(q, k_tail, v_tail, cu_seqlens, seq_start)
    rows, Hq, d = q.shape
    Hkv = k_tail.shape[1]
    if P > 0:
        if pre_row_stride is None:
            _need_cuda(k_pre, v_pre)
            pre_row_stride = Hkv * d
    if out is None:
        out = torch.empty_like(q)
    if lse is None and want_lse:
        lse = torch.empty(Hq, rows, dtype=torch.float32, device=q.device)
    need = attention_workspace_bytes(rows, B, P, Hq, Hkv, d)
    if ws is None:
        ws = new_workspace(need, q.device)
    st = lib().blink_prefix_tail_attention(
        _ptr(q), _ptr(k_pre) if P > 0 else None, _ptr(v_pre) if P > 0 else None, int(pre_row_stride or 0),
        _ptr(k_tail), _ptr(v_tail), _ptr(cu_seqlens), _ptr(seq_start), int(B), int(rows), int(P), int(max_tail),
        int(Hq), int(Hkv), int(d), float(scale), _ptr(out), _ptr(lse), _ptr(ws), ws.numel(), _stream(stream))
    _check(st, "blink_prefix_tail_attention")
    return out, lse, ws


def blink_prefix_tail_attention_multi(q, k_arena, v_arena, k_tail, v_tail, cu_seqlens, B: int, req_rows,
                                      req_prefix_start, req_prefix_len, max_tail: int, seq_start=None,
                                      scale: float = 0.0, out=None, lse=None, want_lse: bool = False, ws=None,
                                      arena_row_stride: int | None = None, stream=None):
    """Several requests in one launch: request r owns rows [req_rows[r], req_rows[r+1]) of q/k_tail/
    v_tail and attends to arena slots [req_prefix_start[r], + req_prefix_len[r]).  The arena tensors
    are [slots, Hkv, d] (or [slots, stride] with `arena_row_stride`).  Returns (out, lse, ws)."""
    import numpy as np
    _need_cuda(q, k_tail, v_tail, cu_seqlens, seq_start)
    rows, Hq, d = q.shape
    Hkv = k_tail.shape[1]
    n_req = len(req_prefix_len)
    h_rows = np.ascontiguousarray(req_rows, dtype=np.int32)
    h_start = np.ascontiguousarray(req_prefix_start, dtype=np.int32)
    h_len = np.ascontiguousarray(req_prefix_len, dtype=np.int32)
    if arena_row_stride is None:
        arena_row_stride = Hkv * d
    slots = int(k_arena.shape[0]) if k_arena is not None else 0
    if out is None:
        out = torch.empty_like(q)
    if lse is None and want_lse:
        lse = torch.empty(Hq, rows, dtype=torch.float32, device=q.device)
    if ws is None:
        ws = new_workspace(attention_workspace_bytes(rows, B, 0, Hq, Hkv, d), q.device)
    st = lib().blink_prefix_tail_attention_multi(
        _ptr(q), _ptr(k_arena), _ptr(v_arena), int(arena_row_stride), slots,
        _ptr(k_tail), _ptr(v_tail), _ptr(cu_seqlens), _ptr(seq_start), int(B), int(rows), int(n_req),
        h_rows.ctypes.data_as(ctypes.c_void_p), h_start.ctypes.data_as(ctypes.c_void_p),
        h_len.ctypes.data_as(ctypes.c_void_p), int(max_tail), int(Hq), int(Hkv), int(d), float(scale), _ptr(out),
        _ptr(lse), _ptr(ws), ws.numel(), _stream(stream))
    _check(st, "blink_prefix_tail_attention_multi")
    return out, lse, ws


def blink_read_device_status(ws: torch.Tensor, clear: bool = True, stream=None) -> int:
    return int(lib().blink_read_device_status(_ptr(ws), 1 if clear else 0, _stream(stream)))


def blink_selftest_wait_timeout(limit_us: int, ws: torch.Tensor, stream=None) -> int:
    """Runs the bounded device wait against a barrier nothing arrives at; returns the status it
    latched (BLINK_DEVICE_TIMEOUT when the failure path works)."""
    return int(lib().blink_selftest_wait_timeout(int(limit_us), _ptr(ws), ws.numel(), _stream(stream)))


# ------------------------------------------------------------------------------------------------ readout
def readout_workspace_bytes(B: int) -> int:
    return int(lib().blink_label_readout_workspace(B))


def blink_label_readout(hidden, last_idx, unembed, label_off, label_ids, temperature: float, probs=None,
                        host_probs=None, logits=None, ws=None, slot_of=None, qtype=None, answers=None,
                        host_answers=None, stream=None):
    """hidden [rows, H] bf16, last_idx int32 (per question, or per slot with `slot_of`), unembed [V, H]
    bf16, CSR label_off [B+1] / label_ids [sum K] int32, all on the device.  Returns (probs, ws); if
    `host_probs` (pinned fp32) is given the call copies into it and synchronises."""
    _need_cuda(hidden, last_idx, unembed, label_off, label_ids, probs, logits, slot_of, qtype, answers)
    rows, H = hidden.shape
    V = unembed.shape[0]
    B = label_off.numel() - 1
    sum_k = label_ids.numel()
    if probs is None:
        probs = torch.empty(sum_k, dtype=torch.float32, device=hidden.device)
    if qtype is not None and answers is None:
        answers = torch.empty(B, 3, dtype=torch.float32, device=hidden.device)
    if ws is None:
        ws = new_workspace(readout_workspace_bytes(B), hidden.device)
    st = lib().blink_label_readout(_ptr(hidden), int(hidden.stride(0)), int(rows), _ptr(last_idx), _ptr(slot_of), _ptr(unembed),
                                   int(V), int(H), _ptr(label_off), _ptr(label_ids), int(B), int(sum_k),
                                   float(temperature), _ptr(probs), _ptr(host_probs), _ptr(logits), _ptr(qtype),
                                   _ptr(answers), _ptr(host_answers), _ptr(ws), ws.numel(), _stream(stream))
    _check(st, "blink_label_readout")
    if answers is not None:
        return probs, ws, answers
    return probs, ws


STATIC_SCRATCH_QUESTIONS = 32768


def blink_label_readout_noalloc(hidden, last_idx, unembed, label_off, label_ids, temperature: float, probs=None,
                                host_probs=None, logits=None, slot_of=None, stream=None):
    """The readout for callers that cannot allocate device memory (the library keeps its scratch in a
    static device array; at most 32768 questions; calls that overlap on the GPU race).  Outputs are
    allocated here only when the caller passes none.

    Device-side errors (a label id outside [0, V), malformed offsets) are reported only when
    `host_probs` is given: the C call then reads the error word back after its copy and this
    wrapper raises BlinkError.  Without `host_probs` the call stays asynchronous and such a
    question's probabilities come back as NaN (or, for malformed offsets, unwritten)."""
    _need_cuda(hidden, last_idx, unembed, label_off, label_ids, probs, logits, slot_of)
    rows, H = hidden.shape
    V = unembed.shape[0]
    B = label_off.numel() - 1
    sum_k = label_ids.numel()
    if probs is None:
        probs = torch.empty(sum_k, dtype=torch.float32, device=hidden.device)
    st = lib().blink_label_readout_noalloc(_ptr(hidden), int(hidden.stride(0)), int(rows), _ptr(last_idx),
                                           _ptr(slot_of), _ptr(unembed), int(V), int(H), _ptr(label_off),
                                           _ptr(label_ids), int(B), int(sum_k), float(temperature), _ptr(probs),
                                           _ptr(host_probs), _ptr(logits), _stream(stream))
    _check(st, "blink_label_readout_noalloc")
    return probs


# ------------------------------------------------------------------------------------------------ prefix side
def blink_shared_prefix_len(tokens, cu, out=None, sync: bool = True, ws=None, stream=None):
    """Shared-prefix length of the sequences in `tokens` (int32, back to back, offsets `cu`)."""
    _need_cuda(tokens, cu)
    n = cu.numel() - 1
    if out is None:
        out = torch.empty(1, dtype=torch.int32, device=tokens.device)
    if ws is None:
        ws = new_workspace(int(lib().blink_shared_prefix_len_workspace()), tokens.device)
    host = torch.empty(1, dtype=torch.int32, pin_memory=True) if sync else None
    st = lib().blink_shared_prefix_len(_ptr(tokens), int(tokens.numel()), _ptr(cu), int(n), _ptr(out), _ptr(host),
                                       _ptr(ws), ws.numel(), _stream(stream))
    _check(st, "blink_shared_prefix_len")
    return int(host.item()) if sync else out


def blink_kv_to_arena(k_src, v_src, k_arena, v_arena, dst_slot: int, stream=None):
    """Write the token rows of k_src / v_src ([n, ...] bf16, rows contiguous) into arena rows
    [dst_slot, dst_slot + n) of k_arena / v_arena ([slots, stride] bf16)."""
    n = k_src.shape[0]
    row_elems = k_src[0].numel() if n else 0
    st = lib().blink_kv_to_arena(_ptr(k_src), _ptr(v_src), int(k_src.stride(0)), int(n), int(row_elems),
                                 _ptr(k_arena), _ptr(v_arena), int(k_arena.stride(0)), int(k_arena.shape[0]),
                                 int(dst_slot), _stream(stream))
    _check(st, "blink_kv_to_arena")


def blink_rotation_debias(logits, pass_off, key_of_pos, question_pass, raw_off, temperature: float, prior=None,
                          raw=None, probs=None, host_probs=None, qtype=None, answers=None, host_answers=None,
                          ws=None, sum_k: int | None = None, stream=None):
    """Per pass log-softmax minus the prior, the mean over each question's passes, then the
    temperature softmax (and optional typed answers).  Returns (probs, raw, answers)."""
    _need_cuda(logits, pass_off, key_of_pos, question_pass, raw_off, prior, raw, probs, qtype, answers)
    n_pass = pass_off.numel() - 1
    B = raw_off.numel() - 1
    if sum_k is None:
        sum_k = int(raw_off[-1].item())  # one small copy; pass sum_k to avoid it
    dev = logits.device
    if probs is None:
        probs = torch.empty(sum_k, dtype=torch.float32, device=dev)
    if raw is None:
        raw = torch.empty(sum_k, dtype=torch.float32, device=dev)
    if qtype is not None and answers is None:
        answers = torch.empty(B, 3, dtype=torch.float32, device=dev)
    if ws is None:
        ws = new_workspace(int(lib().blink_rotation_debias_workspace()), dev)
    st = lib().blink_rotation_debias(_ptr(logits), _ptr(pass_off), _ptr(key_of_pos), int(n_pass), _ptr(question_pass),
                                     _ptr(raw_off), int(B), sum_k, _ptr(prior), float(temperature), _ptr(raw),
                                     _ptr(probs), _ptr(host_probs), _ptr(qtype), _ptr(answers), _ptr(host_answers),
                                     _ptr(ws), ws.numel(), _stream(stream))
    _check(st, "blink_rotation_debias")
    return probs, raw, answers
