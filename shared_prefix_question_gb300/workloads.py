"""Seeded synthetic workloads for the shared-prefix one-pass decision path.

This module only draws random numbers and lays them out; it holds none of the method's
arithmetic, so both the CUDA path and the FP64 oracle can take their inputs from it.

Shapes follow the pages' workloads: blink.py's limits (a token budget of 32768 padded tokens per
forward, up to 512 questions, up to 255 options, inputs up to 131072 tokens) and its
"long multi-question documents" of about 18k tokens.  No dataset is used: the pages measure on
documents that are not available here, and these seeded tensors stand in for them.

Recipe (also written out in the design notes):
  * lengths and label counts: numpy ``default_rng(index)``; uniform integers, bounds inclusive;
  * attention tensors Q, K, V (prefix and tails) and the readout hidden state: N(0, 1) in fp32
    from ``default_rng(1000 + index)``, rounded to bf16 (nearest, ties to even);
  * unembedding: N(0, 0.02) the same way, drawn after the hidden state;
  * label token ids: a seeded table from ``default_rng(2000 + index)``; question b offers the
    first K_b entries of the pool (blink.py renders `self.label_ids[: len(items)]`).
    The tiny case uses ids 0..25 for 'A'..'Z' directly.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

TOKEN_BUDGET = 32768      # padded tokens per forward (blink.py TOKEN_BUDGET)
MAX_QUESTIONS = 512       # blink.py MAX_QUESTIONS
MAX_OPTIONS = 255         # blink.py MAX_OPTIONS
MAX_INPUT_TOKENS = 131072  # blink.py MAX_INPUT_TOKENS
PREFIX_MIN_TOKENS = 256   # blink.py PREFIX_MIN_TOKENS
PREFIX_KV_TOKENS = 131072  # blink.py PREFIX_KV_TOKENS


@dataclass(frozen=True)
class Workload:
    name: str
    index: int
    P: int                  # shared prefix tokens (0 = plain path, no prefix)
    n: int                  # questions
    tail_lo: int            # tail length bounds, inclusive
    tail_hi: int
    Hq: int
    Hkv: int
    d: int
    H: int                  # hidden size
    V: int                  # vocabulary
    k_lo: int               # labels per question, inclusive bounds
    k_hi: int
    temperature: float
    pool: str               # "letters" (ids 0..), "table" (seeded distinct ids), "vocab" (per question)
    fixed_tails: tuple = field(default=())
    description: str = ""


WORKLOADS = {
    "tiny": Workload("tiny", 0, 64, 4, 8, 24, 4, 2, 64, 256, 1024, 2, 5, 1.0, "letters",
                     fixed_tails=(8, 12, 16, 24),
                     description="prefix 64, tails 8/12/16/24, 4/2 heads, d 64, hidden 256, vocab 1024"),
    "2k": Workload("2k", 1, 2048, 16, 32, 128, 32, 8, 128, 2560, 151936, 2, 8, 1.0, "table",
                   description="prefix 2048, 16 tails U[32,128], 32/8 heads, d 128, hidden 2560"),
    "18k": Workload("18k", 2, 18432, 64, 64, 256, 32, 8, 128, 2560, 151936, 2, 26, 0.7, "table",
                    description="long document: prefix 18432, 64 tails U[64,256], 32/8 heads, d 128, "
                                "hidden 2560, 2-26 labels, T 0.7"),
    "plain": Workload("plain", 3, 0, 256, 200, 1000, 32, 8, 128, 2560, 151936, 2, 8, 1.0, "table",
                      description="no prefix: 256 sequences U[200,1000], causal, budget 32768"),
    "max": Workload("max", 4, 131072, 512, 16, 64, 40, 8, 128, 5120, 151936, 2, 255, 1.0, "table",
                    description="max request: prefix 131072, 512 tails U[16,64], 40/8 heads, hidden 5120, "
                                "2-255 labels"),
    "readout_stress": Workload("readout_stress", 5, 0, 512, 1, 1, 40, 8, 128, 5120, 151936, 2, 255, 1.0,
                               "vocab",
                               description="readout stress: 512 questions, K_b U[2,255] ids drawn without "
                                           "replacement from the whole vocabulary, hidden 5120"),
}


def bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round fp32 values to bf16 (nearest, ties to even); returns the uint16 bit patterns."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    u = x.view(np.uint32).astype(np.uint64)
    u = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return u.astype(np.uint16)


def bits_to_f32(b: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns to fp32."""
    return (np.ascontiguousarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def normal_bf16(rng: np.random.Generator, shape, std: float = 1.0, chunk: int = 1 << 24) -> np.ndarray:
    """N(0, std^2) drawn in fp32 and rounded to bf16, in bounded chunks (large tensors)."""
    n = int(np.prod(shape))
    out = np.empty(n, dtype=np.uint16)
    for s in range(0, n, chunk):
        e = min(n, s + chunk)
        x = rng.standard_normal(e - s, dtype=np.float32)
        if std != 1.0:
            x *= np.float32(std)
        out[s:e] = bf16_bits(x)
    return out.reshape(shape)


def tail_lengths(w: Workload) -> np.ndarray:
    """Per-question tail (or, with no prefix, full) lengths in request order."""
    if w.fixed_tails:
        return np.asarray(w.fixed_tails, dtype=np.int32)
    rng = np.random.default_rng(w.index)
    return rng.integers(w.tail_lo, w.tail_hi + 1, size=w.n).astype(np.int32)


def label_counts(w: Workload) -> np.ndarray:
    rng = np.random.default_rng(w.index)
    if not w.fixed_tails:
        rng.integers(w.tail_lo, w.tail_hi + 1, size=w.n)  # same stream position as tail_lengths
    return rng.integers(w.k_lo, w.k_hi + 1, size=w.n).astype(np.int32)


def label_pool(w: Workload, size: int = MAX_OPTIONS) -> np.ndarray:
    """The synthetic verified-label table: the first 26 stand for 'A'..'Z', the rest for the
    two-letter labels.  The real tokenizer's ids are not available here."""
    if w.pool == "letters":
        return np.arange(min(size, w.V), dtype=np.int32)
    rng = np.random.default_rng(2000 + w.index)
    return rng.choice(w.V, size=size, replace=False).astype(np.int32)


def label_csr(w: Workload):
    """(label_off [n+1], label_ids [sum K]) in request order."""
    counts = label_counts(w)
    off = np.zeros(w.n + 1, dtype=np.int32)
    off[1:] = np.cumsum(counts)
    if w.pool == "vocab":
        rng = np.random.default_rng(2000 + w.index)
        ids = np.concatenate([rng.choice(w.V, size=int(k), replace=False) for k in counts]).astype(np.int32)
    else:
        pool = label_pool(w)
        ids = np.concatenate([pool[: int(k)] for k in counts]).astype(np.int32)
    return off, ids


@dataclass
class AttentionInputs:
    q: np.ndarray        # [rows, Hq, d] uint16 (bf16 bits)
    k_pre: np.ndarray    # [P, Hkv, d]
    v_pre: np.ndarray
    k_tail: np.ndarray   # [rows, Hkv, d]
    v_tail: np.ndarray
    seq_start: np.ndarray  # [B] first row of each question
    seq_len: np.ndarray    # [B]
    cu_seqlens: np.ndarray  # [B+1] varlen offsets (valid when the layout is packed)
    rows: int
    P: int
    Hq: int
    Hkv: int
    d: int


def attention_inputs(w: Workload, lengths: np.ndarray | None = None, padded_width: int | None = None,
                     P: int | None = None, seed_offset: int = 0) -> AttentionInputs:
    """Q/K/V for the tails (packed in the given order) and the shared prefix K/V.

    With `padded_width`, question b occupies rows [b*width, b*width + len_b) (right padding);
    otherwise the tails are packed back to back (varlen).
    """
    if lengths is None:
        lengths = tail_lengths(w)
    lengths = np.asarray(lengths, dtype=np.int32)
    P = w.P if P is None else P
    B = int(lengths.shape[0])
    if padded_width is not None:
        seq_start = (np.arange(B, dtype=np.int64) * padded_width).astype(np.int32)
        rows = B * padded_width
    else:
        seq_start = np.zeros(B, dtype=np.int32)
        seq_start[1:] = np.cumsum(lengths)[:-1]
        rows = int(lengths.sum())
    cu = np.zeros(B + 1, dtype=np.int32)
    cu[1:] = np.cumsum(lengths)
    rng = np.random.default_rng(1000 + w.index + seed_offset)
    k_pre = normal_bf16(rng, (P, w.Hkv, w.d))
    v_pre = normal_bf16(rng, (P, w.Hkv, w.d))
    q = normal_bf16(rng, (rows, w.Hq, w.d))
    k_tail = normal_bf16(rng, (rows, w.Hkv, w.d))
    v_tail = normal_bf16(rng, (rows, w.Hkv, w.d))
    return AttentionInputs(q, k_pre, v_pre, k_tail, v_tail, seq_start, lengths.copy(), cu, rows, P,
                           w.Hq, w.Hkv, w.d)


@dataclass
class ReadoutInputs:
    hidden: np.ndarray     # [rows, H] uint16
    last_idx: np.ndarray   # [B]
    unembed: np.ndarray    # [V, H] uint16
    label_off: np.ndarray  # [B+1]
    label_ids: np.ndarray  # [sum K]
    temperature: float


def readout_inputs(w: Workload, rows: int | None = None, last_idx: np.ndarray | None = None,
                   seed_offset: int = 0, unembed: np.ndarray | None = None) -> ReadoutInputs:
    """Hidden states N(0,1) for `rows` tokens, the unembedding N(0, 0.02) and the label CSR.

    `last_idx` defaults to the last token of each question in the varlen packing of the tails.
    A prebuilt `unembed` of the right shape may be passed to avoid redrawing a large matrix.
    """
    lengths = tail_lengths(w)
    if last_idx is None:
        last_idx = (np.cumsum(lengths) - 1).astype(np.int32)
    if rows is None:
        rows = int(lengths.sum())
    rng = np.random.default_rng(1000 + w.index + 500 + seed_offset)
    hidden = normal_bf16(rng, (rows, w.H))
    if unembed is None:
        unembed = normal_bf16(rng, (w.V, w.H), std=0.02)
    off, ids = label_csr(w)
    return ReadoutInputs(hidden, np.asarray(last_idx, dtype=np.int32), unembed, off, ids, w.temperature)


QTYPE_CHOICE, QTYPE_NOUL, QTYPE_SCORE = 0, 1, 2


def question_types(w: Workload, label_off: np.ndarray) -> np.ndarray:
    """Seeded question types consistent with the label counts (blink.py `question_options`):
    a noul offers exactly two labels (yes, no), a score 2 to 10 levels, a choice 1 to 255 options."""
    counts = np.diff(np.asarray(label_off))
    rng = np.random.default_rng(3000 + w.index)
    draw = rng.integers(0, 3, size=counts.shape[0])
    qt = np.full(counts.shape[0], QTYPE_CHOICE, dtype=np.int32)
    qt[(counts == 2) & (draw == 1)] = QTYPE_NOUL
    qt[(counts >= 2) & (counts <= 10) & (draw == 2)] = QTYPE_SCORE
    return qt
