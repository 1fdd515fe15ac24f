"""Question sharding across GPUs (one process per GPU) and the host-side gather of the answers.

Questions are independent once the prefix KV is known, so a request's questions split across
ranks with no exchange in the step: every rank holds the prefix KV, runs the plan, attention
and readout for its own questions, and the probabilities (and typed answers) are gathered on
one rank afterwards, in request order.  (Splitting the prefix across GPUs instead would need an
exchange of (O, LSE) partials; that plan is not used.)

Host logic only (numpy and torch.distributed); the per-rank step is the same C-ABI path.
"""
from __future__ import annotations

import numpy as np


def shard_questions(lengths, world: int) -> list[np.ndarray]:
    """Contiguous shards of the question indices, balanced by tail tokens (a question's attention
    work grows with its tail length).  The cut before shard r is the question boundary nearest to
    r / world of the running token count, kept so that every shard gets at least one question
    when there are at least `world` questions (with fewer, the first ranks get one each and the
    rest none).  Every shard keeps request order."""
    lengths = np.asarray(lengths, dtype=np.int64)
    n = len(lengths)
    if world < 1:
        raise ValueError("world must be >= 1")
    if np.any(lengths < 1):
        raise ValueError("every question needs a tail of at least one token")
    if n < world:
        return [np.arange(r, r + 1, dtype=np.int64) if r < n else np.zeros(0, dtype=np.int64)
                for r in range(world)]
    csum = np.concatenate([[0], np.cumsum(lengths)])
    total = int(csum[-1])
    cuts = [0]
    for r in range(1, world):
        target = total * r / world
        c = int(np.searchsorted(csum, target, side="left"))  # first boundary at or past the target
        if c > 0 and target - csum[c - 1] <= csum[c] - target:
            c -= 1
        c = min(max(c, cuts[-1] + 1), n - (world - r))
        cuts.append(c)
    cuts.append(n)
    return [np.arange(cuts[r], cuts[r + 1], dtype=np.int64) for r in range(world)]


def local_labels(label_off, label_ids, questions):
    """The CSR label lists of a shard's questions, offsets rebased to 0."""
    label_off = np.asarray(label_off, dtype=np.int64)
    label_ids = np.asarray(label_ids)
    questions = np.asarray(questions, dtype=np.int64)
    counts = label_off[questions + 1] - label_off[questions]
    off = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    if len(questions) == 0:
        return off, np.zeros(0, dtype=label_ids.dtype)
    ids = np.concatenate([label_ids[label_off[q]:label_off[q + 1]] for q in questions])
    return off, ids.astype(label_ids.dtype)


def gather_results(questions, local_off, probs, answers=None, dst: int = 0, group=None):
    """Gathers every rank's shard result on rank `dst`: `questions` (request indices), `local_off`
    and `probs` (the shard's CSR probabilities) and optionally `answers` [len(questions), 3].
    Returns, on `dst`, all probabilities in request order (CSR values back to back) and the
    answers [n, 3] (or None); (None, None) elsewhere.  Uses torch.distributed object collectives,
    so any backend works (gloo on the host)."""
    import torch.distributed as dist
    payload = (np.asarray(questions, dtype=np.int64), np.asarray(local_off, dtype=np.int64),
               np.asarray(probs, dtype=np.float32),
               None if answers is None else np.asarray(answers, dtype=np.float32).reshape(-1, 3))
    rank = dist.get_rank(group)
    bucket = [None] * dist.get_world_size(group) if rank == dst else None
    dist.gather_object(payload, bucket, dst=dst, group=group)
    if rank != dst:
        return None, None
    n = sum(len(q) for q, _, _, _ in bucket)
    seen = np.concatenate([q for q, _, _, _ in bucket]) if n else np.zeros(0, dtype=np.int64)
    if not np.array_equal(np.sort(seen), np.arange(n)):
        raise ValueError("the shards do not cover every question exactly once")
    per_q = [None] * n
    ans = np.empty((n, 3), dtype=np.float32) if bucket[0][3] is not None else None
    for q, off, p, a in bucket:
        for j, qi in enumerate(q):
            per_q[qi] = p[off[j]:off[j + 1]]
        if ans is not None and len(q):
            ans[q] = a
    out = np.concatenate(per_q) if n else np.zeros(0, dtype=np.float32)
    return out, ans
