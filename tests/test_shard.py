"""Question sharding across ranks and the host-side gather (host logic, CPU only).

Questions are independent given the prefix KV, so a request splits across GPUs by question with
no exchange in the step; the answers are gathered on one rank.  The two-rank test runs real
`gloo` processes on 127.0.0.1; each rank computes its shard with the FP64 oracle (the per-rank
device step is the same C-ABI path the GPU tests cover), and the gathered result must equal the
unsharded one exactly.
"""
import os
import socket
import sys

import numpy as np
import pytest

from shared_prefix_question_gb300 import shard

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.mark.parametrize("world", [1, 2, 3, 8])
@pytest.mark.parametrize("seed", [0, 1, 2])
def test_shards_cover_in_order_and_balance(world, seed):
    rng = np.random.default_rng(seed)
    lengths = rng.integers(1, 1000, size=int(rng.integers(world, 300)))
    parts = shard.shard_questions(lengths, world)
    assert len(parts) == world
    np.testing.assert_array_equal(np.concatenate(parts), np.arange(len(lengths)))  # contiguous, request order
    assert all(len(p) >= 1 for p in parts)
    tokens = np.array([lengths[p].sum() for p in parts])
    # a cut lands on the question boundary nearest its target, so no shard is off by more than
    # one question's tokens on each side
    assert tokens.max() - lengths.sum() / world <= 2 * lengths.max()


def test_shards_with_fewer_questions_than_ranks():
    parts = shard.shard_questions([5, 9], 4)
    assert [list(p) for p in parts] == [[0], [1], [], []]
    with pytest.raises(ValueError):
        shard.shard_questions([3, 0], 2)


def test_one_long_question_balances_around_it():
    parts = shard.shard_questions([1, 1, 1000, 1, 1], 2)
    np.testing.assert_array_equal(np.concatenate(parts), np.arange(5))
    assert len(parts[0]) >= 1 and len(parts[1]) >= 1


def test_local_labels_rebases_the_csr():
    off = np.array([0, 2, 5, 6, 9], dtype=np.int32)
    ids = np.arange(100, 109, dtype=np.int32)
    loff, lids = shard.local_labels(off, ids, np.array([1, 3]))
    np.testing.assert_array_equal(loff, [0, 3, 6])
    np.testing.assert_array_equal(lids, [102, 103, 104, 106, 107, 108])
    loff, lids = shard.local_labels(off, ids, np.array([], dtype=np.int64))
    np.testing.assert_array_equal(loff, [0])
    assert len(lids) == 0


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, root):
    sys.path.insert(0, root)
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    import torch.distributed as dist
    from oracle import oracle
    from shared_prefix_question_gb300 import shard as sh
    from shared_prefix_question_gb300 import workloads as w
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        rng = np.random.default_rng(5)  # one request: 24 questions, hidden 64, vocabulary 500
        B, H, V = 24, 64, 500
        lengths = rng.integers(1, 40, size=B)
        counts = rng.integers(1, 9, size=B)
        label_off = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
        ins = w.ReadoutInputs(w.normal_bf16(rng, (int(lengths.sum()), H)), (np.cumsum(lengths) - 1).astype(np.int32),
                              w.normal_bf16(rng, (V, H), std=0.05), label_off,
                              rng.integers(0, V, size=int(label_off[-1])).astype(np.int32), 0.7)
        qt = np.where(rng.random(B) < 0.5, oracle.QTYPE_CHOICE, oracle.QTYPE_SCORE)
        mine = sh.shard_questions(lengths, world)[rank]
        off, ids = sh.local_labels(ins.label_off, ins.label_ids, mine)
        _, probs, st = oracle.label_readout(ins.hidden, ins.last_idx[mine], ins.unembed, off, ids, ins.temperature)
        assert st == 0
        ans = np.array([[a["index"], a["confidence"], a["value"]]
                        for a in (oracle.answer(int(qt[q]), probs[off[j]:off[j + 1]]) for j, q in enumerate(mine))],
                       dtype=np.float32).reshape(-1, 3)
        all_probs, all_ans = sh.gather_results(mine, off, probs, ans)
        if rank == 0:
            _, ref, st = oracle.label_readout(ins.hidden, ins.last_idx, ins.unembed, ins.label_off, ins.label_ids,
                                              ins.temperature)
            assert st == 0
            np.testing.assert_array_equal(all_probs, ref.astype(np.float32))
            ref_ans = np.array([[a["index"], a["confidence"], a["value"]] for a in
                                (oracle.answer(int(qt[b]), ref[ins.label_off[b]:ins.label_off[b + 1]])
                                 for b in range(len(lengths)))], dtype=np.float32)
            np.testing.assert_array_equal(all_ans, ref_ans)
        else:
            assert all_probs is None and all_ans is None
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_ranks_gather_equals_unsharded():
    import torch.multiprocessing as mp
    mp.spawn(_rank_main, args=(2, _free_port(), ROOT), nprocs=2, join=True)
