"""The prefix side on the device: the shared-prefix length (blink.py `_shared_prefix_len`,
bit-exact against the oracle), KV rows written into an arena region (simit engine.py's arena,
byte-exact), and the prefix's own causal self-attention (the attention call with no prefix over
one long sequence, against the FP64 oracle on every row)."""
import numpy as np
import pytest
import torch

from oracle import oracle
from shared_prefix_question_gb300 import blink
from shared_prefix_question_gb300 import workloads as wl
from tests.helpers import compare_attention, dev_bf16, dev_i32, run_attention

pytestmark = pytest.mark.gpu


def _lcp_gpu(seqs):
    cu = np.concatenate([[0], np.cumsum([len(s) for s in seqs])]).astype(np.int32)
    toks = np.concatenate([np.asarray(s, dtype=np.int32) for s in seqs])
    return blink.blink_shared_prefix_len(dev_i32(toks), dev_i32(cu))


def test_shared_prefix_len_cases():
    rng = np.random.default_rng(1)
    cases = [[[1, 2, 3]], [[5, 5, 5], [5, 5, 5]], [[7, 8], [7, 8, 9, 10]], [[3, 1], [4, 1]]]
    for n, shared, tail in [(2, 40, 5), (64, 18432, 256), (1000, 300, 50), (7, 0, 9), (3, 100, 1)]:
        pre = rng.integers(0, 151936, size=shared).tolist()
        cases.append([pre + rng.integers(0, 151936, size=int(rng.integers(1, tail + 1))).tolist() for _ in range(n)])
    # sequences that agree beyond a warp's 32-token step, and a divergence at a random point
    pre = rng.integers(0, 5, size=5000).tolist()
    div = [pre[:] for _ in range(9)]
    div[4][3333] += 7
    cases.append(div)
    for seqs in cases:
        assert _lcp_gpu(seqs) == oracle.shared_prefix_len(seqs)


def test_shared_prefix_len_flags_empty_sequence():
    cu = dev_i32(np.array([0, 3, 3, 5], dtype=np.int32))
    toks = dev_i32(np.arange(5, dtype=np.int32))
    with pytest.raises(blink.BlinkError) as e:
        blink.blink_shared_prefix_len(toks, cu)
    assert e.value.status == blink.BLINK_DEVICE_FLAG


def test_kv_rows_into_arena_region():
    rng = np.random.default_rng(2)
    n, Hkv, d, stride, slots, dst = 1000, 8, 128, 8 * 128 + 64, 1500, 321
    k = wl.normal_bf16(rng, (n, Hkv, d))
    v = wl.normal_bf16(rng, (n, Hkv, d))
    ak = torch.zeros(slots, stride, dtype=torch.bfloat16, device="cuda")
    av = torch.zeros_like(ak)
    blink.blink_kv_to_arena(dev_bf16(k), dev_bf16(v), ak, av, dst)
    torch.cuda.synchronize()
    ek = np.zeros((slots, stride), dtype=np.uint16)
    ev = np.zeros((slots, stride), dtype=np.uint16)
    ek[dst:dst + n, :Hkv * d] = k.reshape(n, -1)
    ev[dst:dst + n, :Hkv * d] = v.reshape(n, -1)
    np.testing.assert_array_equal(ak.view(torch.int16).cpu().numpy().view(np.uint16), ek)
    np.testing.assert_array_equal(av.view(torch.int16).cpu().numpy().view(np.uint16), ev)
    with pytest.raises(blink.BlinkError) as e:
        blink.blink_kv_to_arena(dev_bf16(k), dev_bf16(v), ak, av, slots - n + 1)
    assert e.value.status == blink.BLINK_OUT_OF_RANGE


@pytest.mark.parametrize("P,Hq,Hkv,d", [(5000, 8, 2, 128), (18432, 32, 8, 128)])
def test_prefix_self_attention(P, Hq, Hkv, d):
    """Encoding the prefix once (blink.py `_forward_shared`) is one causal pass over its P tokens:
    the attention call with no prefix and a single sequence of length P."""
    w = wl.Workload("prefix-encode", 600 + P % 97, 0, 1, 1, 1, Hq, Hkv, d, 8, 8, 1, 1, 1.0, "letters")
    ins = wl.attention_inputs(w, lengths=np.array([P]), P=0)
    out, lse, st = run_attention(ins)
    assert st == blink.BLINK_OK
    compare_attention(ins, out, lse)
