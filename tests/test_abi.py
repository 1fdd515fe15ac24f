"""The C-ABI library builds, loads and exports every entry point include/blink.h declares; the
host-side argument checks reject bad calls before anything is launched.  CPU only: no call here
reaches a kernel (each is refused by the host validation first)."""
import ctypes
import os
import re

import pytest

from shared_prefix_question_gb300 import blink, build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "blink.h")


@pytest.fixture(scope="module")
def lib():
    build.build()
    return blink.lib()


def _declared():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(blink_[a-z_]+)\s*\(", text)))


def test_header_declares_the_three_path_calls():
    names = _declared()
    for n in ("blink_pack_plan", "blink_prefix_tail_attention", "blink_label_readout"):
        assert n in names


def test_boundary_names_of_the_scope_table(lib):
    """The boundary's calls by name: the status string, the three path calls and the workspace
    query of each that takes a workspace (the planner's returns 0: its scratch is its outputs)."""
    raw = ctypes.CDLL(blink.LIB_PATH)
    for n in ("blink_status_string", "blink_pack_plan_workspace", "blink_pack_plan", "blink_attention_workspace",
              "blink_prefix_tail_attention", "blink_label_readout_workspace", "blink_label_readout"):
        assert n in _declared(), n
        assert hasattr(raw, n), n
    for n in (1, 2048, 2049, 32768):
        assert blink.pack_plan_workspace_bytes(n) == 0


def test_library_exports_every_declared_symbol(lib):
    raw = ctypes.CDLL(blink.LIB_PATH)
    for name in _declared():
        assert hasattr(raw, name), name
    assert sorted(blink.exported_symbols()) == _declared()


def test_status_strings(lib):
    for code in range(7):
        assert blink.status_string(code) not in ("", "unknown status")
    assert blink.status_string(99) == "unknown status"


def test_workspace_sizes(lib):
    assert blink.readout_workspace_bytes(512) >= 256 + 512 * 4
    assert blink.readout_workspace_bytes(0) == 0
    assert blink.attention_workspace_bytes(100, 4, 64, 4, 2, 64) >= 256


FAKE = ctypes.c_void_p(0x1000)  # never dereferenced: every call below is refused on the host


def test_readout_host_checks(lib):
    L = lib
    args = dict(hidden=FAKE, stride=256, rows=4, last=FAKE, W=FAKE, V=1024, H=256, off=FAKE, ids=FAKE, B=2, sum_k=4,
                T=1.0, probs=FAKE, hp=None, logits=None, ws=FAKE, wsb=4096, stream=None)

    def call(**kw):
        a = dict(args, **kw)
        return L.blink_label_readout(a["hidden"], a["stride"], a["rows"], a["last"], None, a["W"], a["V"], a["H"], a["off"],
                                     a["ids"], a["B"], a["sum_k"], a["T"], a["probs"], a["hp"], a["logits"], a.get("qt"),
                                     a.get("ans"), a.get("hans"), a["ws"], a["wsb"], a["stream"])
    for t in (0.0, -0.5, float("inf"), float("nan")):     # blink.py `decide`: temperature must be positive
        assert call(T=t) == blink.BLINK_INVALID_ARG
    assert call(H=100) == blink.BLINK_INVALID_ARG         # not a multiple of 8
    assert call(stride=128) == blink.BLINK_INVALID_ARG    # stride below H
    assert call(B=0) == blink.BLINK_OUT_OF_RANGE
    assert call(B=2, sum_k=2 * 255 + 1) == blink.BLINK_OUT_OF_RANGE  # more than MAX_OPTIONS per question
    assert call(wsb=16) == blink.BLINK_WORKSPACE_TOO_SMALL
    assert call(probs=None) == blink.BLINK_INVALID_ARG
    assert call(qt=FAKE) == blink.BLINK_INVALID_ARG          # question types without an answers buffer
    assert call(hans=FAKE) == blink.BLINK_INVALID_ARG        # host answers without device answers


def test_attention_host_checks(lib):
    L = lib

    def call(P=64, B=4, rows=60, max_tail=24, Hq=4, Hkv=2, d=64, stride=128, ws=4096, kpre=FAKE):
        return L.blink_prefix_tail_attention(FAKE, kpre, kpre, stride, FAKE, FAKE, FAKE, None, B, rows, P, max_tail, Hq,
                                             Hkv, d, 0.0, FAKE, None, FAKE, ws, None)
    assert call(d=96) == blink.BLINK_INVALID_ARG
    assert call(Hq=6, Hkv=4) == blink.BLINK_INVALID_ARG
    assert call(P=131073, max_tail=1) == blink.BLINK_OUT_OF_RANGE   # past MAX_INPUT_TOKENS
    assert call(max_tail=131073) == blink.BLINK_OUT_OF_RANGE
    assert call(B=0) == blink.BLINK_OUT_OF_RANGE
    assert call(stride=100) == blink.BLINK_INVALID_ARG               # stride below Hkv * d
    assert call(kpre=None) == blink.BLINK_INVALID_ARG                # prefix pointers missing
    assert call(ws=8) == blink.BLINK_WORKSPACE_TOO_SMALL
    assert call(rows=0) == blink.BLINK_INVALID_ARG


def test_plan_host_checks(lib):
    L = lib
    f = [FAKE] * 10
    assert L.blink_pack_plan(FAKE, 10, 0, 0, *f, None) == blink.BLINK_INVALID_ARG       # budget < 1
    assert L.blink_pack_plan(FAKE, 10, 100, -1, *f, None) == blink.BLINK_INVALID_ARG    # negative row cap
    assert L.blink_pack_plan(FAKE, 0, 100, 0, *f, None) == blink.BLINK_OUT_OF_RANGE
    assert L.blink_pack_plan(FAKE, 32769, 100, 0, *f, None) == blink.BLINK_OUT_OF_RANGE


def test_selftest_wait_host_checks(lib):
    assert lib.blink_selftest_wait_timeout(1000, None, 256, None) == blink.BLINK_INVALID_ARG
    assert lib.blink_selftest_wait_timeout(1000, FAKE, 16, None) == blink.BLINK_WORKSPACE_TOO_SMALL
    assert lib.blink_selftest_wait_timeout(0, FAKE, 256, None) == blink.BLINK_OUT_OF_RANGE
    assert lib.blink_selftest_wait_timeout(2000000, FAKE, 256, None) == blink.BLINK_OUT_OF_RANGE
