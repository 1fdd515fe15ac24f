#!/usr/bin/env python
"""Benchmark of the shared-prefix one-pass decision hot path on GB300.

One step = one pass of the whole path over one batch: the token-budget pack plan, the
prefix-tail attention of every question's tail against the shared prefix (one attention layer),
the label readout with its temperature softmax and typed answers, and the forward's one host
transfer of the probabilities and answers.  Default workload: the long-document case
(prefix 18432 tokens, 64 questions with tails U[64,256], 32/8 heads, d 128, hidden 2560,
vocabulary 151936, 2-26 labels, T 0.7), synthetic and seeded.

Prints one JSON line (rank 0).  `--impl reference` times the FP64 CPU oracle on the host cores
instead, on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "questions/sec and prefill tokens/sec at 1 GB300; % BF16 TC peak and % HBM BW"
FLUSH_BYTES = 512 << 20  # flushed between timed steps: larger than the 129 MB L2
# Spec-sheet figures of the part, reported beside the fractions of the measured peaks (the
# measured copy bandwidth and bf16 GEMM rate are the roofline denominators).
SPEC_TFLOPS = 2500.0  # dense bf16, TFLOP/s
SPEC_GBS = 8000.0     # HBM3e, GB/s


def flush_l2(buf):
    """Evicts L2 between timed steps: write a buffer larger than L2, then read it back, so the
    write-back of the dirty flush lines happens here and not inside the next timed region."""
    buf.zero_()
    buf.view(-1, 4096).amax(dim=1)


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="18k")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-stress", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=15.0, help="target CPU work of the oracle sample")
    ap.add_argument("--no-cpu-configs", action="store_true",
                    help="skip the oracle timings on every workload of the table (about a minute of CPU work)")
    ap.add_argument("--no-rows", action="store_true", help="skip the measurements of the other path rows")
    ap.add_argument("--only", choices=["readout_stress", "attention", "pack_plan"], default=None,
                    help="run one sub-measurement alone (for profiling) and print its JSON: the readout on "
                         "its stress input, the attention on --workload (optionally --questions / --tails), or "
                         "the pack plan at 32768 lengths")
    ap.add_argument("--questions", type=int, default=0,
                    help="with --only attention: the first N questions of the workload (0: all)")
    ap.add_argument("--tails", default="",
                    help="with --only attention: comma-separated tail lengths instead of the workload's")
    return ap.parse_args()


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), float(p["bf16_tflops"]), float(p.get("bf16_tflops_sustained", 0)), "measured"
    except Exception:
        return 6800.0, 1900.0, 1700.0, "fallback"


def attention_flops(lengths: np.ndarray, P: int, Hq: int, d: int) -> float:
    """Algorithmic FLOPs: QK^T and PV over every prefix key once per tail row, causal tail only."""
    t = lengths.astype(np.float64)
    return 4.0 * Hq * d * (t.sum() * P + (t * (t + 1) / 2).sum())


def traffic_record(kernel_src: str, key: str):
    """DRAM bytes per launch from a committed ncu summary, only if the kernel source is unchanged."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f)[key]
        with open(kernel_src, "rb") as f:
            sha = hashlib.sha256(f.read()).hexdigest()
        if rec.get("source_sha256") == sha:
            return float(rec["bytes_per_launch"])
    except Exception:
        pass
    return None


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str):
        self.gpu_id = gpu_id
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "100",
                 "-i", self.gpu_id], stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
            return
        t0 = time.time()
        while time.time() - t0 < 5 and os.path.getsize(self.path) == 0:
            time.sleep(0.02)

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    rows.append(parts)
                except Exception:
                    pass
        os.unlink(self.path)
        if not rows:
            return None
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows)}


def wl_question_types(w, label_off):
    from shared_prefix_question_gb300 import workloads as wl
    return wl.question_types(w, label_off)


def build_workload(name: str):
    from shared_prefix_question_gb300 import workloads as wl
    w = wl.WORKLOADS[name]
    lengths = wl.tail_lengths(w)                       # request order
    slot_lengths = np.sort(lengths, kind="stable")     # the tails packed in the plan's slot order
    ins = wl.attention_inputs(w, lengths=slot_lengths)
    rd = wl.readout_inputs(w, rows=ins.rows, last_idx=np.zeros(w.n, dtype=np.int32))
    return w, lengths, ins, rd


def cpu_baseline(w, lengths, ins, rd, target_s: float, n_threads: int = 0):
    """The oracle, as it stands, on a bounded sample: the plan over every question, the attention
    of the first q questions' tails (every head, every row) and their label readout."""
    from oracle import oracle
    cores = n_threads or os.cpu_count()

    def run(q):
        t0 = time.perf_counter()
        oracle.pack_plan(lengths, 32768, 0)
        toks = np.concatenate([np.arange(ins.seq_start[b], ins.seq_start[b] + ins.seq_len[b]) for b in range(q)])
        tok = np.repeat(toks, ins.Hq).astype(np.int32)
        head = np.tile(np.arange(ins.Hq), len(toks)).astype(np.int32)
        oracle.prefix_tail_attention(ins.q, ins.k_pre, ins.v_pre, ins.k_tail, ins.v_tail, ins.seq_start, ins.seq_len,
                                     ins.P, ins.Hq, ins.Hkv, ins.d, select=(tok, head), n_threads=cores)
        last = (ins.cu_seqlens[1:q + 1] - 1).astype(np.int32)
        oracle.label_readout(rd.hidden, last, rd.unembed, rd.label_off[:q + 1], rd.label_ids[:rd.label_off[q]],
                             rd.temperature)
        return time.perf_counter() - t0

    t1 = run(1)
    q = int(max(1, min(w.n, target_s / max(t1, 1e-3))))
    if q > 1:
        tq = run(q)
    else:
        tq = t1
    # one core: the first 16 tail tokens of question 0 (every head), scaled to whole questions
    n_tok = int(min(16, ins.seq_len[0]))
    toks = np.arange(ins.seq_start[0], ins.seq_start[0] + n_tok)
    t0 = time.perf_counter()
    oracle.prefix_tail_attention(ins.q, ins.k_pre, ins.v_pre, ins.k_tail, ins.v_tail, ins.seq_start, ins.seq_len,
                                 ins.P, ins.Hq, ins.Hkv, ins.d,
                                 select=(np.repeat(toks, ins.Hq).astype(np.int32),
                                         np.tile(np.arange(ins.Hq), n_tok).astype(np.int32)), n_threads=1)
    t_one = time.perf_counter() - t0
    per_question = t_one / n_tok * float(np.mean(ins.seq_len))
    return {"value": q / tq, "unit": "questions/s", "cores": cores, "kind": "oracle",
            "sample": f"{q} of {w.n} questions (all heads and tail rows; plan over all {w.n}), "
                      f"{tq:.1f} s of FP64 CPU work",
            "single_core": {"value": 1.0 / per_question, "unit": "questions/s",
                            "sample": f"attention of {n_tok} tail tokens x {ins.Hq} heads of question 0 on one "
                                      f"core ({t_one:.1f} s), scaled to the mean tail length"}}, q, tq


def _oracle_flops(ins, tok, head):
    """Algorithmic FLOPs of the oracle's attention rows (token, head): 4 d (P + i + 1) each."""
    owner = np.searchsorted(ins.seq_start, tok, side="right") - 1
    i = tok - ins.seq_start[owner]
    return float(4.0 * ins.d * (ins.P + i + 1).astype(np.float64).sum())


def cpu_baseline_per_config(cores: int, max_questions: int = 2, names=("tiny", "2k", "18k", "plain", "max")):
    """The oracle, as it stands, on every workload of the table: the plan, the attention of every
    tail row and head, and the label readout of every question.  Tiny, 2k, 18k and plain run in
    full on all host cores; the largest request on its first `max_questions` questions (plan and
    readout over all), extrapolated to all 512 by attention FLOPs.  Beside each, one core on a
    sample (the attention of question 0's last 8 tail rows, every head), scaled by FLOPs to the
    whole workload."""
    from oracle import oracle
    from shared_prefix_question_gb300 import workloads as wl
    out = {}
    for name in names:
        w = wl.WORKLOADS[name]
        lengths = wl.tail_lengths(w)
        ins = wl.attention_inputs(w, lengths=lengths)
        rd = wl.readout_inputs(w, rows=ins.rows)
        total_flops = attention_flops(lengths, w.P, w.Hq, w.d)
        q = w.n if name != "max" else max_questions
        t0 = time.perf_counter()
        oracle.pack_plan(lengths, wl.TOKEN_BUDGET, 0)
        if q == w.n:
            oracle.prefix_tail_attention(ins.q, ins.k_pre, ins.v_pre, ins.k_tail, ins.v_tail, ins.seq_start,
                                         ins.seq_len, ins.P, ins.Hq, ins.Hkv, ins.d, n_threads=cores)
            sub_flops = total_flops
        else:
            toks = np.concatenate([np.arange(ins.seq_start[b], ins.seq_start[b] + ins.seq_len[b]) for b in range(q)])
            tok = np.repeat(toks, ins.Hq).astype(np.int32)
            head = np.tile(np.arange(ins.Hq), len(toks)).astype(np.int32)
            oracle.prefix_tail_attention(ins.q, ins.k_pre, ins.v_pre, ins.k_tail, ins.v_tail, ins.seq_start,
                                         ins.seq_len, ins.P, ins.Hq, ins.Hkv, ins.d, select=(tok, head),
                                         n_threads=cores)
            sub_flops = _oracle_flops(ins, tok, head)
        oracle.label_readout(rd.hidden, rd.last_idx, rd.unembed, rd.label_off, rd.label_ids, rd.temperature)
        t = time.perf_counter() - t0
        t_full = t * total_flops / sub_flops  # the plan and readout are < 1 % of the oracle's time
        # one core: question 0's last 8 tail rows, every head
        L0 = int(ins.seq_len[0])
        toks = np.arange(ins.seq_start[0] + max(0, L0 - 8), ins.seq_start[0] + L0)
        tok = np.repeat(toks, ins.Hq).astype(np.int32)
        head = np.tile(np.arange(ins.Hq), len(toks)).astype(np.int32)
        t1 = time.perf_counter()
        oracle.prefix_tail_attention(ins.q, ins.k_pre, ins.v_pre, ins.k_tail, ins.v_tail, ins.seq_start,
                                     ins.seq_len, ins.P, ins.Hq, ins.Hkv, ins.d, select=(tok, head), n_threads=1)
        t1 = time.perf_counter() - t1
        rate1 = _oracle_flops(ins, tok, head) / max(t1, 1e-9)
        prefill = w.P + int(lengths.sum())
        out[name] = {"questions_per_s": w.n / t_full, "prefill_tokens_per_s": prefill / t_full,
                     "seconds": t, "cores": cores,
                     "timed": "in full" if q == w.n else
                              f"first {q} of {w.n} questions ({sub_flops:.3g} of {total_flops:.3g} attention FLOP), "
                              f"extrapolated by FLOPs to {t_full:.0f} s",
                     "single_core_questions_per_s": w.n / (total_flops / rate1),
                     "single_core_sample": f"{len(toks)} tail rows x {ins.Hq} heads of question 0 in {t1:.2f} s "
                                           f"({rate1 / 1e9:.2f} GFLOP/s), scaled by FLOPs"}
    return out


def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    w, lengths, ins, rd = build_workload(args.workload)
    from oracle import oracle
    oracle.build()
    cores = os.cpu_count()
    # each step: the oracle on one question's tail (all heads), its readout and the whole plan
    times = []
    for i in range(args.warmup + args.steps):
        b = i % w.n
        t0 = time.perf_counter()
        oracle.pack_plan(lengths, 32768, 0)
        toks = np.arange(ins.seq_start[b], ins.seq_start[b] + ins.seq_len[b])
        tok = np.repeat(toks, ins.Hq).astype(np.int32)
        head = np.tile(np.arange(ins.Hq), len(toks)).astype(np.int32)
        oracle.prefix_tail_attention(ins.q, ins.k_pre, ins.v_pre, ins.k_tail, ins.v_tail, ins.seq_start,
                                     ins.seq_len, ins.P, ins.Hq, ins.Hkv, ins.d, select=(tok, head), n_threads=cores)
        lo, hi = rd.label_off[b], rd.label_off[b + 1]
        oracle.label_readout(rd.hidden, np.array([ins.cu_seqlens[b + 1] - 1], dtype=np.int32), rd.unembed,
                             np.array([0, hi - lo], dtype=np.int32), rd.label_ids[lo:hi].copy(), rd.temperature)
        if i >= args.warmup:
            times.append(time.perf_counter() - t0)
    t = sum(times)
    value = args.steps / t
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "questions/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1000 * t / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": f"{w.name}: {w.description}", "P": w.P, "questions": w.n,
                       "sample_per_step": "one question's tail rows x all heads, its readout, the full plan"},
            "cpu_baseline": {"value": value, "unit": "questions/s", "cores": cores, "kind": "oracle",
                             "sample": "one question per step"},
            "e2e": {"value": value, "unit": "questions/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main():
    args = parse()
    if args.impl == "reference":
        run_reference(args)
        return
    import torch
    import torch.distributed as dist

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        dist.init_process_group("nccl", device_id=dev)

    from shared_prefix_question_gb300 import blink, build
    build.build()
    hbm_peak, tc_peak, tc_sustained, peak_kind = peaks()
    if args.only == "readout_stress":
        flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)
        print(json.dumps(readout_stress(blink, dev, hbm_peak, peak_kind, flush, args)), flush=True)
        return
    if args.only == "attention":
        from shared_prefix_question_gb300 import workloads as wl
        flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)
        if args.tails:
            lengths = np.array([int(x) for x in args.tails.split(",")], dtype=np.int32)
        else:
            lengths = wl.tail_lengths(wl.WORKLOADS[args.workload]).astype(np.int32)
            if args.questions:
                lengths = lengths[:args.questions]
        row = attention_config_row(blink, dev, args.workload, tc_peak, hbm_peak, flush, lengths=lengths)
        print(json.dumps({"only": "attention", "workload": args.workload, **row}), flush=True)
        return
    if args.only == "pack_plan":
        flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)
        print(json.dumps({"only": "pack_plan", **pack_plan_row(blink, dev, flush)}), flush=True)
        return

    w, lengths, ins, rd = build_workload(args.workload)

    def bf(a):
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(dev)

    def i32(a):
        return torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).to(dev)

    # ---- device-resident inputs
    d_len = i32(lengths)
    q, kt, vt = bf(ins.q), bf(ins.k_tail), bf(ins.v_tail)
    kp, vp = (bf(ins.k_pre), bf(ins.v_pre)) if ins.P else (None, None)
    hidden, W = bf(rd.hidden), bf(rd.unembed)
    off, ids = i32(rd.label_off), i32(rd.label_ids)
    qtype = i32(wl_question_types(w, rd.label_off))
    n, sum_k = w.n, len(rd.label_ids)
    answers = torch.empty(n, 3, dtype=torch.float32, device=dev)
    max_tail = int(lengths.max())
    plan = {k: torch.empty(n + (1 if k in ("fwd_slot_start", "cu_seqlens") else 0), dtype=torch.int32, device=dev)
            for k in ("order", "slot_of", "fwd_of_slot", "fwd_slot_start", "fwd_width", "cu_seqlens", "last_varlen",
                      "last_padded")}
    plan["n_forwards_dev"] = torch.empty(1, dtype=torch.int32, device=dev)
    out = torch.empty_like(q)
    probs = torch.empty(sum_k, dtype=torch.float32, device=dev)
    ws_a = blink.new_workspace(blink.attention_workspace_bytes(ins.rows, n, ins.P, ins.Hq, ins.Hkv, ins.d), dev)
    ws_r = blink.new_workspace(blink.readout_workspace_bytes(n), dev)
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()

    # the forward's one host transfer: probabilities and answers into pinned host memory (issued
    # on the stream without a host wait, as a server overlapping forwards would)
    h_probs = torch.empty(sum_k, dtype=torch.float32, pin_memory=True)
    h_answers = torch.empty(n, 3, dtype=torch.float32, pin_memory=True)

    def step(ev=None):
        if ev:
            ev[0].record(stream)
        blink.blink_pack_plan(d_len, 32768, 0, out=plan)
        if ev:
            ev[1].record(stream)
        blink.blink_prefix_tail_attention(q, kp, vp, kt, vt, plan["cu_seqlens"], B=n, P=ins.P, max_tail=max_tail,
                                          out=out, ws=ws_a)
        if ev:
            ev[2].record(stream)
        blink.blink_label_readout(hidden, plan["last_varlen"], W, off, ids, rd.temperature, probs=probs, ws=ws_r,
                                  slot_of=plan["slot_of"], qtype=qtype, answers=answers)
        if ev:
            ev[3].record(stream)
        h_probs.copy_(probs, non_blocking=True)
        h_answers.copy_(answers, non_blocking=True)
        if ev:
            ev[4].record(stream)

    for _ in range(args.warmup):
        flush_l2(flush)
        step()
    torch.cuda.synchronize()
    st = blink.blink_read_device_status(ws_a)
    st_r = blink.blink_read_device_status(ws_r)
    if st != 0 or st_r != 0:
        raise SystemExit(f"device status after warm-up: attention {st}, readout {st_r}")

    # ---- timed region: K steps, L2 flushed before each, per-kernel events on the launching stream
    gpu_uuid = str(torch.cuda.get_device_properties(dev).uuid)
    sampler = ClockSampler(gpu_uuid if gpu_uuid.startswith("GPU-") else f"GPU-{gpu_uuid}")
    if rank == 0:
        sampler.start()
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(5)] for _ in range(args.steps)]
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    for k in range(args.steps):
        flush_l2(flush)
        step(evs[k])
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    clocks = sampler.stop() if rank == 0 else None
    plan_ms = [e[0].elapsed_time(e[1]) for e in evs]
    attn_ms = [e[1].elapsed_time(e[2]) for e in evs]
    read_ms = [e[2].elapsed_time(e[3]) for e in evs]
    d2h_ms = [e[3].elapsed_time(e[4]) for e in evs]
    step_ms = [e[0].elapsed_time(e[4]) for e in evs]
    total_ms = sum(step_ms)
    if world > 1:
        t = torch.tensor([total_ms], dtype=torch.float64, device=dev)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        total_ms = float(t.item())
    ms_per_step = total_ms / args.steps
    value = world * n / (ms_per_step / 1000.0)
    prefill_tokens = ins.P + int(lengths.sum())  # blink.py `_prefill_tokens`: the shared prefix counted once

    # ---- roofline of the dominant kernel (attention: a dense contraction on the tensor cores)
    flops = attention_flops(lengths, ins.P, ins.Hq, ins.d)
    attn_mean = statistics.mean(attn_ms)
    achieved = flops / (attn_mean / 1000.0) / 1e12
    traffic = traffic_record(os.path.join(ROOT, "shared_prefix_question_gb300", "csrc", "attention.cu"),
                             f"attention_{w.name}")
    roofline = {"bound": "tensor", "achieved": achieved, "peak": tc_peak, "unit": "TFLOP/s",
                "frac": achieved / tc_peak, "traffic": traffic,
                "spec_peak": SPEC_TFLOPS, "frac_spec": achieved / SPEC_TFLOPS,
                "kernel": "attention_kernel<128>", "peak_kind": f"{peak_kind} bf16 burst (kernel timed alone)",
                "flops_per_launch": flops}

    line = {"metric": METRIC, "value": value, "unit": "questions/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": f"{w.name}: {w.description}", "P": ins.P, "questions": n,
                       "tail_tokens": int(lengths.sum()), "Hq": ins.Hq, "Hkv": ins.Hkv, "d": ins.d, "H": w.H,
                       "V": w.V, "labels": sum_k, "temperature": w.temperature, "budget": 32768,
                       "l2": f"flushed before every step ({FLUSH_BYTES >> 20} MiB written then read back)",
                       "parallelism": f"replicas x{world}, questions sharded, no collective in the step"},
            "prefill_tokens_per_s": world * prefill_tokens / (ms_per_step / 1000.0),
            "tail_tokens_per_s": world * int(lengths.sum()) / (ms_per_step / 1000.0),
            "kernels_ms": {"plan": statistics.mean(plan_ms), "attention": attn_mean,
                           "readout": statistics.mean(read_ms), "d2h_probs_answers": statistics.mean(d2h_ms)},
            "spread_ms": {"step": spread(step_ms), "attention": spread(attn_ms)},
            "roofline": roofline, "gpu_launches": 3 * args.steps, "clocks": clocks}

    # ---- readout on the stress input (HBM-bound at scale)
    if not args.no_stress and rank == 0:
        line["roofline_readout_stress"] = readout_stress(blink, dev, hbm_peak, peak_kind, flush, args)

    # ---- the other rows of the path, each timed alone (CUDA events, L2 flushed before each launch)
    if not args.no_rows and rank == 0:
        line["rows"] = other_rows(blink, dev, w, ins, flush, hbm_peak, tc_peak, peak_kind)

    # ---- end to end through the C ABI with host buffers (copies inside the timed region)
    if not args.no_e2e:
        line["e2e"] = e2e(blink, dev, w, lengths, ins, rd, flush, args, world)

    if rank == 0:
        if not args.no_cpu_baseline:
            line["cpu_baseline"] = cpu_baseline(w, lengths, ins, rd, args.cpu_seconds)[0]
            if not args.no_cpu_configs:
                line["cpu_baseline"]["per_config"] = cpu_baseline_per_config(os.cpu_count())
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def _time_all(fn, flush, reps=10):
    """Device times (ms) of fn() over reps launches, L2 flushed before each."""
    import torch
    fn()
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()
    evs = []
    for _ in range(reps):
        flush_l2(flush)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        fn()
        e1.record(stream)
        evs.append((e0, e1))
    torch.cuda.synchronize()
    return [a.elapsed_time(b) for a, b in evs]


def _time(fn, flush, reps=10):
    """Mean device time (ms) of fn() over reps launches, L2 flushed before each."""
    return statistics.mean(_time_all(fn, flush, reps))


def spread(ms):
    """Median and 10th / 90th percentiles of a list of times."""
    q = np.percentile(np.asarray(ms, dtype=np.float64), [10, 50, 90])
    return {"p10": float(q[0]), "median": float(q[1]), "p90": float(q[2])}


def attention_config_row(blink, dev, name, tc_peak, hbm_peak, flush, lengths=None, header_only_ws=False):
    """The prefix-tail attention on one of the other workloads (lengths and shapes from the
    workload table, values drawn on the device): FLOP fraction, and for the plain causal
    workload, which sits near the ridge, the byte fraction too (Q, K, V read and O written once)."""
    import torch
    from shared_prefix_question_gb300 import workloads as wl
    w = wl.WORKLOADS[name]
    if lengths is None:
        lengths = wl.tail_lengths(w).astype(np.int32)
    rows = int(lengths.sum())
    g = torch.Generator(device=dev)
    g.manual_seed(100 + w.index)
    bf = torch.bfloat16
    q = torch.randn(rows, w.Hq, w.d, generator=g, device=dev).to(bf)
    kt = torch.randn(rows, w.Hkv, w.d, generator=g, device=dev).to(bf)
    vt = torch.randn(rows, w.Hkv, w.d, generator=g, device=dev).to(bf)
    kp = torch.randn(w.P, w.Hkv, w.d, generator=g, device=dev).to(bf) if w.P else None
    vp = torch.randn(w.P, w.Hkv, w.d, generator=g, device=dev).to(bf) if w.P else None
    cu = torch.tensor(np.concatenate([[0], np.cumsum(lengths)]), dtype=torch.int32, device=dev)
    o = torch.empty_like(q)
    # a header-only workspace leaves no room for prefix chunks: the unsplit kernel, for comparison
    ws = blink.new_workspace(256 if header_only_ws else
                             blink.attention_workspace_bytes(rows, len(lengths), w.P, w.Hq, w.Hkv, w.d), dev)
    ms_all = _time_all(lambda: blink.blink_prefix_tail_attention(q, kp, vp, kt, vt, cu, B=len(lengths), P=w.P,
                                                                 max_tail=int(lengths.max()), out=o, ws=ws), flush)
    ms = statistics.mean(ms_all)
    fl = attention_flops(lengths, w.P, w.Hq, w.d)
    row = {"ms": ms, **spread(ms_all), "tflops": fl / ms / 1e9, "frac": fl / ms / 1e9 / tc_peak,
           "frac_spec": fl / ms / 1e9 / SPEC_TFLOPS,
           "shape": w.description if len(lengths) == w.n else f"{len(lengths)} question(s), tails {list(lengths)}, "
                                                                 f"prefix {w.P}, {w.Hq}/{w.Hkv} heads"}
    if not w.P:
        nbytes = rows * (2 * w.Hq + 2 * w.Hkv) * w.d * 2
        row.update({"bytes": nbytes, "GBs": nbytes / ms / 1e6, "byte_frac": nbytes / ms / 1e6 / hbm_peak,
                    "byte_frac_spec": nbytes / ms / 1e6 / SPEC_GBS})
    return row


def other_rows(blink, dev, w, ins, flush, hbm_peak, tc_peak, peak_kind):
    """The prefix side, several requests per launch and the log-space readout, on inputs shaped
    like the long-document workload (synthetic, drawn on the device: timing only; parity is in
    the tests)."""
    import torch
    g = torch.Generator(device=dev)
    g.manual_seed(11)
    bf = torch.bfloat16
    out = {}
    # 0. the attention on the other workloads of the table (the 18k one is the step above), and
    # one question against the 18k prefix (a small grid: the prefix is split into chunks)
    for name in ("2k", "plain", "max"):
        out[f"attention_{name}"] = attention_config_row(blink, dev, name, tc_peak, hbm_peak, flush)
    out["attention_one_question_18k"] = attention_config_row(blink, dev, "18k", tc_peak, hbm_peak, flush,
                                                             lengths=np.array([128], dtype=np.int32))
    out["attention_one_question_18k_unsplit"] = attention_config_row(
        blink, dev, "18k", tc_peak, hbm_peak, flush, lengths=np.array([128], dtype=np.int32), header_only_ws=True)
    P, Hq, Hkv, d = w.P, w.Hq, w.Hkv, w.d
    # 1. the prefix's own causal self-attention: one sequence of P tokens, no prefix
    q = torch.randn(P, Hq, d, generator=g, device=dev).to(bf)
    k = torch.randn(P, Hkv, d, generator=g, device=dev).to(bf)
    v = torch.randn(P, Hkv, d, generator=g, device=dev).to(bf)
    cu1 = torch.tensor([0, P], dtype=torch.int32, device=dev)
    o = torch.empty_like(q)
    ws = blink.new_workspace(256, dev)
    ms = _time(lambda: blink.blink_prefix_tail_attention(q, None, None, k, v, cu1, B=1, P=0, max_tail=P, out=o, ws=ws),
               flush)
    fl = attention_flops(np.array([P]), 0, Hq, d)
    out["prefix_self_attention"] = {"ms": ms, "tflops": fl / ms / 1e9, "frac": fl / ms / 1e9 / tc_peak,
                                    "frac_spec": fl / ms / 1e9 / SPEC_TFLOPS,
                                    "shape": f"one causal sequence of {P} tokens, {Hq}/{Hkv} heads, d {d}"}
    # 2. the prefix K/V rows written into an arena region
    slots = P + 4096
    ak = torch.empty(slots, Hkv * d, dtype=bf, device=dev)
    av = torch.empty_like(ak)
    ms = _time(lambda: blink.blink_kv_to_arena(k, v, ak, av, 1024), flush)
    nbytes = 2 * 2 * P * Hkv * d * 2
    out["kv_to_arena"] = {"ms": ms, "GBs": nbytes / ms / 1e6, "frac": nbytes / ms / 1e6 / hbm_peak,
                          "frac_spec": nbytes / ms / 1e6 / SPEC_GBS,
                          "bytes": nbytes, "shape": f"{P} rows of K and V ({Hkv}x{d} bf16) read and written"}
    del q, o
    # 3. shared-prefix length over the questions' full prompts (prefix + tail each)
    lengths = wl_tail_lengths(w)
    pre = torch.randint(0, w.V, (P,), generator=g, device=dev, dtype=torch.int32)
    seqs = [torch.cat([pre, torch.randint(0, w.V, (int(L),), generator=g, device=dev, dtype=torch.int32)])
            for L in lengths]
    toks = torch.cat(seqs)
    cu = torch.tensor(np.concatenate([[0], np.cumsum([P + int(L) for L in lengths])]), dtype=torch.int32, device=dev)
    lout = torch.empty(1, dtype=torch.int32, device=dev)
    lws = blink.new_workspace(256, dev)
    ms = _time(lambda: blink.blink_shared_prefix_len(toks, cu, out=lout, sync=False, ws=lws), flush)
    out["shared_prefix_len"] = {"ms": ms, "tokens": int(toks.numel()),
                                "shape": f"{len(lengths)} prompts sharing {P} tokens"}
    # 4. several requests in one launch: 8 requests, each a 2048-token prefix with 16 tails U[32,128]
    rng = np.random.default_rng(21)
    n_req, Pr = 8, 2048
    tails = [rng.integers(32, 129, size=16) for _ in range(n_req)]
    lens = np.concatenate(tails).astype(np.int32)
    rows = int(lens.sum())
    arena_k = torch.randn(n_req * Pr, Hkv, d, generator=g, device=dev).to(bf)
    arena_v = torch.randn(n_req * Pr, Hkv, d, generator=g, device=dev).to(bf)
    qm = torch.randn(rows, Hq, d, generator=g, device=dev).to(bf)
    km = torch.randn(rows, Hkv, d, generator=g, device=dev).to(bf)
    vm = torch.randn(rows, Hkv, d, generator=g, device=dev).to(bf)
    cum = torch.tensor(np.concatenate([[0], np.cumsum(lens)]), dtype=torch.int32, device=dev)
    req_rows = np.concatenate([[0], np.cumsum([t.sum() for t in tails])]).astype(np.int32)
    om = torch.empty_like(qm)
    mws = blink.new_workspace(256, dev)
    ms = _time(lambda: blink.blink_prefix_tail_attention_multi(
        qm, arena_k, arena_v, km, vm, cum, B=len(lens), req_rows=req_rows,
        req_prefix_start=[r * Pr for r in range(n_req)], req_prefix_len=[Pr] * n_req, max_tail=128, out=om, ws=mws),
        flush)
    fl = sum(attention_flops(t, Pr, Hq, d) for t in tails)
    out["several_requests"] = {"ms": ms, "tflops": fl / ms / 1e9, "frac": fl / ms / 1e9 / tc_peak,
                               "frac_spec": fl / ms / 1e9 / SPEC_TFLOPS,
                               "shape": f"{n_req} requests x (prefix {Pr}, 16 tails U[32,128]) in one launch"}
    # 5. the pack plan at its largest size: 64 requests x 512 questions (32768 lengths U[16,1024])
    out["pack_plan_32768"] = pack_plan_row(blink, dev, flush)
    # 6. log-space readout over option orders: 512 questions x 4 orders x up to 26 options
    B = 512
    K = rng.integers(2, 27, size=B)
    R = 4
    pass_k = np.repeat(K, R)
    pass_off = torch.tensor(np.concatenate([[0], np.cumsum(pass_k)]), dtype=torch.int32, device=dev)
    keys = torch.tensor(np.concatenate([[(pos + r) % k for pos in range(k)] for k in K for r in range(R)]),
                        dtype=torch.int32, device=dev)
    logits = torch.randn(int(pass_k.sum()), generator=g, device=dev)
    qpass = torch.arange(0, B * R + 1, R, dtype=torch.int32, device=dev)
    raw_off = torch.tensor(np.concatenate([[0], np.cumsum(K)]), dtype=torch.int32, device=dev)
    prior = torch.randn(255 * 255, generator=g, device=dev)
    pr = torch.empty(int(K.sum()), dtype=torch.float32, device=dev)
    rw = torch.empty_like(pr)
    dws = blink.new_workspace(256, dev)
    sk = int(K.sum())
    ms = _time(lambda: blink.blink_rotation_debias(logits, pass_off, keys, qpass, raw_off, 1.0, prior=prior, raw=rw,
                                                   probs=pr, ws=dws, sum_k=sk), flush)
    out["rotation_debias"] = {"ms": ms, "shape": f"{B} questions x {R} orders x 2-26 options"}
    return out


def pack_plan_row(blink, dev, flush):
    """The pack plan at its largest size: 64 requests x 512 questions (32768 lengths U[16,1024])."""
    import torch
    g = torch.Generator(device=dev)
    g.manual_seed(12)
    plan_len = torch.randint(16, 1025, (32768,), generator=g, device=dev, dtype=torch.int32)
    pout = blink.blink_pack_plan(plan_len, 32768, 0)
    ms = _time(lambda: blink.blink_pack_plan(plan_len, 32768, 0, out=pout, sync=False), flush)
    return {"ms": ms, "shape": "32768 lengths U[16,1024], budget 32768 (64 requests x 512)"}


def wl_tail_lengths(w):
    from shared_prefix_question_gb300 import workloads as wl
    return wl.tail_lengths(w)


def readout_stress(blink, dev, hbm_peak, peak_kind, flush, args):
    import torch
    from shared_prefix_question_gb300 import workloads as wl
    w = wl.WORKLOADS["readout_stress"]
    off, ids = wl.label_csr(w)
    g = torch.Generator(device=dev)
    g.manual_seed(5)
    W = (torch.randn(w.V, w.H, generator=g, device=dev) * 0.02).to(torch.bfloat16)
    hidden = torch.randn(w.n, w.H, generator=g, device=dev).to(torch.bfloat16)
    last = torch.arange(w.n, dtype=torch.int32, device=dev)
    d_off = torch.from_numpy(off).to(dev)
    d_ids = torch.from_numpy(ids).to(dev)
    probs = torch.empty(len(ids), dtype=torch.float32, device=dev)
    ws = blink.new_workspace(blink.readout_workspace_bytes(w.n), dev)
    stream = torch.cuda.current_stream()
    for _ in range(3):
        blink.blink_label_readout(hidden, last, W, d_off, d_ids, 1.0, probs=probs, ws=ws)
    times = []
    for _ in range(max(10, args.steps)):
        flush_l2(flush)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        blink.blink_label_readout(hidden, last, W, d_off, d_ids, 1.0, probs=probs, ws=ws)
        e1.record(stream)
        times.append((e0, e1))
    torch.cuda.synchronize()
    ms = statistics.mean(a.elapsed_time(b) for a, b in times)
    distinct = len(np.unique(ids))
    nbytes = distinct * w.H * 2 + w.n * w.H * 2 + len(ids) * 4
    achieved = nbytes / (ms / 1000.0) / 1e9
    del W
    return {"bound": "hbm", "achieved": achieved, "peak": hbm_peak, "unit": "GB/s", "frac": achieved / hbm_peak,
            "spec_peak": SPEC_GBS, "frac_spec": achieved / SPEC_GBS,
            "traffic": traffic_record(os.path.join(ROOT, "shared_prefix_question_gb300", "csrc", "readout.cu"),
                                      "readout_stress"),
            "kernel": "readout_kernel", "ms": ms, "algorithmic_bytes": nbytes,
            "input": f"512 questions, {len(ids)} labels ({distinct} distinct rows) drawn per question without "
                     f"replacement from {w.V}, hidden {w.H}; the whole call is timed (logit launch and "
                     f"softmax launch)",
            "peak_kind": f"{peak_kind} copy bandwidth"}


def e2e(blink, dev, w, lengths, ins, rd, flush, args, world):
    """Same step through the C ABI with HOST inputs: every step copies its inputs from pinned host
    memory and reads its probabilities and answers back into pinned host memory.  Serving-style
    double buffering: step i + 1's inputs are copied into the second device buffer set on a copy
    stream while step i computes, and step i's results are copied back asynchronously and read by
    the host before their buffer set is reused, so the host stays a step ahead and the timed loop
    runs the steps back to back; every step's copy-in and read-back stays inside it.  The inputs
    of a step (260 MB on the 18k workload) are larger than L2, so no flush between steps."""
    import torch
    import torch.distributed as dist

    def pinned(a, dtype):
        t = torch.from_numpy(np.ascontiguousarray(a).view(dtype)).pin_memory()
        return t

    host = {"len": pinned(lengths.astype(np.int32), np.int32), "q": pinned(ins.q, np.int16),
            "kt": pinned(ins.k_tail, np.int16), "vt": pinned(ins.v_tail, np.int16),
            "hid": pinned(rd.hidden, np.int16), "off": pinned(rd.label_off, np.int32),
            "ids": pinned(rd.label_ids, np.int32), "qt": pinned(wl_question_types(w, rd.label_off), np.int32)}
    if ins.P:
        host["kp"] = pinned(ins.k_pre, np.int16)
        host["vp"] = pinned(ins.v_pre, np.int16)
    devb = [{k: torch.empty(v.shape, dtype=v.dtype, device=dev) for k, v in host.items()} for _ in range(2)]
    W = torch.from_numpy(np.ascontiguousarray(rd.unembed).view(np.int16)).view(torch.bfloat16).to(dev)  # resident
    # results: device outputs, read back asynchronously into one of two pinned host buffer sets
    h_probs = [torch.empty(len(rd.label_ids), dtype=torch.float32, pin_memory=True) for _ in range(2)]
    h_answers = [torch.empty(w.n, 3, dtype=torch.float32, pin_memory=True) for _ in range(2)]
    d_probs = torch.empty(len(rd.label_ids), dtype=torch.float32, device=dev)
    d_answers = torch.empty(w.n, 3, dtype=torch.float32, device=dev)
    n = w.n
    plan = None
    out = torch.empty(ins.q.shape, dtype=torch.bfloat16, device=dev)
    ws_a = blink.new_workspace(blink.attention_workspace_bytes(ins.rows, n, ins.P, ins.Hq, ins.Hkv, ins.d), dev)
    ws_r = blink.new_workspace(blink.readout_workspace_bytes(n), dev)
    bf = torch.bfloat16
    compute = torch.cuda.current_stream()
    copier = torch.cuda.Stream(device=dev)
    copied = [torch.cuda.Event() for _ in range(2)]
    consumed = [torch.cuda.Event() for _ in range(2)]
    read_back = [torch.cuda.Event() for _ in range(2)]
    pending = [False, False]
    checksum = [0.0]

    def copy_in(i):
        s = i % 2
        with torch.cuda.stream(copier):
            copier.wait_event(consumed[s])  # the step that last read this buffer set has finished
            for k in host:
                devb[s][k].copy_(host[k], non_blocking=True)
            copied[s].record(copier)

    def step(i):
        nonlocal plan
        d = devb[i % 2]
        compute.wait_event(copied[i % 2])
        plan = blink.blink_pack_plan(d["len"], 32768, 0, out=plan)
        blink.blink_prefix_tail_attention(d["q"].view(bf), d["kp"].view(bf) if ins.P else None,
                                          d["vp"].view(bf) if ins.P else None, d["kt"].view(bf),
                                          d["vt"].view(bf), plan["cu_seqlens"], B=n, P=ins.P,
                                          max_tail=int(lengths.max()), out=out, ws=ws_a)
        blink.blink_label_readout(d["hid"].view(bf), plan["last_varlen"], W, d["off"], d["ids"],
                                  rd.temperature, probs=d_probs, ws=ws_r, slot_of=plan["slot_of"],
                                  qtype=d["qt"], answers=d_answers)
        consumed[i % 2].record(compute)
        # step i's result to the host; the host reads it once the copy has landed (below, before
        # the buffer set is reused, and at the end)
        h = i % 2
        if pending[h]:
            read_back[h].synchronize()
            checksum[0] += float(h_answers[h][0, 0])
        h_probs[h].copy_(d_probs, non_blocking=True)
        h_answers[h].copy_(d_answers, non_blocking=True)
        read_back[h].record(compute)
        pending[h] = True

    def drain():
        for h in range(2):
            if pending[h]:
                read_back[h].synchronize()
                checksum[0] += float(h_answers[h][0, 0])
                pending[h] = False

    def run(k):
        copy_in(0)
        for i in range(k):
            if i + 1 < k:
                copy_in(i + 1)
            step(i)
        drain()

    for e in consumed:
        e.record(compute)
    run(max(3, args.warmup))
    steps = max(5, min(args.steps, 30))
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    t0 = time.perf_counter()
    run(steps)
    torch.cuda.synchronize()
    sec = (time.perf_counter() - t0) / steps
    if blink.blink_read_device_status(ws_a) != 0 or blink.blink_read_device_status(ws_r) != 0:
        raise SystemExit("device status after the end-to-end steps is not OK")
    if world > 1:
        t = torch.tensor([sec], dtype=torch.float64, device=dev)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        sec = float(t.item())
    h2d = sum(v.numel() * v.element_size() for v in host.values())
    return {"value": world * n / sec, "unit": "questions/s", "h2d_bytes_per_step": int(h2d),
            "d2h_bytes_per_step": int(h_probs[0].numel() * 4 + h_answers[0].numel() * 4), "ms_per_step": sec * 1000,
            "steps": steps,
            "pipelined": "step i + 1's inputs copied on a second stream while step i computes; step i's "
                         "probabilities and answers copied to pinned host buffers asynchronously and read "
                         "by the host before the buffer is reused (two sets) and at the end",
            "resident": "unembedding (model weight) stays on the device"}


if __name__ == "__main__":
    main()
