#!/usr/bin/env python3
"""Throughput of the segmented KDA forward on GB300: one JSON line.

A step is one pass of the whole hot path -- kda_segment_forward (chunk forward +
summaries), kda_compose_summaries (scan) and kda_apply_boundary (fix-up) -- over
one batch of the synthetic workload, inputs resident in HBM.  The L2 cache is
flushed (a 256 MiB write) before every step, outside the timed events.  Each
timed step is bracketed by one event pair, so its three calls run as they do
for a user (each kernel a programmatic dependent of the one before); the
per-kernel breakdown comes from a second pass of as many steps with events
between the calls.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]
                  [--path fix_up|two_pass]

N > 1 is launched with torch.distributed.run: every rank runs its own copy of
the workload (independent problems, no collective on the data path), so the
value is the tokens of all ranks over the slowest rank's time ("weak" scaling).
``--impl reference`` times the fp64 CPU oracle on the host cores instead.
``--path two_pass`` times kda_forward_two_pass (the forward from preceding
summaries, no fix-up) in place of the three calls, for comparison.
"""
from __future__ import annotations

import argparse
import hashlib
import re
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from context_kda_gb300.inputs import HEADLINE, bf16_to_f32, make_workload, workloads  # noqa: E402

METRIC = "segmented KDA fwd tokens/sec (H=16,K=V=128) on 1 GB300; % of roofline"
UNIT = "tokens/s"
K_DIM = V_DIM = 128
CH = 64
# algorithmic work per token-head (minimal counts of the chunkwise algebra): the state columns of the
# chunk forward, and the transition columns a continuing token adds
FLOPS_STATE = 6 * CH * K_DIM + 4 * CH * V_DIM + 6 * K_DIM * V_DIM          # 180,224
FLOPS_TRANSITION = 6 * K_DIM * K_DIM + 2 * CH * K_DIM                      # 114,688
# algorithmic HBM bytes of the chunk forward: per token-head q, k, v (bf16), g (fp32), beta (fp32)
# read and the bf16 output written; per continuing token-head the bf16 qhat written; per segment-head
# the fp32 summaries A (K x K) and B (K x V) written; per sequence-head the fp32 final state written
# and, when given, h0 read
BYTES_TOKEN = 3 * K_DIM * 2 + K_DIM * 4 + 4 + V_DIM * 2                  # 1,540
BYTES_CONT = K_DIM * 2                                                   # 256
BYTES_SEGMENT = (K_DIM * K_DIM + K_DIM * V_DIM) * 4                      # 131,072
BYTES_SEQ_STATE = K_DIM * V_DIM * 4                                      # 65,536
# tensor work the chunk stage issues (bf16 M=128 MMAs, split passes included), as 2 * 128 * N * K
# per product: the preparation, once per (chunk, head): [KK; QK] 3 x (N 64, K 128), W 3 x (64, 64),
# Ut 2 x (64, 64); the state pass, per chunk and work item: W X 3 x (64, 128), Qt X 1 x (64, 128),
# QK U 1 x (64, 64), Kh^T U 3 x (128, 64)
ISSUED_PREP_PER_CHUNK = 2 * 128 * (3 * 64 * 128 + 3 * 64 * 64 + 2 * 64 * 64)
ISSUED_STATE_PER_CHUNK = 2 * 128 * (3 * 64 * 128 + 64 * 128 + 64 * 64 + 3 * 128 * 64)
CHUNK_KERNEL_SRCS = [os.path.join(ROOT, "context_kda_gb300", "csrc", f) for f in ("chunk_prep.cu", "chunk_state.cu")]
PROFILE_SUMMARY = os.path.join(ROOT, "profiles", "chunk_forward_t8192_h16_s4.txt")


def _peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return {"hbm_gbs": d["hbm_gbs"], "bf16_tflops": d["bf16_tflops"],
                "bf16_tflops_sustained": d.get("bf16_tflops_sustained"), "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}


def _profile_values(kernel_srcs):
    """Figures recorded in the committed ncu summary, if it was taken on the current sources."""
    if not os.path.exists(PROFILE_SUMMARY):
        return {}
    h = hashlib.sha256()
    for src in kernel_srcs:
        h.update(open(src, "rb").read())
    sha = h.hexdigest()[:16]
    vals = {}
    for line in open(PROFILE_SUMMARY):
        if line.startswith("- ") and ":" in line:
            key, _, val = line[2:].partition(":")
            m = re.search(r"`([^`]*)`", val)   # the value is the first backticked token
            vals[key.strip()] = m.group(1) if m else val.strip()
    return vals if vals.get("kernel_source_sha256_16") == sha else {}


class ClockSampler:
    """nvidia-smi samples (200 ms) during the timed region."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
            time.sleep(0.3)
        except OSError:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.thread.join(timeout=2)

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for n, p in zip(names, parts[4:8]):
                if p.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


def _oracle_pass(inp, nthreads):
    import oracle
    q, k, v = bf16_to_f32(inp.q), bf16_to_f32(inp.k), bf16_to_f32(inp.v)
    t = time.perf_counter()
    oracle.forward(inp.cu_seqlens, q, k, v, inp.g, inp.beta, h0=inp.h0, nthreads=nthreads, want_final=False)
    return time.perf_counter() - t


def cpu_baseline(inp, budget_s=10.0, max_passes=8):
    """The fp64 oracle (monolithic recurrence) on the host cores: full passes over the
    workload until about budget_s seconds have been spent."""
    import oracle
    oracle.build()
    cores = len(os.sched_getaffinity(0))
    times = []
    while len(times) < max_passes and (not times or sum(times) < budget_s):
        times.append(_oracle_pass(inp, cores))
    tasks = inp.num_seqs * inp.heads
    return {"value": inp.tokens / statistics.median(times), "unit": UNIT, "cores": min(cores, tasks),
            "kind": "oracle",
            "sample": f"full workload ({inp.tokens} tokens x {inp.heads} heads), fp64 token recurrence, "
                      f"{len(times)} pass(es), median; OpenMP over {tasks} (sequence, head) tasks"}


def _config(w, n):
    return {"workload": w.name, "tokens": w.tokens, "heads": w.heads, "segments": w.segments,
            "sequences": len(w.seqlens), "K": K_DIM, "V": V_DIM, "chunk": CH, "g_range": [w.g_lo, w.g_hi],
            "h0_std": w.h0_std, "l2": "flushed before every step (256 MiB write)", "parallelism": f"replicas{n}"}


def max_over_ranks(values, world, device=None):
    """Each rank's timings (ms) -> the slowest rank's, element by element; every rank gets them.
    With one rank the values come back unchanged."""
    import torch
    t = torch.tensor([float(x) for x in values], dtype=torch.float64, device=device)
    if world > 1:
        import torch.distributed as dist
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(x) for x in t.cpu()]


def aggregate_rate(world, tokens_per_rank, ms):
    """Whole-job tokens/s: every rank processes its own copy of the workload (weak scaling), and
    the job takes the slowest rank's time."""
    return world * tokens_per_rank / (ms / 1e3)


def run_reference(args, w, rank):
    if rank != 0:
        return
    import oracle
    oracle.build()
    inp = make_workload(w)
    cores = len(os.sched_getaffinity(0))
    # each step is one full pass of the oracle over the workload
    for _ in range(args.warmup):
        _oracle_pass(inp, cores)
    times = [_oracle_pass(inp, cores) for _ in range(args.steps)]
    ms = 1e3 * sum(times) / len(times)
    value = inp.tokens / (ms / 1e3)
    tasks = inp.num_seqs * inp.heads
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": _config(w, args.gpus),
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": min(cores, tasks), "kind": "oracle",
                             "sample": f"full workload per step ({inp.tokens} tokens x {inp.heads} heads)"},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def kernel_bytes(plan, H, h0_given):
    """Algorithmic HBM bytes of each kernel of one step:
    chunk stage  q, k, v, g, beta read and o written per token-head, qhat written per continuing
                 token-head, A and B written per segment-head, the final state written (and h0 read)
                 per sequence-head;
    composition  A and B read and S_in written per segment-head;
    fix-up       qhat read and o read and written per continuing token-head, S_in read per
                 (segment, head) with a continuing piece, and per final-state transition the
                 transition and the final state read and the final state written."""
    T, N, S, T_cont, n_fin = int(plan[3]), int(plan[4]), int(plan[5]), int(plan[9]), int(plan[10])
    n_cont, cont_off = int(plan[8]), int(plan[20])
    segs_with_cont = len({int(plan[cont_off + 4 * i + 1]) for i in range(n_cont)})
    chunk = (T * H * BYTES_TOKEN + T_cont * H * BYTES_CONT + S * H * BYTES_SEGMENT
             + N * H * BYTES_SEQ_STATE * (2 if h0_given else 1))
    compose = S * H * (BYTES_SEGMENT + BYTES_SEQ_STATE)
    fixup = T_cont * H * 3 * V_DIM * 2 + segs_with_cont * H * BYTES_SEQ_STATE + n_fin * H * 3 * BYTES_SEQ_STATE
    return {"chunk_forward": chunk, "compose": compose, "boundary": fixup}


class Problem:
    """One workload resident on the device: inputs, plan, workspace and outputs."""

    def __init__(self, w, dev, inp=None, refined=False):
        import torch
        from context_kda_gb300 import binding as kda
        self.kda = kda
        self.w = w
        self.inp = inp if inp is not None else make_workload(w)
        inp = self.inp
        self.T, self.H, self.N, self.S = inp.tokens, inp.heads, inp.num_seqs, inp.segments
        to = lambda a, dt: torch.from_numpy(np.ascontiguousarray(a)).view(dt)
        self.host = {"q": to(inp.q, torch.bfloat16), "k": to(inp.k, torch.bfloat16),
                     "v": to(inp.v, torch.bfloat16), "g": to(inp.g, torch.float32),
                     "beta": to(inp.beta, torch.float32)}
        if inp.h0 is not None:
            self.host["h0"] = to(inp.h0, torch.float32)
        self.d = {k_: v_.to(dev) for k_, v_ in self.host.items()}
        self.h0 = self.d.get("h0")
        if refined:   # the chunk-level split within the segments, sized for this device
            sms = __import__("torch").cuda.get_device_properties(dev).multi_processor_count
            self.plan = kda.kda_plan_segments_refined(inp.cu_seqlens, self.S, self.H, sms)
            self.S = int(self.plan[5])
        else:
            self.plan = kda.kda_plan_segments(inp.cu_seqlens, self.S)
        self.plan_dev = kda.upload_plan(self.plan, dev)
        off = kda.kda_workspace_layout(self.plan, self.H)
        self.ws = torch.empty(off[6], dtype=torch.uint8, device=dev)
        self.A = self.ws[off[3]:off[4]].view(torch.float32)
        self.B = self.ws[off[4]:off[5]].view(torch.float32)
        self.S_in = self.ws[off[5]:off[6]].view(torch.float32)
        self.o = torch.empty((self.T, self.H, V_DIM), dtype=torch.bfloat16, device=dev)
        self.fin = torch.empty((self.N, self.H, K_DIM, V_DIM), dtype=torch.float32, device=dev)
        n_cont, n_fin = int(self.plan[8]), int(self.plan[10])
        self.launches_per_step = 3 + (1 if (n_cont + n_fin) > 0 else 0)   # prep, state, compose (+ fix-up)

    def step(self, stream, evs=None, two_pass=False):
        kda, d, H = self.kda, self.d, self.H
        if two_pass:   # one call: the whole step is its first interval
            if evs:
                evs[0].record(stream)
            kda.kda_forward_two_pass(self.plan, self.plan_dev, H, d["q"], d["k"], d["v"], d["g"], d["beta"],
                                     self.h0, 1.0, self.o, self.fin, self.ws, stream)
            if evs:
                for e in evs[1:]:
                    e.record(stream)
            return
        if evs:
            evs[0].record(stream)
        kda.kda_segment_forward(self.plan, self.plan_dev, H, d["q"], d["k"], d["v"], d["g"], d["beta"], self.h0,
                                1.0, self.o, self.A, self.B, self.fin, self.ws, stream)
        if evs:
            evs[1].record(stream)
        kda.kda_compose_summaries(self.plan, self.plan_dev, H, self.A, self.B, self.h0, self.S_in, stream)
        if evs:
            evs[2].record(stream)
        kda.kda_apply_boundary(self.plan, self.plan_dev, H, self.S_in, self.ws, self.o, self.fin, stream)
        if evs:
            evs[3].record(stream)

    def time_steps(self, stream, flush, steps, warmup, two_pass=False):
        """Per-kernel CUDA-event times (ms) of 'steps' steps after 'warmup' untimed ones, the L2
        flushed (a 256 MiB write) before every step outside the events: array [steps, 3]."""
        import torch
        for _ in range(warmup):
            flush.fill_(1)
            self.step(stream, two_pass=two_pass)
        evsets = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(steps)]
        for i in range(steps):
            flush.fill_(1)
            self.step(stream, evsets[i], two_pass=two_pass)
        torch.cuda.synchronize()
        return np.array([[e[j].elapsed_time(e[j + 1]) for j in range(3)] for e in evsets])

    def time_whole(self, stream, flush, steps, warmup, two_pass=False):
        """CUDA-event times (ms) of whole steps, one event pair around each step and none between its
        kernels (so each kernel may launch as a programmatic dependent of the one before), after 'warmup'
        untimed steps; the L2 flushed before every step outside the events."""
        import torch
        for _ in range(warmup):
            flush.fill_(1)
            self.step(stream, two_pass=two_pass)
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
        for e0, e1 in evs:
            flush.fill_(1)
            e0.record(stream)
            self.step(stream, two_pass=two_pass)
            e1.record(stream)
        torch.cuda.synchronize()
        return np.array([e0.elapsed_time(e1) for e0, e1 in evs])

    def free(self):
        for name in ("d", "ws", "A", "B", "S_in", "o", "fin", "plan_dev", "h0"):
            setattr(self, name, None)


def pages_protocol(prob, stream, flush, warmup=20, iters=60, repeats=5):
    """The timing protocol of cuLA PR #110 §Performance: 20 warm-up iterations, then 5 repeats of 60
    timed iterations; the median of each repeat, then the median of the repeats (one rank, so the
    rank-max is the value itself).  The L2 is flushed before every iteration, outside the events."""
    step = prob.time_whole(stream, flush, iters * repeats, warmup).reshape(repeats, iters)
    return float(np.median(np.median(step, axis=1)))


def run_ours(args, w, rank, world, local_rank):
    import torch
    import torch.distributed as dist

    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    prob = Problem(w, dev)
    inp, plan = prob.inp, prob.plan
    T, H = prob.T, prob.H
    flush = torch.empty(256 * 2 ** 20, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    two_pass = args.path == "two_pass"
    launches_per_step = 4 if two_pass else prob.launches_per_step   # two-pass: prep, summary pass, compose, output pass

    for _ in range(args.warmup):
        flush.fill_(1)
        prob.step(stream, two_pass=two_pass)
    torch.cuda.synchronize(dev)
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize(dev)
    with ClockSampler(local_rank) as clk:
        # the timed region is short, so clocks are sampled over a ~1 s soak of identical
        # (untimed) steps right before it as well as during it
        soak0 = time.perf_counter()
        while time.perf_counter() - soak0 < args.clock_soak_s:
            for _ in range(8):
                flush.fill_(1)
                prob.step(stream, two_pass=two_pass)
            torch.cuda.synchronize(dev)
        wall0 = time.perf_counter()
        for e0, e1 in evs:
            flush.fill_(1)
            e0.record(stream)
            prob.step(stream, two_pass=two_pass)
            e1.record(stream)
        torch.cuda.synchronize(dev)
        wall = time.perf_counter() - wall0
        # the per-kernel breakdown: the same number of steps again, with events between the kernels
        # (they serialise the programmatic dependent launches, so these sum to more than a step)
        per = prob.time_steps(stream, flush, args.steps, 0, two_pass=two_pass)   # ms [steps, 3]
    if world > 1:
        dist.barrier()
    step_ms = float(np.mean([e0.elapsed_time(e1) for e0, e1 in evs]))
    kern_ms = per.mean(axis=0)
    protocol_ms = None if (two_pass or args.no_extra) else pages_protocol(prob, stream, flush)

    # end to end through the public entry point: every step uploads its inputs from pinned host
    # memory and reads its outputs and final states back.  Two lanes (own stream, device buffers
    # and workspace each) alternate steps, so one step's upload overlaps the previous step's
    # compute and read-back; the copies of every step stay inside the timed region.
    kda = prob.kda
    d, o, fin, ws = prob.d, prob.o, prob.fin, prob.ws
    pinned = {k_: v_.pin_memory() for k_, v_ in prob.host.items()}
    h2d = sum(v_.numel() * v_.element_size() for v_ in pinned.values())
    d2h = o.numel() * o.element_size() + fin.numel() * fin.element_size()
    lanes = []
    for li in range(2):
        lane = {"stream": torch.cuda.Stream(dev), "d": d if li == 0 else {k_: torch.empty_like(v_) for k_, v_ in d.items()},
                "o": o if li == 0 else torch.empty_like(o), "fin": fin if li == 0 else torch.empty_like(fin),
                "ws": ws if li == 0 else torch.empty_like(ws),
                "o_host": torch.empty(o.shape, dtype=o.dtype).pin_memory(),
                "f_host": torch.empty(fin.shape, dtype=fin.dtype).pin_memory()}
        lanes.append(lane)

    def e2e_step(i):
        ln = lanes[i % 2]
        with torch.cuda.stream(ln["stream"]):
            dd = ln["d"]
            for k_ in pinned:
                dd[k_].copy_(pinned[k_], non_blocking=True)
            run = kda.kda_forward_two_pass if two_pass else kda.kda_forward_segmented
            run(plan, prob.plan_dev, H, dd["q"], dd["k"], dd["v"], dd["g"], dd["beta"], dd.get("h0"), 1.0,
                ln["o"], ln["fin"], ln["ws"], ln["stream"])
            ln["o_host"].copy_(ln["o"], non_blocking=True)
            ln["f_host"].copy_(ln["fin"], non_blocking=True)

    torch.cuda.synchronize(dev)
    for i in range(args.warmup):
        e2e_step(i)
    torch.cuda.synchronize(dev)
    e_start = torch.cuda.Event(enable_timing=True)
    e_start.record(stream)
    for ln in lanes:
        ln["stream"].wait_event(e_start)
    for i in range(args.steps):
        e2e_step(i)
    ends = []
    for ln in lanes:
        ev = torch.cuda.Event(enable_timing=True)
        ev.record(ln["stream"])
        ends.append(ev)
    torch.cuda.synchronize(dev)
    e2e_ms = max(e_start.elapsed_time(ev) for ev in ends) / args.steps

    # the host link alone: the step's input uploads with nothing else running (median of 5), which
    # bounds the end-to-end rate from above; and one 1 GiB pinned upload, the link's own rate
    def timed_copies(pairs, reps=5):
        out = []
        for _ in range(reps):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for dst, src in pairs:
                dst.copy_(src, non_blocking=True)
            e1.record(stream)
            torch.cuda.synchronize(dev)
            out.append(e0.elapsed_time(e1))
        return float(statistics.median(out))
    h2d_ms = timed_copies([(d[k_], pinned[k_]) for k_ in pinned])
    big_host = torch.empty(2 ** 30, dtype=torch.uint8).pin_memory()
    big_dev = torch.empty(2 ** 30, dtype=torch.uint8, device=dev)
    big_ms = timed_copies([(big_dev, big_host)])
    del big_host, big_dev, lanes

    step_ms, e2e_ms = max_over_ranks([step_ms, e2e_ms], world, dev)
    if rank != 0:
        return
    peaks = _peaks()
    T_cont = int(plan[9])
    flops = T * H * FLOPS_STATE + T_cont * H * FLOPS_TRANSITION
    kb = kernel_bytes(plan, H, w.h0_std > 0)
    algo_bytes = kb["chunk_forward"]
    # the binding roof is the larger of bytes / HBM bandwidth and flops / tensor peak
    t_hbm = algo_bytes / (peaks["hbm_gbs"] * 1e9)
    t_tensor = flops / (peaks["bf16_tflops"] * 1e12)
    sec = kern_ms[0] / 1e3
    achieved_gbs = algo_bytes / sec / 1e9
    achieved_tflops = flops / sec / 1e12
    items_off, pieces_off = int(plan[18]), int(plan[17])
    issued = int(plan[11]) * H * ISSUED_PREP_PER_CHUNK   # every (chunk, head) is prepared once
    for i in range(int(plan[12])):
        pc = int(plan[items_off + 2 * i])
        ln = int(plan[pieces_off + 8 * pc + 1])
        issued += ((ln + CH - 1) // CH) * ISSUED_STATE_PER_CHUNK * H
    prof = _profile_values(CHUNK_KERNEL_SRCS)
    traffic = float(prof["dram_bytes_per_launch"]) if "dram_bytes_per_launch" in prof and not two_pass else None
    shares = (kern_ms / kern_ms.sum()).tolist()
    kernel = "two_pass_forward" if two_pass else "chunk_forward"
    if two_pass:   # the issued-flop count below is the fix-up path's
        issued = None
    line = {
        "metric": METRIC, "value": aggregate_rate(world, T, step_ms), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": step_ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16 in, f32 state", "data": "synthetic",
        "config": _config(w, world) | ({"path": "two_pass"} if two_pass else {}),
        "kernels_ms": ({"two_pass_forward": kern_ms[0]} if two_pass else
                       {"chunk_forward": kern_ms[0], "compose": kern_ms[1], "boundary": kern_ms[2]}),
        "kernel_timing": ("ms_per_step: one event pair around each whole step; kernels_ms: a second pass of "
                          "as many steps with events between the kernels, which serialises their "
                          "programmatic dependent launches (sum %.4f ms)" % float(kern_ms.sum())),
        "kernel_shares": ({"two_pass_forward": 1.0} if two_pass else
                          {"chunk_forward": shares[0], "compose": shares[1], "boundary": shares[2]}),
        "kernel_hbm_frac": (None if two_pass else
                            {k_: kb[k_] / (kern_ms[i] / 1e3) / 1e9 / peaks["hbm_gbs"]
                             for i, k_ in enumerate(("chunk_forward", "compose", "boundary"))}),
        "roofline": ({"bound": "hbm", "kernel": kernel, "achieved": achieved_gbs,
                      "peak": peaks["hbm_gbs"], "unit": "GB/s", "frac": achieved_gbs / peaks["hbm_gbs"],
                      "peak_source": f"{peaks['source']} HBM copy"}
                     if t_hbm >= t_tensor else
                     {"bound": "tensor", "kernel": kernel, "achieved": achieved_tflops,
                      "peak": peaks["bf16_tflops"], "unit": "TFLOP/s", "frac": achieved_tflops / peaks["bf16_tflops"],
                      "peak_source": f"{peaks['source']} bf16 dense (burst)"})
        | {"traffic": traffic, "algorithmic_bytes_per_launch": algo_bytes,
           "algorithmic_flops_per_launch": flops, "tensor_frac": achieved_tflops / peaks["bf16_tflops"],
           "issued_tensor_flops_per_launch": issued,
           "issued_frac": None if issued is None else issued / sec / 1e12 / peaks["bf16_tflops"],
           "hbm_peak_gbs": peaks["hbm_gbs"],
           "bf16_peak_tflops": peaks["bf16_tflops"]},
        "pages_protocol_ms_per_step": protocol_ms,
        "e2e": {"value": aggregate_rate(world, T, e2e_ms), "unit": UNIT, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "h2d_gbs_alone": h2d / (h2d_ms / 1e3) / 1e9,
                "h2d_gbs_one_1gib_copy": 2 ** 30 / (big_ms / 1e3) / 1e9,
                "upload_bound_value": aggregate_rate(world, T, h2d_ms),
                "pipeline": "2 lanes: step i+1 uploads its inputs while step i computes and reads back"},
        "gpu_launches": launches_per_step * args.steps,
        "clocks": dict(clk.summary(), window=f"{args.clock_soak_s:g} s soak of identical steps + timed region"),
        "wall_s_timed_region": wall,
    }
    if world == 1 and not two_pass and not args.no_extra:
        line["backward"] = time_backward(prob, stream, flush)
        line["workloads"] = extra_workloads(args, dev, stream, flush, peaks)
        line["chunk_level_split"] = refined_comparison(args, dev, stream, flush)
    if world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(inp)
    print(json.dumps(line), flush=True)


EXTRA_WORKLOADS = ("packed65536_h32_s64", "t131072_h32_s64", "t32768_h2_s64")


def time_scans(prob, stream, flush, steps=10, warmup=3):
    """The composition alone, by the chain and by the two-level scan, from the summaries of one step:
    mean CUDA-event ms of each (L2 flushed before every run)."""
    import torch
    kda = prob.kda
    prob.step(stream)
    scan_ws = torch.empty(max(1, kda.kda_scan_workspace_bytes(prob.plan, prob.H)), dtype=torch.uint8,
                          device=prob.o.device)
    out = {}
    for name in ("chain", "blocked"):
        def run():
            if name == "chain":
                kda.kda_compose_summaries(prob.plan, prob.plan_dev, prob.H, prob.A, prob.B, prob.h0, prob.S_in, stream)
            else:
                kda.kda_compose_summaries_blocked(prob.plan, prob.plan_dev, prob.H, prob.A, prob.B, prob.h0,
                                                  prob.S_in, scan_ws, stream)
        for _ in range(warmup):
            flush.fill_(1)
            run()
        ms = []
        for _ in range(steps):
            flush.fill_(1)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            run()
            e1.record(stream)
            torch.cuda.synchronize()
            ms.append(e0.elapsed_time(e1))
        out[name] = float(np.mean(ms))
    del scan_ws
    return out


REFINED_WORKLOADS = ("t1024_h4_s2", "t8192_h16_s4", "t131072_h2_s1")


def refined_comparison(args, dev, stream, flush):
    """The chunk-level split within a segment: each workload's step on its own plan and on the refined
    plan (kda_plan_segments_refined for this device), per-kernel ms and tokens/s of both."""
    import torch
    out = {}
    for name in REFINED_WORKLOADS:
        w = workloads()[name]
        inp = make_workload(w)
        row = {}
        for label, refined in (("plan", False), ("refined", True)):
            prob = Problem(w, dev, inp=inp, refined=refined)
            per = prob.time_steps(stream, flush, args.extra_steps, 3)
            kern = per.mean(axis=0)
            ms = float(prob.time_whole(stream, flush, args.extra_steps, 3).mean())
            row[label] = {"segments": prob.S, "ms_per_step": ms, "tokens_per_s": prob.T / (ms / 1e3),
                          "kernels_ms": {n: float(kern[i]) for i, n in enumerate(("chunk_forward", "compose", "boundary"))}}
            prob.free()
            del prob
            torch.cuda.empty_cache()
        out[name] = row
    return out


def time_backward(prob, stream, flush, steps=5, warmup=2):
    """kda_backward_segmented on the problem (seeded output gradients, inputs resident in HBM): mean
    CUDA-event ms and tokens/s.  It includes the forward's local pass and composition it runs first."""
    import torch
    from context_kda_gb300.inputs import draw_output_grads
    kda, dev = prob.kda, prob.o.device
    do_bits, dfinal = draw_output_grads(prob.inp, seed=1)
    dout = torch.from_numpy(np.ascontiguousarray(do_bits)).view(torch.bfloat16).to(dev)
    df = torch.from_numpy(dfinal).to(dev)
    T, H, N = prob.T, prob.H, prob.N
    grads = [torch.empty((T, H, K_DIM), device=dev), torch.empty((T, H, K_DIM), device=dev),
             torch.empty((T, H, V_DIM), device=dev), torch.empty((T, H, K_DIM), device=dev),
             torch.empty((T, H), device=dev), torch.empty((N, H, K_DIM, V_DIM), device=dev)]
    ws = torch.empty(kda.kda_backward_workspace_bytes(prob.plan, H), dtype=torch.uint8, device=dev)
    d = prob.d

    def run():
        kda.kda_backward_segmented(prob.plan, prob.plan_dev, H, d["q"], d["k"], d["v"], d["g"], d["beta"], prob.h0,
                                   1.0, dout, df, *grads, ws, stream)
    for _ in range(warmup):
        flush.fill_(1)
        run()
    ms = []
    for _ in range(steps):
        flush.fill_(1)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        run()
        e1.record(stream)
        torch.cuda.synchronize()
        ms.append(e0.elapsed_time(e1))
    m = float(np.mean(ms))
    del ws, grads
    return {"ms_per_step": m, "tokens_per_s": T / (m / 1e3), "steps": steps, "warmup": warmup,
            "note": "FP32 matrices, products on tcgen05 as a 3-term bf16 split; includes the forward's local pass and composition"}


def scan_bytes(S, H):
    """Algorithmic HBM bytes of the two schedules of the composition: the chain reads A and B and writes
    S_in per segment-head; the two-level scan adds the group totals (written, then read) and the group
    incoming states (written, then read) and reads A and B twice."""
    import math
    m = math.isqrt(S - 1) + 1 if S > 1 else 1
    G = (S + m - 1) // m
    seg = S * H * (BYTES_SEGMENT + BYTES_SEQ_STATE)
    totals = G * H * BYTES_SEGMENT
    entry = G * H * BYTES_SEQ_STATE
    return {"chain": seg, "blocked": seg + S * H * BYTES_SEGMENT + 2 * totals + 2 * entry}


def extra_workloads(args, dev, stream, flush, peaks):
    """The packed and long-context workloads, timed after the headline's timed region in the same
    run: per-kernel CUDA-event times (mean of the timed steps), tokens/s and each kernel's fraction
    of the measured HBM copy bandwidth on its algorithmic bytes."""
    import torch
    out = {}
    for name in EXTRA_WORKLOADS:
        w = workloads()[name]
        prob = Problem(w, dev)
        per = prob.time_steps(stream, flush, args.extra_steps, 3)
        kern = per.mean(axis=0)
        ms = float(prob.time_whole(stream, flush, args.extra_steps, 3).mean())
        kb = kernel_bytes(prob.plan, prob.H, w.h0_std > 0)
        names = ("chunk_forward", "compose", "boundary")
        out[name] = {
            "tokens_per_s": prob.T / (ms / 1e3), "ms_per_step": ms, "steps": args.extra_steps, "warmup": 3,
            "kernels_ms": {n: float(kern[i]) for i, n in enumerate(names)},
            "kernel_hbm_frac": {n: kb[n] / (kern[i] / 1e3) / 1e9 / peaks["hbm_gbs"] for i, n in enumerate(names)},
            "algorithmic_bytes": kb, "config": _config(w, 1),
        }
        scans = time_scans(prob, stream, flush)
        sb = scan_bytes(prob.S, prob.H)
        out[name]["compose_schedules_ms"] = scans
        out[name]["compose_schedules_hbm_frac"] = {k_: sb[k_] / (scans[k_] / 1e3) / 1e9 / peaks["hbm_gbs"]
                                                   for k_ in scans}
        prob.free()
        del prob
        torch.cuda.empty_cache()
    return out


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default=HEADLINE, choices=sorted(workloads().keys()))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-extra", action="store_true",
                    help="skip the pages' timing protocol and the packed / long-context workloads")
    ap.add_argument("--extra-steps", type=int, default=10)
    ap.add_argument("--clock-soak-s", type=float, default=1.0)
    ap.add_argument("--path", default="fix_up", choices=["fix_up", "two_pass"],
                    help="fix_up: the three calls (local forward, composition, fix-up); two_pass: "
                         "kda_forward_two_pass (state pass from the preceding summaries, no fix-up)")
    args = ap.parse_args()
    args.warmup = max(3, args.warmup)   # at least 3 untimed warm-up steps
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    w = workloads()[args.workload]
    if args.impl == "reference":
        run_reference(args, w, rank)
        return
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    try:
        run_ours(args, w, rank, world, local_rank)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
