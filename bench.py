#!/usr/bin/env python3
"""Throughput of the segmented KDA forward on GB300: one JSON line.

A step is one pass of the whole hot path -- kda_segment_forward (chunk forward +
summaries), kda_compose_summaries (scan) and kda_apply_boundary (fix-up) -- over
one batch of the synthetic workload, inputs resident in HBM.  The L2 cache is
flushed (a 256 MiB write) before every step, outside the timed events.

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


def run_ours(args, w, rank, world, local_rank):
    import torch
    import torch.distributed as dist
    from context_kda_gb300 import binding as kda

    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    inp = make_workload(w)
    T, H, N, S = inp.tokens, inp.heads, inp.num_seqs, inp.segments
    to = lambda a, dt: torch.from_numpy(np.ascontiguousarray(a)).view(dt)
    host = {"q": to(inp.q, torch.bfloat16), "k": to(inp.k, torch.bfloat16), "v": to(inp.v, torch.bfloat16),
            "g": to(inp.g, torch.float32), "beta": to(inp.beta, torch.float32)}
    if inp.h0 is not None:
        host["h0"] = to(inp.h0, torch.float32)
    d = {k_: v_.to(dev) for k_, v_ in host.items()}
    h0 = d.get("h0")
    plan = kda.kda_plan_segments(inp.cu_seqlens, S)
    plan_dev = kda.upload_plan(plan, dev)
    off = kda.kda_workspace_layout(plan, H)
    ws = torch.empty(off[6], dtype=torch.uint8, device=dev)
    A = ws[off[3]:off[4]].view(torch.float32)
    B = ws[off[4]:off[5]].view(torch.float32)
    S_in = ws[off[5]:off[6]].view(torch.float32)
    o = torch.empty((T, H, V_DIM), dtype=torch.bfloat16, device=dev)
    fin = torch.empty((N, H, K_DIM, V_DIM), dtype=torch.float32, device=dev)
    flush = torch.empty(256 * 2 ** 20, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    n_cont, n_fin = int(plan[8]), int(plan[10])
    launches_per_step = 3 + (1 if (n_cont + n_fin) > 0 else 0)   # prep, state, compose (+ fix-up)
    two_pass = args.path == "two_pass"
    if two_pass:
        launches_per_step = 4   # prep, summary pass, compose, output pass

    def step(evs=None):
        if two_pass:   # one call: the whole step is its first interval
            if evs:
                evs[0].record(stream)
            kda.kda_forward_two_pass(plan, plan_dev, H, d["q"], d["k"], d["v"], d["g"], d["beta"], h0, 1.0, o, fin,
                                     ws, stream)
            if evs:
                for e in evs[1:]:
                    e.record(stream)
            return
        if evs:
            evs[0].record(stream)
        kda.kda_segment_forward(plan, plan_dev, H, d["q"], d["k"], d["v"], d["g"], d["beta"], h0, 1.0, o, A, B,
                                fin, ws, stream)
        if evs:
            evs[1].record(stream)
        kda.kda_compose_summaries(plan, plan_dev, H, A, B, h0, S_in, stream)
        if evs:
            evs[2].record(stream)
        kda.kda_apply_boundary(plan, plan_dev, H, S_in, ws, o, fin, stream)
        if evs:
            evs[3].record(stream)

    for _ in range(args.warmup):
        flush.fill_(1)
        step()
    torch.cuda.synchronize(dev)
    evsets = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(args.steps)]
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
                step()
            torch.cuda.synchronize(dev)
        wall0 = time.perf_counter()
        for i in range(args.steps):
            flush.fill_(1)
            step(evsets[i])
        torch.cuda.synchronize(dev)
        wall = time.perf_counter() - wall0
    if world > 1:
        dist.barrier()
    per = np.array([[e[j].elapsed_time(e[j + 1]) for j in range(3)] for e in evsets])  # ms
    step_ms = float(np.mean(per.sum(axis=1)))
    kern_ms = per.mean(axis=0)

    # end to end through the public entry point: every step uploads its inputs from pinned host
    # memory and reads its outputs and final states back.  Two lanes (own stream, device buffers
    # and workspace each) alternate steps, so one step's upload overlaps the previous step's
    # compute and read-back; the copies of every step stay inside the timed region.
    pinned = {k_: v_.pin_memory() for k_, v_ in host.items()}
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
            run(plan, plan_dev, H, dd["q"], dd["k"], dd["v"], dd["g"], dd["beta"], dd.get("h0"), 1.0, ln["o"],
                ln["fin"], ln["ws"], ln["stream"])
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
    # bounds the end-to-end rate from above
    link = []
    for _ in range(5):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for k_ in pinned:
            d[k_].copy_(pinned[k_], non_blocking=True)
        e1.record(stream)
        torch.cuda.synchronize(dev)
        link.append(e0.elapsed_time(e1))
    h2d_ms = float(statistics.median(link))

    step_ms, e2e_ms = max_over_ranks([step_ms, e2e_ms], world, dev)
    if rank != 0:
        return
    peaks = _peaks()
    T_cont = int(plan[9])
    flops = T * H * FLOPS_STATE + T_cont * H * FLOPS_TRANSITION
    n_seq, n_seg = int(plan[4]), int(plan[5])
    algo_bytes = (T * H * BYTES_TOKEN + T_cont * H * BYTES_CONT + n_seg * H * BYTES_SEGMENT
                  + n_seq * H * BYTES_SEQ_STATE * (2 if w.h0_std > 0 else 1))
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
        "kernel_shares": ({"two_pass_forward": 1.0} if two_pass else
                          {"chunk_forward": shares[0], "compose": shares[1], "boundary": shares[2]}),
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
        "e2e": {"value": aggregate_rate(world, T, e2e_ms), "unit": UNIT, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "h2d_gbs_alone": h2d / (h2d_ms / 1e3) / 1e9,
                "upload_bound_value": aggregate_rate(world, T, h2d_ms),
                "pipeline": "2 lanes: step i+1 uploads its inputs while step i computes and reads back"},
        "gpu_launches": launches_per_step * args.steps,
        "clocks": dict(clk.summary(), window=f"{args.clock_soak_s:g} s soak of identical steps + timed region"),
        "wall_s_timed_region": wall,
    }
    if world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(inp)
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default=HEADLINE, choices=sorted(workloads().keys()))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
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
