"""Helpers shared by the GPU tests: move a drawn problem to the device, run the
CUDA path through the C ABI, and compute the oracle's values for comparison.

Tolerances (the same in every GPU test):
  outputs  max_{t,h,v} |o_gpu - o_oracle| <= 2e-2 (bf16 outputs vs fp64 oracle)
  states   per (segment or sequence, head) matrix:
           ||x - y||_F <= 1e-4 * max(||y||_F, 1e-6 * sqrt(K))
"""
from __future__ import annotations

import numpy as np

import oracle
from context_kda_gb300.inputs import bf16_to_f32

O_TOL = 2e-2
REL_TOL = 1e-4
K = V = 128


def rel_err(x, y):
    """Largest per-matrix relative Frobenius error over the leading axes."""
    x = np.asarray(x, dtype=np.float64)
    y = np.asarray(y, dtype=np.float64)
    x = x.reshape(-1, x.shape[-2] * x.shape[-1])
    y = y.reshape(-1, y.shape[-2] * y.shape[-1])
    num = np.linalg.norm(x - y, axis=1)
    den = np.maximum(np.linalg.norm(y, axis=1), 1e-6 * np.sqrt(K))
    return float(np.max(num / den)) if num.size else 0.0


def to_device(inp, device="cuda"):
    import torch
    t = lambda a, dt: torch.from_numpy(np.ascontiguousarray(a)).view(dt).to(device)
    return {
        "q": t(inp.q, torch.bfloat16), "k": t(inp.k, torch.bfloat16), "v": t(inp.v, torch.bfloat16),
        "g": t(inp.g, torch.float32), "beta": t(inp.beta, torch.float32),
        "h0": None if inp.h0 is None else t(inp.h0, torch.float32),
    }


def plan_bounds(plan, S):
    off = int(plan[14])
    return [int(x) for x in plan[off:off + S + 1]]


def gpu_forward(inp, scale=1.0, path="fused", seg_bounds=None, dev=None):
    """Run the CUDA path ("fused": kda_forward_segmented; "split": its three calls; "two_pass":
    kda_forward_two_pass); returns numpy o (fp32 of the bf16 bits), final, A, B, S_in."""
    import torch
    from context_kda_gb300 import binding as kda
    dev = dev or to_device(inp)
    T, H, N = inp.tokens, inp.heads, inp.num_seqs
    S = inp.segments if seg_bounds is None else len(seg_bounds) - 1
    plan = kda.kda_plan_segments(inp.cu_seqlens, S, seg_bounds)
    plan_dev = kda.upload_plan(plan)
    off = kda.kda_workspace_layout(plan, H)
    ws = torch.empty(off[6], dtype=torch.uint8, device="cuda")
    o = torch.empty((T, H, V), dtype=torch.bfloat16, device="cuda")
    fin = torch.empty((N, H, K, V), dtype=torch.float32, device="cuda")
    if path in ("fused", "two_pass"):
        run = kda.kda_forward_segmented if path == "fused" else kda.kda_forward_two_pass
        run(plan, plan_dev, H, dev["q"], dev["k"], dev["v"], dev["g"], dev["beta"], dev["h0"], scale, o, fin, ws)
        view = lambda a, shape: ws[a:a + 4 * int(np.prod(shape))].view(torch.float32).view(*shape)
        A = view(off[3], (S, H, K, K))
        B = view(off[4], (S, H, K, V))
        S_in = view(off[5], (S, H, K, V))
    else:
        A = torch.empty((S, H, K, K), dtype=torch.float32, device="cuda")
        B = torch.empty((S, H, K, V), dtype=torch.float32, device="cuda")
        S_in = torch.empty((S, H, K, V), dtype=torch.float32, device="cuda")
        kda.kda_segment_forward(plan, plan_dev, H, dev["q"], dev["k"], dev["v"], dev["g"], dev["beta"],
                                dev["h0"], scale, o, A, B, fin, ws)
        kda.kda_compose_summaries(plan, plan_dev, H, A, B, dev["h0"], S_in)
        kda.kda_apply_boundary(plan, plan_dev, H, S_in, ws, o, fin)
    torch.cuda.synchronize()
    return {"o": o.float().cpu().numpy(), "final": fin.cpu().numpy(), "A": A.cpu().numpy(),
            "B": B.cpu().numpy(), "S_in": S_in.cpu().numpy(), "plan": plan, "bounds": plan_bounds(plan, S),
            "o_bits": o.view(torch.int16).cpu().numpy()}


def f32_inputs(inp):
    return bf16_to_f32(inp.q), bf16_to_f32(inp.k), bf16_to_f32(inp.v), inp.g, inp.beta


def oracle_forward(inp, heads=None, scale=1.0):
    q, k, v, g, b = f32_inputs(inp)
    return oracle.forward(inp.cu_seqlens, q, k, v, g, b, h0=inp.h0, scale=scale, heads=heads)


def oracle_segment(inp, bounds, j, h, want_s_in=True):
    """(A_j, B_j, S_in[j]) of segment j, head h, straight from the definitions:
    A_j/B_j from a zero-start run with the transition tracked (A_j = 0 when a sequence
    starts inside the segment), S_in[j] from the monolithic run up to b_j."""
    q, k, v, g, b = f32_inputs(inp)
    cu = [int(x) for x in inp.cu_seqlens]
    a, e = bounds[j], bounds[j + 1]
    starts = [c for c in cu[:-1] if a <= c < e]
    h0 = lambda s: None if inp.h0 is None else inp.h0[s, h].astype(np.float64)
    if starts:
        s_last = cu.index(max(starts))
        r = oracle.run_range(max(starts), e, h, q, k, v, g, b, S0=h0(s_last), want_o=False)
        A, B = np.zeros((K, K)), r["S"]
    else:
        r = oracle.run_range(a, e, h, q, k, v, g, b, S0=None, track_transition=True, want_o=False)
        A, B = r["P"], r["S"]
    S_in = None
    if want_s_in:
        s = max(i for i in range(len(cu) - 1) if cu[i] <= a)
        if cu[s] == a:
            S_in = np.zeros((K, V)) if inp.h0 is None else h0(s)
        else:
            S_in = oracle.run_range(cu[s], a, h, q, k, v, g, b, S0=h0(s), want_o=False)["S"]
    return A, B, S_in


def oracle_summaries(inp, bounds, heads=None, threads=None):
    """A, B and S_in of every segment for the listed heads (default all), from the definitions,
    one head per task on a thread pool (the oracle's C runner releases the GIL):
      S_in[j]  the state of the monolithic run at b_j (h0 of a sequence starting there);
      A_j, B_j the map of the segment: a zero-start run from a with the transition tracked when no
               sequence starts inside [a, e); otherwise A_j = 0 and B_j is the monolithic state at e.
    Returns arrays [S,H,K,K], [S,H,K,V], [S,H,K,V] (NaN for heads not listed)."""
    import concurrent.futures as cf
    import os
    q, k, v, g, b = f32_inputs(inp)
    cu = [int(x) for x in inp.cu_seqlens]
    S = len(bounds) - 1
    H = inp.heads
    heads = list(range(H)) if heads is None else list(heads)
    A = np.full((S, H, K, K), np.nan)
    B = np.full((S, H, K, V), np.nan)
    S_in = np.full((S, H, K, V), np.nan)
    starts = set(cu[:-1])

    def h0(s, h):
        return np.zeros((K, V)) if inp.h0 is None else inp.h0[s, h].astype(np.float64)

    def one_head(h):
        # monolithic states at every segment bound, sequence by sequence
        at = {}
        for s in range(len(cu) - 1):
            cuts = [x for x in bounds if cu[s] < x <= cu[s + 1]]
            St, t = h0(s, h), cu[s]
            for x in cuts:
                St = oracle.run_range(t, x, h, q, k, v, g, b, S0=St, want_o=False)["S"]
                t = x
                at[(s, x)] = St
        for j in range(S):
            a, e = bounds[j], bounds[j + 1]
            s_a = max(i for i in range(len(cu) - 1) if cu[i] <= a)
            S_in[j, h] = h0(s_a, h) if cu[s_a] == a else at[(s_a, a)]
            inside = [c for c in cu[:-1] if a <= c < e]
            if inside:
                s_e = max(i for i in range(len(cu) - 1) if cu[i] < e)
                A[j, h] = 0.0
                B[j, h] = at[(s_e, e)]
            else:
                r = oracle.run_range(a, e, h, q, k, v, g, b, S0=None, track_transition=True, want_o=False)
                A[j, h], B[j, h] = r["P"], r["S"]

    n = threads or max(1, min(len(heads), os.cpu_count() or 1))
    with cf.ThreadPoolExecutor(max_workers=n) as ex:
        list(ex.map(one_head, heads))
    return A, B, S_in


def gpu_scan_both(inp, seg_bounds=None):
    """The three-call path, with S_in computed both by the chain (kda_compose_summaries) and by the
    two-level scan (kda_compose_summaries_blocked) from the same device summaries.  Returns numpy
    S_in_chain, S_in_blocked, A, B and the segment bounds."""
    import torch
    from context_kda_gb300 import binding as kda
    dev = to_device(inp)
    T, H, N = inp.tokens, inp.heads, inp.num_seqs
    S = inp.segments if seg_bounds is None else len(seg_bounds) - 1
    plan = kda.kda_plan_segments(inp.cu_seqlens, S, seg_bounds)
    plan_dev = kda.upload_plan(plan)
    off = kda.kda_workspace_layout(plan, H)
    ws = torch.empty(off[6], dtype=torch.uint8, device="cuda")
    scan_ws = torch.empty(kda.kda_scan_workspace_bytes(plan, H), dtype=torch.uint8, device="cuda")
    o = torch.empty((T, H, V), dtype=torch.bfloat16, device="cuda")
    fin = torch.empty((N, H, K, V), dtype=torch.float32, device="cuda")
    A = torch.empty((S, H, K, K), dtype=torch.float32, device="cuda")
    B = torch.empty((S, H, K, V), dtype=torch.float32, device="cuda")
    S1 = torch.full((S, H, K, V), float("nan"), dtype=torch.float32, device="cuda")
    S2 = torch.full((S, H, K, V), float("nan"), dtype=torch.float32, device="cuda")
    kda.kda_segment_forward(plan, plan_dev, H, dev["q"], dev["k"], dev["v"], dev["g"], dev["beta"], dev["h0"],
                            1.0, o, A, B, fin, ws)
    kda.kda_compose_summaries(plan, plan_dev, H, A, B, dev["h0"], S1)
    kda.kda_compose_summaries_blocked(plan, plan_dev, H, A, B, dev["h0"], S2, scan_ws)
    torch.cuda.synchronize()
    return {"S_in_chain": S1.cpu().numpy(), "S_in_blocked": S2.cpu().numpy(), "A": A.cpu().numpy(),
            "B": B.cpu().numpy(), "bounds": plan_bounds(plan, S)}


def gpu_backward(inp, do_bits, dfinal, scale=1.0, want_dh0=True):
    """kda_backward_segmented through the C ABI; returns numpy dq, dk, dv, dg, dbeta, dh0 (fp32)."""
    import torch
    from context_kda_gb300 import binding as kda
    dev = to_device(inp)
    T, H, N = inp.tokens, inp.heads, inp.num_seqs
    plan = kda.kda_plan_segments(inp.cu_seqlens, inp.segments)
    plan_dev = kda.upload_plan(plan)
    ws = torch.empty(kda.kda_backward_workspace_bytes(plan, H), dtype=torch.uint8, device="cuda")
    dout = torch.from_numpy(np.ascontiguousarray(do_bits)).view(torch.bfloat16).to("cuda")
    df = None if dfinal is None else torch.from_numpy(np.ascontiguousarray(dfinal)).to("cuda")
    nan = float("nan")
    out = {"dq": torch.full((T, H, K), nan, device="cuda"), "dk": torch.full((T, H, K), nan, device="cuda"),
           "dv": torch.full((T, H, V), nan, device="cuda"), "dg": torch.full((T, H, K), nan, device="cuda"),
           "dbeta": torch.full((T, H), nan, device="cuda"),
           "dh0": torch.full((N, H, K, V), nan, device="cuda") if want_dh0 else None}
    kda.kda_backward_segmented(plan, plan_dev, H, dev["q"], dev["k"], dev["v"], dev["g"], dev["beta"], dev["h0"],
                               scale, dout, df, out["dq"], out["dk"], out["dv"], out["dg"], out["dbeta"],
                               out["dh0"], ws)
    torch.cuda.synchronize()
    return {k_: (None if t is None else t.cpu().numpy()) for k_, t in out.items()}


def oracle_backward(inp, do_bits, dfinal, scale=1.0, heads=None):
    """The fp64 backward of the monolithic recurrence (oracle/backward.py) on the same values."""
    from oracle import backward as bw
    q, k, v, g, b = f32_inputs(inp)
    return bw.backward(inp.cu_seqlens, q, k, v, g, b, bf16_to_f32(do_bits), dfinal=dfinal, h0=inp.h0,
                       scale=scale, heads=heads)


def grad_rel_err(x, y, axis_heads=1):
    """Largest per-head relative Frobenius error of a gradient tensor (heads on axis 1)."""
    x = np.asarray(x, dtype=np.float64)
    y = np.asarray(y, dtype=np.float64)
    worst = 0.0
    for h in range(y.shape[axis_heads]):
        xs, ys = np.take(x, h, axis=axis_heads), np.take(y, h, axis=axis_heads)
        den = max(float(np.linalg.norm(ys)), 1e-30)
        worst = max(worst, float(np.linalg.norm(xs - ys)) / den)
    return worst
