"""Segment-parallel reading of KDA, built on the oracle's token-range runner.

Test infrastructure only (see ``oracle/__init__.py``).

The context-parallel design of the pages is followed literally, with segments
of one packed token stream standing in for CP ranks:

* Each segment is cut at sequence boundaries into pieces.  A piece that starts a
  sequence runs from that sequence's initial state, so its outputs are final.
  A piece that continues a sequence begun in an earlier segment runs from a
  zero state and also tracks the transition P from the identity.
* Each segment's affine boundary summary is the map S_start -> A S_start + B of
  the state crossing its end (cuLA PR #110, "feat(cp): add opt-in NVSHMEM CP
  state handoff", §Motivation: each producer publishes its affine recurrence
  state; cuLA PR #136, "feat(kda): add cuDNN concatenated-summary Kimi CP",
  §Summary: preceding_state_update / preceding_transition).  A segment in
  which some sequence starts forgets its incoming state, so A = 0 there.
* Summaries are composed in order, (A2,B2) o (A1,B1) = (A2 A1, A2 B1 + B2)
  (PR #136 §Summary: affine summary composition in FP32 -- done here in fp64),
  seeded by the initial state of the first sequence and reset to a sequence's
  initial state where that sequence starts exactly at a segment start.
* Continuing outputs are then corrected with the incoming state S_in:
  o_t = o_local,t + S_in^T qhat_t, where qhat_t = scale P_t^T q_t.

The result must equal the monolithic recurrence (PR #136 §Walkthrough: the
distributed outputs are compared with a monolithic reference).
"""
from __future__ import annotations

import numpy as np

from . import run_range


def compose(later, earlier):
    """(A2,B2) o (A1,B1) = (A2 A1, A2 B1 + B2); ``earlier`` acts first on the state."""
    A2, B2 = later
    A1, B1 = earlier
    return A2 @ A1, A2 @ B1 + B2


def apply_summary(summary, S):
    A, B = summary
    return A @ S + B


def balanced_bounds(T: int, S: int):
    """Segment j covers tokens [floor(j T / S), floor((j+1) T / S))."""
    return [(j * T) // S for j in range(S + 1)]


def pieces_of_segment(cu, a, b):
    """(sequence, start, end) for every sequence overlapping tokens [a, b), in order."""
    out = []
    for s in range(len(cu) - 1):
        lo, hi = max(a, int(cu[s])), min(b, int(cu[s + 1]))
        if lo < hi:
            out.append((s, lo, hi))
    return out


def segmented_forward(cu, q, k, v, g, beta, h0=None, seg_bounds=None, num_segments=None,
                      scale=1.0, heads=None):
    """Returns dict with o, final [N,H,K,V], A [S,H,K,K], B [S,H,K,V], S_in [S,H,K,V],
    o_local [T,H,V], qhat (dict (token, head) -> vector is avoided: array [T,H,K] with
    NaN outside continuing pieces).  Only heads in ``heads`` (default all) are filled."""
    cu = [int(x) for x in cu]
    T, H, K = q.shape
    V = v.shape[2]
    N = len(cu) - 1
    if seg_bounds is None:
        seg_bounds = balanced_bounds(T, num_segments)
    Sg = len(seg_bounds) - 1
    heads = range(H) if heads is None else heads
    o = np.full((T, H, V), np.nan)
    o_local = np.full((T, H, V), np.nan)
    qhat = np.full((T, H, K), np.nan)
    final = np.full((N, H, K, V), np.nan)
    A = np.full((Sg, H, K, K), np.nan)
    B = np.full((Sg, H, K, V), np.nan)
    S_in = np.full((Sg, H, K, V), np.nan)
    seq_starts = set(cu[:-1])

    def init_state(s, h):
        return np.zeros((K, V)) if h0 is None else np.asarray(h0[s, h], dtype=np.float64)

    for h in heads:
        cont = {}          # segment -> (seq, start, end, run result)
        for j in range(Sg):
            a, b = seg_bounds[j], seg_bounds[j + 1]
            ps = pieces_of_segment(cu, a, b)
            has_reset = False
            last = None
            for (s, lo, hi) in ps:
                if lo == cu[s]:
                    has_reset = True
                    r = run_range(lo, hi, h, q, k, v, g, beta, S0=init_state(s, h), scale=scale)
                    o[lo:hi, h] = r["o"]
                    o_local[lo:hi, h] = r["o"]
                    if hi == cu[s + 1]:
                        final[s, h] = r["S"]
                else:
                    r = run_range(lo, hi, h, q, k, v, g, beta, S0=None, track_transition=True, scale=scale)
                    o_local[lo:hi, h] = r["o"]
                    qhat[lo:hi, h] = r["qhat"]
                    cont[j] = (s, lo, hi, r)
                last = r
            A[j, h] = 0.0 if has_reset else cont[j][3]["P"]
            B[j, h] = last["S"]
        # sequential composition, seeded by the first sequence's initial state
        prefix = (np.zeros((K, K)), init_state(0, h))
        S_in[0, h] = prefix[1]
        for j in range(1, Sg):
            bj = seg_bounds[j]
            if bj in seq_starts:
                e = (np.zeros((K, K)), init_state(cu.index(bj), h))
            else:
                e = (A[j - 1, h], B[j - 1, h])
            prefix = compose(e, prefix)
            S_in[j, h] = prefix[1]
        # fix-up of continuing pieces and of the final states they end
        for j, (s, lo, hi, r) in cont.items():
            o[lo:hi, h] = r["o"] + r["qhat"] @ S_in[j, h]
            if hi == cu[s + 1]:
                final[s, h] = apply_summary((r["P"], r["S"]), S_in[j, h])
    return {"o": o, "final": final, "A": A, "B": B, "S_in": S_in, "o_local": o_local, "qhat": qhat,
            "seg_bounds": list(seg_bounds)}
