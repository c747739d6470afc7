"""Backward of the KDA recurrence: gradients of q, k, v, g, beta and h0 -- test infrastructure.

Only the test suite may import this module (see ``oracle/__init__.py``); nothing of the CUDA
library uses it.

The forward is the recurrence the oracle's C code runs (cuLA PR #110, "feat(cp): add opt-in
NVSHMEM CP state handoff", §Supported configuration: BF16 inputs, FP32 recurrent state), written
per token t of one (sequence, head) as

    St_t = Diag(exp g_t) S_{t-1}             (decay first)
    u_t  = v_t - St_t^T k_t                  (delta-rule residual)
    S_t  = St_t + beta_t k_t u_t^T           (= (I - beta k k^T) Diag(exp g) S + beta k v^T)
    o_t  = scale S_t^T q_t

and the loss whose gradients are taken is L = sum_t <do_t, o_t> + sum_seq <dfinal, S_end>.  The
pages say only that the backward needs the "following" FP32 summaries (cuLA PR #136, "feat(kda):
add cuDNN concatenated-summary Kimi CP", §Summary and the walkthrough's sequence diagram: the
following summaries are gathered during backward); which gradients exist is from PR #110
§Correctness (output and Q/K/V/g/beta gradients checked).  Everything else here is the chain rule
applied to the four lines above, in reverse token order:

    dS    += scale q_t do_t^T                (o_t reads S_t)
    dq_t   = scale S_t do_t
    du     = beta_t dS^T k_t,   dbeta_t = k_t^T dS u_t,   dk_t = beta_t dS u_t
    dv_t   = du,   dSt = dS - k_t du^T,   dk_t -= St_t du
    dg_t   = rowsum(dSt * St_t)              (d St[i, :] / d g_t[i] = St[i, :])
    dS     = Diag(exp g_t) dSt               (the gradient reaching S_{t-1})

with dS starting at dfinal of the sequence and ending as dh0.

``segmented_backward`` is the pages' context-parallel reading of the same gradients: the
gradient reaching each segment's end state is composed from the segments after it through their
summaries alone (transposed transitions and the qhat of their continuing tokens), and each piece
then runs the local backward above from its true incoming state.  It must equal ``backward``.

Arithmetic is fp64 throughout.  Functions take any K and V (the tests use small ones for finite
differences).
"""
from __future__ import annotations

import numpy as np

# Planted mistakes for the tests that show the pins catch them (0 = the definition).
MUTATIONS = {
    "none": 0,
    "dk_without_state_term": 1,     # drops dk_t -= St_t du
    "dg_sign": 2,                   # dg_t negated
    "ds_without_residual_term": 3,  # drops the -k_t du^T term of dSt
    "dq_without_scale": 4,          # dq_t = S_t do_t
    "decay_not_applied_to_ds": 5,   # dS = dSt (no Diag(exp g_t))
}


def _f64(a):
    return np.asarray(a, dtype=np.float64)


def forward_range(t0, t1, h, q, k, v, g, beta, S0=None, scale=1.0):
    """States and outputs of tokens [t0, t1) of head h from S0 (zeros if None), by the four
    lines of the module docstring.  Returns (states [(n+1), K, V] with states[0] = S0, o [n, V])."""
    q, k, v, g, beta = _f64(q), _f64(k), _f64(v), _f64(g), _f64(beta)
    K, V = q.shape[2], v.shape[2]
    n = int(t1 - t0)
    states = np.empty((n + 1, K, V))
    states[0] = np.zeros((K, V)) if S0 is None else _f64(S0)
    o = np.empty((n, V))
    for i in range(n):
        t = t0 + i
        St = np.exp(g[t, h])[:, None] * states[i]
        u = v[t, h] - St.T @ k[t, h]
        S = St + beta[t, h] * np.outer(k[t, h], u)
        states[i + 1] = S
        o[i] = scale * (S.T @ q[t, h])
    return states, o


def backward_range(t0, t1, h, q, k, v, g, beta, do, S0=None, dS_end=None, scale=1.0, mutate=0):
    """Gradients over tokens [t0, t1) of head h, run from state S0 with dS_end the gradient of the
    state after token t1 - 1 (zeros if None) and do [T, H, V] the output gradients.  Returns dict
    with dq, dk, dg [n, K], dv [n, V], dbeta [n] and dS0 (the gradient of the starting state)."""
    q, k, v, g, beta, do = _f64(q), _f64(k), _f64(v), _f64(g), _f64(beta), _f64(do)
    K, V = q.shape[2], v.shape[2]
    n = int(t1 - t0)
    states, _ = forward_range(t0, t1, h, q, k, v, g, beta, S0=S0, scale=scale)
    dS = np.zeros((K, V)) if dS_end is None else _f64(dS_end).copy()
    dq, dk, dg = np.empty((n, K)), np.empty((n, K)), np.empty((n, K))
    dv, dbeta = np.empty((n, V)), np.empty(n)
    for i in range(n - 1, -1, -1):
        t = t0 + i
        qt, kt, gt, bt, dot = q[t, h], k[t, h], g[t, h], beta[t, h], do[t, h]
        e = np.exp(gt)
        S, Sp = states[i + 1], states[i]
        St = e[:, None] * Sp
        u = v[t, h] - St.T @ kt
        dS = dS + scale * np.outer(qt, dot)
        dq[i] = (S @ dot) if mutate == 4 else scale * (S @ dot)
        du = bt * (dS.T @ kt)
        dbeta[i] = kt @ dS @ u
        dki = bt * (dS @ u)
        dv[i] = du
        dSt = dS if mutate == 3 else dS - np.outer(kt, du)
        if mutate != 1:
            dki = dki - St @ du
        dk[i] = dki
        dgi = np.sum(dSt * St, axis=1)
        dg[i] = -dgi if mutate == 2 else dgi
        dS = dSt if mutate == 5 else e[:, None] * dSt
    return {"dq": dq, "dk": dk, "dv": dv, "dg": dg, "dbeta": dbeta, "dS0": dS}


def backward(cu_seqlens, q, k, v, g, beta, do, dfinal=None, h0=None, scale=1.0, heads=None, mutate=0):
    """Gradients of L = sum <do, o> + sum <dfinal, final> for packed sequences (the definition):
    q, k, g [T, H, K], v [T, H, V], beta [T, H], do [T, H, V], dfinal and h0 [N, H, K, V] or
    None.  Returns dict dq, dk, dg [T, H, K], dv [T, H, V], dbeta [T, H], dh0 [N, H, K, V];
    heads not listed in ``heads`` are left as NaN."""
    cu = [int(x) for x in cu_seqlens]
    T, H, K = np.shape(q)
    V = np.shape(v)[2]
    N = len(cu) - 1
    heads = range(H) if heads is None else heads
    out = {"dq": np.full((T, H, K), np.nan), "dk": np.full((T, H, K), np.nan),
           "dg": np.full((T, H, K), np.nan), "dv": np.full((T, H, V), np.nan),
           "dbeta": np.full((T, H), np.nan), "dh0": np.full((N, H, K, V), np.nan)}
    for h in heads:
        for s in range(N):
            r = backward_range(cu[s], cu[s + 1], h, q, k, v, g, beta, do,
                               S0=None if h0 is None else h0[s, h],
                               dS_end=None if dfinal is None else dfinal[s, h], scale=scale, mutate=mutate)
            for key in ("dq", "dk", "dg", "dv", "dbeta"):
                out[key][cu[s]:cu[s + 1], h] = r[key]
            out["dh0"][s, h] = r["dS0"]
    return out


def segmented_backward(cu_seqlens, q, k, v, g, beta, do, dfinal=None, h0=None, seg_bounds=None,
                       num_segments=None, scale=1.0, heads=None):
    """The same gradients, segment-parallel.  The forward summaries come from the segmented
    oracle (A, S_in and the continuing tokens' qhat).  Then, per head:

    * following summaries, last segment first: the gradient of the state crossing the end of
      segment j is dfinal of the sequence that ends there, or else the gradient of segment
      j + 1's incoming state, which is sum_t qhat_t do_t^T over j + 1's continuing piece plus
      the transposed map of that piece applied to the gradient at its end (A^T of the segment,
      or P_end^T of a piece that ends its sequence inside the segment, applied to dfinal);
    * every piece runs the local backward from its true incoming state (S_in of its segment for
      a continuing piece, h0 for a piece that starts its sequence) with that end gradient.

    Returns the dict of ``backward`` plus dS_out [S, H, K, V] (the gradient of each segment's
    end state), dS_in [S, H, K, V] (of its incoming state, from the following summaries; NaN where
    a sequence starts at the segment start) and dS_in_local (the same gradient as the continuing
    piece's own local backward returns it).  The forward summaries come from the C oracle, which
    reads fp32 inputs: pass fp32-representable values."""
    from . import run_range
    from .segmented import balanced_bounds, pieces_of_segment, segmented_forward

    cu = [int(x) for x in cu_seqlens]
    T, H, K = np.shape(q)
    V = np.shape(v)[2]
    N = len(cu) - 1
    if seg_bounds is None:
        seg_bounds = balanced_bounds(T, num_segments)
    Sg = len(seg_bounds) - 1
    heads = list(range(H)) if heads is None else list(heads)
    fw = segmented_forward(cu, q, k, v, g, beta, h0=h0, seg_bounds=seg_bounds, scale=scale, heads=heads)
    do64 = _f64(do)
    out = {"dq": np.full((T, H, K), np.nan), "dk": np.full((T, H, K), np.nan),
           "dg": np.full((T, H, K), np.nan), "dv": np.full((T, H, V), np.nan),
           "dbeta": np.full((T, H), np.nan), "dh0": np.full((N, H, K, V), np.nan),
           "dS_out": np.full((Sg, H, K, V), np.nan), "dS_in": np.full((Sg, H, K, V), np.nan),
           "dS_in_local": np.full((Sg, H, K, V), np.nan)}
    seq_end_at = {cu[s + 1]: s for s in range(N)}
    zero = np.zeros((K, V))

    def dfin(s, h):
        return zero if dfinal is None else _f64(dfinal[s, h])

    for h in heads:
        # following summaries: the end-state gradient of every segment, from the later segments'
        # summaries only
        for j in range(Sg - 1, -1, -1):
            b = seg_bounds[j + 1]
            if b in seq_end_at:
                out["dS_out"][j, h] = dfin(seq_end_at[b], h)
                continue
            nxt = j + 1
            a2, b2 = seg_bounds[nxt], seg_bounds[nxt + 1]
            s, lo, hi = pieces_of_segment(cu, a2, b2)[0]          # the continuing piece of j + 1
            qh = fw["qhat"][lo:hi, h]
            g_in = qh.T @ do64[lo:hi, h]
            if hi == cu[s + 1]:                                    # it ends its sequence in j + 1
                P_end = run_range(lo, hi, h, q, k, v, g, beta, S0=None, track_transition=True,
                                  scale=scale, want_o=False)["P"]
                g_in = g_in + P_end.T @ dfin(s, h)
            else:                                                  # it spans j + 1
                g_in = g_in + fw["A"][nxt, h].T @ out["dS_out"][nxt, h]
            out["dS_in"][nxt, h] = g_in
            out["dS_out"][j, h] = g_in
        # local backward of every piece from its true incoming state
        for j in range(Sg):
            a, b = seg_bounds[j], seg_bounds[j + 1]
            for (s, lo, hi) in pieces_of_segment(cu, a, b):
                starts_seq = lo == cu[s]
                S0 = (None if h0 is None else h0[s, h]) if starts_seq else fw["S_in"][j, h]
                dS_end = dfin(s, h) if hi == cu[s + 1] else out["dS_out"][j, h]
                r = backward_range(lo, hi, h, q, k, v, g, beta, do, S0=S0, dS_end=dS_end, scale=scale)
                for key in ("dq", "dk", "dg", "dv", "dbeta"):
                    out[key][lo:hi, h] = r[key]
                if starts_seq:
                    out["dh0"][s, h] = r["dS0"]
                else:
                    out["dS_in_local"][j, h] = r["dS0"]
    return out
