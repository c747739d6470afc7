"""Pins of the backward oracle (oracle/backward.py) -- CPU only.

The backward is the chain rule through the token recurrence; nothing on the pages prints a
gradient value, so it is pinned by what the mathematics fixes:
  * central finite differences of the forward loss, element by element, on tiny problems;
  * its own forward against the C oracle's recurrence;
  * closed forms: beta = 0 and g = 0 (a static state), and do = 0 (the gradient of the initial
    state is the sequence's transposed transition applied to dfinal);
  * the pages' segment-parallel reading (cuLA PR #136, "feat(kda): add cuDNN concatenated-summary
    Kimi CP", §Summary: following summaries gathered during backward) equals the monolithic one;
  * every planted mistake is caught by the finite-difference pin.
"""
import numpy as np
import pytest

import oracle
from oracle import backward as bw


def _problem(seqlens, H, K, V, seed, h0=True, fp32=False, g_lo=-0.3, g_hi=-0.01):
    rng = np.random.default_rng(seed)
    T = int(sum(seqlens))
    N = len(seqlens)
    cu = np.concatenate([[0], np.cumsum(seqlens)]).astype(np.int64)
    x = {
        "q": rng.standard_normal((T, H, K)) / np.sqrt(K),
        "k": rng.standard_normal((T, H, K)) / np.sqrt(K),
        "v": rng.standard_normal((T, H, V)),
        "g": rng.uniform(g_lo, g_hi, (T, H, K)),
        "beta": 1.0 / (1.0 + np.exp(-rng.standard_normal((T, H)))),
        "h0": 0.3 * rng.standard_normal((N, H, K, V)) if h0 else None,
        "do": rng.standard_normal((T, H, V)),
        "dfinal": rng.standard_normal((N, H, K, V)),
    }
    if fp32:
        x = {k_: (None if a is None else a.astype(np.float32).astype(np.float64)) for k_, a in x.items()}
    return cu, x


def _loss(cu, x, scale):
    """L = sum <do, o> + sum <dfinal, final>, from the backward module's own forward."""
    H = x["q"].shape[1]
    total = 0.0
    for h in range(H):
        for s in range(len(cu) - 1):
            S0 = None if x["h0"] is None else x["h0"][s, h]
            states, o = bw.forward_range(cu[s], cu[s + 1], h, x["q"], x["k"], x["v"], x["g"], x["beta"],
                                         S0=S0, scale=scale)
            total += float(np.sum(x["do"][cu[s]:cu[s + 1], h] * o))
            total += float(np.sum(x["dfinal"][s, h] * states[-1]))
    return total


def _grads(cu, x, scale, mutate=0):
    return bw.backward(cu, x["q"], x["k"], x["v"], x["g"], x["beta"], x["do"], dfinal=x["dfinal"],
                       h0=x["h0"], scale=scale, mutate=mutate)


def _finite_differences(cu, x, scale, eps=1e-6):
    fd = {}
    for name, key in (("dq", "q"), ("dk", "k"), ("dv", "v"), ("dg", "g"), ("dbeta", "beta"), ("dh0", "h0")):
        arr = x[key]
        grad = np.zeros_like(arr)
        for idx in np.ndindex(arr.shape):
            keep = arr[idx]
            arr[idx] = keep + eps
            up = _loss(cu, x, scale)
            arr[idx] = keep - eps
            dn = _loss(cu, x, scale)
            arr[idx] = keep
            grad[idx] = (up - dn) / (2 * eps)
        fd[name] = grad
    return fd


def _rel(a, b):
    a, b = np.asarray(a, dtype=np.float64), np.asarray(b, dtype=np.float64)
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-30))


FD_CASE = dict(seqlens=[5, 3], H=2, K=3, V=2, seed=21)


@pytest.fixture(scope="module")
def fd_case():
    cu, x = _problem(FD_CASE["seqlens"], FD_CASE["H"], FD_CASE["K"], FD_CASE["V"], FD_CASE["seed"])
    scale = 0.7
    return cu, x, scale, _finite_differences(cu, x, scale)


def test_gradients_match_central_differences(fd_case):
    cu, x, scale, fd = fd_case
    gr = _grads(cu, x, scale)
    for name in fd:
        assert _rel(gr[name], fd[name]) <= 1e-7, name


@pytest.mark.parametrize("name", [m for m in bw.MUTATIONS if m != "none"])
def test_planted_mistake_is_caught(fd_case, name):
    cu, x, scale, fd = fd_case
    gr = _grads(cu, x, scale, mutate=bw.MUTATIONS[name])
    assert max(_rel(gr[n], fd[n]) for n in fd) > 1e-3, name


def test_own_forward_matches_the_c_oracle():
    cu, x = _problem([17, 1, 30], H=2, K=8, V=8, seed=22, fp32=True)
    scale = 0.6
    o_ref, f_ref = oracle.forward(cu.astype(np.int32), x["q"], x["k"], x["v"], x["g"], x["beta"], h0=x["h0"],
                                  scale=scale)
    for h in range(2):
        for s in range(3):
            states, o = bw.forward_range(cu[s], cu[s + 1], h, x["q"], x["k"], x["v"], x["g"], x["beta"],
                                         S0=x["h0"][s, h], scale=scale)
            assert np.max(np.abs(o - o_ref[cu[s]:cu[s + 1], h])) <= 1e-12
            assert np.max(np.abs(states[-1] - f_ref[s, h])) <= 1e-12


def test_static_state_closed_form():
    """beta = 0, g = 0: S_t = h0 for every t.  Then dq_t = scale h0 do_t, dk = dv = 0,
    dS_t = dfinal + scale sum_{s >= t} q_s do_s^T, dg_t = rowsum(dS_t * h0),
    dbeta_t = k_t^T dS_t (v_t - h0^T k_t), and dh0 = dS_1."""
    cu, x = _problem([9], H=1, K=4, V=3, seed=23)
    x["beta"][:] = 0.0
    x["g"][:] = 0.0
    scale = 0.8
    gr = _grads(cu, x, scale)
    S0, q, k, v, do, dfin = x["h0"][0, 0], x["q"][:, 0], x["k"][:, 0], x["v"][:, 0], x["do"][:, 0], x["dfinal"][0, 0]
    T = 9
    dS = [dfin + scale * sum(np.outer(q[s], do[s]) for s in range(t, T)) for t in range(T)]
    np.testing.assert_allclose(gr["dq"][:, 0], scale * do @ S0.T, rtol=1e-12, atol=1e-13)
    assert np.all(gr["dk"][:, 0] == 0) and np.all(gr["dv"][:, 0] == 0)
    np.testing.assert_allclose(gr["dg"][:, 0], [np.sum(dS[t] * S0, axis=1) for t in range(T)], rtol=1e-12,
                               atol=1e-13)
    np.testing.assert_allclose(gr["dbeta"][:, 0], [k[t] @ dS[t] @ (v[t] - S0.T @ k[t]) for t in range(T)],
                               rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(gr["dh0"][0, 0], dS[0], rtol=1e-12, atol=1e-13)


def test_initial_state_gradient_is_the_transposed_transition():
    """With do = 0 the loss is <dfinal, P h0 + B>, so dh0 = P^T dfinal, P the sequence's
    transition as the C oracle tracks it."""
    cu, x = _problem([40], H=1, K=8, V=8, seed=24, fp32=True)
    x["do"][:] = 0.0
    gr = _grads(cu, x, 1.0)
    P = oracle.run_range(0, 40, 0, x["q"], x["k"], x["v"], x["g"], x["beta"], track_transition=True,
                         want_o=False)["P"]
    np.testing.assert_allclose(gr["dh0"][0, 0], P.T @ x["dfinal"][0, 0], rtol=1e-10, atol=1e-12)


@pytest.mark.parametrize("seqlens,S", [
    ([40], 1),
    ([40], 3),                     # continuing pieces spanning whole segments
    ([23, 5, 31, 12], 4),          # resets inside segments, continuing pieces ending mid-segment
    ([7, 7, 7], 3),                # segment bounds at sequence starts
    ([3, 1, 2, 6], 10),            # one-token segments
])
def test_segmented_backward_equals_monolithic(seqlens, S):
    cu, x = _problem(seqlens, H=2, K=6, V=5, seed=25, fp32=True)
    scale = 0.9
    mono = _grads(cu, x, scale)
    seg = bw.segmented_backward(cu, x["q"], x["k"], x["v"], x["g"], x["beta"], x["do"], dfinal=x["dfinal"],
                                h0=x["h0"], num_segments=S, scale=scale)
    for name in ("dq", "dk", "dv", "dg", "dbeta", "dh0"):
        assert _rel(seg[name], mono[name]) <= 1e-10, name
    have = ~np.isnan(seg["dS_in"])
    # the incoming-state gradient from the following summaries is the one the piece's own
    # backward produces
    assert np.array_equal(have, ~np.isnan(seg["dS_in_local"]))
    if have.any():
        assert _rel(seg["dS_in"][have], seg["dS_in_local"][have]) <= 1e-10


def test_segmented_backward_catches_a_dropped_following_summary():
    """The pin above is not vacuous: without the transposed transition of the next segment the
    gradients of earlier segments change."""
    cu, x = _problem([40], H=1, K=6, V=5, seed=26, fp32=True)
    mono = _grads(cu, x, 1.0)
    seg = bw.segmented_backward(cu, x["q"], x["k"], x["v"], x["g"], x["beta"], x["do"], dfinal=x["dfinal"],
                                h0=x["h0"], num_segments=3, scale=1.0)
    # redo segment 0's local backward with only the next segment's qhat term
    bounds = [0, 13, 26, 40]
    qh = oracle.run_range(13, 26, 0, x["q"], x["k"], x["v"], x["g"], x["beta"], track_transition=True,
                          want_o=True)["qhat"]
    wrong_end = qh.T @ x["do"][13:26, 0]
    r = bw.backward_range(0, 13, 0, x["q"], x["k"], x["v"], x["g"], x["beta"], x["do"], S0=x["h0"][0, 0],
                          dS_end=wrong_end)
    assert bounds[1] == 13
    for name in ("dk", "dv", "dg", "dbeta"):   # dq reads only the forward states
        assert _rel(r[name], mono[name][0:13, 0]) > 1e-6, name
        assert _rel(seg[name][0:13, 0], mono[name][0:13, 0]) <= 1e-10, name
