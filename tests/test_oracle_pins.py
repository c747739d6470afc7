"""Pins for the CPU oracle: closed forms, brute-force dense products, invariants.

Each pin ties the oracle to something other than itself.  The last test plants
each plausible mistake in the oracle (its test-only 'mutate' switch) and checks
that at least one pin catches it.

The recurrence pinned is the KDA gated delta rule with a K x V state
(cuLA PR #110, "feat(cp): add opt-in NVSHMEM CP state handoff", §Supported
configuration: BF16 inputs, FP32 recurrent state, non-transposed layout):
S_t = (I - b_t k_t k_t^T) Diag(exp g_t) S_{t-1} + b_t k_t v_t^T,
o_t = scale S_t^T q_t.
"""
import numpy as np
import pytest

import oracle
from oracle import MUTATIONS
from oracle.segmented import apply_summary, balanced_bounds, compose, segmented_forward


def _rand_problem(rng, T, H, K, V, g_scale=0.2):
    q = rng.standard_normal((T, H, K)).astype(np.float32)
    k = rng.standard_normal((T, H, K)).astype(np.float32)
    k /= np.linalg.norm(k, axis=-1, keepdims=True)
    v = rng.standard_normal((T, H, V)).astype(np.float32)
    g = (-g_scale * rng.random((T, H, K))).astype(np.float32)
    beta = rng.random((T, H)).astype(np.float32)
    return q, k, v, g, beta


# ---------------------------------------------------------------- pins, each returns True when it holds

def pin_static_state(mutate=0):
    """beta = 0, g = 0: the state never moves, o_t = scale S_0^T q_t, final = S_0."""
    rng = np.random.default_rng(1)
    T, H, K, V = 9, 2, 5, 7
    q, k, v, g, beta = _rand_problem(rng, T, H, K, V)
    g[:] = 0
    beta[:] = 0
    S0 = rng.standard_normal((K, V))
    r = oracle.run_range(0, T, 1, q, k, v, g, beta, S0=S0, scale=0.5, mutate=mutate)
    want = 0.5 * q[:, 1].astype(np.float64) @ S0
    return np.allclose(r["o"], want, rtol=0, atol=1e-12) and np.allclose(r["S"], S0, rtol=0, atol=1e-14)


def pin_decay_only(mutate=0):
    """beta = 0: S_t = Diag(exp Gamma_t) S_0, so o_t = S_0^T (exp(Gamma_t) * q_t) and the
    transition is Diag(exp sum g)."""
    rng = np.random.default_rng(2)
    T, H, K, V = 11, 1, 6, 6
    q, k, v, g, beta = _rand_problem(rng, T, H, K, V, g_scale=0.5)
    beta[:] = 0
    S0 = rng.standard_normal((K, V))
    r = oracle.run_range(0, T, 0, q, k, v, g, beta, S0=S0, track_transition=True, mutate=mutate)
    gam = np.cumsum(g[:, 0].astype(np.float64), axis=0)
    want = (np.exp(gam) * q[:, 0]) @ S0
    ok = np.allclose(r["o"], want, rtol=1e-12, atol=1e-13)
    ok &= np.allclose(r["P"], np.diag(np.exp(gam[-1])), rtol=1e-12, atol=1e-14)
    return bool(ok)


def pin_overwrite(mutate=0):
    """g = 0, beta = 1, q_t = k_t = a standard basis vector: each token overwrites one row of
    the state with v_t exactly, so o_t = v_t (delta-rule overwrite)."""
    rng = np.random.default_rng(3)
    T, H, K, V = 14, 1, 6, 6
    q, k, v, g, beta = _rand_problem(rng, T, H, K, V)
    g[:] = 0
    beta[:] = 1
    idx = rng.integers(0, K, size=T)
    k[:] = 0
    k[np.arange(T), 0, idx] = 1
    q[:] = k
    S0 = rng.standard_normal((K, V))
    r = oracle.run_range(0, T, 0, q, k, v, g, beta, S0=S0, mutate=mutate)
    ok = np.allclose(r["o"], v[:, 0], rtol=0, atol=1e-12)
    # rows never keyed keep S0; keyed rows hold the last value written with that key
    want = S0.copy()
    for t in range(T):
        want[idx[t]] = v[t, 0]
    return bool(ok and np.allclose(r["S"], want, rtol=0, atol=1e-12))


def pin_scalar(mutate=0):
    """K = V = 1: s_t = a_t s_{t-1} + b_t with a_t = (1 - beta k^2) e^g, b_t = beta k v;
    s_T = (prod a) s_0 + sum_t (prod_{u>t} a_u) b_t."""
    rng = np.random.default_rng(4)
    T = 13
    q = rng.standard_normal((T, 1, 1)).astype(np.float32)
    k = rng.uniform(-1, 1, (T, 1, 1)).astype(np.float32)
    v = rng.standard_normal((T, 1, 1)).astype(np.float32)
    g = (-0.3 * rng.random((T, 1, 1))).astype(np.float32)
    beta = rng.random((T, 1)).astype(np.float32)
    s0 = 0.7
    r = oracle.run_range(0, T, 0, q, k, v, g, beta, S0=np.array([[s0]]), mutate=mutate)
    kk, vv, gg, bb, qq = (x.reshape(T).astype(np.float64) for x in (k, v, g, beta[:, :, None], q))
    a = (1 - bb * kk * kk) * np.exp(gg)
    b = bb * kk * vv
    outs = []
    for t in range(T):
        st = np.prod(a[:t + 1]) * s0 + sum(np.prod(a[u + 1:t + 1]) * b[u] for u in range(t + 1))
        outs.append(st * qq[t])
    return bool(np.allclose(r["o"][:, 0], outs, rtol=1e-12, atol=1e-14))


def _dense_step(kt, gt, bt):
    K = kt.shape[0]
    kt = kt.astype(np.float64)
    return (np.eye(K) - float(bt) * np.outer(kt, kt)) @ np.diag(np.exp(gt.astype(np.float64)))


def pin_bruteforce(mutate=0):
    """Explicit dense products on tiny T with K != V: A = M_T ... M_1 with
    M_t = (I - b_t k_t k_t^T) Diag(exp g_t), B = sum_t (M_T ... M_{t+1}) b_t k_t v_t^T;
    the runner's transition, zero-start state, random-start state, outputs and qhat must
    all agree."""
    rng = np.random.default_rng(5)
    T, H, K, V = 12, 3, 5, 7
    q, k, v, g, beta = _rand_problem(rng, T, H, K, V, g_scale=0.6)
    h = 2
    S0 = rng.standard_normal((K, V))
    Ms = [_dense_step(k[t, h], g[t, h], beta[t, h]) for t in range(T)]
    A = np.eye(K)
    Bz = np.zeros((K, V))
    outs, qh = [], []
    for t in range(T):
        A = Ms[t] @ A
        Bz = Ms[t] @ Bz + float(beta[t, h]) * np.outer(k[t, h].astype(np.float64), v[t, h].astype(np.float64))
        St = A @ S0 + Bz
        outs.append(0.75 * St.T @ q[t, h].astype(np.float64))
        qh.append(0.75 * A.T @ q[t, h].astype(np.float64))
    r0 = oracle.run_range(0, T, h, q, k, v, g, beta, S0=None, track_transition=True, scale=0.75,
                          mutate=mutate)
    r1 = oracle.run_range(0, T, h, q, k, v, g, beta, S0=S0, scale=0.75, mutate=mutate)
    ok = np.allclose(r0["P"], A, rtol=1e-12, atol=1e-13)
    ok &= np.allclose(r0["S"], Bz, rtol=1e-12, atol=1e-13)
    ok &= np.allclose(r1["S"], A @ S0 + Bz, rtol=1e-12, atol=1e-13)
    ok &= np.allclose(r1["o"], np.array(outs), rtol=1e-11, atol=1e-12)
    ok &= np.allclose(r0["qhat"], np.array(qh), rtol=1e-11, atol=1e-12)
    return bool(ok)


PINS = [pin_static_state, pin_decay_only, pin_overwrite, pin_scalar, pin_bruteforce]


@pytest.mark.parametrize("pin", PINS, ids=lambda p: p.__name__)
def test_pin_holds(pin):
    assert pin(0)


@pytest.mark.parametrize("name", [m for m in MUTATIONS if m != "none"])
def test_planted_mistake_is_caught(name):
    caught = [p.__name__ for p in PINS if not p(MUTATIONS[name])]
    assert caught, f"mutation {name} escaped every pin"


# ---------------------------------------------------------------- invariants

def test_compose_associative_and_semantic():
    rng = np.random.default_rng(6)
    K, V = 6, 4
    es = [(rng.standard_normal((K, K)), rng.standard_normal((K, V))) for _ in range(3)]
    left = compose(compose(es[2], es[1]), es[0])
    right = compose(es[2], compose(es[1], es[0]))
    assert np.allclose(left[0], right[0], atol=1e-12) and np.allclose(left[1], right[1], atol=1e-12)
    S = rng.standard_normal((K, V))
    step = apply_summary(es[1], apply_summary(es[0], S))
    assert np.allclose(apply_summary(compose(es[1], es[0]), S), step, atol=1e-12)
    # the identity summary is neutral
    ident = (np.eye(K), np.zeros((K, V)))
    c = compose(ident, es[0])
    assert np.array_equal(c[0], es[0][0]) and np.array_equal(c[1], es[0][1])


def _small_varlen(rng, seqlens, H=2, K=6, V=5):
    T = sum(seqlens)
    cu = np.concatenate([[0], np.cumsum(seqlens)]).astype(np.int32)
    q, k, v, g, beta = _rand_problem(rng, T, H, K, V, g_scale=0.3)
    h0 = rng.standard_normal((len(seqlens), H, K, V))
    return cu, q, k, v, g, beta, h0


@pytest.mark.parametrize("nseg", [1, 2, 4, 7, 16])
def test_segmented_equals_monolithic(nseg):
    """The segment-parallel result equals the monolithic sequence (cuLA PR #136,
    §Walkthrough: distributed outputs compared with a monolithic reference)."""
    rng = np.random.default_rng(10 + nseg)
    cu, q, k, v, g, beta, h0 = _small_varlen(rng, [17, 5, 30, 1, 12])
    o_ref, f_ref = oracle.forward(cu, q, k, v, g, beta, h0=h0, scale=0.9)
    seg = segmented_forward(cu, q, k, v, g, beta, h0=h0, num_segments=nseg, scale=0.9)
    assert np.allclose(seg["o"], o_ref, rtol=1e-10, atol=1e-11)
    assert np.allclose(seg["final"], f_ref, rtol=1e-10, atol=1e-11)


def test_segmented_custom_bounds_and_structural_zeros():
    rng = np.random.default_rng(20)
    cu, q, k, v, g, beta, h0 = _small_varlen(rng, [40, 23, 3, 34])
    bounds = [0, 9, 40, 41, 66, 70, 100]
    o_ref, f_ref = oracle.forward(cu, q, k, v, g, beta, h0=h0)
    seg = segmented_forward(cu, q, k, v, g, beta, h0=h0, seg_bounds=bounds)
    assert np.allclose(seg["o"], o_ref, rtol=1e-10, atol=1e-11)
    assert np.allclose(seg["final"], f_ref, rtol=1e-10, atol=1e-11)
    starts = set(int(x) for x in cu[:-1])
    for j in range(len(bounds) - 1):
        has_reset = any(bounds[j] <= s < bounds[j + 1] for s in starts)
        assert (np.all(seg["A"][j] == 0.0)) == has_reset


def test_summary_reproduces_segment_state():
    """A_j S + B_j is the state at the segment end for any incoming state S."""
    rng = np.random.default_rng(21)
    cu, q, k, v, g, beta, _ = _small_varlen(rng, [64])
    seg = segmented_forward(cu, q, k, v, g, beta, num_segments=4)
    b = seg["seg_bounds"]
    for h in range(q.shape[1]):
        S = rng.standard_normal((q.shape[2], v.shape[2]))
        r = oracle.run_range(b[1], b[2], h, q, k, v, g, beta, S0=S)
        assert np.allclose(seg["A"][1, h] @ S + seg["B"][1, h], r["S"], rtol=1e-11, atol=1e-12)


def test_resume_from_final_state():
    """forward(T1) then forward(T2, h0 = final) equals forward(T1 + T2)."""
    rng = np.random.default_rng(22)
    q, k, v, g, beta = _rand_problem(rng, 50, 2, 6, 5)
    o_all, f_all = oracle.forward([0, 50], q, k, v, g, beta)
    o1, f1 = oracle.forward([0, 20], q[:20], k[:20], v[:20], g[:20], beta[:20])
    o2, f2 = oracle.forward([0, 30], q[20:], k[20:], v[20:], g[20:], beta[20:], h0=f1)
    assert np.allclose(np.concatenate([o1, o2]), o_all, rtol=1e-11, atol=1e-12)
    assert np.allclose(f2, f_all, rtol=1e-11, atol=1e-12)


def test_head_independence_and_head_subset():
    rng = np.random.default_rng(23)
    q, k, v, g, beta = _rand_problem(rng, 30, 3, 6, 5)
    o_a, _ = oracle.forward([0, 30], q, k, v, g, beta)
    q2, k2 = q.copy(), k.copy()
    q2[:, 1] += 1.0
    k2[:, 1] *= -1.0
    o_b, _ = oracle.forward([0, 30], q2, k2, v, g, beta)
    assert np.array_equal(o_a[:, 0], o_b[:, 0]) and np.array_equal(o_a[:, 2], o_b[:, 2])
    o_c, _ = oracle.forward([0, 30], q, k, v, g, beta, heads=[2])
    assert np.array_equal(o_c[:, 2], o_a[:, 2]) and np.all(np.isnan(o_c[:, 0]))


def test_sequences_do_not_leak():
    """State resets at each sequence start: a packed run equals separate runs."""
    rng = np.random.default_rng(24)
    cu, q, k, v, g, beta, h0 = _small_varlen(rng, [10, 15])
    o_p, f_p = oracle.forward(cu, q, k, v, g, beta, h0=h0)
    o_2, f_2 = oracle.forward([0, 15], q[10:], k[10:], v[10:], g[10:], beta[10:], h0=h0[1:])
    assert np.array_equal(o_p[10:], o_2) and np.array_equal(f_p[1], f_2[0])


def test_thread_count_does_not_change_results():
    rng = np.random.default_rng(25)
    cu, q, k, v, g, beta, h0 = _small_varlen(rng, [33, 31], H=4)
    a = oracle.forward(cu, q, k, v, g, beta, h0=h0, nthreads=1)
    b = oracle.forward(cu, q, k, v, g, beta, h0=h0, nthreads=4)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])
