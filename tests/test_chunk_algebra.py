"""The chunkwise algebra that the CUDA kernels implement, checked in fp64 against the oracle (CPU).

The kernels do not run the token recurrence.  Per 64-token chunk they use the closed form of the
KDA gated delta rule (cuLA PR #110, "feat(cp): add opt-in NVSHMEM CP state handoff",
§Supported configuration: BF16 inputs, FP32 recurrent state) unrolled over the chunk:

    Gamma_r = sum_{i<=r} g_i,  kt = e^Gamma k,  kh = e^-Gamma k,  qt = scale e^Gamma q
    M = (Diag(beta) Kt Kh^T) strictly lower,  T = (I + M)^-1
    W = T Diag(beta) Kt,  Ut = T Diag(beta) V,  QK = (Qt Kh^T) lower incl. the diagonal
    U = Ut - W X,  O = Qt X + QK U,  X' = Diag(e^Gamma_C) (X + Kh^T U)

with T assembled from 16 x 16 diagonal blocks as the preparation does, and the transition
columns running the same map on P from P = I with zero values, so that their outputs are qhat.
These tests write that algebra out in plain numpy (no CUDA code is shared) and check it equals the
token recurrence of the oracle to fp64 rounding, so the GPU's remaining error is rounding only.
They also check the error model of the three-term bf16 split used for the state-feeding products,
and the chunkwise form of the backward (the next row of the work) against the backward oracle.
"""
import numpy as np
import pytest

import oracle
from oracle import backward as bw

C = 64


def _problem(seqlens, H, K, V, seed, g_lo=-0.2, g_hi=-0.001, h0_std=0.3):
    rng = np.random.default_rng(seed)
    T = int(sum(seqlens))
    f32 = lambda a: a.astype(np.float32).astype(np.float64)
    q = rng.standard_normal((T, H, K))
    k = rng.standard_normal((T, H, K))
    q /= np.linalg.norm(q, axis=-1, keepdims=True)
    k /= np.linalg.norm(k, axis=-1, keepdims=True)
    x = {"q": f32(q), "k": f32(k), "v": f32(rng.standard_normal((T, H, V))),
         "g": f32(rng.uniform(g_lo, g_hi, (T, H, K))),
         "beta": f32(1.0 / (1.0 + np.exp(-rng.standard_normal((T, H))))),
         "h0": f32(h0_std * rng.standard_normal((len(seqlens), H, K, V)))}
    cu = np.concatenate([[0], np.cumsum(seqlens)]).astype(np.int32)
    return cu, x


def blocked_inverse(M):
    """(I + M)^-1 for strictly lower M (n <= 64, zero-padded to 64) as the preparation builds it:
    16 x 16 diagonal blocks by forward substitution, each 32 x 32 half as [t0 0; -t1 M10 t0  t1],
    the whole as [T_lo 0; -T_hi M_hi,lo T_lo  T_hi]."""
    n = M.shape[0]
    Mp = np.zeros((C, C))
    Mp[:n, :n] = M
    Tm = np.zeros((C, C))
    for b in range(4):
        s = slice(16 * b, 16 * b + 16)
        blk = Mp[s, s]
        t = np.zeros((16, 16))
        for j in range(16):                 # column j: x_r = -sum_{i<r} blk[r, i] x_i, x_j = 1
            x = np.zeros(16)
            x[j] = 1.0
            for r in range(j + 1, 16):
                x[r] = -blk[r, :r] @ x[:r]
            t[:, j] = x
        Tm[s, s] = t
    for h in range(2):                      # 32 x 32 halves
        lo, hi = slice(32 * h, 32 * h + 16), slice(32 * h + 16, 32 * h + 32)
        Tm[hi, lo] = -Tm[hi, hi] @ Mp[hi, lo] @ Tm[lo, lo]
    lo, hi = slice(0, 32), slice(32, 64)
    Tm[hi, lo] = -Tm[hi, hi] @ Mp[hi, lo] @ Tm[lo, lo]
    return Tm[:n, :n]


def chunk_terms(q, k, v, g, beta, scale):
    """Everything about one chunk that does not depend on the state (the preparation)."""
    Gam = np.cumsum(g, axis=0)
    kt, kh, qt = np.exp(Gam) * k, np.exp(-Gam) * k, scale * np.exp(Gam) * q
    n = q.shape[0]
    M = np.tril(beta[:, None] * (kt @ kh.T), -1)
    T = blocked_inverse(M)
    return {"Gam": Gam, "kt": kt, "kh": kh, "qt": qt, "M": M, "T": T, "W": T @ (beta[:, None] * kt),
            "Ut": T @ (beta[:, None] * v), "QK": np.tril(qt @ kh.T), "gc": np.exp(Gam[-1]), "n": n}


def chunk_step(p, X, zero_values=False):
    """The state pass of one chunk: outputs and the next state."""
    U = (0.0 if zero_values else p["Ut"]) - p["W"] @ X
    O = p["qt"] @ X + p["QK"] @ U
    return O, p["gc"][:, None] * (X + p["kh"].T @ U)


def chunkwise_range(t0, t1, h, x, X0, scale, transition=False):
    """Tokens [t0, t1) of head h in chunks of 64 from the piece start t0."""
    K = x["q"].shape[2]
    X = np.eye(K) if transition else X0.copy()
    outs = []
    for c0 in range(t0, t1, C):
        c1 = min(c0 + C, t1)
        p = chunk_terms(x["q"][c0:c1, h], x["k"][c0:c1, h], x["v"][c0:c1, h], x["g"][c0:c1, h],
                        x["beta"][c0:c1, h], scale)
        O, X = chunk_step(p, X, zero_values=transition)
        outs.append(O)
    return np.concatenate(outs), X


@pytest.mark.parametrize("n", [1, 5, 16, 17, 40, 64])
def test_blocked_inverse_is_the_inverse(n):
    rng = np.random.default_rng(n)
    M = np.tril(0.3 * rng.standard_normal((n, n)), -1)
    np.testing.assert_allclose(blocked_inverse(M), np.linalg.inv(np.eye(n) + M), rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("seqlens", [[64], [200], [1, 63, 65, 130]])
def test_chunkwise_forward_is_the_recurrence(seqlens):
    cu, x = _problem(seqlens, H=2, K=16, V=12, seed=31)
    scale = 0.8
    o_ref, f_ref = oracle.forward(cu, x["q"], x["k"], x["v"], x["g"], x["beta"], h0=x["h0"], scale=scale)
    for h in range(2):
        for s in range(len(seqlens)):
            o, X = chunkwise_range(cu[s], cu[s + 1], h, x, x["h0"][s, h], scale)
            np.testing.assert_allclose(o, o_ref[cu[s]:cu[s + 1], h], rtol=1e-10, atol=1e-11)
            np.testing.assert_allclose(X, f_ref[s, h], rtol=1e-10, atol=1e-11)


def test_transition_columns_give_qhat_and_the_transition():
    cu, x = _problem([150], H=1, K=16, V=12, seed=32)
    scale = 0.7
    qh, P = chunkwise_range(0, 150, 0, x, None, scale, transition=True)
    r = oracle.run_range(0, 150, 0, x["q"], x["k"], x["v"], x["g"], x["beta"], track_transition=True,
                         scale=scale)
    np.testing.assert_allclose(qh, r["qhat"], rtol=1e-10, atol=1e-11)
    np.testing.assert_allclose(P, r["P"], rtol=1e-10, atol=1e-11)


# ---- the three-term bf16 split of the state-feeding products

def _bf16(x):
    """Round fp32 values to bf16 (round to nearest, ties to even), returned as float64."""
    b = np.asarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    b = (b + 0x7FFF + ((b >> 16) & 1)) >> 16 << 16
    return b.astype(np.uint32).view(np.float32).astype(np.float64)


def test_bf16_rounding_helper():
    assert _bf16(np.float32(1.0)) == 1.0
    assert _bf16(np.float32(1.0 + 2.0 ** -8)) == 1.0            # tie -> even
    assert _bf16(np.float32(1.0 + 3 * 2.0 ** -8)) == 1.0 + 2.0 ** -6
    assert _bf16(np.float32(1.0 + 2.0 ** -7)) == 1.0 + 2.0 ** -7


def test_three_term_split_product_error():
    """a = ah + al, b = bh + bl with bf16 parts: ah bh + ah bl + al bh leaves only al bl and the
    rounding of the lo parts, about 2^-16 of |a||b| per term, against 2^-8 for one bf16 term.
    Checked on 128-long dot products of the sizes the state pass multiplies; the sums are exact
    here, and the tensor core's fp32 accumulation adds about 2^-24 per term on top."""
    rng = np.random.default_rng(33)
    a = rng.standard_normal((256, 128)).astype(np.float32).astype(np.float64)
    b = rng.standard_normal((128, 128)).astype(np.float32).astype(np.float64)
    ah, bh = _bf16(a), _bf16(b)
    al, bl = _bf16(a - ah), _bf16(b - bh)
    exact = a @ b
    scale = np.abs(a) @ np.abs(b)
    one = ah @ bh
    three = ah @ bh + ah @ bl + al @ bh
    e1 = np.max(np.abs(one - exact) / scale)
    e3 = np.max(np.abs(three - exact) / scale)
    assert 2.0 ** -11 < e1 < 2.0 ** -7
    assert e3 < 2.0 ** -14
    assert e3 < e1 / 100


# ---- the chunkwise backward (for the backward kernels that come next)

def chunk_backward(p, X, dO, G, k, v, beta):
    """Gradients through one chunk_step (and chunk_terms) by the chain rule: given the chunk-start
    state X, the output gradient dO and the gradient G of the next state, returns dq, dk, dv, dg,
    dbeta of the chunk's rows and the gradient of X."""
    kt, kh, qt, T, W, QK = p["kt"], p["kh"], p["qt"], p["T"], p["W"], p["QK"]
    n = p["n"]
    U = p["Ut"] - W @ X
    DG = p["gc"][:, None] * G                       # X' = Dc (X + Kh^T U)
    dX = DG.copy()
    dU = kh @ DG
    dkh = U @ DG.T
    dGamC = np.sum(G * (p["gc"][:, None] * (X + kh.T @ U)), axis=1)
    dX += qt.T @ dO                                 # O = Qt X + QK U
    dqt = dO @ X.T
    dQK = np.tril(dO @ U.T)
    dU += QK.T @ dO
    dqt += dQK @ kh
    dkh += dQK.T @ qt
    dUt = dU                                        # U = Ut - W X
    dW = -dU @ X.T
    dX += -W.T @ dU
    bkt, bv = beta[:, None] * kt, beta[:, None] * v  # W = T B Kt, Ut = T B V
    dT = dW @ bkt.T + dUt @ bv.T
    dbkt = T.T @ dW
    dbv = T.T @ dUt
    dv = beta[:, None] * dbv
    dkt = beta[:, None] * dbkt
    dbeta = np.sum(dbkt * kt, axis=1) + np.sum(dbv * v, axis=1)
    dM = np.tril(-T.T @ dT @ T.T, -1)              # T = (I + M)^-1
    S = kt @ kh.T                                   # M = strictly lower(B Kt Kh^T)
    dbeta += np.sum(dM * S, axis=1)
    dkt += beta[:, None] * (dM @ kh)
    dkh += dM.T @ (beta[:, None] * kt)
    E, Ei = np.exp(p["Gam"]), np.exp(-p["Gam"])   # kt = E k, kh = Ei k, qt = scale E q
    dk = E * dkt + Ei * dkh
    dGam = kt * dkt - kh * dkh + qt * dqt
    dGam[n - 1] += dGamC
    dg = np.cumsum(dGam[::-1], axis=0)[::-1]        # Gamma_r = sum_{i<=r} g_i
    return {"dqt": dqt, "dk": dk, "dv": dv, "dg": dg, "dbeta": dbeta, "dX": dX, "E": E}


def test_chunkwise_backward_is_the_token_backward():
    seqlens = [150]
    cu, x = _problem(seqlens, H=1, K=8, V=6, seed=34)
    scale = 0.9
    rng = np.random.default_rng(35)
    do = rng.standard_normal((150, 1, 6))
    dfinal = rng.standard_normal((1, 1, 8, 6))
    ref = bw.backward(cu, x["q"], x["k"], x["v"], x["g"], x["beta"], do, dfinal=dfinal, h0=x["h0"], scale=scale)
    # forward, keeping each chunk's terms and start state
    h, X = 0, x["h0"][0, 0].copy()
    chunks = []
    for c0 in range(0, 150, C):
        c1 = min(c0 + C, 150)
        p = chunk_terms(x["q"][c0:c1, h], x["k"][c0:c1, h], x["v"][c0:c1, h], x["g"][c0:c1, h],
                        x["beta"][c0:c1, h], scale)
        chunks.append((c0, c1, p, X))
        _, X = chunk_step(p, X)
    # backward, last chunk first
    G = dfinal[0, 0].copy()
    got = {name: np.zeros_like(ref[name][:, 0]) for name in ("dq", "dk", "dv", "dg", "dbeta")}
    for c0, c1, p, X0 in reversed(chunks):
        r = chunk_backward(p, X0, do[c0:c1, 0], G, x["k"][c0:c1, h], x["v"][c0:c1, h], x["beta"][c0:c1, h])
        got["dq"][c0:c1] = scale * r["E"] * r["dqt"]
        for name in ("dk", "dv", "dg", "dbeta"):
            got[name][c0:c1] = r[name]
        G = r["dX"]
    for name in got:
        np.testing.assert_allclose(got[name], ref[name][:, 0], rtol=1e-9, atol=1e-10, err_msg=name)
    np.testing.assert_allclose(G, ref["dh0"][0, 0], rtol=1e-9, atol=1e-10)
