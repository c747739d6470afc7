"""CPU oracle for segmented Kimi Delta Attention (KDA) -- test infrastructure.

Only the test suite, ``__graft_entry__.smoke()`` and the benchmark's CPU
baseline leg (``bench.py``) may import this package.  The CUDA library does
not link, include or call anything here, and nothing here imports the CUDA
package: the two share no code.  The seeded input generator
(``context_kda_gb300.inputs``) is the only module both sides use, and it holds
none of the method's arithmetic.

Contents
  * ``kda_oracle.c`` -- the fp64 token-by-token recurrence (monolithic forward,
    and a single token-range runner that also tracks the transition P).
  * ``segmented.py`` -- the segment-parallel reading built from that runner:
    per-segment affine summaries (transition A, state update B), their
    sequential composition, and the fix-up of continuing outputs.
  * ``plan.py`` -- an independent Python planner producing the packed-THD
    segment plan word for word.
  * ``backward.py`` -- gradients of q, k, v, g, beta and h0 by the chain rule
    through the same recurrence (fp64, any K and V), and their segment-parallel
    reading through the following summaries.  No CUDA path computes them yet.

Parity pins (tests/test_oracle_*.py) tie the oracle to closed forms,
brute-force dense products and invariants; see each function's docstring.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "kda_oracle.c")
_LIB_PATH = os.path.join(_HERE, "libkda_oracle.so")
_lock = threading.Lock()
_lib = None

MUTATIONS = {
    "none": 0,
    "decay_after_delta": 1,
    "output_old_state": 2,
    "output_transposed": 3,
    "project_undecayed": 4,
    "decay_sign": 5,
    "drop_beta": 6,
    "decay_on_value_axis": 7,
}


def build(force: bool = False) -> str:
    """Compile the C oracle with gcc + OpenMP (portable flags, no FMA contraction)."""
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O3", "-ffp-contract=off", "-fno-fast-math", "-fopenmp", "-fPIC", "-shared",
               "-std=c11", _SRC, "-o", tmp, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB_PATH)
            P = ctypes.c_void_p
            lib.oracle_kda_run.argtypes = [ctypes.c_int64, ctypes.c_int64, ctypes.c_int32, ctypes.c_int32,
                                           ctypes.c_int32, ctypes.c_int32, P, P, P, P, P, ctypes.c_double,
                                           P, P, P, P, ctypes.c_int]
            lib.oracle_kda_run.restype = ctypes.c_int
            lib.oracle_kda_forward.argtypes = [ctypes.c_int32, P, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
                                               P, P, P, P, P, P, ctypes.c_double, P, ctypes.c_int32,
                                               P, P, ctypes.c_int, ctypes.c_int]
            lib.oracle_kda_forward.restype = ctypes.c_int
            lib.oracle_max_threads.restype = ctypes.c_int
            _lib = lib
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _f32(a):
    return np.ascontiguousarray(a, dtype=np.float32)


def max_threads() -> int:
    return int(_load().oracle_max_threads())


def as_f32(inputs):
    """fp32 views of one drawn problem: (q, k, v, g, beta) with bf16 decoded exactly."""
    from context_kda_gb300.inputs import bf16_to_f32
    return (bf16_to_f32(inputs.q), bf16_to_f32(inputs.k), bf16_to_f32(inputs.v),
            _f32(inputs.g), _f32(inputs.beta))


def forward(cu_seqlens, q, k, v, g, beta, h0=None, scale=1.0, heads=None, nthreads=0, mutate=0,
            want_o=True, want_final=True):
    """Monolithic recurrence (the definition).  q,k,g [T,H,K], v [T,H,V], beta [T,H] as
    fp32 arrays; h0 [N,H,K,V] or None.  Returns (o [T,H,V] f64, final [N,H,K,V] f64);
    heads not listed in ``heads`` are left as NaN."""
    lib = _load()
    q, k, v, g, beta = _f32(q), _f32(k), _f32(v), _f32(g), _f32(beta)
    cu = np.ascontiguousarray(cu_seqlens, dtype=np.int32)
    T, H, K = q.shape
    V = v.shape[2]
    N = cu.shape[0] - 1
    h0d = None if h0 is None else np.ascontiguousarray(h0, dtype=np.float64)
    hl = None if heads is None else np.ascontiguousarray(heads, dtype=np.int32)
    o = np.full((T, H, V), np.nan) if want_o else None
    fin = np.full((N, H, K, V), np.nan) if want_final else None
    rc = lib.oracle_kda_forward(N, _ptr(cu), H, K, V, _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta),
                                _ptr(h0d), float(scale), _ptr(hl), 0 if hl is None else len(hl),
                                _ptr(o), _ptr(fin), int(nthreads), int(mutate))
    if rc != 0:
        raise ValueError("oracle_kda_forward rejected its arguments")
    return o, fin


def run_range(t0, t1, h, q, k, v, g, beta, S0=None, track_transition=False, scale=1.0,
              want_o=True, mutate=0):
    """Run tokens [t0, t1) of head h from state S0 (zeros if None) and, when asked,
    the transition from the identity.  Returns dict with S (state at t1), o
    [(t1-t0),V], and if tracked P (transition at t1) and qhat [(t1-t0),K]."""
    lib = _load()
    q, k, v, g, beta = _f32(q), _f32(k), _f32(v), _f32(g), _f32(beta)
    T, H, K = q.shape
    V = v.shape[2]
    S = np.zeros((K, V)) if S0 is None else np.array(S0, dtype=np.float64, copy=True, order="C")
    P = np.eye(K) if track_transition else None
    n = int(t1 - t0)
    o = np.empty((n, V)) if want_o else None
    qh = np.empty((n, K)) if track_transition and want_o else None
    rc = lib.oracle_kda_run(int(t0), int(t1), int(h), H, K, V, _ptr(q), _ptr(k), _ptr(v), _ptr(g),
                            _ptr(beta), float(scale), _ptr(S), _ptr(P), _ptr(o), _ptr(qh), int(mutate))
    if rc != 0:
        raise ValueError("oracle_kda_run rejected its arguments")
    out = {"S": S, "o": o}
    if track_transition:
        out["P"] = P
        out["qhat"] = qh
    return out
