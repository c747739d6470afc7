"""Host-side checks of the C ABI (no GPU needed): exported symbols, the C++
planner against the independent Python planner (bit-exact), error codes, the
workspace layout, and argument validation that rejects calls before any
device work is enqueued."""
import ctypes
import os
import re
import subprocess

import numpy as np
import pytest

from context_kda_gb300.inputs import workloads
from oracle.plan import PlanError, plan_segments

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def kda():
    import __graft_entry__
    __graft_entry__._load_build_module().build()
    from context_kda_gb300 import binding
    return binding


def _declared_functions():
    names = []
    for hdr in sorted(os.listdir(os.path.join(ROOT, "include"))):
        src = open(os.path.join(ROOT, "include", hdr)).read()
        src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
        names += re.findall(r"\b(kda_[a-z_0-9]+)\s*\(", src)
    return sorted(set(names))


def test_header_declares_the_entry_points():
    names = _declared_functions()
    for want in ("kda_plan_segments", "kda_segment_forward", "kda_compose_summaries", "kda_apply_boundary",
                 "kda_forward_segmented", "kda_workspace_bytes", "kda_workspace_layout", "kda_status_string",
                 "kda_last_cuda_error", "kda_device_status", "kda_selftest_wait_expiry", "kda_forward_two_pass",
                 "kda_plan_check"):
        assert want in names


def test_library_exports_every_declared_symbol(kda):
    lib = ctypes.CDLL(kda.LIB_PATH)
    for name in _declared_functions():
        assert hasattr(lib, name), name
    out = subprocess.run(["nm", "-D", "--defined-only", kda.LIB_PATH], capture_output=True, text=True).stdout
    exported = set(line.split()[-1] for line in out.splitlines() if line.strip())
    for name in _declared_functions():
        assert name in exported, name


def _cu(seqlens):
    return [0] + [int(x) for x in np.cumsum(seqlens)]


@pytest.mark.parametrize("name", list(workloads().keys()))
def test_planner_bit_exact_on_workloads(kda, name):
    w = workloads()[name]
    cu = _cu(w.seqlens)
    got = kda.kda_plan_segments(cu, w.segments)
    want = np.array(plan_segments(cu, w.segments), dtype=np.int32)
    assert got.dtype == np.int32 and np.array_equal(got, want)


def test_planner_bit_exact_random(kda):
    rng = np.random.default_rng(7)
    for _ in range(200):
        n = int(rng.integers(1, 12))
        cu = _cu(rng.integers(1, 300, size=n))
        T = cu[-1]
        S = int(rng.integers(1, min(T, 40) + 1))
        assert np.array_equal(kda.kda_plan_segments(cu, S), np.array(plan_segments(cu, S), dtype=np.int32))
        inner = sorted(set(int(x) for x in rng.integers(1, T, size=int(rng.integers(0, 6))))) if T > 1 else []
        b = [0] + inner + [T]
        assert np.array_equal(kda.kda_plan_segments(cu, len(b) - 1, b),
                              np.array(plan_segments(cu, len(b) - 1, b), dtype=np.int32))


@pytest.mark.parametrize("cu,S,bounds,chunk", [
    ([1, 5], 1, None, 64), ([0, 5, 5], 1, None, 64), ([0, 4], 5, None, 64), ([0, 4], 0, None, 64),
    ([0, 8], 2, [0, 4, 7], 64), ([0, 8], 2, [0, 9, 8], 64), ([0, 8], 2, [0, 4, 4], 64), ([0, 128], 2, None, 32),
])
def test_planner_rejects_like_the_oracle(kda, cu, S, bounds, chunk):
    with pytest.raises(PlanError) as e:
        plan_segments(cu, S, bounds, chunk)
    with pytest.raises(kda.KDAError) as f:
        kda.kda_plan_segments(cu, S, bounds, chunk)
    want = {"invalid": kda.KDA_ERR_INVALID_ARG, "unsupported": kda.KDA_ERR_UNSUPPORTED}[e.value.code]
    assert f.value.status == want


def test_planner_capacity_and_query(kda):
    lib = kda._lib
    cu = np.array([0, 100, 300], dtype=np.int32)
    n = ctypes.c_size_t(0)
    assert lib.kda_plan_segments(cu.ctypes.data_as(ctypes.c_void_p), 2, 3, None, 64, None, ctypes.byref(n)) == 0
    need = n.value
    small = np.zeros(need - 1, dtype=np.int32)
    n2 = ctypes.c_size_t(need - 1)
    rc = lib.kda_plan_segments(cu.ctypes.data_as(ctypes.c_void_p), 2, 3, None, 64,
                               small.ctypes.data_as(ctypes.c_void_p), ctypes.byref(n2))
    assert rc == kda.KDA_ERR_WORKSPACE and n2.value == need


def test_summary_workspace_matches_the_pages(kda):
    """The A + B regions equal S*H*(K*K + K*V)*4 bytes: 256 MiB at CP64, H=32, K=V=128
    (cuLA PR #136, §Latest cuDNN compatibility; fixture tests/golden/pages_summary_workspace.txt)."""
    rows = [l.split() for l in open(os.path.join(ROOT, "tests", "golden", "pages_summary_workspace.txt"))
            if l.strip() and not l.startswith("#")]
    S, H, K, V, want = (int(x) for x in rows[0])
    assert (K, V) == (128, 128)
    w = workloads()["packed65536_h32_s64"]
    assert (w.segments, w.heads) == (S, H)
    plan = kda.kda_plan_segments(_cu(w.seqlens), S)
    off = kda.kda_workspace_layout(plan, H)
    a_bytes, b_bytes = off[4] - off[3], off[5] - off[4]
    assert a_bytes + b_bytes == want == 256 * 2 ** 20
    assert a_bytes == S * H * K * K * 4 and b_bytes == S * H * K * V * 4
    assert kda.kda_workspace_bytes(plan, H) == off[6]
    assert all(o % 256 == 0 for o in off)


@pytest.mark.parametrize("name", list(workloads().keys()))
def test_workspace_regions_hold_what_the_header_documents(kda, name):
    """qhat H*T_cont*K bf16 (per piece, 128-row tile images), fin fp32 [n_fin][H][K][K], packages [H][n_chunks] of
    KDA_PACKAGE_BYTES, then A, B, S_in, and from 16 segments on the two-level scan's scratch
    (G H K (K + V) fp32 group totals, then G H K V fp32 incoming states, G = ceil(S / ceil(sqrt S)));
    each region starts on a 256-byte boundary."""
    w = workloads()[name]
    plan = kda.kda_plan_segments(_cu(w.seqlens), w.segments)
    H, K = w.heads, 128
    off = kda.kda_workspace_layout(plan, H)
    up = lambda x: (x + 255) // 256 * 256
    T_cont, n_fin, n_chunks, S = int(plan[9]), int(plan[10]), int(plan[11]), int(plan[5])
    sizes = [H * T_cont * K * 2, n_fin * H * K * K * 4, n_chunks * H * 123392, S * H * K * K * 4,
             S * H * K * K * 4, S * H * K * K * 4]
    if S >= 16:
        m = next(x for x in range(1, S + 1) if x * x >= S)
        G = (S + m - 1) // m
        sizes[5] = up(sizes[5]) + up(G * H * K * 256 * 4) + G * H * K * K * 4
        assert kda.kda_scan_workspace_bytes(plan, H) == up(G * H * K * 256 * 4) + G * H * K * K * 4
    assert off[0] == 0
    for i, n in enumerate(sizes):
        assert off[i + 1] - off[i] == up(n), i


def test_layout_rejects_bad_plan_and_heads(kda):
    plan = kda.kda_plan_segments([0, 256], 2)
    with pytest.raises(kda.KDAError):
        kda.kda_workspace_layout(plan, 0)
    bad = plan.copy()
    bad[0] = 0
    with pytest.raises(kda.KDAError):
        kda.kda_workspace_layout(bad, 4)
    assert kda.kda_workspace_bytes(bad, 4) == 0


def test_entry_points_reject_bad_arguments_before_any_device_work(kda):
    """Null or misaligned pointers and short workspaces are refused on the host; these
    calls return before touching the GPU, so they run here without one."""
    lib = kda._lib
    plan = kda.kda_plan_segments([0, 256], 2)
    pp = plan.ctypes.data_as(ctypes.c_void_p)
    fake = ctypes.c_void_p(1 << 20)          # never dereferenced: validation fails first
    odd = ctypes.c_void_p((1 << 20) + 8)
    ws_need = kda.kda_workspace_bytes(plan, 2)
    args = [pp, fake, 2, fake, fake, fake, fake, fake, None, ctypes.c_float(1.0), fake, fake, fake, ws_need, None]
    for i in (3, 4, 5, 6, 7, 10, 11, 12):
        a = list(args)
        a[i] = None
        assert lib.kda_forward_segmented(*a) == kda.KDA_ERR_INVALID_ARG
        a[i] = odd
        assert lib.kda_forward_segmented(*a) == kda.KDA_ERR_INVALID_ARG
    a = list(args)
    a[13] = ws_need - 1
    assert lib.kda_forward_segmented(*a) == kda.KDA_ERR_WORKSPACE
    for i in (3, 4, 5, 6, 7, 10, 11, 12):   # the two-pass entry takes the same arguments
        a = list(args)
        a[i] = None
        assert lib.kda_forward_two_pass(*a) == kda.KDA_ERR_INVALID_ARG
        a[i] = odd
        assert lib.kda_forward_two_pass(*a) == kda.KDA_ERR_INVALID_ARG
    a = list(args)
    a[13] = ws_need - 1
    assert lib.kda_forward_two_pass(*a) == kda.KDA_ERR_WORKSPACE
    a = list(args)
    a[1] = None
    assert lib.kda_forward_segmented(*a) == kda.KDA_ERR_INVALID_ARG
    a = list(args)
    a[2] = 0
    assert lib.kda_forward_segmented(*a) == kda.KDA_ERR_INVALID_ARG
    assert lib.kda_compose_summaries(pp, fake, 2, None, fake, None, fake, None) == kda.KDA_ERR_INVALID_ARG
    assert lib.kda_apply_boundary(pp, fake, 2, fake, fake, 0, fake, fake, None) == kda.KDA_ERR_WORKSPACE
    assert lib.kda_segment_forward(pp, fake, 2, fake, fake, fake, fake, fake, None, ctypes.c_float(1.0), fake,
                                   None, fake, fake, fake, ws_need, None) == kda.KDA_ERR_INVALID_ARG
    assert kda.kda_status_string(kda.KDA_ERR_WORKSPACE) == "buffer too small"


def test_state_abort_selftest_refuses_plans_without_a_second_chunk(kda):
    lib = kda._lib
    plan = kda.kda_plan_segments([0, 64, 128], 2)       # every piece one chunk long
    pp = plan.ctypes.data_as(ctypes.c_void_p)
    fake = ctypes.c_void_p(1 << 20)                     # never dereferenced: validation fails first
    assert lib.kda_selftest_state_abort(pp, fake, 2, fake, fake, fake, fake, fake, None, ctypes.c_float(1.0), fake,
                                        fake, fake, fake, fake, 1 << 30, None) == kda.KDA_ERR_INVALID_ARG
